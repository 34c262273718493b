// ffn.cu -- the token-chunked feed-forward block.
//
// The noflash-attention forum post (ai-navigate-news, section "The DIY
// approach", list "What worked") lists FFN chunking, with a runtime safety
// check, next to the tiled attention: the feed-forward block acts on every
// token on its own, so running it a slice of tokens at a time never holds the
// [tokens x d_ff] intermediate of the whole sequence.  Per token row x:
//     h = act(x W1^T + b1),   y = h W2^T + b2
// (swiglu: W1 = [Wg; Wu], h = silu(x Wg^T + bg) * (x Wu^T + bu)).
//
// Both products run in one persistent tcgen05 kernel with a fused epilogue:
// each CTA walks its tiles of 128 rows x 128..256 columns (the width that pads
// the product's columns least), accumulating in fp32 in one of two TMEM
// buffers (TMA ring of 4 stages of 64-wide K slices, one elected lane issuing
// M=128 MMAs as wide as the tile) while four warps empty the other
// buffer: add the bias, apply the activation, round to the 16-bit dtype and
// store.  For swiglu the 256 columns are 128 gate columns and the same 128
// up columns, so the epilogue combines them in registers.  The host loop runs
// chunk after chunk through a caller-sized intermediate buffer.  Every output
// element is one fixed-order K reduction of its own row, so a chunked run is
// bit-identical to an unchunked one; ffn_check_chunking verifies that at run
// time.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/ffn.h"
#include "attn_internal.h"
#include "ptx.cuh"

namespace tme {

// Defined in abi.cu: device set-up (context, architecture, status word,
// tensor-map encoder) and the 3-D TMA map over a [groups][rows][cols] tensor.
int device_setup_public(unsigned int** status);
int make_map_public(CUtensorMap* map, const void* base, bool bf16, int cols, int64_t rows,
                    int64_t groups);

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kGemmThreads = 192;  // warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer
constexpr int kProducerWarp = 4, kMmaWarp = 5;   // warps 0-3: epilogue
constexpr int kEpiThreads = 128;
constexpr int kTileA = kBM * kBK * 2;              // 16 KiB
constexpr int kTileB = kBN * kBK * 2;              // 32 KiB
constexpr int kStageBytes = kTileA + kTileB;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kGemmSmem = kBarOff + 256 + 1024;    // barriers + alignment slack

struct GemmParams {
    void* c;              // output rows of this launch, [M][ldc] 16-bit
    const void* bias;     // 16-bit, or nullptr (swiglu: gate biases, then up biases)
    unsigned int* status;
    int M, N, K;          // rows, output columns, reduction length
    int a_row0;           // first row of A (TMA coordinate)
    int ldc;              // output row stride in elements
    int glu_off;          // swiglu: first B row of the up projection (= d_ff)
    int bn;               // output columns of a tile: 128 for swiglu, else 128..256
};

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The activations from their definitions (gelu: the tanh form of Hendrycks
// and Gimpel; silu: a / (1 + e^-a), with e^-a = 2^(-a log2 e)).
template <int ACT>
__device__ __forceinline__ float act_fn(float a) {
    if constexpr (ACT == FFN_ACT_RELU) return fmaxf(a, 0.0f);
    if constexpr (ACT == FFN_ACT_GELU_TANH) {
        const float u = 0.7978845608028654f * fmaf(0.044715f * a, a * a, a);
        return 0.5f * a * (1.0f + tanh_approx(u));
    }
    if constexpr (ACT == FFN_ACT_SILU || ACT == FFN_ACT_SWIGLU)
        return __fdividef(a, 1.0f + ex2_ftz(-1.4426950408889634f * a));
    return a;
}

template <bool BF16>
__device__ __forceinline__ float load16(const void* base, int i) {
    const uint16_t h = static_cast<const uint16_t*>(base)[i];
    if constexpr (BF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
    return __half2float(__ushort_as_half(h));
}

template <int ACT, bool BF16>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
    constexpr bool GLU = ACT == FFN_ACT_SWIGLU;
    const int out_n = p.bn;   // output columns of a tile (the MMA's N unless swiglu)
    // The second 128-row box of B is needed for swiglu (the up rows) and for
    // tiles wider than 128 columns.
    const bool two_b = GLU || out_n > 128;
    const uint32_t stage_tx = two_b ? kStageBytes : kTileA + kTileB / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);   // [kStages]
    uint64_t* empty = full + kStages;                               // [kStages]
    uint64_t* acc_full = empty + kStages;                           // [2] accumulator b written
    uint64_t* acc_empty = acc_full + 2;                             // [2] accumulator b read
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_mt = (p.M + kBM - 1) / kBM;
    const int n_tiles = n_mt * ((p.N + out_n - 1) / out_n);
    const int n_kb = (p.K + kBK - 1) / kBK;
    // Persistent CTAs: tiles blockIdx.x, blockIdx.x + gridDim.x, ...; the
    // row tiles of one column tile are adjacent (B stays in L2).
    auto tile_m0 = [&](int t) { return (t % n_mt) * kBM; };
    auto tile_n0 = [&](int t) { return (t / n_mt) * out_n; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiThreads);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int g = 0;   // K slices issued by this CTA (ring position)
            bool okp = true;
            for (int t = blockIdx.x; okp && t < n_tiles; t += gridDim.x) {
                const int m0 = tile_m0(t), n0 = tile_n0(t);
                const int b1 = GLU ? p.glu_off + n0 : n0 + 128;   // second 128-row box of B
                for (int kb = 0; kb < n_kb; ++kb, ++g) {
                    const int s = g % kStages;
                    if (g >= kStages &&
                        !mbar_wait(&empty[s], ((g / kStages) - 1) & 1, abort_flag, p.status)) {
                        okp = false;
                        break;
                    }
                    uint8_t* sA = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], stage_tx);
                    tma_load_3d(&tmA, &full[s], sA, kb * kBK, p.a_row0 + m0, 0);
                    tma_load_3d(&tmB, &full[s], sA + kTileA, kb * kBK, n0, 0);
                    if (two_b)
                        tma_load_3d(&tmB, &full[s], sA + kTileA + kTileB / 2, kb * kBK, b1, 0);
                }
            }
            // never leave a copy in flight into shared memory about to be released
            for (int n = (g > kStages ? g - kStages : 0); n < g; ++n)
                mbar_wait_bounded(&full[n % kStages], (n / kStages) & 1, p.status);
        }
    } else if (warp == kMmaWarp) {
        // swiglu: N = 256 (128 gate + 128 up columns); else N = the tile width
        const uint32_t idesc = idesc_f16(kBM, GLU ? kBN : out_n, BF16, false);
        int g = 0, i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            const int b = i & 1;
            if (i >= 2) {   // the epilogue has read this accumulator's previous tile
                warp_wait(&acc_empty[b], ((i >> 1) - 1) & 1, abort_flag, p.status);
                tc_fence_after();
            }
            for (int kb = 0; kb < n_kb; ++kb, ++g) {
                const int s = g % kStages;
                warp_wait(&full[s], (g / kStages) & 1, abort_flag, p.status);
                tc_fence_after();
                const uint32_t a = smem_u32(smem + s * kStageBytes);
                mma_ss_k64(tmem + 256 * b, smem_desc_sw128(a, 16, 1024),
                           smem_desc_sw128(a + kTileA, 16, 1024), idesc, kb > 0 ? 1u : 0u);
                mma_commit_elect(&empty[s]);
            }
            mma_commit_elect(&acc_full[b]);
        }
    } else {
        // epilogue: thread = output row (TMEM lane)
        const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
        int i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            const int b = i & 1;
            const int m0 = tile_m0(t), n0 = tile_n0(t);
            const int row = m0 + warp * 32 + lane;
            const bool ok = warp_wait(&acc_full[b], (i >> 1) & 1, abort_flag, p.status) &&
                            *abort_flag == 0;
            tc_fence_after();
            const uint32_t tacc = tmem + lb + 256 * b;
            uint16_t* crow = static_cast<uint16_t*>(p.c) + static_cast<int64_t>(row) * p.ldc;
#pragma unroll 1
            for (int c = 0; c < out_n / 32; ++c) {   // out_n is a multiple of 32
                const int col0 = n0 + 32 * c;
                uint32_t a[32];
                tmem_ld32(tacc + 32 * c, a);
                float h[32];
                if constexpr (GLU) {
                    uint32_t u[32];
                    tmem_ld32(tacc + 128 + 32 * c, u);
                    tmem_wait_ld();
                    reg_fence(a);
                    reg_fence(u);
                    if (c == out_n / 32 - 1) {   // the accumulator is read: release it
                        tc_fence_before();
                        mbar_arrive(&acc_empty[b]);
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float gt = __uint_as_float(a[e]), v = __uint_as_float(u[e]);
                        if (p.bias && col0 + e < p.N) {
                            gt += load16<BF16>(p.bias, col0 + e);
                            v += load16<BF16>(p.bias, p.glu_off + col0 + e);
                        }
                        h[e] = act_fn<ACT>(gt) * v;
                    }
                } else {
                    tmem_wait_ld();
                    reg_fence(a);
                    if (c == out_n / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive(&acc_empty[b]);
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float v = __uint_as_float(a[e]);
                        if (p.bias && col0 + e < p.N) v += load16<BF16>(p.bias, col0 + e);
                        h[e] = act_fn<ACT>(v);
                    }
                }
                if (ok && row < p.M) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {   // 8 columns per 16-byte store; N % 8 == 0
                        if (col0 + 8 * q + 8 > p.N) break;
                        const uint4 w = make_uint4(pack2<BF16>(h[8 * q], h[8 * q + 1]),
                                                   pack2<BF16>(h[8 * q + 2], h[8 * q + 3]),
                                                   pack2<BF16>(h[8 * q + 4], h[8 * q + 5]),
                                                   pack2<BF16>(h[8 * q + 6], h[8 * q + 7]));
                        *reinterpret_cast<uint4*>(crow + col0 + 8 * q) = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int ACT, bool BF16>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p,
                        cudaStream_t stream) {
    auto kern = ffn_gemm_kernel<ACT, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGemmSmem);
    if (e != cudaSuccess) return e;
    const long long tiles = static_cast<long long>((p.M + kBM - 1) / kBM) * ((p.N + p.bn - 1) / p.bn);
    // persistent: one CTA per SM at most (its shared memory and 512 TMEM columns)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    const long long ctas = tiles < sms ? tiles : sms;
    return launch_kernel(kern, dim3(static_cast<unsigned>(ctas)), dim3(kGemmThreads), kGemmSmem,
                         stream, tmA, tmB, p);
}

cudaError_t gemm(int act, bool bf16, const CUtensorMap& tmA, const CUtensorMap& tmB,
                 const GemmParams& p, cudaStream_t stream) {
#define TME_GEMM(a)                                                                 \
    if (act == a) return bf16 ? launch_gemm<a, true>(tmA, tmB, p, stream)          \
                              : launch_gemm<a, false>(tmA, tmB, p, stream);
    TME_GEMM(FFN_ACT_NONE)
    TME_GEMM(FFN_ACT_RELU)
    TME_GEMM(FFN_ACT_GELU_TANH)
    TME_GEMM(FFN_ACT_SILU)
    TME_GEMM(FFN_ACT_SWIGLU)
#undef TME_GEMM
    return cudaErrorInvalidValue;
}

// Sets *flag when two 16-bit buffers differ anywhere.
__global__ void compare_kernel(const uint16_t* a, const uint16_t* b, int64_t n,
                               unsigned int* flag) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        if (a[i] != b[i]) {
            atomicOr(flag, 1u);
            return;
        }
}

__device__ unsigned int g_mismatch;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_args(const void* x, const void* w1, const void* b1, const void* w2, const void* b2,
               const void* y, int T, int d_model, int d_ff, int act, int chunk, int dtype) {
    if (!x || !w1 || !w2 || !y) return ATTN_ERR_INVALID;
    if (T <= 0 || d_model <= 0 || d_ff <= 0 || chunk <= 0) return ATTN_ERR_INVALID;
    if (act < FFN_ACT_NONE || act > FFN_ACT_SWIGLU) return ATTN_ERR_INVALID;
    if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
    if (d_model % 8 || d_ff % 8) return ATTN_ERR_UNSUPPORTED;   // 16-byte rows for TMA and stores
    if (d_ff > (1 << 28) || d_model > (1 << 28)) return ATTN_ERR_UNSUPPORTED;
    const void* ptrs[] = {x, w1, w2, y};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return ATTN_ERR_ALIGN;
    return ATTN_OK;
}

// Tile width of a product with n output columns: the multiple of 32 in
// [128, 256] that pads n least, the widest on a tie (d_model = 896 runs as
// four 224-column tiles rather than four 256-column ones, 1/8 of them idle).
int tile_width(int n) {
    int best = 256;
    long long best_pad = (static_cast<long long>(n) + 255) / 256 * 256;
    for (int w = 224; w >= 128; w -= 32) {
        const long long pad = (static_cast<long long>(n) + w - 1) / w * w;
        if (pad < best_pad) best = w, best_pad = pad;
    }
    return best;
}

int run(const void* x, const void* w1, const void* b1, const void* w2, const void* b2, void* y,
        int T, int d_model, int d_ff, int act, int chunk, void* workspace, size_t workspace_bytes,
        int dtype, cudaStream_t stream) {
    int rc = check_args(x, w1, b1, w2, b2, y, T, d_model, d_ff, act, chunk, dtype);
    if (rc != ATTN_OK) return rc;
    if (chunk > T) chunk = T;
    if (!workspace) return ATTN_ERR_INVALID;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    if (workspace_bytes < static_cast<size_t>(chunk) * d_ff * 2) return ATTN_ERR_WORKSPACE;
    unsigned int* status = nullptr;
    rc = device_setup_public(&status);
    if (rc != ATTN_OK) return rc;
    const bool bf16 = dtype == ATTN_BF16;
    const bool glu = act == FFN_ACT_SWIGLU;
    CUtensorMap tmX, tmW1, tmH, tmW2;
    if (make_map_public(&tmX, x, bf16, d_model, T, 1) != ATTN_OK ||
        make_map_public(&tmW1, w1, bf16, d_model, glu ? 2 * static_cast<int64_t>(d_ff) : d_ff, 1) !=
            ATTN_OK ||
        make_map_public(&tmH, workspace, bf16, d_ff, chunk, 1) != ATTN_OK ||
        make_map_public(&tmW2, w2, bf16, d_ff, d_model, 1) != ATTN_OK)
        return ATTN_ERR_CUDA;
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int m = T - t0 < chunk ? T - t0 : chunk;
        GemmParams g1{workspace, b1, status, m, d_ff, d_model, t0, d_ff, glu ? d_ff : 0,
                      glu ? 128 : tile_width(d_ff)};
        cudaError_t e = gemm(act, bf16, tmX, tmW1, g1, stream);
        if (e != cudaSuccess) return ATTN_ERR_CUDA;
        GemmParams g2{static_cast<uint16_t*>(y) + static_cast<int64_t>(t0) * d_model, b2, status, m,
                      d_model, d_ff, 0, d_model, 0, tile_width(d_model)};
        e = gemm(FFN_ACT_NONE, bf16, tmH, tmW2, g2, stream);
        if (e != cudaSuccess) return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace
}  // namespace tme

using namespace tme;

extern "C" size_t ffn_workspace_size(int T, int d_ff, int chunk) {
    if (T <= 0 || d_ff <= 0 || chunk <= 0) return 0;
    const int c = chunk < T ? chunk : T;
    return (static_cast<size_t>(c) * d_ff * 2 + 255) & ~static_cast<size_t>(255);
}

extern "C" int ffn_forward(const void* x, const void* w1, const void* b1, const void* w2,
                           const void* b2, void* y, int T, int d_model, int d_ff, int act,
                           int chunk, void* workspace, size_t workspace_bytes, int dtype,
                           void* stream) {
    return run(x, w1, b1, w2, b2, y, T, d_model, d_ff, act, chunk, workspace, workspace_bytes,
               dtype, static_cast<cudaStream_t>(stream));
}

extern "C" int ffn_check_chunking(const void* x, const void* w1, const void* b1, const void* w2,
                                  const void* b2, void* y, void* y_ref, int T, int d_model,
                                  int d_ff, int act, int chunk, void* workspace,
                                  size_t workspace_bytes, int dtype, void* stream) {
    if (!y_ref) return ATTN_ERR_INVALID;
    if (!aligned16(y_ref)) return ATTN_ERR_ALIGN;
    if (workspace_bytes < ffn_workspace_size(T, d_ff, T)) return ATTN_ERR_WORKSPACE;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = run(x, w1, b1, w2, b2, y, T, d_model, d_ff, act, chunk, workspace, workspace_bytes,
                 dtype, st);
    if (rc != ATTN_OK) return rc;
    rc = run(x, w1, b1, w2, b2, y_ref, T, d_model, d_ff, act, T, workspace, workspace_bytes, dtype,
             st);
    if (rc != ATTN_OK) return rc;
    void* flag = nullptr;
    if (cudaGetSymbolAddress(&flag, g_mismatch) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemsetAsync(flag, 0, sizeof(unsigned int), st) != cudaSuccess) return ATTN_ERR_CUDA;
    const int64_t n = static_cast<int64_t>(T) * d_model;
    if (launch_kernel(compare_kernel, dim3(1024), dim3(256), 0, st,
                      static_cast<const uint16_t*>(y), static_cast<const uint16_t*>(y_ref), n,
                      static_cast<unsigned int*>(flag)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, flag, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return host ? ATTN_ERR_MISMATCH : ATTN_OK;
}
