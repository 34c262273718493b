// vconv.cu -- the value tensor of a bf16 forward as fp16, once per call.
//
// The PV product takes P as 16-bit values.  fp16 P carries 11 significant
// bits against bf16's 8, which the tolerances on O need where a few keys
// share a row's weight, but the tensor core takes P and V in the same
// format.  attn_fwd_ws therefore writes an fp16 copy of V into the caller's
// workspace first: one CTA per (KV head, 128-key tile) reads the tile once
// into registers, finds its largest bf16 exponent, and writes the tile as
// fp16 when fp16 represents it well -- largest magnitude in [2^-8, 2^16) (every
// bf16 value down to 2^-14 is exact in fp16, smaller ones are off by at most
// 2^-25, under 2^-17 of the tile's largest value), or a tile of zeros and
// bf16 subnormals.  Its flag byte says which: 0 = fp16 copy written, 1 = the
// tile stays bf16 (a magnitude of 2^16 or more, an inf or NaN, or only
// values below 2^-8).  The forward then reads the fp16 copy for every CTA
// whose key tiles all have flag 0, and the bf16 original otherwise.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_internal.h"
#include "ptx.cuh"

namespace tme {
namespace {

constexpr int kConvThreads = 256;

template <int D>
__global__ void __launch_bounds__(kConvThreads) v_to_f16_kernel(const uint16_t* __restrict__ v,
                                                               uint16_t* __restrict__ v16,
                                                               uint8_t* __restrict__ flags, int Nk,
                                                               int n_ktiles) {
    constexpr int kPer = 128 * D / 8 / kConvThreads;  // 16-byte chunks per thread (4 or 8)
    const int group = static_cast<int>(blockIdx.x / n_ktiles);
    const int kt = static_cast<int>(blockIdx.x % n_ktiles);
    const int rows = min(128, Nk - kt * 128);
    const int chunks = rows * (D / 8);
    const int64_t off = (static_cast<int64_t>(group) * Nk + static_cast<int64_t>(kt) * 128) * D;
    const uint4* src = reinterpret_cast<const uint4*>(v + off);
    uint4 w[kPer];
    uint32_t ex = 0u;   // largest exponent field of each 16-bit half
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = threadIdx.x + i * kConvThreads;
        w[i] = c < chunks ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        ex = __vmaxu2(ex, __vmaxu2(__vmaxu2(w[i].x & 0x7f807f80u, w[i].y & 0x7f807f80u),
                                   __vmaxu2(w[i].z & 0x7f807f80u, w[i].w & 0x7f807f80u)));
    }
    __shared__ uint32_t s_max[kConvThreads / 32];
    uint32_t e = __reduce_max_sync(0xffffffffu, max(ex & 0xffffu, ex >> 16) >> 7);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = e;
    __syncthreads();
    e = 0u;
#pragma unroll
    for (int i = 0; i < kConvThreads / 32; ++i) e = max(e, s_max[i]);
    // exponent field 119..142: largest magnitude in [2^-8, 2^16); 0: zeros and
    // subnormals (below 2^-126, which fp16 rounds to zero)
    const bool ok = e == 0u || (e >= 119u && e <= 142u);
    if (ok) {
        uint4* dst = reinterpret_cast<uint4*>(v16 + off);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int c = threadIdx.x + i * kConvThreads;
            if (c < chunks)
                dst[c] = make_uint4(bf16x2_to_f16x2(w[i].x), bf16x2_to_f16x2(w[i].y),
                                    bf16x2_to_f16x2(w[i].z), bf16x2_to_f16x2(w[i].w));
        }
    }
    if (threadIdx.x == 0) flags[blockIdx.x] = ok ? 0 : 1;
}

}  // namespace

cudaError_t launch_v_to_f16(int D, const void* v, void* v16, uint8_t* flags, int64_t groups, int Nk,
                            cudaStream_t stream) {
    const int n_ktiles = (Nk + 127) / 128;
    const long long blocks = groups * n_ktiles;
    if (blocks <= 0 || blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    const uint16_t* src = static_cast<const uint16_t*>(v);
    uint16_t* dst = static_cast<uint16_t*>(v16);
    if (D == 128)
        return launch_kernel(v_to_f16_kernel<128>, dim3(static_cast<unsigned>(blocks)),
                             dim3(kConvThreads), 0, stream, src, dst, flags, Nk, n_ktiles);
    if (D == 64)
        return launch_kernel(v_to_f16_kernel<64>, dim3(static_cast<unsigned>(blocks)),
                             dim3(kConvThreads), 0, stream, src, dst, flags, Nk, n_ktiles);
    return cudaErrorInvalidValue;
}

}  // namespace tme
