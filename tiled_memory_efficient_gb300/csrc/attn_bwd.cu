// attn_bwd.cu -- backward of tiled scaled-dot-product attention for sm_103a.
//
// The autograd tier of the method (noflash-attention forum post,
// ai-navigate-news, section "Other areas where this could be useful": the
// tiled attention supports autograd, so its memory savings carry over to
// training).  Like the forward it never forms the N x N matrices: scores and
// probabilities are recomputed tile by tile from the forward's LSE.
//
// With s = scale * q.k, P = exp(s - LSE), dP = dO V^T, Delta = rowsum(dO * O):
//   dS = P * (dP - Delta),  dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K.
// Three kernels, all deterministic (no atomics):
//   1. statistics: -Delta and -LSE*log2(e) per query row into the workspace;
//   2. dK/dV, KV-stationary: one CTA per (KV group, 128-key tile) loops over
//      the query tiles of every head of the group (so GQA gradients are summed
//      inside the CTA): S^T = K Q^T and dP^T = V dO^T on the tensor core, P^T
//      and dS^T elementwise (one thread per key row), then dV += P^T dO and
//      dK += dS^T Q with P^T / dS^T read from TMEM;
//   3. dQ, Q-stationary: one CTA per (KV group, 128-row query tile) loops over
//      key tiles: S = Q K^T, dP = dO V^T, dS elementwise, dQ += dS K.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_internal.h"
#include "bias.cuh"
#include "ptx.cuh"

namespace tme {
namespace {

constexpr int kRows = 128;
// dQ kernel: EW elementwise warps (EW / 4 warpgroups, each owning 512 / EW of
// the 128 columns of a tile) + producer (warp EW) + MMA issuer (warp EW + 1).
// 16 warps of 32 columns (four warps per SM sub-partition hide more of the
// elementwise chain's latency than two), except with a general mask at D = 128:
// 8 warps of 64 columns there (measured faster with its staged bias and the
// 2-deep K ring it leaves).
template <int MK, int D>
constexpr int dq_ew() { return (MK == 1 && D == 128) ? 8 : 16; }

// Key-only keep bytes of the 32 keys from key0 (a multiple of 32): a dropped
// key's score becomes -inf.  Whole 32-byte runs inside [0, Nk) are read as two
// 16-byte vectors (every lane of the warp reads the same bytes) and skipped at
// once when no byte is zero; the ragged end goes key by key (keys >= Nk are
// masked later with the causal limit).
__device__ __forceinline__ void keep_fold32(uint32_t (&s)[32], const uint8_t* row, int key0,
                                            int Nk) {
    if (key0 + 32 <= Nk) {
        const uint4 a = reinterpret_cast<const uint4*>(row + key0)[0];
        const uint4 b = reinterpret_cast<const uint4*>(row + key0)[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t z = 0u;   // (v - 0x01..01) & ~v & 0x80..80 is nonzero exactly when a byte of v is 0
#pragma unroll
        for (int i = 0; i < 8; ++i) z |= (w[i] - 0x01010101u) & ~w[i] & 0x80808080u;
        if (z == 0u) return;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (((w[i >> 2] >> (8 * (i & 3))) & 0xffu) == 0u) s[i] = __float_as_uint(-INFINITY);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (key0 + i < Nk && row[key0 + i] == 0) s[i] = __float_as_uint(-INFINITY);
    }
}
template <int MK, int D>
constexpr int dq_threads() { return (dq_ew<MK, D>() + 2) * 32; }
// dK/dV kernel: 16 elementwise warps (warp w: key rows 32(w%4).., query half
// (w/4)%2, 32-query chunk w/8 of that half) + producer + MMA issuer.
constexpr int kKvThreads = 18 * 32;
constexpr int kKvProducerWarp = 16;
constexpr int kKvMmaWarp = 17;
constexpr float kLog2e = 1.4426950408889634f;

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<const __half2*>(&w);
        return __half22float2(h);
    }
}

// Low-order bf16 parts of two fp32 values whose bf16 roundings are packed in
// hi (first value in the low half): bf16(x - x_hi), so that x_hi + x_lo holds x
// to about 16 significant bits (the subtraction is exact in fp32).
__device__ __forceinline__ uint32_t bf16x2_residual(float x0, float x1, uint32_t hi) {
    return pack2<true>(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

// ---------------------------------------------------------------- statistics
// One query row per D/8 lanes (16-byte loads): ndelta = -sum_d dO * O in fp32,
// nlse2 = -LSE * log2(e).  Output rows go to the per-group padded layout.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_stats_kernel(const BwdParams p) {
    constexpr int LPR = D / 8;
    const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = gt / LPR;
    const int sub = static_cast<int>(gt % LPR);
    float acc = 0.0f;
    if (row < p.total_rows) {
        const uint4 o = *reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(p.out) + row * D + sub * 8);
        const uint4 g = *reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(p.dout) + row * D + sub * 8);
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = unpack2<BF16>(ow[i]);
            const float2 b = unpack2<BF16>(gw[i]);
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
        }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < p.total_rows && sub == 0) {
        const int64_t g = row / p.rows_per_group, r = row % p.rows_per_group;
        p.ndelta[g * p.rows_pad + r] = -acc;
        // A row whose every key was masked (LSE = -inf) gets P = 0 everywhere.
        const float lse = p.lse[row];
        p.nlse2[g * p.rows_pad + r] = lse == -INFINITY ? -INFINITY : -lse * kLog2e;
    }
}

// Query position of column q of a 128-row tile whose first row has position
// `base` (rows are head-major within the group, so positions wrap at Nq).
__device__ __forceinline__ int tile_pos(int base, int q, int Nq) {
    const int ps = base + q;
    if (Nq >= kRows) return ps >= Nq ? ps - Nq : ps;  // at most one wrap per tile
    return ps % Nq;
}

// Largest query position in the tile that starts at `row0`.
__device__ __forceinline__ int tile_max_pos(int64_t row0, const BwdParams& p) {
    const int64_t last = min(row0 + kRows - 1, p.rows_per_group - 1);
    return (row0 / p.Nq == last / p.Nq) ? static_cast<int>(last % p.Nq) : p.Nq - 1;
}

// The same from the position `pos` of the tile's first row, without any
// division (the dK/dV kernel walks all query tiles of a group in order).
__device__ __forceinline__ int tile_max_pos_at(int qi, int pos, const BwdParams& p) {
    const int64_t left = p.rows_per_group - static_cast<int64_t>(qi) * kRows;  // rows from row0 on
    const int span = left < kRows ? static_cast<int>(left) - 1 : kRows - 1;    // last - row0
    return pos + span < p.Nq ? pos + span : p.Nq - 1;
}

// Position of the first row of the next 128-row tile.
__device__ __forceinline__ int next_tile_pos(int pos, int Nq) {
    pos += kRows;
    if (pos >= Nq) pos = Nq >= kRows ? pos - Nq : pos % Nq;  // at most one wrap when Nq >= 128
    return pos;
}

// The same, also tracking the head (within the group) of that row.
__device__ __forceinline__ void next_tile(int& pos, int& head, int Nq) {
    pos += kRows;
    if (pos >= Nq) {
        if (Nq >= kRows) {
            pos -= Nq;
            ++head;
        } else {
            head += pos / Nq;
            pos %= Nq;
        }
    }
}

// dK/dV layout: a thread owns one key; the bias of its 32 query rows
// (first row at head `head`, position `pos`, all of them real if rows_left
// >= 32, else only rows below `rows_left`) runs down a column of the mask.
// bias_load_column reads that column (raw 16-bit values or bytes; rows and
// keys outside the problem get the neutral 0 / keep); when the 32 rows lie in
// one head the addresses are one stride apart.  bias_fold_column then turns
// the scores in x, in place, into natural-log logits s * scale + b (additive;
// the caller's softmax scale becomes log2 e) or leaves them raw / -inf
// (boolean).
__device__ __forceinline__ void bias_load_column(uint32_t (&r)[32], const BwdParams& p,
                                                 int64_t b_off, int head, int pos, int key,
                                                 int rows_left) {
    const uint8_t* base = static_cast<const uint8_t*>(p.mask);
    const bool add = p.mask_kind == 2;
    const int esz = add ? 2 : 1;
    int64_t off = b_off + static_cast<int64_t>(head) * p.msh + static_cast<int64_t>(pos) * p.msq;
    if (pos + 32 <= p.Nq && rows_left >= 32 && key < p.Nk) {
        const uint8_t* e = base + (off + key) * esz;
        const int64_t step = p.msq * esz;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            r[i] = add ? static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(e + i * step))
                       : static_cast<uint32_t>(e[i * step]);
        return;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        uint32_t v = add ? 0u : 1u;
        if (i < rows_left && key < p.Nk) {
            if (add)
                v = *reinterpret_cast<const uint16_t*>(base + (off + key) * 2);
            else
                v = base[off + key];
        }
        r[i] = v;
        if (++pos == p.Nq) {   // the next row starts the next head
            pos = 0;
            off += p.msh - static_cast<int64_t>(p.Nq - 1) * p.msq;
        } else {
            off += p.msq;
        }
    }
}

template <bool BF16>
__device__ __forceinline__ void bias_fold_column(uint32_t (&x)[32], const uint32_t (&r)[32],
                                                 int kind, float scale) {
    if (kind == 2) {
        const uint64_t sc2 = f2(scale, scale);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint64_t t = ffma2(f2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])), sc2,
                                     f2(half_to_float<BF16>(r[i]), half_to_float<BF16>(r[i + 1])));
            x[i] = __float_as_uint(f2lo(t));
            x[i + 1] = __float_as_uint(f2hi(t));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (r[i] == 0u) x[i] = __float_as_uint(-INFINITY);
    }
}

constexpr int kDqKStages = 3;  // dQ kernel: K ring (live from S_j to dQ_j)
constexpr int kDqVStages = 2;  // dQ kernel: V ring (live until dP_j)
// K stages of the dQ kernel: one fewer at D = 128 with a staged general mask
// (its bias takes that stage's shared memory).
template <int D, bool STAGE>
constexpr int dq_kstages() { return (STAGE && D == 128) ? kDqKStages - 1 : kDqKStages; }

template <int D>
struct BwdCfg {
    static constexpr int kTileBytes = kRows * D * 2;
    static constexpr int kKB = D / 64;
};

// ---------------------------------------------------------------- dK / dV
// Each 128-query tile is processed as two halves of 64 queries, one per pair
// of elementwise warpgroups, so that the tensor core works on one half while
// the other half's P^T / dS^T are computed.  TMEM: half u holds S^T_u at
// [128u, 128u+64) and dP^T_u at [128u+64, 128u+128) (M = 128 keys, N = 64
// queries).  The warp of 32-query chunk c of the half packs its P^T / dS^T
// into the first 16 of its own 32 columns ([128u+32c, +16) and
// [128u+64+32c, +16)), which it has already read, so the products read A
// from two column ranges.  dV at [256, 256+D), dK at [256+D, 256+2D).
// bf16: P^T has 8 significant bits, too few for dV = sum_i P_i dO_i over many
// queries; the chunk's warp also packs the low-order part of P^T (bf16(p -
// P^T)) into the other 16 of its 32 S^T columns, and a second product adds
// it, so dV sees P to about 16 bits.
// MMA order per tile n: for u = 0, 1: dV/dK += (half u of tile n) as soon as
// its P^T / dS^T are in TMEM, then S^T / dP^T of half u of tile n+1 into the
// same columns (the tensor pipe runs in order, so the products of tile n have
// read them first).
template <int D, bool BF16, bool CAUSAL, bool MASK>
__global__ void __launch_bounds__(kKvThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const BwdParams p) {
    using C = BwdCfg<D>;
    constexpr int TB = C::kTileBytes, KB = C::kKB, QS = 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;
    uint8_t* sV = sK + TB;
    uint8_t* sQ = sV + TB;             // [QS]
    uint8_t* sDO = sQ + QS * TB;       // [QS]
    float* sL = reinterpret_cast<float*>(sDO + QS * TB);  // [QS][128] -lse2 of the query tile
    float* sDl = sL + QS * kRows;                          // [QS][128] -delta
    uint64_t* bars = reinterpret_cast<uint64_t*>(sDl + QS * kRows);
    uint64_t* kv_full = bars;
    uint64_t* q_full = kv_full + 1;    // [QS]
    uint64_t* q_empty = q_full + QS;   // [QS]
    uint64_t* s_full = q_empty + QS;   // [2] S^T_u and dP^T_u in TMEM
    uint64_t* p_full = s_full + 2;     // [2] P^T_u and dS^T_u in TMEM (128 arrivals)
    uint64_t* acc_full = p_full + 2;   // last dV / dK product done
    uint64_t* mma_done = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Heaviest first: under the causal mask low key tiles meet the most queries.
    // CTA (group, key tile kt, query range sp): consecutive CTAs share a key
    // tile; range sp takes query tiles [qi0, qi1).
    const int unit = static_cast<int>(blockIdx.x / p.kv_splits);
    const int sp = static_cast<int>(blockIdx.x % p.kv_splits);
    const int group = unit / p.n_ktiles;
    const int kt = unit % p.n_ktiles;
    const int key0 = kt * kRows;
    const int qi0 = sp * p.qtiles_per_split;
    const int qi1 = min(p.n_qtiles, qi0 + p.qtiles_per_split);
    // head (within the group) and position of the first row of query tile qi0
    const int64_t r0 = static_cast<int64_t>(qi0) * kRows;
    const int head_0 = static_cast<int>(r0 / p.Nq);
    const int pos_0 = static_cast<int>(r0 % p.Nq);
    // Query tile qi (first-row position pos) meets this key tile.
    // A boolean mask that depends on the key alone (one row of keep bytes per
    // KV group, as a padding mask is) may remove every key of this tile: then
    // no query tile is visited and dK, dV of the tile are zero.
    const bool key_only = MASK && p.mask_kind == 1 && p.msq == 0 && (p.msh == 0 || p.G == 1);
    volatile int* tile_kept = reinterpret_cast<volatile int*>(abort_flag + 1);
    if (key_only && warp == 0) {
        const uint8_t* krow = static_cast<const uint8_t*>(p.mask) + (group / p.Hkv) * p.msb +
                              (group % p.Hkv) * p.msh;
        const int last = last_kept_key(krow, key0, min(p.Nk, key0 + kRows), lane);
        if (lane == 0) *tile_kept = last >= 0 ? 1 : 0;
    }
    bool any_kept = true;   // set after the set-up barrier
    auto visit = [&](int qi, int pos) {
        return any_kept && (!CAUSAL || tile_max_pos_at(qi, pos, p) >= key0);
    };

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < QS; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
        for (int u = 0; u < 2; ++u) {
            mbar_init(&s_full[u], 1);
            mbar_init(&p_full[u], 256);
        }
        mbar_init(acc_full, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kKvMmaWarp) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (key_only) any_kept = *tile_kept != 0;

    if (warp == kKvProducerWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmDO);
            mbar_arrive_expect_tx(kv_full, 2 * TB);
            for (int kb = 0; kb < KB; ++kb) {
                tma_load_3d(&tmK, kv_full, sK + kb * (kRows * 128), kb * 64, key0, group);
                tma_load_3d(&tmV, kv_full, sV + kb * (kRows * 128), kb * 64, key0, group);
            }
            int n = 0;
            for (int qi = qi0, pos = pos_0; qi < qi1; ++qi, pos = next_tile_pos(pos, p.Nq)) {
                if (!visit(qi, pos)) continue;
                const int slot = n % QS;
                if (!mbar_wait(&q_empty[slot], ((n / QS) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&q_full[slot], 2 * TB + 2 * kRows * 4);
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_3d(&tmQ, &q_full[slot], sQ + slot * TB + kb * (kRows * 128), kb * 64,
                                qi * kRows, group);
                    tma_load_3d(&tmDO, &q_full[slot], sDO + slot * TB + kb * (kRows * 128),
                                kb * 64, qi * kRows, group);
                }
                const int64_t w0 = static_cast<int64_t>(group) * p.rows_pad + qi * kRows;
                bulk_load(sL + slot * kRows, p.nlse2 + w0, kRows * 4, &q_full[slot]);
                bulk_load(sDl + slot * kRows, p.ndelta + w0, kRows * 4, &q_full[slot]);
                ++n;
            }
            mbar_wait_bounded(kv_full, 0, p.status);
            for (int m = (n > QS ? n - QS : 0); m < n; ++m)
                mbar_wait_bounded(&q_full[m % QS], (m / QS) & 1, p.status);
        }
    } else if (warp == kKvMmaWarp) {
        constexpr uint32_t idesc_s = idesc_f16(kRows, 64, BF16, false);  // 128 keys x 64 queries
        constexpr uint32_t idesc_g = idesc_f16(kRows, D, BF16, true);
        constexpr uint64_t kStep = TB >> 4;
        constexpr uint64_t kBlk = (kRows * 128) >> 4;
        // 64 rows of a 128-byte-swizzled tile, in 16-byte descriptor units:
        // query half u starts 64u rows into the Q / dO tiles (the N rows of
        // the K-major view, the K rows of the MN-major view).
        constexpr uint64_t kHalf = (64 * 128) >> 4;
        const uint64_t dK_ = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dV_ = smem_desc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t dQk = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dDOk = smem_desc_sw128(smem_u32(sDO), 16, 1024);
        const uint64_t dQm = smem_desc_sw128(smem_u32(sQ), kRows * 128, 1024);
        const uint64_t dDOm = smem_desc_sw128(smem_u32(sDO), kRows * 128, 1024);
        // S^T_u = K Q_u^T and dP^T_u = V dO_u^T of the tile in `slot`.
        auto issue_sdp = [&](int slot, int u) {
            const uint32_t d = tmem + 128 * u;
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                mma_ss_k64(d, dK_ + kb * kBlk, dQk + slot * kStep + kb * kBlk + u * kHalf, idesc_s,
                           kb > 0 ? 1u : 0u);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                mma_ss_k64(d + 64, dV_ + kb * kBlk, dDOk + slot * kStep + kb * kBlk + u * kHalf,
                           idesc_s, kb > 0 ? 1u : 0u);
            mma_commit_elect(&s_full[u]);
        };
        int n_vis = 0;   // query tiles this key tile meets (the producer loads them in order)
        for (int qi = qi0, pos = pos_0; qi < qi1; ++qi, pos = next_tile_pos(pos, p.Nq))
            n_vis += visit(qi, pos) ? 1 : 0;
        warp_wait(kv_full, 0, abort_flag, p.status);
        if (n_vis > 0) {
            warp_wait(&q_full[0], 0, abort_flag, p.status);
            tc_fence_after();
            issue_sdp(0, 0);
            issue_sdp(0, 1);
        }
        // A wait that times out sets the abort flag and later waits return at
        // once, so the loop runs to its end without blocking.
        for (int n = 0; n < n_vis; ++n) {
            const int slot = n % QS, nslot = (n + 1) % QS;
#pragma unroll 1
            for (int u = 0; u < 2; ++u) {
                warp_wait(&p_full[u], n & 1, abort_flag, p.status);
                tc_fence_after();
                const uint32_t acc = (n > 0 || u > 0) ? 1u : 0u;
                // dV += P^T_u dO_u, dK += dS^T_u Q_u (K = the 64 queries of half u)
                const uint32_t pu = tmem + 128 * u;
                mma_ts_k64_split(tmem + 256, pu, pu + 32, dDOm + slot * kStep + u * kHalf, idesc_g,
                                 acc);
                if constexpr (BF16)   // dV += (low-order part of P^T_u) dO_u
                    mma_ts_k64_split(tmem + 256, pu + 16, pu + 48, dDOm + slot * kStep + u * kHalf,
                                     idesc_g, 1u);
                mma_ts_k64_split(tmem + 256 + D, pu + 64, pu + 96, dQm + slot * kStep + u * kHalf,
                                 idesc_g, acc);
                if (u == 1) mma_commit_elect(&q_empty[slot]);
                if (n + 1 < n_vis) {
                    if (u == 0) {
                        warp_wait(&q_full[nslot], ((n + 1) / QS) & 1, abort_flag, p.status);
                        tc_fence_after();
                    }
                    issue_sdp(nslot, u);
                }
            }
        }
        mma_commit_elect(acc_full);
        mma_commit_elect(mma_done);
        mbar_wait_bounded(mma_done, 0, p.status);
    } else {
        // One thread per key row and 32-query chunk: warp w reads TMEM lanes
        // 32(w%4) .. 32(w%4)+31, query half hq = (w/4)%2, chunk cc = w/8 of it.
        const int quad = warp & 3, hq = (warp >> 2) & 1, cc = warp >> 3;
        const int c = 2 * hq + cc;   // 32-query chunk of the tile
        const int key = key0 + quad * 32 + lane;
        const uint32_t lb = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lb + 128 * hq + 32 * cc, tDP = tS + 64;
        const float sl2 = p.scale_log2;
        // scale still to apply to the scores read below: an additive bias
        // leaves natural-log logits (log2 e), a boolean one raw scores
        const float sc = (MASK && p.mask_kind == 2) ? kLog2e : sl2;
        const int64_t b_off = MASK ? static_cast<int64_t>(group / p.Hkv) * p.msb : 0;
        const int head0 = MASK ? (group % p.Hkv) * p.G : 0;
        int n = 0;
        int head = head_0;   // head within the group of the current tile's first row
        for (int qi = qi0, pos = pos_0; qi < qi1; ++qi, next_tile(pos, head, p.Nq)) {
            if (!visit(qi, pos)) continue;
            const int slot = n % QS;
            // This chunk's bias column, requested before the waits for the
            // tile's Q and S (their latency hides the loads').
            uint32_t bcol[MASK ? 32 : 1];
            if constexpr (MASK) {
                int cpos = pos + 32 * c, chead = head;   // first query row of the chunk
                while (cpos >= p.Nq) {
                    cpos -= p.Nq;
                    ++chead;
                }
                const int64_t left = p.rows_per_group - static_cast<int64_t>(qi) * kRows - 32 * c;
                bias_load_column(bcol, p, b_off, head0 + chead, cpos, key,
                                 left <= 0 ? 0 : left < 32 ? static_cast<int>(left) : 32);
            }
            warp_wait(&q_full[slot], (n / QS) & 1, abort_flag, p.status);
            warp_wait(&s_full[hq], n & 1, abort_flag, p.status);
            tc_fence_after();
            if constexpr (MASK) {
                // this chunk's scores -> logits with the bias, in place in TMEM
                uint32_t x[32];
                tmem_ld32(tS, x);
                tmem_wait_ld();
                reg_fence(x);
                bias_fold_column<BF16>(x, bcol, p.mask_kind, p.scale);
                tmem_st32(tS, x);
                tmem_wait_st();
            }
            uint32_t sv[32], dp[32];
            tmem_ld32(tS, sv);
            tmem_ld32(tDP, dp);
            const int64_t row0 = static_cast<int64_t>(qi) * kRows;
            const int base = pos;
            const float* L = sL + slot * kRows + c * 32;
            const float* Dl = sDl + slot * kRows + c * 32;
            // No mask anywhere in this warp's 32 x 32 block: every column is a
            // real row of the group, every key exists, and (causal) the warp's
            // last key is at or before the chunk's first query position.
            const int wkey_last = key0 + quad * 32 + 31;
            const int q_first = c * 32;
            bool fast = (row0 + q_first + 32 <= p.rows_per_group) && (wkey_last < p.Nk);
            if (CAUSAL)
                fast = fast && (base + q_first + 32 <= p.Nq) && (wkey_last <= base + q_first);
            const uint64_t sl22 = f2(sc, sc);
            tmem_wait_ld();
            reg_fence(sv);
            reg_fence(dp);
            uint32_t pw[16], dw[16];
            uint32_t plw[BF16 ? 16 : 1];   // bf16: low-order parts of P^T
            if (fast) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(L + i);
                    const float4 d4 = *reinterpret_cast<const float4*>(Dl + i);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int e = i + 2 * h;
                        const uint64_t x = ffma2(f2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                 sl22, h ? f2(l4.z, l4.w) : f2(l4.x, l4.y));
                        const float p0 = ex2_ftz(f2lo(x)), p1 = ex2_ftz(f2hi(x));
                        const uint64_t dd = fmul2(
                            f2(p0, p1),
                            fadd2(f2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                  h ? f2(d4.z, d4.w) : f2(d4.x, d4.y)));
                        pw[e >> 1] = pack2<BF16>(p0, p1);
                        dw[e >> 1] = pack2<BF16>(f2lo(dd), f2hi(dd));
                        if constexpr (BF16) plw[e >> 1] = bf16x2_residual(p0, p1, pw[e >> 1]);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float pp[2], dd[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int q = q_first + i + u;
                        bool ok = (row0 + q < p.rows_per_group) && (key < p.Nk);
                        if (CAUSAL) ok = ok && key <= tile_pos(base, q, p.Nq);
                        const float pr = ex2_ftz(fmaf(__uint_as_float(sv[i + u]), sc, L[i + u]));
                        pp[u] = ok ? pr : 0.0f;
                        dd[u] = ok ? pr * (__uint_as_float(dp[i + u]) + Dl[i + u]) : 0.0f;
                    }
                    pw[i >> 1] = pack2<BF16>(pp[0], pp[1]);
                    dw[i >> 1] = pack2<BF16>(dd[0], dd[1]);
                    if constexpr (BF16) plw[i >> 1] = bf16x2_residual(pp[0], pp[1], pw[i >> 1]);
                }
            }
            // The packed P^T / dS^T of this chunk go to the first 16 of its own
            // 32 columns, which are already read into registers.
            tmem_st16(tS, pw);
            tmem_st16(tDP, dw);
            if constexpr (BF16) tmem_st16(tS + 16, plw);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[hq]);
            ++n;
        }
        // epilogue: dV and scale * dK of this key row, D/4 columns per warp
        constexpr int CW = D / 4;   // 32 (D = 128) or 16 (D = 64)
        const int col0 = (hq + 2 * cc) * CW;
        const bool ok = *abort_flag == 0;
        const int64_t grow = static_cast<int64_t>(group) * p.Nk + key;
        uint16_t* dvp = static_cast<uint16_t*>(p.dv) + grow * D + col0;
        uint16_t* dkp = static_cast<uint16_t*>(p.dk) + grow * D + col0;
        if (n > 0) warp_wait(acc_full, 0, abort_flag, p.status);
        tc_fence_after();
        // dV first, then dK, so only one accumulator chunk is live at a time.
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            uint32_t a[CW];
            if (n > 0) {
                const uint32_t src = tmem + lb + 256 + which * D + col0;
                if constexpr (CW == 32) tmem_ld32(src, a);
                else tmem_ld16(src, a);
                tmem_wait_ld();
                reg_fence(a);
            } else {
#pragma unroll
                for (int i = 0; i < CW; ++i) a[i] = 0u;
            }
            if (ok && key < p.Nk && p.kv_splits > 1) {
                // this query range's fp32 partial sum (dK unscaled)
                float* dst = (which ? p.dk_part : p.dv_part) +
                             (static_cast<int64_t>(sp) * p.n_groups * p.Nk + grow) * D + col0;
#pragma unroll
                for (int i = 0; i < CW / 4; ++i)
                    reinterpret_cast<float4*>(dst)[i] =
                        make_float4(__uint_as_float(a[4 * i]), __uint_as_float(a[4 * i + 1]),
                                    __uint_as_float(a[4 * i + 2]), __uint_as_float(a[4 * i + 3]));
            } else if (ok && key < p.Nk) {
                const float sc = which ? p.scale : 1.0f;
                uint32_t w[CW / 2];
#pragma unroll
                for (int i = 0; i < CW / 2; ++i)
                    w[i] = pack2<BF16>(__uint_as_float(a[2 * i]) * sc, __uint_as_float(a[2 * i + 1]) * sc);
                uint4* dst = reinterpret_cast<uint4*>(which ? dkp : dvp);
#pragma unroll
                for (int i = 0; i < CW / 8; ++i)
                    dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kKvMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // Launched as a programmatic dependent of the dQ kernel (whose results it
    // does not read): it does not end before dQ has, so whatever follows in the
    // stream sees both.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// General bias, dQ layout: the next key tile's bias for a warp's 32 rows x 32
// keys [key0, key0 + 32) (inside [0, Nk)), staged with cp.async, whole rows
// per instruction (4 16-byte chunks per row for a 16-bit additive bias, 2 for
// a boolean one).  Chunk q of row r sits at chunk position q ^ ((r >> 1) & 3)
// (additive, 64-byte rows) or q ^ ((r >> 2) & 1) (boolean, 32-byte rows), so
// the fold's reads (one row per lane, 16 bytes at a time) meet every bank once
// per 8 lanes.  Rows r >= nvalid (1 <= nvalid <= 32) copy row nvalid - 1.
// Wait with cp_async_wait_all and then __syncwarp before reading.
__device__ __forceinline__ void bias_prefetch32(uint32_t buf, const uint8_t* row_ptr, int kind,
                                                int key0, int nvalid, int lane) {
    const unsigned long long mine = reinterpret_cast<uintptr_t>(row_ptr);
    const bool add = kind == 2;
    const int cshift = add ? 2 : 1;   // log2 chunks per row
    const int q = lane & ((1 << cshift) - 1);
    const int n_ins = add ? 4 : 2;    // 32 rows / (32 >> cshift) rows per instruction
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i >= n_ins) break;
        const int r = (i << (5 - cshift)) + (lane >> cshift);
        const unsigned long long base = __shfl_sync(0xffffffffu, mine, min(r, nvalid - 1));
        const uint8_t* src = reinterpret_cast<const uint8_t*>(base) +
                             static_cast<int64_t>(key0) * (add ? 2 : 1) + 16 * q;
        const int slot = add ? (q ^ ((r >> 1) & 3)) : (q ^ ((r >> 2) & 1));
        cp_async16(buf + r * (add ? 64 : 32) + (slot << 4), src);
    }
    cp_async_commit();
}

// This lane's staged 32 bias values folded into its 32 scores: natural-log
// logits u = s * scale + b (additive) or raw scores / -inf (boolean), the
// arithmetic of the forward's fold.
template <bool BF16>
__device__ __forceinline__ void bias_fold_smem32(uint32_t (&s)[32], uint32_t buf, int kind,
                                                 float scale, int lane) {
    if (kind == 2) {
        const uint32_t rbase = buf + lane * 64;
        const int sw = (lane >> 1) & 3;
        const uint64_t sc2 = f2(scale, scale);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(rbase + ((q ^ sw) << 4)));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 8 * q + 2 * e;
                const uint64_t t =
                    ffma2(f2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), sc2,
                          f2(half_to_float<BF16>(w[e] & 0xffffu), half_to_float<BF16>(w[e] >> 16)));
                s[k] = __float_as_uint(f2lo(t));
                s[k + 1] = __float_as_uint(f2hi(t));
            }
        }
    } else {
        const uint32_t rbase = buf + lane * 32;
        const int sw = (lane >> 2) & 1;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(rbase + ((q ^ sw) << 4)));
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (((w[i >> 2] >> (8 * (i & 3))) & 0xffu) == 0u)
                    s[16 * q + i] = __float_as_uint(-INFINITY);
        }
    }
}

// The same fold read from the bias row key by key (keys >= Nk and unreal rows:
// no bias), for a key tile that reaches past Nk.
template <bool BF16>
__device__ __forceinline__ void bias_fold_direct32(uint32_t (&s)[32], const uint8_t* row, int kind,
                                                   int key0, int Nk, float scale, bool row_ok) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int key = key0 + i;
        const bool in = row_ok && key < Nk;
        if (kind == 2) {
            const float b =
                in ? half_to_float<BF16>(reinterpret_cast<const uint16_t*>(row)[key]) : 0.0f;
            s[i] = __float_as_uint(fmaf(__uint_as_float(s[i]), scale, b));
        } else if (in && row[key] == 0) {
            s[i] = __float_as_uint(-INFINITY);
        }
    }
}

// ---------------------------------------------------------------- dQ
// TMEM: S [0,128), dP [128,256), dQ [256,256+D), dS [384,448) (packed 16-bit).
// Warpgroup h owns key columns [32 CPW h, 32 CPW (h+1)).  dS has its own columns, so once
// every warpgroup has read S_j and dP_j into registers (s_free) the tensor
// core computes S_{j+1} and dP_{j+1} while the elementwise work on j runs.
template <int D, bool BF16, bool CAUSAL, int MK>
__global__ void __launch_bounds__(dq_threads<MK, D>(), 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const BwdParams p) {
    using C = BwdCfg<D>;
    // MK: 0 no mask, 1 a general bias, 2 a boolean mask that depends on the
    // key alone (the same keep bytes for every row: read directly, served to
    // the whole warp at once).
    constexpr bool MASK = MK != 0, STAGE = MK == 1;
    // K lives from S_j to dQ_j, V only until dP_j: separate rings, K deeper.
    // A general mask stages each warp's next 32 x 64 bias block in shared
    // memory (8 warps x 4 KB); at D = 128 the K ring gives a stage for it.
    constexpr int TB = C::kTileBytes, KB = C::kKB, VS = kDqVStages;
    constexpr int KS = dq_kstages<D, STAGE>();
    constexpr int EW = dq_ew<MK, D>();
    constexpr int CPW = 128 / (EW / 4) / 32;   // 32-column chunks per elementwise warp
    constexpr int kProducerWarp = EW, kMmaWarp = EW + 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sDO = sQ + TB;
    uint8_t* sK = sDO + TB;           // [KS]
    uint8_t* sV = sK + KS * TB;       // [VS]
    uint8_t* sB = sV + VS * TB;       // [8 warps][32 rows][64 keys x 2 bytes] (STAGE)
    float* sL = reinterpret_cast<float*>(sB + (STAGE ? 8 * 4096 : 0));
    float* sDl = sL + kRows;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sDl + kRows);
    uint64_t* q_full = bars;
    uint64_t* k_full = q_full + 1;    // [KS]
    uint64_t* k_empty = k_full + KS;  // [KS]
    uint64_t* v_full = k_empty + KS;  // [VS]
    uint64_t* v_empty = v_full + VS;  // [VS]
    uint64_t* s_full = v_empty + VS;  // S_j and dP_j in TMEM
    uint64_t* s_free = s_full + 1;     // S_j and dP_j read by all 256 threads
    uint64_t* p_full = s_free + 1;     // dS_j in TMEM (256 arrivals)
    uint64_t* dq_done = p_full + 1;    // dQ += dS_j K_j done (dS columns free)
    uint64_t* acc_full = dq_done + 1;
    uint64_t* mma_done = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = static_cast<int>(blockIdx.x / p.n_qtiles);
    const int qi = p.n_qtiles - 1 - static_cast<int>(blockIdx.x % p.n_qtiles);
    const int64_t row0 = static_cast<int64_t>(qi) * kRows;
    int nkv = (p.Nk + kRows - 1) / kRows;
    if (CAUSAL) {
        const int keys = min(tile_max_pos(row0, p) + 1, p.Nk);
        nkv = (keys + kRows - 1) / kRows;
    }
    // A boolean mask that depends on the key alone: the key tiles past its last
    // kept key contribute nothing to dQ (at least one tile is kept, so rows with
    // no kept key still end with dQ = 0).
    const bool key_only = MASK && p.mask_kind == 1 && p.msq == 0 && (p.msh == 0 || p.G == 1);
    volatile int* key_lim = reinterpret_cast<volatile int*>(abort_flag + 1);
    if (key_only && warp == 0 && nkv > 0) {
        const uint8_t* krow = static_cast<const uint8_t*>(p.mask) + (group / p.Hkv) * p.msb +
                              (group % p.Hkv) * p.msh;
        const int last = last_kept_key(krow, 0, min(p.Nk, nkv * kRows), lane);
        if (lane == 0) *key_lim = last < 0 ? 1 : last / kRows + 1;
    }

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < KS; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
        for (int i = 0; i < VS; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
        mbar_init(s_full, 1);
        mbar_init(s_free, EW * 32);
        mbar_init(p_full, EW * 32);
        mbar_init(dq_done, 1);
        mbar_init(acc_full, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (key_only && nkv > 0) nkv = min(nkv, *key_lim);
    // Launched as a programmatic dependent of the statistics kernel: its set-up
    // above overlaps that kernel's end; nothing below runs before its results
    // are complete.  Then the dK/dV kernel, which reads nothing this one
    // writes, may start on the SMs this grid leaves idle once every CTA here
    // has passed this point (so it, too, sees the statistics).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == kProducerWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(q_full, 2 * TB + 2 * kRows * 4);
            for (int kb = 0; kb < KB; ++kb) {
                tma_load_3d(&tmQ, q_full, sQ + kb * (kRows * 128), kb * 64, qi * kRows, group);
                tma_load_3d(&tmDO, q_full, sDO + kb * (kRows * 128), kb * 64, qi * kRows, group);
            }
            const int64_t w0 = static_cast<int64_t>(group) * p.rows_pad + row0;
            bulk_load(sL, p.nlse2 + w0, kRows * 4, q_full);
            bulk_load(sDl, p.ndelta + w0, kRows * 4, q_full);
            int nk = 0, nv = 0;
            for (int j = 0; j < nkv; ++j) {
                const int ks = j % KS, vs = j % VS;
                if (!mbar_wait(&k_empty[ks], ((j / KS) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&k_full[ks], TB);
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d(&tmK, &k_full[ks], sK + ks * TB + kb * (kRows * 128), kb * 64,
                                j * kRows, group);
                ++nk;
                if (!mbar_wait(&v_empty[vs], ((j / VS) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&v_full[vs], TB);
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d(&tmV, &v_full[vs], sV + vs * TB + kb * (kRows * 128), kb * 64,
                                j * kRows, group);
                ++nv;
            }
            mbar_wait_bounded(q_full, 0, p.status);
            for (int m = (nk > KS ? nk - KS : 0); m < nk; ++m)
                mbar_wait_bounded(&k_full[m % KS], (m / KS) & 1, p.status);
            for (int m = (nv > VS ? nv - VS : 0); m < nv; ++m)
                mbar_wait_bounded(&v_full[m % VS], (m / VS) & 1, p.status);
        }
    } else if (warp == kMmaWarp) {
        constexpr uint32_t idesc_s = idesc_f16(kRows, kRows, BF16, false);
        constexpr uint32_t idesc_g = idesc_f16(kRows, D, BF16, true);
        constexpr uint64_t kStep = TB >> 4;
        constexpr uint64_t kBlk = (kRows * 128) >> 4;
        const uint64_t dQk = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dDOk = smem_desc_sw128(smem_u32(sDO), 16, 1024);
        const uint64_t dKk = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dVk = smem_desc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t dKm = smem_desc_sw128(smem_u32(sK), kRows * 128, 1024);
        // S_j = Q K_j^T and dP_j = dO V_j^T, one commit for both.
        auto issue_s_dp = [&](int j) {
            const int ks = j % KS, vs = j % VS;
            warp_wait(&k_full[ks], (j / KS) & 1, abort_flag, p.status);
            warp_wait(&v_full[vs], (j / VS) & 1, abort_flag, p.status);
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                mma_ss_k64(tmem, dQk + kb * kBlk, dKk + ks * kStep + kb * kBlk, idesc_s,
                           kb > 0 ? 1u : 0u);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                mma_ss_k64(tmem + 128, dDOk + kb * kBlk, dVk + vs * kStep + kb * kBlk, idesc_s,
                           kb > 0 ? 1u : 0u);
            mma_commit_elect(s_full);
            mma_commit_elect(&v_empty[vs]);   // V_j is only read by dP_j
        };
        warp_wait(q_full, 0, abort_flag, p.status);
        if (nkv > 0) issue_s_dp(0);
        for (int j = 0; j < nkv; ++j) {
            const int ks = j % KS;
            if (j + 1 < nkv) {
                warp_wait(s_free, j & 1, abort_flag, p.status);
                issue_s_dp(j + 1);
            }
            warp_wait(p_full, j & 1, abort_flag, p.status);
            tc_fence_after();
            mma_ts_k128(tmem + 256, tmem + 384, dKm + ks * kStep, idesc_g, j > 0 ? 1u : 0u);
            mma_commit_elect(dq_done);
            mma_commit_elect(&k_empty[ks]);
        }
        mma_commit_elect(acc_full);
        mma_commit_elect(mma_done);
        mbar_wait_bounded(mma_done, 0, p.status);
    } else {
        const int hq = warp >> 2, quad = warp & 3;   // column group, TMEM lane quadrant
        const int64_t row = row0 + quad * 32 + lane;
        const bool row_ok = row < p.rows_per_group;
        const int pos = static_cast<int>(row % p.Nq);
        const uint32_t lb = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lb, tDP = tmem + lb + 128;
        const float sl2 = p.scale_log2;
        warp_wait(q_full, 0, abort_flag, p.status);
        const float nl = sL[quad * 32 + lane];   // -lse2 of this row
        const float nd = sDl[quad * 32 + lane];  // -delta of this row
        const int lim = CAUSAL ? min(p.Nk, pos + 1) : p.Nk;  // keys [0, lim) allowed
        // Smallest position among this warp's rows: key tiles past it (or past
        // Nk) need the mask.  Rows past the group only feed their own dQ rows,
        // which are never stored, so they need none.
        const int64_t wr0 = row0 + quad * 32;
        const int64_t wr1 = min(wr0 + 31, p.rows_per_group - 1);
        const int warp_min_pos = (wr0 / p.Nq == wr1 / p.Nq) ? static_cast<int>(wr0 % p.Nq) : 0;
        // scale still to apply to the scores read below: an additive bias
        // leaves natural-log logits (log2 e), a boolean one raw scores
        const float sc = (MASK && p.mask_kind == 2) ? kLog2e : sl2;
        const uint64_t sl22 = f2(sc, sc), nl2 = f2(nl, nl), nd2 = f2(nd, nd);
        const uint32_t tDS = tmem + lb + 384;
        // This row's bias: query head hkv*G + row/Nq of batch group/Hkv.
        const uint8_t* mrow = nullptr;
        if constexpr (MASK) {
            const int64_t h = static_cast<int64_t>(group % p.Hkv) * p.G + row / p.Nq;
            const int64_t b = group / p.Hkv;
            mrow = static_cast<const uint8_t*>(p.mask) +
                   (b * p.msb + h * p.msh + pos * p.msq) * (p.mask_kind == 2 ? 2 : 1);
        }
        // Staged bias (MK = 1): this warp's 32 rows x the 32 CPW keys of its
        // column group of each key tile, one tile ahead, nvalid rows real; a
        // group past Nk reads its bias directly.
        const int64_t wleft = p.rows_per_group - wr0;
        const int nvalid = wleft <= 0 ? 0 : wleft >= 32 ? 32 : static_cast<int>(wleft);
        const uint32_t bbuf = smem_u32(sB) + warp * (CPW * 2048);
        auto staged = [&](int jj) {
            return STAGE && nvalid > 0 && jj * kRows + 32 * CPW * (hq + 1) <= p.Nk;
        };
        auto prefetch = [&](int key0) {
            if constexpr (CPW == 2) bias_prefetch<64>(bbuf, mrow, p.mask_kind, key0, nvalid, lane);
            else bias_prefetch32(bbuf, mrow, p.mask_kind, key0, nvalid, lane);
        };
        if constexpr (STAGE)
            if (nkv > 0 && staged(0)) prefetch(32 * CPW * hq);
        for (int j = 0; j < nkv; ++j) {
            const int k0 = j * kRows;
            warp_wait(s_full, j & 1, abort_flag, p.status);
            tc_fence_after();
            const bool need_mask = (k0 + kRows > p.Nk) || (CAUSAL && k0 + kRows - 1 > warp_min_pos);
            uint32_t sv[CPW][32], dp[CPW][32];
#pragma unroll
            for (int cc = 0; cc < CPW; ++cc) {
                tmem_ld32(tS + (CPW * hq + cc) * 32, sv[cc]);
                tmem_ld32(tDP + (CPW * hq + cc) * 32, dp[cc]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < CPW; ++cc) {
                reg_fence(sv[cc]);
                reg_fence(dp[cc]);
            }
            // S_j and dP_j are in registers: the next S and dP may overwrite them.
            tc_fence_before();
            mbar_arrive(s_free);
            if constexpr (MK == 2 && CPW == 1) {
                keep_fold32(sv[0], mrow, k0 + 32 * hq, p.Nk);
            } else if constexpr (MASK) {
                // this group's scores -> logits with the bias; then the next
                // key tile's bias is requested into the same rows
                if (staged(j)) {
                    cp_async_wait_all();
                    __syncwarp();
                    if constexpr (CPW == 2) bias_fold_smem64<BF16>(sv, bbuf, p.mask_kind, p.scale, lane);
                    else bias_fold_smem32<BF16>(sv[0], bbuf, p.mask_kind, p.scale, lane);
                    __syncwarp();
                } else {
                    if constexpr (CPW == 2)
                        bias_fold_direct64<BF16>(sv, mrow, p.mask_kind, k0 + 64 * hq, p.Nk, p.scale,
                                                 row_ok);
                    else
                        bias_fold_direct32<BF16>(sv[0], mrow, p.mask_kind, k0 + 32 * hq, p.Nk,
                                                 p.scale, row_ok);
                }
                if (j + 1 < nkv && staged(j + 1)) prefetch(k0 + kRows + 32 * CPW * hq);
            }
            // dS columns still feed dQ += dS_{j-1} K_{j-1}.
            if (j > 0) {
                warp_wait(dq_done, (j - 1) & 1, abort_flag, p.status);
                tc_fence_after();
            }
#pragma unroll
            for (int cc = 0; cc < CPW; ++cc) {
                const int c = CPW * hq + cc;   // 32-column chunk of the tile
                uint32_t dw[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const uint64_t x = ffma2(f2(__uint_as_float(sv[cc][i]), __uint_as_float(sv[cc][i + 1])),
                                             sl22, nl2);
                    float p0 = ex2_ftz(f2lo(x)), p1 = ex2_ftz(f2hi(x));
                    if (need_mask) {
                        const int kk = k0 + c * 32 + i;
                        p0 = kk < lim ? p0 : 0.0f;
                        p1 = kk + 1 < lim ? p1 : 0.0f;
                    }
                    const uint64_t dd = fmul2(
                        f2(p0, p1),
                        fadd2(f2(__uint_as_float(dp[cc][i]), __uint_as_float(dp[cc][i + 1])), nd2));
                    dw[i >> 1] = pack2<BF16>(f2lo(dd), f2hi(dd));
                }
                tmem_st16(tDS + 16 * c, dw);   // keys 32c.. -> dS columns 16c..
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // No bias copy may still be in flight when the CTA gives up its shared memory.
        if constexpr (STAGE) cp_async_wait_all();
        const bool ok = *abort_flag == 0;
        if (nkv > 0) warp_wait(acc_full, 0, abort_flag, p.status);
        tc_fence_after();
        uint16_t* dqp = static_cast<uint16_t*>(p.dq) + (static_cast<int64_t>(group) * p.rows_per_group + row) * D;
        // this warpgroup's dQ columns: a contiguous half with 8 warps, every
        // fourth 32-column chunk with 16
        constexpr int kC0 = EW == 8 ? D / 64 : 1, kCStep = EW == 8 ? 1 : EW / 4;
#pragma unroll 1
        for (int c = hq * kC0; c < (EW == 8 ? (hq + 1) * kC0 : D / 32); c += kCStep) {
            uint32_t a[32];
            tmem_ld32(tmem + lb + 256 + c * 32, a);
            tmem_wait_ld();
            reg_fence(a);
            if (ok && row_ok) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack2<BF16>(__uint_as_float(a[2 * i]) * p.scale,
                                       __uint_as_float(a[2 * i + 1]) * p.scale);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    reinterpret_cast<uint4*>(dqp + c * 32)[i] =
                        make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
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

template <int D>
constexpr int dkdv_smem() { return 2 * BwdCfg<D>::kTileBytes + 4 * BwdCfg<D>::kTileBytes + 2 * 2 * kRows * 4 + 256 + 1024; }
template <int D, bool STAGE>
constexpr int dq_smem() {
    return (2 + dq_kstages<D, STAGE>() + kDqVStages) * BwdCfg<D>::kTileBytes +
           (STAGE ? 8 * 4096 : 0) + 2 * kRows * 4 + 256 + 1024;
}

// Sum of the kv_splits partial dV / dK (fp32, in range order) into dv / dk
// in the input dtype (dK scaled): 8 consecutive elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_dkdv_reduce_kernel(const BwdParams p, int64_t n8) {
    // Launched as a programmatic dependent of the dK/dV kernel: wait for its
    // partial sums (and, through its own wait, for the dQ kernel).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const int64_t stride = n8 * 8;   // elements per range
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
        const float* src = (which ? p.dk_part : p.dv_part) + i * 8;
        float4 a = reinterpret_cast<const float4*>(src)[0];
        float4 b = reinterpret_cast<const float4*>(src)[1];
        for (int s = 1; s < p.kv_splits; ++s) {
            const float4 c = reinterpret_cast<const float4*>(src + s * stride)[0];
            const float4 d = reinterpret_cast<const float4*>(src + s * stride)[1];
            a = make_float4(a.x + c.x, a.y + c.y, a.z + c.z, a.w + c.w);
            b = make_float4(b.x + d.x, b.y + d.y, b.z + d.z, b.w + d.w);
        }
        const float sc = which ? p.scale : 1.0f;
        reinterpret_cast<uint4*>(which ? p.dk : p.dv)[i] =
            make_uint4(pack2<BF16>(a.x * sc, a.y * sc), pack2<BF16>(a.z * sc, a.w * sc),
                       pack2<BF16>(b.x * sc, b.y * sc), pack2<BF16>(b.z * sc, b.w * sc));
    }
}

// Launch as a programmatic dependent of the previous kernel in the stream:
// the grid may start before that kernel has ended, and waits for it on the
// device (griddepcontrol.wait) where it needs its results.
template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern kern, long long ctas, int threads, int smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D, bool BF16, bool CAUSAL, int MK>
cudaError_t launch_dq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                      const CUtensorMap& tmDO, const BwdParams& p, cudaStream_t stream) {
    auto kern = bwd_dq_kernel<D, BF16, CAUSAL, MK>;
    constexpr int smem = dq_smem<D, MK == 1>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.n_groups) * p.n_qtiles;
    return launch_dependent(kern, ctas, dq_threads<MK, D>(), smem, stream, tmQ, tmDO, tmK, tmV, p);
}

template <int D, bool BF16, bool CAUSAL, bool MASK>
cudaError_t launch_one(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmDO, const BwdParams& p, cudaStream_t stream) {
    {
        const int64_t threads = p.total_rows * (D / 8);
        const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
        cudaError_t e = launch_kernel(bwd_stats_kernel<D, BF16>, dim3(blocks), dim3(256), 0, stream, p);
        if (e != cudaSuccess) return e;
    }
    // Statistics, then dQ, then dK/dV, each a programmatic dependent of the
    // one before: dQ sets up while the statistics kernel ends; dQ and dK/dV
    // read the same inputs and statistics and write disjoint outputs, so
    // dK/dV's CTAs take the SMs that dQ's last wave leaves idle (dK/dV waits
    // for dQ only at its end); the partial sums' reduction sets up while
    // dK/dV ends.  A key-only boolean mask takes its own dQ instantiation (no
    // staging).
    const bool key_only = MASK && p.mask_kind == 1 && p.msq == 0 && (p.msh == 0 || p.G == 1);
    {
        const cudaError_t e =
            key_only ? launch_dq<D, BF16, CAUSAL, MASK ? 2 : 0>(tmQ, tmK, tmV, tmDO, p, stream)
                     : launch_dq<D, BF16, CAUSAL, MASK ? 1 : 0>(tmQ, tmK, tmV, tmDO, p, stream);
        if (e != cudaSuccess) return e;
    }
    auto kern = bwd_dkdv_kernel<D, BF16, CAUSAL, MASK>;
    constexpr int smem = dkdv_smem<D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.n_groups) * p.n_ktiles * p.kv_splits;
    e = launch_dependent(kern, ctas, kKvThreads, smem, stream, tmQ, tmDO, tmK, tmV, p);
    if (e != cudaSuccess) return e;
    if (p.kv_splits > 1) {
        const int64_t n8 = static_cast<int64_t>(p.n_groups) * p.Nk * D / 8;
        e = launch_dependent(bwd_dkdv_reduce_kernel<BF16>, (n8 + 255) / 256, 256, 0, stream, p, n8);
    }
    return e;
}

}  // namespace

cudaError_t launch_bwd(int D, bool bf16, bool causal, const CUtensorMap& tmQ,
                       const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                       const BwdParams& p, cudaStream_t stream) {
    const bool mask = p.mask != nullptr;
#define TME_CASE(d, b, c, m)                              \
    if (D == d && bf16 == b && causal == c && mask == m)  \
        return launch_one<d, b, c, m>(tmQ, tmK, tmV, tmDO, p, stream);
#define TME_CASES(m)              \
    TME_CASE(64, false, false, m)  \
    TME_CASE(64, false, true, m)   \
    TME_CASE(64, true, false, m)   \
    TME_CASE(64, true, true, m)    \
    TME_CASE(128, false, false, m) \
    TME_CASE(128, false, true, m)  \
    TME_CASE(128, true, false, m)  \
    TME_CASE(128, true, true, m)
    TME_CASES(false)
    TME_CASES(true)
#undef TME_CASES
#undef TME_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tme
