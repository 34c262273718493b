// bias.cuh -- the attention bias (the SDPA call's attn_mask) applied to a
// row of scores, shared by the forward and backward kernels.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace tme {

// Last kept key in [lo, hi) of a row of boolean keep bytes (row 16-byte
// aligned, lo a multiple of 16), or -1 if none: warp-collective, scanning from
// the top down -- the ragged tail byte by byte, then 16-byte chunks, 2 KB per
// warp per round -- so trailing padding costs one round per 2 KB of it.
__device__ __forceinline__ int last_kept_key(const uint8_t* row, int lo, int hi, int lane) {
    const int hi16 = hi & ~15;
    int found = -1;
    for (int k = hi16 + lane; k < hi; k += 32)
        if (row[k] != 0) found = k;
    int last = __reduce_max_sync(0xffffffffu, found);
    for (int top = hi16; last < 0 && top > lo; top -= 2048) {
        found = -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c0 = top - 16 * (1 + lane + 32 * u);
            if (c0 >= lo) {
                const uint4 w = *reinterpret_cast<const uint4*>(row + c0);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 3; q >= 0; --q)
                    if (ws[q] != 0u && found < 0) found = c0 + 4 * q + 3 - (__clz(ws[q]) >> 3);
            }
        }
        last = __reduce_max_sync(0xffffffffu, found);
    }
    return last;
}

// Attention bias (SDPA attn_mask) of one 32-key chunk of a row, applied in
// the log2 domain: t = s * sl2 + b * log2(e) for an additive bias (16-bit,
// the input dtype), t = s * sl2 or -inf for a boolean keep-mask (bytes).
struct BiasChunk {
    uint4 w[4];
};

__device__ __forceinline__ void bias_load(BiasChunk& b, const uint8_t* row, int kind, int key,
                                          bool full) {
    if (!full) return;
    if (kind == 2) {
        const uint4* src = reinterpret_cast<const uint4*>(row + 2 * static_cast<int64_t>(key));
        b.w[0] = src[0];
        b.w[1] = src[1];
        b.w[2] = src[2];
        b.w[3] = src[3];
    } else {
        const uint4* src = reinterpret_cast<const uint4*>(row + key);
        b.w[0] = src[0];
        b.w[1] = src[1];
    }
}

template <bool BF16>
__device__ __forceinline__ float half_to_float(uint32_t h) {
    if constexpr (BF16) return __uint_as_float(h << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// `full`: the 32 keys are in range and the row is real, and b holds them.
// Otherwise keys are read one by one (keys >= Nk and unreal rows: no bias).
template <bool BF16>
__device__ __forceinline__ void bias_apply(uint32_t (&s)[32], const BiasChunk& b,
                                           const uint8_t* row, int kind, int key, int Nk,
                                           float sl2, bool full, bool row_ok) {
    constexpr float kLog2e = 1.4426950408889634f;
    if (full) {
        if (kind == 2) {
            const uint64_t sl22 = f2(sl2, sl2), l2e2 = f2(kLog2e, kLog2e);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint4 q4 = b.w[i >> 2];
                const uint32_t w = (i & 3) == 0 ? q4.x : (i & 3) == 1 ? q4.y : (i & 3) == 2 ? q4.z : q4.w;
                const uint64_t bb = fmul2(f2(half_to_float<BF16>(w & 0xffffu), half_to_float<BF16>(w >> 16)),
                                          l2e2);
                const uint64_t t = ffma2(f2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                         sl22, bb);
                s[2 * i] = __float_as_uint(f2lo(t));
                s[2 * i + 1] = __float_as_uint(f2hi(t));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint4 q4 = b.w[i >> 4];
                const int wi = (i >> 2) & 3;
                const uint32_t w = wi == 0 ? q4.x : wi == 1 ? q4.y : wi == 2 ? q4.z : q4.w;
                const bool keep = ((w >> (8 * (i & 3))) & 0xffu) != 0u;
                s[i] = __float_as_uint(keep ? __uint_as_float(s[i]) * sl2 : -INFINITY);
            }
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float t = __uint_as_float(s[i]) * sl2;
        if (row_ok && key + i < Nk) {
            if (kind == 2) {
                const uint16_t h = reinterpret_cast<const uint16_t*>(row)[key + i];
                t += half_to_float<BF16>(h) * kLog2e;
            } else if (row[key + i] == 0) {
                t = -INFINITY;
            }
        }
        s[i] = __float_as_uint(t);
    }
}

// Shared-memory staging of the bias of one key tile (KEYS = 128 keys, or the
// 64 keys of one half of a 128-key tile) for the 32 rows of a warp, one row
// per lane.  Row r occupies KEYS * 2 bytes at buf + r * KEYS * 2 (room for a
// 16-bit additive bias; a boolean one uses the first half), its 16-byte chunk
// q stored at chunk position q ^ (r & 7): the eight lanes of one quarter-warp
// read the same chunk of eight consecutive rows from eight different bank
// groups.
//
// bias_prefetch (warp-collective) issues the copies of the keys [key0, key0 +
// KEYS) with cp.async, whole rows per instruction (a row's chunks on
// consecutive lanes), so each instruction touches whole 64- or 128-byte
// spans.  row_ptr is the lane's own bias row; rows r >= nvalid (1 <= nvalid
// <= 32) copy row nvalid - 1, so every staged value is a real bias value.
// The keys must lie inside [0, Nk).  Wait with cp_async_wait_all and then
// __syncwarp before reading.
template <int KEYS>
__device__ __forceinline__ void bias_prefetch(uint32_t buf, const uint8_t* row_ptr, int kind,
                                              int key0, int nvalid, int lane) {
    const unsigned long long mine = reinterpret_cast<uintptr_t>(row_ptr);
    const int esz = kind == 2 ? 2 : 1;
    const int cshift = kind == 2 ? (KEYS == 128 ? 4 : 3) : (KEYS == 128 ? 3 : 2);  // log2 chunks per row
    const int q = lane & ((1 << cshift) - 1);
    const int n_ins = 1 << cshift;   // instructions: 32 rows / (32 >> cshift) rows each
#pragma unroll 2
    for (int i = 0; i < n_ins; ++i) {
        const int r = (i << (5 - cshift)) + (lane >> cshift);
        const unsigned long long base = __shfl_sync(0xffffffffu, mine, min(r, nvalid - 1));
        const uint8_t* src = reinterpret_cast<const uint8_t*>(base) +
                             static_cast<int64_t>(key0) * esz + 16 * q;
        cp_async16(buf + r * (2 * KEYS) + ((q ^ (r & 7)) << 4), src);
    }
    cp_async_commit();
}

// Adds this lane's staged bias row to its 128 scores in registers: the
// scores become log2-domain logits t = s * sl2 + b * log2(e) (additive) or
// t = s * sl2 / -inf (boolean), the same arithmetic as bias_apply.
template <bool BF16>
__device__ __forceinline__ void bias_fold_smem(uint32_t (&s)[4][32], uint32_t buf, int kind,
                                               float sl2, int lane) {
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t rbase = buf + lane * 256;
    const int sw = lane & 7;
    if (kind == 2) {
        const uint64_t sl22 = f2(sl2, sl2), l2e2 = f2(kLog2e, kLog2e);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(rbase + ((q ^ sw) << 4)));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 8 * q + 2 * e;  // keys k, k + 1 of the tile
                uint32_t& a = s[k >> 5][k & 31];
                uint32_t& b = s[k >> 5][(k & 31) + 1];
                const uint64_t bb = fmul2(
                    f2(half_to_float<BF16>(w[e] & 0xffffu), half_to_float<BF16>(w[e] >> 16)), l2e2);
                const uint64_t t = ffma2(f2(__uint_as_float(a), __uint_as_float(b)), sl22, bb);
                a = __float_as_uint(f2lo(t));
                b = __float_as_uint(f2hi(t));
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(rbase + ((q ^ sw) << 4)));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = 16 * q + i;
                const bool keep = ((w[i >> 2] >> (8 * (i & 3))) & 0xffu) != 0u;
                s[k >> 5][k & 31] =
                    __float_as_uint(keep ? __uint_as_float(s[k >> 5][k & 31]) * sl2 : -INFINITY);
            }
        }
    }
}

// Split layout (each row's 128-key tile in two halves of 64 keys, one per
// warp): the half's 64 scores become natural-log-domain logits u = s * scale
// + b (additive; the softmax then takes 2^(u * log2 e - m)) or stay raw
// scores / -inf (boolean; the softmax keeps its scale * log2 e).
// bias_fold_smem64 reads the staged half-row (bias_prefetch<64>),
// bias_fold_direct64 reads the bias row directly key by key (keys >= Nk and
// unreal rows: no bias).  Both compute the same fused multiply-add.
template <bool BF16>
__device__ __forceinline__ void bias_fold_smem64(uint32_t (&s)[2][32], uint32_t buf, int kind,
                                                 float scale, int lane) {
    const uint32_t rbase = buf + lane * 128;
    const int sw = lane & 7;
    if (kind == 2) {
        const uint64_t sc2 = f2(scale, scale);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(rbase + ((q ^ sw) << 4)));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 8 * q + 2 * e;
                uint32_t& a = s[k >> 5][k & 31];
                uint32_t& b = s[k >> 5][(k & 31) + 1];
                const uint64_t t =
                    ffma2(f2(__uint_as_float(a), __uint_as_float(b)), sc2,
                          f2(half_to_float<BF16>(w[e] & 0xffffu), half_to_float<BF16>(w[e] >> 16)));
                a = __float_as_uint(f2lo(t));
                b = __float_as_uint(f2hi(t));
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(rbase + ((q ^ sw) << 4)));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = 16 * q + i;
                if (((w[i >> 2] >> (8 * (i & 3))) & 0xffu) == 0u)
                    s[k >> 5][k & 31] = __float_as_uint(-INFINITY);
            }
        }
    }
}

template <bool BF16>
__device__ __forceinline__ void bias_fold_direct64(uint32_t (&s)[2][32], const uint8_t* row,
                                                   int kind, int key0, int Nk, float scale,
                                                   bool row_ok) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int key = key0 + 32 * c + i;
            const bool in = row_ok && key < Nk;
            if (kind == 2) {
                const float b =
                    in ? half_to_float<BF16>(reinterpret_cast<const uint16_t*>(row)[key]) : 0.0f;
                s[c][i] = __float_as_uint(fmaf(__uint_as_float(s[c][i]), scale, b));
            } else if (in && row[key] == 0) {
                s[c][i] = __float_as_uint(-INFINITY);
            }
        }
}

}  // namespace tme
