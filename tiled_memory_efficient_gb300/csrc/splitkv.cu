// splitkv.cu -- merge step of the split-key forward.
//
// For short query blocks against long key sequences (LLM decode against a KV
// cache: the forum post's table "PyTorch LLM Inference -- Qwen 2.5 0.5B (GQA,
// FP16)" runs exactly that model family), one CTA per (KV group, pair of Q
// tiles) leaves most SMs idle.  The forward kernel then cuts the keys into
// ranges, one CTA per range, and every range r leaves a normalised partial
// output O_r and its log-sum-exp L_r.  Softmax over the union of the ranges is
//     L = M + ln(sum_r e^(L_r - M)),   O = sum_r e^(L_r - L) O_r,
// with M = max_r L_r (the same online-softmax identity the tiles use, applied
// once per range).  This file combines the partials: one warp per output row
// of the split units (all rows, or the rows of the last units of a grid whose
// first units ran whole), fp32 throughout, the result rounded once to the
// output dtype.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx.cuh"

namespace tme {
namespace {

constexpr int kMergeWarps = 8;

template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeWarps * 32)
    splitkv_merge_kernel(const FwdParams p) {
    constexpr int V = D / 32;  // columns per lane
    // partial row pr = output row part_row0 + pr
    const int64_t pr = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    const int64_t row = p.part_row0 + pr;
    const int lane = threadIdx.x & 31;
    // Launched as a programmatic dependent of the split kernel: wait here
    // until that grid has finished and its partials are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (pr >= p.part_rows) return;

    // Every lane holds the LSE of ranges lane, lane + 32, ...: the maximum and
    // the weights need no further loads, so all partial-output loads below
    // are independent of each other.
    float ls[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int s = lane + 32 * u;
        ls[u] = s < p.n_splits ? p.lse_part[static_cast<int64_t>(s) * p.part_rows + pr]
                               : -INFINITY;
    }
    float M = ls[0];
#pragma unroll
    for (int u = 1; u < 8; ++u) M = fmaxf(M, ls[u]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float w[8];
    float wsum = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        w[u] = (M == -INFINITY || ls[u] == -INFINITY) ? 0.0f : expf(ls[u] - M);
        wsum += w[u];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);

    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    const float* src = p.o_part + pr * D + lane * V;
    const int64_t step = p.part_rows * D;   // one range further (kMaxSplits = 256 = 8 x 32)
#pragma unroll
    for (int u = 0; u < 8; ++u) {   // ranges 32u .. 32u + 31, weight from lane s - 32u
        if (32 * u >= p.n_splits) break;
        const int cnt = p.n_splits - 32 * u < 32 ? p.n_splits - 32 * u : 32;
#pragma unroll 4
        for (int l = 0; l < cnt; ++l) {
            const float ws = __shfl_sync(0xffffffffu, w[u], l);
            const float* r = src + (32 * u + l) * step;
            if constexpr (V == 4) {
                const float4 o = *reinterpret_cast<const float4*>(r);
                acc[0] += ws * o.x;
                acc[1] += ws * o.y;
                acc[2] += ws * o.z;
                acc[3] += ws * o.w;
            } else {
                const float2 o = *reinterpret_cast<const float2*>(r);
                acc[0] += ws * o.x;
                acc[1] += ws * o.y;
            }
        }
    }
    const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
    uint16_t* out = static_cast<uint16_t*>(p.out) + row * D + lane * V;
    if constexpr (V == 4) {
        const uint2 o = make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv),
                                   pack2<BF16>(acc[2] * inv, acc[3] * inv));
        *reinterpret_cast<uint2*>(out) = o;
    } else {
        *reinterpret_cast<uint32_t*>(out) = pack2<BF16>(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) p.lse[row] = wsum > 0.0f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_splitkv_merge(int D, bool bf16, const FwdParams& p, cudaStream_t stream) {
    const long long blocks = (p.part_rows + kMergeWarps - 1) / kMergeWarps;
    // Programmatic dependent launch: the merge grid is set up while the split
    // kernel drains, and waits for it on the device (griddepcontrol.wait).
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
#define TME_MERGE(d, b) \
    if (D == d && bf16 == b) return cudaLaunchKernelEx(&cfg, splitkv_merge_kernel<d, b>, p);
    TME_MERGE(64, false)
    TME_MERGE(64, true)
    TME_MERGE(128, false)
    TME_MERGE(128, true)
#undef TME_MERGE
    return cudaErrorInvalidValue;
}

}  // namespace tme
