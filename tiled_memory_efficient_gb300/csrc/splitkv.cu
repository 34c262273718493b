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
// once per range).  This file combines the partials: one warp per output row,
// fp32 throughout, the result rounded once to the output dtype.
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
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.total_rows) return;

    float M = -INFINITY;
    for (int s = lane; s < p.n_splits; s += 32)
        M = fmaxf(M, p.lse_part[static_cast<int64_t>(s) * p.total_rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    float wsum = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < p.n_splits; ++s) {
            const int64_t idx = static_cast<int64_t>(s) * p.total_rows + row;
            const float ls = p.lse_part[idx];
            if (ls == -INFINITY) continue;  // an empty range (same for the whole warp)
            const float w = expf(ls - M);
            const float* src = p.o_part + idx * D + lane * V;
            if constexpr (V == 4) {
                const float4 o = *reinterpret_cast<const float4*>(src);
                acc[0] += w * o.x;
                acc[1] += w * o.y;
                acc[2] += w * o.z;
                acc[3] += w * o.w;
            } else {
                const float2 o = *reinterpret_cast<const float2*>(src);
                acc[0] += w * o.x;
                acc[1] += w * o.y;
            }
            wsum += w;
        }
    }
    const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
    uint16_t* out = static_cast<uint16_t*>(p.out) + row * D + lane * V;
    if constexpr (V == 4) {
        const uint2 w = make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv),
                                   pack2<BF16>(acc[2] * inv, acc[3] * inv));
        *reinterpret_cast<uint2*>(out) = w;
    } else {
        *reinterpret_cast<uint32_t*>(out) = pack2<BF16>(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) p.lse[row] = wsum > 0.0f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_splitkv_merge(int D, bool bf16, const FwdParams& p, cudaStream_t stream) {
    const long long blocks = (p.total_rows + kMergeWarps - 1) / kMergeWarps;
    const dim3 grid(static_cast<unsigned>(blocks)), block(kMergeWarps * 32);
#define TME_MERGE(d, b) \
    if (D == d && bf16 == b) return launch_kernel(splitkv_merge_kernel<d, b>, grid, block, 0, stream, p);
    TME_MERGE(64, false)
    TME_MERGE(64, true)
    TME_MERGE(128, false)
    TME_MERGE(128, true)
#undef TME_MERGE
    return cudaErrorInvalidValue;
}

}  // namespace tme
