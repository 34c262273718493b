// attn_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tme {

// Launches `kern` and returns the status of this launch itself (unlike
// cudaGetLastError, which would also report an unrelated earlier error left
// in the calling thread).
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, Args... args) {
    void* ptrs[] = {static_cast<void*>(&args)...};
    return cudaLaunchKernel(reinterpret_cast<const void*>(kern), grid, block, ptrs, smem, stream);
}

// Forward launch parameters (everything the kernel needs besides the three
// tensor maps).  Row indices are "flattened": within KV group g of batch b the
// G query heads that share that KV head form G*Nq consecutive rows, head-major.
struct FwdParams {
    void* out;               // [B, Hq, Nq, D] fp16/bf16
    float* lse;              // [B, Hq, Nq] fp32, natural log
    unsigned int* status;    // device status word
    int64_t rows_per_group;  // G * Nq
    int Nq, Nk;
    int n_groups;            // B * Hkv
    int n_pairs;             // ceil(rows_per_group / 256): CTAs per group
    float scale_log2;        // scale * log2(e)
};

// Launches the forward kernel for one (D, dtype, causal) instantiation.
cudaError_t launch_fwd(int D, bool bf16, bool causal, const CUtensorMap& tmQ,
                       const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                       cudaStream_t stream);

// Backward launch parameters.  The workspace holds two fp32 arrays laid out
// per KV group with rows_pad = n_qtiles * 128 rows each (so every 128-row
// tile of per-row statistics is one aligned 512-byte block), stored negated
// so each enters its use as a single fused add: nlse2 = -LSE * log2(e) and
// ndelta = -rowsum(dO * O).
struct BwdParams {
    const void* out;         // forward output O, [B, Hq, Nq, D]
    const void* dout;        // upstream gradient dO, [B, Hq, Nq, D]
    const float* lse;        // forward LSE, [B, Hq, Nq]
    float* nlse2;            // workspace [n_groups][rows_pad]
    float* ndelta;           // workspace [n_groups][rows_pad]
    void* dq;                // [B, Hq, Nq, D]
    void* dk;                // [B, Hkv, Nk, D]
    void* dv;                // [B, Hkv, Nk, D]
    unsigned int* status;
    int64_t rows_per_group;  // G * Nq
    int64_t rows_pad;        // n_qtiles * 128
    int64_t total_rows;      // B * Hq * Nq
    int Nq, Nk;
    int n_groups;            // B * Hkv
    int n_qtiles;            // ceil(rows_per_group / 128)
    int n_ktiles;            // ceil(Nk / 128)
    float scale;
    float scale_log2;
};

// Launches the three backward kernels (statistics, dK/dV, dQ) in order.
cudaError_t launch_bwd(int D, bool bf16, bool causal, const CUtensorMap& tmQ,
                       const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                       const BwdParams& p, cudaStream_t stream);

}  // namespace tme
