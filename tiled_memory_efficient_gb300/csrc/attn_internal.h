// attn_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tme {

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

}  // namespace tme
