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
// With n_splits > 1 the keys of the split units are cut into n_splits ranges
// of tiles_per_split 128-key tiles, one CTA per (unit, range); each such CTA
// writes its range's normalised partial output and LSE in fp32 to o_part /
// lse_part ([n_splits][part_rows][D] and [n_splits][part_rows]) instead of
// out / lse, and splitkv_merge combines them.
struct FwdParams {
    void* out;               // [B, Hq, Nq, D] fp16/bf16
    float* lse;              // [B, Hq, Nq] fp32, natural log
    float* o_part;           // split mode: partial outputs (fp32)
    float* lse_part;         // split mode: partial LSEs (fp32)
    unsigned int* status;    // device status word
    int64_t rows_per_group;  // G * Nq
    int64_t total_rows;      // n_groups * rows_per_group
    int Nq, Nk;
    int causal_off;          // causal: position i sees keys j <= i + causal_off
    int n_groups;            // B * Hkv
    int n_pairs;             // ceil(rows_per_group / 256): CTAs per group and key range
    int n_splits;            // key ranges (1: no split)
    int tiles_per_split;     // 128-key tiles per range
    // Units [0, n_whole) run whole (every key tile, output to out / lse); the
    // CTAs after them take the n_splits key ranges of units n_whole, n_whole
    // + 1, ...  Their partials hold rows [part_row0, part_row0 + part_rows) of
    // the flattened output (those units' rows, contiguous): partial row
    // grow - part_row0 of range s at index s * part_rows + grow - part_row0.
    int n_whole;
    int64_t part_row0, part_rows;
    float scale_log2;        // scale * log2(e)
    float scale;             // softmax scale (a general additive bias is added after it)
    // Optional attention bias (masked kernels only): element (b, h, i, j) at
    // mask + b*msb + h*msh + i*msq + j elements; kind 1: bytes, nonzero keeps
    // the key; kind 2: additive, 16-bit in the input dtype.
    const void* mask;
    int mask_kind;
    int64_t msb, msh, msq;
    int Hkv, G;              // KV heads, query heads per KV head
    // bf16 with an fp16 copy of V (attn_fwd_ws): one flag byte per (KV group,
    // 128-key tile), 0 when the copy holds that tile.
    const uint8_t* vflags;
    int n_ktiles;            // ceil(Nk / 128)
    // Causal mask with Nq % 256 == 0 and no key ranges (n_splits == 1): the
    // n_half_pos heaviest pair positions of every head run as two CTAs per
    // pair, one per Q tile (n_groups * G * n_half_pos more CTAs); 0: none.
    int n_half_pos;
};

// Launches the forward kernel for one (D, dtype, causal) instantiation.
// p.mask != nullptr selects the masked instantiation; tmV16 (with p.vflags)
// the bf16 instantiation that reads the fp16 copy of V where it exists.
cudaError_t launch_fwd(int D, bool bf16, bool causal, const CUtensorMap& tmQ,
                       const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                       cudaStream_t stream, const CUtensorMap* tmV16 = nullptr);

// Writes the fp16 copy of a bf16 value tensor [groups][Nk][D] and one flag
// byte per (group, 128-key tile) (vconv.cu).
cudaError_t launch_v_to_f16(int D, const void* v, void* v16, uint8_t* flags, int64_t groups,
                            int Nk, cudaStream_t stream);

// Combines the n_splits partial results of a split forward into out / lse.
cudaError_t launch_splitkv_merge(int D, bool bf16, const FwdParams& p, cudaStream_t stream);

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
    // Optional attention bias, as in FwdParams (masked kernels only).
    const void* mask;
    int mask_kind;
    int64_t msb, msh, msq;
    int Hkv, G;
    // dK/dV with the query tiles of a key tile cut into kv_splits ranges of
    // qtiles_per_split tiles (kv_splits > 1: when B * Hkv * n_ktiles CTAs
    // would leave SMs idle): each range's CTA writes fp32 partial sums to
    // dv_part / dk_part ([kv_splits][n_groups * Nk][D]; dK not yet scaled)
    // and a last kernel adds them in range order.
    int kv_splits;
    int qtiles_per_split;
    float* dv_part;
    float* dk_part;
};

// Workspace bytes of the backward without the split of dK/dV (the per-row
// statistics only), and the bytes the partial sums of `splits` ranges add.
size_t bwd_stats_bytes(int B, int Hq, int Hkv, int Nq);
size_t bwd_split_bytes(int B, int Hkv, int Nk, int D, int splits);

// Launches the three backward kernels (statistics, dK/dV, dQ) in order;
// p.mask != nullptr selects the masked instantiations.
cudaError_t launch_bwd(int D, bool bf16, bool causal, const CUtensorMap& tmQ,
                       const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmDO,
                       const BwdParams& p, cudaStream_t stream);

}  // namespace tme
