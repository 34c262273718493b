// bwd_noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// attn_bwd needs a few bytes of device scratch per query row (the per-row
// statistics the backward kernels read), and takes it from the caller.  Some
// callers have no way to provide it: for example a plugin or operator that is
// handed its input and output buffers by a host framework that owns every
// device allocation itself, or code that must not call cudaMalloc/cudaFree
// because those calls can synchronise the device and must not be mixed into
// another allocator's pool.  This entry point serves them from a fixed scratch
// array that lives in the library's own device image, so the call itself
// allocates nothing.
//
// Costs and rules of that array:
//   * It is kScratchBytes (4 MiB) on every GPU that loads the library, held
//     until the process exits.
//   * Problems whose per-row statistics (the first part of
//     attn_bwd_workspace_size) exceed that are rejected with
//     ATTN_ERR_WORKSPACE before anything is launched; the rest of the array
//     holds as many of attn_bwd's partial dK/dV sums as fit.
//   * All calls on a device share the one array.  Calls that can run on the
//     GPU at the same time (for example on two streams without ordering
//     between them) race on it and produce wrong gradients; order them.
//   * The array keeps whatever the last call left in it.  Nothing needs to
//     start at zero: the backward writes every scratch entry it later reads
//     without masking, before reading it.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code `g_bwd_scratch` only names the symbol; its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
int scratch_address(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                                int causal, int dtype, void* stream) {
    if (attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, dtype) == 0)
        return ATTN_ERR_INVALID;   // sizes attn_bwd would reject
    // The per-row statistics must fit; attn_bwd splits the dK/dV work over
    // more CTAs only as far as the rest of the array holds its partial sums.
    if (tme::bwd_stats_bytes(B, Hq, Hkv, Nq) > kScratchBytes) return ATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != ATTN_OK) return rc;
    return attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, scratch, kScratchBytes, B, Hq, Hkv, Nq,
                    Nk, D, scale, causal, dtype, stream);
}
