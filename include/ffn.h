/*
 * ffn.h -- C ABI of the token-chunked feed-forward block (sm_103a).
 *
 * The noflash-attention forum post (ai-navigate-news, section "The DIY
 * approach", list "What worked") lists FFN chunking with a runtime safety
 * check as a further memory saving next to the tiled attention.  The
 * feed-forward block of a transformer acts on each token on its own:
 *     h = act(x W1^T + b1),   y = h W2^T + b2
 * so it can run a chunk of tokens at a time, holding only [chunk, d_ff] of the
 * intermediate h (in `workspace`, in the 16-bit dtype) instead of [T, d_ff].
 *
 * Conventions (as in attn.h): device pointers owned by the caller, dense
 * row-major, 16-bit dtype ATTN_F16 / ATTN_BF16 with fp32 accumulation; work
 * enqueued on `stream` (0 = legacy default stream); no allocation.
 *   x, y : [T, d_model]         W1 : [n1, d_model]   (PyTorch Linear layout)
 *   W2   : [d_model, d_ff]      b1 : [n1] or NULL    b2 : [d_model] or NULL
 * with n1 = d_ff, or 2*d_ff for FFN_ACT_SWIGLU (rows [0, d_ff) the gate
 * projection, rows [d_ff, 2*d_ff) the up projection; h = silu(gate) * up).
 * Requirements: d_model and d_ff multiples of 8; x, W1, W2, y, workspace
 * 16-byte aligned; chunk >= 1 (chunk >= T runs unchunked).
 * Errors: ATTN_ERR_INVALID (null pointer, size <= 0, unknown act / dtype),
 * ATTN_ERR_UNSUPPORTED (d_model or d_ff not a multiple of 8), ATTN_ERR_ALIGN,
 * ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA.
 */
#ifndef TME_FFN_H
#define TME_FFN_H

#include <stddef.h>

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FFN_ACT_NONE = 0,
    FFN_ACT_RELU = 1,
    FFN_ACT_GELU_TANH = 2, /* 0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3))) */
    FFN_ACT_SILU = 3,      /* a / (1 + e^-a) */
    FFN_ACT_SWIGLU = 4     /* silu(gate) * up, W1 = [Wg; Wu] */
} ffn_act_t;

/* Workspace bytes ffn_forward needs: min(chunk, T) * d_ff 16-bit values,
 * rounded up to 256.  0 for invalid sizes.  Host-only. */
size_t ffn_workspace_size(int T, int d_ff, int chunk);

/* y = FFN(x), min(chunk, T) tokens at a time. */
int ffn_forward(const void* x, const void* w1, const void* b1, const void* w2, const void* b2,
                void* y, int T, int d_model, int d_ff, int act, int chunk, void* workspace,
                size_t workspace_bytes, int dtype, void* stream);

/*
 * The runtime safety check of chunking: runs ffn_forward with `chunk` into y
 * and unchunked (one chunk of T tokens) into y_ref, compares the two bit for
 * bit on the device, synchronises `stream` and returns ATTN_OK when they are
 * identical, ATTN_ERR_MISMATCH when not.  workspace must hold the unchunked
 * intermediate: ffn_workspace_size(T, d_ff, T) bytes, so callers run it on a
 * probe batch of T tokens.
 */
int ffn_check_chunking(const void* x, const void* w1, const void* b1, const void* w2,
                       const void* b2, void* y, void* y_ref, int T, int d_model, int d_ff,
                       int act, int chunk, void* workspace, size_t workspace_bytes, int dtype,
                       void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TME_FFN_H */
