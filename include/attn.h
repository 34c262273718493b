/*
 * attn.h -- C ABI of the tiled, memory-efficient attention library (sm_103a).
 *
 * The operation is scaled-dot-product attention computed the way the
 * noflash-attention forum post describes it (ai-navigate-news, section "The
 * DIY approach", list "What worked"): the N x N score matrix is never formed;
 * Q is tiled along queries and K/V along keys with an online softmax (running
 * max and sum); the query heads of a GQA group are flattened onto their shared
 * KV head instead of broadcasting K/V; negligible softmax terms are flushed to
 * zero; a causal mask is optional.  Its "Other areas where this could be
 * useful" section adds the autograd tier used for training (attn_bwd).  The
 * call mirrors the SDPA call the post patches, scaled_dot_product_attention
 * over [batch, heads, seq_len, dim] tensors (the ai-manual.ru page, section
 * "2 PyTorch SDPA", and its chunked snippet's default scale 1/sqrt(dim)).
 *
 * Conventions for every entry point
 *   - Pointers named q, k, v, out, dout, dq, dk, dv, lse, workspace are DEVICE
 *     pointers owned by the caller; the library never allocates, frees or
 *     retains them past the call.  Layouts are dense row-major:
 *         q, out, dout, dq : [B, Hq, Nq, D]      (dtype)
 *         k, v, dk, dv     : [B, Hkv, Nk, D]     (dtype)
 *         lse              : [B, Hq, Nq]         (fp32, natural log)
 *     dtype is ATTN_F16 or ATTN_BF16; accumulation is fp32.
 *   - Query head h uses KV head h / (Hq / Hkv) (contiguous groups).
 *   - causal selects the mask (attn_causal_t): ATTN_CAUSAL_NONE, or
 *     ATTN_CAUSAL_TOP_LEFT (query position i sees keys j <= i; the is_causal
 *     convention of the SDPA call), or, forward only, ATTN_CAUSAL_BOTTOM_RIGHT
 *     (i sees j <= i + Nk - Nq: the Nq queries are the last Nq positions of a
 *     sequence whose first Nk positions are in K/V, as when decoding against
 *     a KV cache; requires Nq <= Nk).  Other values are ATTN_ERR_INVALID.
 *   - scale multiplies q.k; it must be finite and > 0 (1/sqrt(D) is the usual).
 *   - Work is enqueued on `stream` (a cudaStream_t; 0 = legacy default) and the
 *     call returns without synchronising.  The return value reports argument
 *     validation and launch errors only.  A device-side wait that gives up
 *     (after about 2 s) sets a status word that attn_sync_status() reports.
 *   - Requirements: D in {64, 128}; every pointer 16-byte aligned (lse and
 *     workspace: 16 bytes too); Hq % Hkv == 0; all sizes > 0; the current
 *     device is an sm_103 GPU.  Violations return an error without launching.
 */
#ifndef TME_ATTN_H
#define TME_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

typedef enum {
    ATTN_CAUSAL_NONE = 0,
    ATTN_CAUSAL_TOP_LEFT = 1,
    ATTN_CAUSAL_BOTTOM_RIGHT = 2
} attn_causal_t;

typedef enum { ATTN_MASK_BOOL = 1, ATTN_MASK_ADDITIVE = 2 } attn_mask_kind_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,     /* null pointer, non-positive size, Hq % Hkv, bad scale/dtype */
    ATTN_ERR_UNSUPPORTED = 2, /* D not in {64,128}, sizes beyond the kernel's index range, not sm_103 */
    ATTN_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    ATTN_ERR_TIMEOUT = 5,     /* a device wait gave up (reported by attn_sync_status) */
    ATTN_ERR_WORKSPACE = 6,   /* workspace too small */
    ATTN_ERR_MISMATCH = 7     /* a run-time check found two results that must agree differ (ffn.h) */
} attn_status_t;

/*
 * Forward: out = softmax(scale * q k^T [masked]) v per query row, and
 * lse = log(sum_j exp(scale * q.k_j)) over the allowed keys.
 * (Forum post, "The DIY approach": tiled attention with online softmax.)
 * Nq and Nk need not be equal nor multiples of 128.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int Nq, int Nk, int D, float scale, int causal, int dtype, void* stream);

/*
 * Forward with a caller workspace.  The same operation, arguments, layouts and
 * errors as attn_fwd, plus workspace / workspace_bytes.
 *
 * Why: the PV product takes P as 16-bit values, and the tensor core takes P
 * in the format of V.  fp16 P carries 11 significant bits, bf16 P only 8, and
 * where a few keys share a row's weight the bf16 rounding of P moves O by up
 * to about 0.4% of the spread of their value rows (the forum post's
 * "What worked": online softmax, "same math" -- the result should be the
 * softmax attention itself).  So for bf16 inputs the value tiles are used as
 * fp16.  attn_fwd does that conversion inside every CTA that reads a tile;
 * this call does it once, in a first kernel, into the workspace: an fp16 copy
 * of v (same layout) plus one flag byte per (KV head, 128-key tile).  A tile
 * is copied when fp16 represents it well (largest magnitude in [2^-8, 2^16),
 * or only zeros); a CTA whose key tiles are all copied reads the copy, any
 * other reads v and packs P as bf16.  The results agree with attn_fwd's to
 * rounding; this call runs about 20% faster at D = 128.
 *
 * The workspace also lets this call even out the grid (both dtypes).  attn_fwd
 * runs one CTA per SM-sized unit (KV group, pair of 128-row query tiles), so a
 * grid of U units runs as ceil(U / SMs) waves.  When cutting the last wave's
 * units into 2 to 4 key ranges shortens that wave by more than the extra CTAs
 * and the merge cost (no causal mask, >= 8 key tiles; ranges of >= 4), or when
 * the whole grid is under one wave (every unit cut into ranges of >= 16 key
 * tiles), the cut units write fp32 partial results to the workspace and a
 * second kernel merges them (the online-softmax identity of attn_fwd_splitkv).
 * The rows of uncut units are attn_fwd's bit for bit (fp16); merged rows agree
 * with them to rounding.
 *
 * workspace: a 16-byte-aligned device buffer of at least
 * attn_fwd_workspace_size() bytes (ATTN_ERR_WORKSPACE if smaller, checked
 * before anything is launched); its contents on entry do not matter, and the
 * call writes it.  When that size is 0 (fp16 with no cut) it may be NULL.
 */
int attn_fwd_ws(const void* q, const void* k, const void* v, void* out, float* lse,
                void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nk,
                int D, float scale, int causal, int dtype, void* stream);

/*
 * Workspace bytes attn_fwd_ws needs: for bf16, B*Hkv*Nk*D*2 (the fp16 copy of
 * v) plus B*Hkv*ceil(Nk/128) flag bytes; for a grid that is cut (above), S
 * ranges times R rows of D + 1 fp32 values (the cut units' partial outputs and
 * LSEs); each part padded to 256 bytes.  0 for invalid sizes.  The cut depends
 * on the SM count of the current device (queried here; no cut without a
 * device) and is planned for the non-causal case, which covers the causal
 * one.  Host-only.
 */
size_t attn_fwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int D, int dtype);

/*
 * Key ranges attn_fwd_ws cuts its cut units into for this shape and causal
 * mode on a device of num_sms SMs (<= 0: the current device, as attn_fwd_ws
 * does): 1 when the grid is not cut (one forward kernel, plus the value
 * conversion for bf16), > 1 when a merge kernel follows.  0 for invalid
 * sizes.  Host-only.
 */
int attn_fwd_ws_splits(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal, int num_sms);

/*
 * Causal mask, D = 64, fp16, Nq a multiple of 256: how many of the heaviest
 * 256-row pair positions of every head attn_fwd (and attn_fwd_ws, when it
 * does not cut keys into ranges) runs as two CTAs per pair, one per 128-row
 * Q tile, on a device of num_sms SMs (<= 0: the current device; 0 without
 * one).  A pair's work grows with its position under the causal mask, and
 * at short sequences the last pairs of each head outlast the average work
 * per SM; the split changes no result bit.  0 for every other shape, -1 for
 * invalid sizes or causal mode.  Host-only.
 */
int attn_fwd_half_positions(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal, int dtype,
                            int num_sms);

/*
 * Forward with an attention bias: the attn_mask argument of the SDPA call
 * that the forum post patches ("Other areas where this could be useful":
 * every SDPA call, e.g. from HuggingFace Transformers, which pass padding and
 * causal masks this way).  Element (b, h, i, j) of the mask is at
 *     mask + b*mask_stride_b + h*mask_stride_h + i*mask_stride_q + j
 * elements (h = query head; a stride of 0 broadcasts that dimension; keys are
 * contiguous).  ATTN_MASK_BOOL: one byte per element, nonzero keeps key j.
 * ATTN_MASK_ADDITIVE: 16-bit values in `dtype`, added to scale * q.k (natural
 * log units; -inf removes the key).  The causal mask, if any, applies on top.
 * A row whose every key is removed gets out = 0 and lse = -inf.
 * Requirements beyond attn_fwd's: mask 16-byte aligned and every stride times
 * the element size a multiple of 16 bytes (ATTN_ERR_ALIGN otherwise); the
 * mask is read, never written, and must stay valid until the work completes.
 * Speed: at D = 64 a boolean mask that depends on the key alone (stride_q 0,
 * and stride_h 0 unless Hq == Hkv: a padding mask) runs in the unmasked
 * forward's layout and skips key tiles past the last kept key; any other mask
 * stages each key tile's bias in shared memory and folds it into the scores
 * (D = 64 fp16: in the unmasked layout; bf16 D = 64: one thread per query
 * row), at about half the unmasked speed; at D = 128 each row reads its bias
 * directly.
 */
int attn_fwd_masked(const void* q, const void* k, const void* v, void* out, float* lse,
                    const void* mask, int mask_kind, long long mask_stride_b,
                    long long mask_stride_h, long long mask_stride_q, int B, int Hq, int Hkv,
                    int Nq, int Nk, int D, float scale, int causal, int dtype, void* stream);

/*
 * Split-key forward for short query blocks against long key sequences (LLM
 * decode against a KV cache, the workload of the forum post's table "PyTorch
 * LLM Inference -- Qwen 2.5 0.5B (GQA, FP16)").  attn_fwd runs one CTA per KV
 * group and pair of 128-row query tiles, which leaves most of the GPU idle
 * when B * Hkv * ceil(G * Nq / 256) is small.  This call also cuts the keys
 * into num_splits ranges of whole 128-key tiles (fewer if the keys run out:
 * every range gets ceil(tiles / num_splits) tiles), runs one CTA per range,
 * writes each range's normalised partial output and log-sum-exp to the
 * workspace in fp32, and merges them into out / lse with a second kernel:
 *     lse = M + ln sum_r e^(lse_r - M),  out = sum_r e^(lse_r - lse) out_r,
 * M = max_r lse_r.  The result is the attention of attn_fwd up to rounding
 * (out is rounded once, from fp32).
 *
 * num_splits: 1..256.  With one effective range the call is attn_fwd (no
 * workspace is touched and it may be NULL).  Otherwise workspace must be a
 * 16-byte-aligned device buffer of at least
 * attn_fwd_splitkv_workspace_size(..., num_splits) bytes (ATTN_ERR_WORKSPACE
 * if smaller); its contents on entry do not matter.  Other arguments, layouts
 * and errors are those of attn_fwd.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq,
                     int Nk, int D, float scale, int causal, int dtype, int num_splits,
                     void* stream);

/*
 * Workspace bytes attn_fwd_splitkv needs: fp32 partial outputs and LSEs of
 * every range, each array padded to 256 bytes.  0 when one range results, or
 * for invalid sizes / num_splits outside 1..256.  Host-only.
 */
size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                       int num_splits);

/*
 * A range count for attn_fwd_splitkv: 1 when the unsplit grid already has at
 * least one CTA per SM, else enough ranges to fill one wave of num_sms CTAs,
 * keeping at least two key tiles per range.  num_sms <= 0 asks the current
 * device for its SM count.  Returns 1 for invalid sizes.  Host-only apart
 * from that query.
 */
int attn_fwd_num_splits(int B, int Hq, int Hkv, int Nq, int Nk, int D, int num_sms);

/*
 * Bytes of device workspace for attn_bwd at these sizes: the fp32 per-row
 * statistics, 2 * B*Hkv * ceil(G*Nq/128)*128 * 4 bytes (G = Hq/Hkv; padded to
 * 256), plus -- when B*Hkv*ceil(Nk/128) dK/dV CTAs would leave SMs of the
 * current device idle (small batches, GQA) -- fp32 partial sums of dK and dV
 * for the S query ranges the dK/dV work is cut into, 2 * S * B*Hkv*Nk*D * 4
 * bytes (S of the causal plan, which covers the plain one: attn_bwd_splits).  Returns 0 for invalid sizes.  Needs the current device only for its
 * SM count (without one: the statistics alone).
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int D, int dtype);

/*
 * The number S of query ranges attn_bwd cuts the dK/dV work into at these
 * sizes and causal mode on a device of num_sms SMs (<= 0: the current one,
 * as attn_bwd does), given the workspace
 * attn_bwd_workspace_size() recommends: 1 (three kernels: statistics, dQ,
 * dK/dV) or more (a fourth adds the ranges' partial sums).  Without the causal
 * mask, as many ranges as fill one wave of CTAs; with it, enough that the
 * CTAs of the first key tile (which meets every query tile) do no more than
 * the average work per SM.  0 for invalid sizes.  Host-only.
 */
int attn_bwd_splits(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal, int num_sms);

/*
 * Backward of attn_fwd (forum post, "Other areas where this could be useful":
 * the autograd tier for training).  Inputs: q, k, v, the forward's out and
 * lse, and the upstream gradient dout.  Outputs dq [B,Hq,Nq,D], and dk, dv
 * [B,Hkv,Nk,D] summed over the query heads of each group (overwritten, not
 * accumulated).  workspace: caller-owned device memory of at least the
 * statistics part of attn_bwd_workspace_size() (ATTN_ERR_WORKSPACE otherwise);
 * the dK/dV work is cut into as many query ranges as the rest of the given
 * bytes hold partial sums for (at most the count that size was computed
 * with), summed in a fixed order by a last kernel, so the result is
 * deterministic for a given workspace size.  Its contents on entry do not
 * matter.
 * causal: ATTN_CAUSAL_NONE or ATTN_CAUSAL_TOP_LEFT (bottom-right returns
 * ATTN_ERR_UNSUPPORTED).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
             int causal, int dtype, void* stream);

/*
 * Backward of attn_fwd_masked: the same bias (same mask, kind and strides)
 * enters the recomputed scores; rows whose every key was masked (forward LSE
 * -inf) contribute nothing.  Other arguments, layouts and errors are those of
 * attn_bwd and attn_fwd_masked.
 */
int attn_bwd_masked(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv,
                    void* workspace, size_t workspace_bytes, const void* mask, int mask_kind,
                    long long mask_stride_b, long long mask_stride_h, long long mask_stride_q,
                    int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                    int dtype, void* stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory (for example an operator handed its buffers by a framework
 * that owns every device allocation, or code that must not call cudaMalloc /
 * cudaFree because they can synchronise the device).  The pages have no
 * counterpart: this is a packaging convenience of this library.
 *
 * The scratch comes from one fixed 4 MiB array inside the library's device
 * image (present on every GPU that loads the library until the process
 * exits); nothing is allocated per call.  Problems whose per-row statistics
 * (the first part of attn_bwd_workspace_size()) exceed 4 MiB return
 * ATTN_ERR_WORKSPACE without launching; invalid or unsupported sizes return
 * ATTN_ERR_INVALID.  The result equals attn_bwd's with a 4 MiB workspace.  All calls
 * on a device share the array, so calls that may run on the GPU at the same
 * time (e.g. unordered streams) race and must be ordered by the caller.  The
 * array keeps the last call's contents; nothing in it needs to start at zero.
 * The first call on each device looks up the array's address; make that first
 * call before any stream capture.  Other arguments, layouts and errors are
 * those of attn_bwd.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                     int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal, int dtype,
                     void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of the
 * current device: ATTN_ERR_TIMEOUT if any kernel's bounded wait gave up since
 * the last call, ATTN_ERR_CUDA if the synchronisation failed, else ATTN_OK.
 */
int attn_sync_status(void* stream);

/*
 * Self-test of the bounded-wait path: enqueues one tiny kernel that waits on
 * an mbarrier nothing will ever arrive on, for at most `wait_ns` nanoseconds
 * (clamped to [1000, 10^8]), then records a timeout in the status word.  A
 * following attn_sync_status() must return ATTN_ERR_TIMEOUT.  It touches no
 * caller memory.
 */
int attn_selftest_timeout(unsigned long long wait_ns, void* stream);

/* Static, human-readable text for a status code. */
const char* attn_strerror(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TME_ATTN_H */
