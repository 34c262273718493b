// abi.cu -- the extern "C" entry points of include/attn.h: argument
// validation, TMA tensor-map construction, the device status word, and the
// kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "ptx.cuh"

namespace tme {

// One status word per device (a static device variable; nothing is allocated).
__device__ unsigned int g_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 256;  // key ranges of one split forward, at most
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_cc_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Device set-up, once per device with that device current: check the
// architecture and look up the status word's device address.
int device_setup(unsigned int** status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    // The tensor-map encoder is a driver call and needs a current context; a
    // thread whose only runtime call so far was cudaGetDevice (autograd's
    // worker thread, for one) has none.  Make the device's primary context
    // current once per thread and device.
    thread_local int tl_current_dev = -1;
    if (tl_current_dev != dev) {
        if (cudaSetDevice(dev) != cudaSuccess) return ATTN_ERR_CUDA;
        tl_current_dev = dev;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_cc_ok[dev] != 1) return ATTN_ERR_UNSUPPORTED;
    if (!g_status_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return ATTN_ERR_CUDA;
        g_status_ptr[dev] = static_cast<unsigned int*>(ptr);
    }
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return ATTN_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *status = g_status_ptr[dev];
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D map over a [groups][rows][D] 16-bit tensor, boxes of 64 columns x 128
// rows x 1 group, 128-byte swizzle, zero fill outside the tensor.
int make_map(CUtensorMap* map, const void* base, bool bf16, int D, int64_t rows, int64_t groups) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(groups)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(rows) * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                3, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Shape checks shared by forward and backward.
int check_shape(int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale, int dtype) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || D <= 0) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    const int64_t G = Hq / Hkv;
    const int64_t rows = G * static_cast<int64_t>(Nq);
    // TMA coordinates and row indices are 32-bit signed inside the kernels.
    if (rows > (1ll << 31) - 512 || Nk > (1 << 30)) return ATTN_ERR_UNSUPPORTED;
    const int64_t groups = static_cast<int64_t>(B) * Hkv;
    const int64_t pairs = (rows + 255) / 256;
    if (groups * pairs > 0x7fffffffll || groups > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

__global__ void selftest_timeout_kernel(unsigned long long wait_ns, unsigned int* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    // Nothing ever arrives on `bar`: the wait must give up by itself.
    const uint32_t a = smem_u32(&bar);
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(a, 0)) return;  // cannot happen
        if ((it & 63u) == 63u && global_ns() - t0 > wait_ns) {
            atomicOr(status, kStatusTimeout);
            return;
        }
    }
}

}  // namespace

// For the other translation units of the library (ffn.cu).
int device_setup_public(unsigned int** status) { return device_setup(status); }
int make_map_public(CUtensorMap* map, const void* base, bool bf16, int cols, int64_t rows,
                    int64_t groups) {
    return make_map(map, base, bf16, cols, rows, groups);
}

}  // namespace tme

using namespace tme;

namespace tme {
namespace {

int64_t key_tiles(int Nk) { return (static_cast<int64_t>(Nk) + 127) / 128; }

// Ranges actually used for a requested count: every range gets
// ceil(tiles / requested) key tiles, and no range is left empty.
int effective_splits(int Nk, int requested) {
    const int64_t tiles = key_tiles(Nk);
    if (requested <= 1) return 1;
    if (requested > tiles) requested = static_cast<int>(tiles);
    const int64_t per = (tiles + requested - 1) / requested;
    return static_cast<int>((tiles + per - 1) / per);
}

// SM count of the current device (0 without one, leaving no error behind).
int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

// Launch plan of attn_fwd_ws: units [0, n_whole) run whole, the keys of the
// rest are cut into `splits` ranges of `tps` key tiles (FwdParams).
struct FwdPlan {
    int64_t n_whole = 0;
    int splits = 1;
    int tps = 0;
};

// One CTA per SM (shared memory and the 512 TMEM columns), so a grid of U
// equal units runs as ceil(U / SMs) waves.
//  * Several waves (no causal mask, whose units are laid out so that the last
//    ones cover the last output rows; at least 8 key tiles): the last wave's
//    units are cut into S = 2, 3 or 4 key ranges (each of at least 4 key
//    tiles) when that shortens the last wave: its pieces run in ceil(tail * S
//    / SMs) rounds of 1/S of a unit, each round after the first costing ~15 us
//    (CTA set-up, ramp, the extra partials) and the cut ~4 us of merge,
//    against a unit of about 1.1 us (D = 64) or 2.2 us (D = 128) per key tile
//    (measured: N = 8192 of the sweep, a tail of 56, gains 8% in halves; N =
//    16384, a tail of 112, lost 1% in quarters; video-DiT N = 75600 gains 1-2%
//    in quarters).  N = 4096 (104) is not cut.
//  * Under one wave: every unit's keys are cut into as many ranges as fill
//    the SMs, each of at least 16 key tiles (a range costs a CTA's fixed
//    set-up and its share of the merge: two ranges of 4 key tiles made N =
//    1024 (B = 1, H = 16, D = 64) 19% slower).
FwdPlan fwd_plan(int B, int Hq, int Hkv, int Nq, int Nk, int causal, int D, int sms = 0) {
    FwdPlan pl;
    if (sms <= 0) sms = device_sms();
    if (sms <= 0) return pl;
    const int64_t rows = static_cast<int64_t>(Hq / Hkv) * Nq;
    const int64_t units = static_cast<int64_t>(B) * Hkv * ((rows + 255) / 256);
    const int64_t tiles = key_tiles(Nk);
    if (units >= sms) {
        if (causal != ATTN_CAUSAL_NONE || tiles < 8) return pl;
        const int64_t waves = (units + sms - 1) / sms;
        const int64_t tail = units - (waves - 1) * sms;
        if (waves < 2) return pl;
        const double unit_us = static_cast<double>(tiles) * (D == 128 ? 2.2 : 1.1);
        const double fixed = 15.0 / unit_us, merge = 4.0 / unit_us;
        double best = 1.0;
        int best_s = 1;
        for (int S = 2; S <= 4 && tiles >= 4 * S; ++S) {
            const int64_t rounds = (tail * S + sms - 1) / sms;
            const double cost = static_cast<double>(rounds) / S + (rounds - 1) * fixed + merge;
            if (cost < best - 0.02) {
                best = cost;
                best_s = S;
            }
        }
        if (best_s < 2) return pl;
        pl.n_whole = units - tail;
        pl.tps = static_cast<int>((tiles + best_s - 1) / best_s);
        pl.splits = static_cast<int>((tiles + pl.tps - 1) / pl.tps);
        return pl;
    }
    int64_t want = sms / units;
    if (want > tiles / 16) want = tiles / 16;
    if (want > kMaxSplits) want = kMaxSplits;
    if (want < 2) return pl;
    pl.tps = static_cast<int>((tiles + want - 1) / want);
    pl.splits = static_cast<int>((tiles + pl.tps - 1) / pl.tps);
    if (pl.splits < 2) pl = FwdPlan{};
    return pl;
}

// First output row and row count of the split units' partials.
void plan_rows(const FwdPlan& pl, int B, int Hq, int Hkv, int Nq, int64_t* row0,
               int64_t* nrows) {
    const int64_t rows = static_cast<int64_t>(Hq / Hkv) * Nq;
    const int64_t total = rows * B * Hkv;
    const int64_t n_pairs = (rows + 255) / 256;
    const int64_t first = (pl.n_whole / n_pairs) * rows + (pl.n_whole % n_pairs) * 256;
    *row0 = pl.n_whole > 0 ? first : 0;
    *nrows = total - *row0;
}

size_t pad256(size_t b) { return (b + 255) & ~size_t(255); }

// Causal forward, D = 64 fp16, Nq a multiple of 256, no key ranges: how many
// of the heaviest pair positions run as two CTAs per pair, one per Q tile
// (FwdParams::n_half_pos).  Under the causal mask a pair's work grows with
// its position, and the grid runs heaviest first, so at short sequences the
// last pairs of each head outlast the average work per SM.  A one-tile CTA
// runs its key tiles in kHalfTime of the pair's time (half the tensor work,
// and each SM sub-partition runs two softmax warps instead of four); every
// CTA costs kCtaTiles key-tile times more (set-up, first loads, last PV,
// epilogue).  The plan simulates the hardware's in-order assignment of CTAs to
// the first free SM for every count of split positions and keeps the
// shortest, unless it saves under 2% (grids of more than 8 waves of pairs are
// not split: the spread of their pairs no longer matters).  The constants are
// fitted to GQA 14:2 prefill launches on a 152-SM GB300 (N = 1024 .. 16384,
// 0 to all positions split) so that the plan's pick is the measured best at
// every N: 2 / 3 / 1 / 0 / 0 positions, 18.4 -> 16.4 us at N = 1024, 28.7 ->
// 22.5 us at N = 2048 and 49.2 -> 47.1 us at N = 4096; at N >= 8192 every
// split measured slower.
constexpr double kHalfTime = 0.70;
constexpr double kCtaTiles = 2.5;

int plan_half_positions(int64_t heads, int Nq, int Nk, int causal, int sms) {
    const int m = Nq / 256;
    const int64_t off = causal == ATTN_CAUSAL_BOTTOM_RIGHT ? static_cast<int64_t>(Nk) - Nq : 0;
    std::vector<double> t(m);   // key tiles of the later Q tile of the pair at position i from the top
    for (int i = 0; i < m; ++i) {
        int64_t keys = static_cast<int64_t>(m - 1 - i) * 256 + 256 + off;
        if (keys > Nk) keys = Nk;
        t[i] = keys <= 0 ? 0.0 : static_cast<double>((keys + 127) / 128);
    }
    double best = 0.0;
    int best_h = 0;
    for (int h = 0; h <= m; ++h) {
        std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
        for (int s_ = 0; s_ < sms; ++s_) free_at.push(0.0);
        double end = 0.0;
        auto run = [&](double cost) {
            const double t0 = free_at.top();
            free_at.pop();
            free_at.push(t0 + cost);
            if (t0 + cost > end) end = t0 + cost;
        };
        for (int i = 0; i < m; ++i)
            for (int64_t r = 0; r < heads; ++r) {
                if (i < h) {
                    run(kHalfTime * t[i] + kCtaTiles);
                    run(kHalfTime * t[i] + kCtaTiles);
                } else {
                    run(t[i] + kCtaTiles);
                }
            }
        if (h == 0 || end < 0.98 * best) {
            best = end;
            best_h = h;
        }
    }
    return best_h;
}

// The plan above, remembered per shape (the simulation costs up to a few
// hundred microseconds of host time, which a launch must not wait for).
int half_positions(int B, int Hq, int Nq, int Nk, int causal, int D, int dtype, int sms) {
    if (causal == ATTN_CAUSAL_NONE || D != 64 || dtype != ATTN_F16 || Nq % 256 != 0) return 0;
    if (sms <= 0) sms = device_sms();
    if (sms <= 0) return 0;
    const int64_t heads = static_cast<int64_t>(B) * Hq;
    if (heads * (Nq / 256) > 8LL * sms) return 0;
    struct Entry {
        int64_t heads;
        int Nq, Nk, causal, sms, h;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n_cached = 0, next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_cached; ++i) {
            const Entry& e = cache[i];
            if (e.heads == heads && e.Nq == Nq && e.Nk == Nk && e.causal == causal && e.sms == sms)
                return e.h;
        }
    }
    const int h = plan_half_positions(heads, Nq, Nk, causal, sms);
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{heads, Nq, Nk, causal, sms, h};
    next = (next + 1) % 64;
    if (n_cached < 64) ++n_cached;
    return h;
}

// Bytes of the split partials of a plan (0 without a split).
size_t plan_bytes(const FwdPlan& pl, int B, int Hq, int Hkv, int Nq, int D) {
    if (pl.splits < 2) return 0;
    int64_t row0 = 0, nrows = 0;
    plan_rows(pl, B, Hq, Hkv, Nq, &row0, &nrows);
    return pad256(static_cast<size_t>(pl.splits) * nrows * D * sizeof(float)) +
           pad256(static_cast<size_t>(pl.splits) * nrows * sizeof(float));
}

// Checks shared by the mask entry points: kind, strides, alignment of the
// 16-byte vector loads of bias rows.
int check_mask(const void* mask, int kind, long long sb, long long sh, long long sq) {
    if (!mask) return ATTN_ERR_INVALID;
    if (kind != ATTN_MASK_BOOL && kind != ATTN_MASK_ADDITIVE) return ATTN_ERR_INVALID;
    if (sb < 0 || sh < 0 || sq < 0) return ATTN_ERR_INVALID;
    const long long esz = kind == ATTN_MASK_ADDITIVE ? 2 : 1;
    if (!aligned16(mask) || (sb * esz) % 16 || (sh * esz) % 16 || (sq * esz) % 16)
        return ATTN_ERR_ALIGN;
    return ATTN_OK;
}

// Checks shared by the forward entry points; fills everything in FwdParams
// but the split fields.
int fwd_prepare(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal, int dtype,
                CUtensorMap* tmQ, CUtensorMap* tmK, CUtensorMap* tmV, FwdParams* p) {
    if (!q || !k || !v || !out || !lse) return ATTN_ERR_INVALID;
    int rc = check_shape(B, Hq, Hkv, Nq, Nk, D, scale, dtype);
    if (rc != ATTN_OK) return rc;
    if (causal < ATTN_CAUSAL_NONE || causal > ATTN_CAUSAL_BOTTOM_RIGHT) return ATTN_ERR_INVALID;
    if (causal == ATTN_CAUSAL_BOTTOM_RIGHT && Nq > Nk) return ATTN_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return ATTN_ERR_ALIGN;
    unsigned int* status = nullptr;
    rc = device_setup(&status);
    if (rc != ATTN_OK) return rc;

    const bool bf16 = dtype == ATTN_BF16;
    const int64_t G = Hq / Hkv;
    const int64_t rows = G * Nq;
    const int64_t groups = static_cast<int64_t>(B) * Hkv;
    if (make_map(tmQ, q, bf16, D, rows, groups) != ATTN_OK ||
        make_map(tmK, k, bf16, D, Nk, groups) != ATTN_OK ||
        make_map(tmV, v, bf16, D, Nk, groups) != ATTN_OK)
        return ATTN_ERR_CUDA;

    *p = FwdParams{};
    p->out = out;
    p->lse = lse;
    p->status = status;
    p->rows_per_group = rows;
    p->total_rows = rows * groups;
    p->Nq = Nq;
    p->Nk = Nk;
    p->causal_off = causal == ATTN_CAUSAL_BOTTOM_RIGHT ? Nk - Nq : 0;
    p->n_groups = static_cast<int>(groups);
    p->n_pairs = static_cast<int>((rows + 255) / 256);
    p->n_splits = 1;
    p->tiles_per_split = static_cast<int>(key_tiles(Nk));
    p->n_whole = 0;
    p->part_row0 = 0;
    p->part_rows = p->total_rows;
    p->scale_log2 = scale * 1.4426950408889634f;
    p->scale = scale;
    p->mask = nullptr;
    p->Hkv = Hkv;
    p->G = Hq / Hkv;
    return ATTN_OK;
}

}  // namespace
}  // namespace tme

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                        int dtype, void* stream) {
    CUtensorMap tmQ, tmK, tmV;
    FwdParams p;
    const int rc = fwd_prepare(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype,
                               &tmQ, &tmK, &tmV, &p);
    if (rc != ATTN_OK) return rc;
    p.n_half_pos = half_positions(B, Hq, Nq, Nk, causal, D, dtype, 0);
    const cudaError_t e = launch_fwd(D, dtype == ATTN_BF16, causal != ATTN_CAUSAL_NONE, tmQ, tmK,
                                     tmV, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" size_t attn_fwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                          int dtype) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, dtype) != ATTN_OK) return 0;
    size_t bytes = 0;
    if (dtype == ATTN_BF16) {
        const size_t groups = static_cast<size_t>(B) * Hkv;
        bytes = pad256(groups * Nk * D * 2) + pad256(groups * static_cast<size_t>(key_tiles(Nk)));
    }
    // The plan without the causal mask cuts at least as much as with it.
    return bytes + plan_bytes(fwd_plan(B, Hq, Hkv, Nq, Nk, ATTN_CAUSAL_NONE, D), B, Hq, Hkv, Nq, D);
}

extern "C" int attn_fwd_ws(const void* q, const void* k, const void* v, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                           int Nq, int Nk, int D, float scale, int causal, int dtype,
                           void* stream) {
    int rc = check_shape(B, Hq, Hkv, Nq, Nk, D, scale, dtype);
    if (rc != ATTN_OK) return rc;
    const FwdPlan pl = fwd_plan(B, Hq, Hkv, Nq, Nk, causal, D);
    const bool bf16 = dtype == ATTN_BF16;
    // Workspace checks come before any device call.
    const size_t need = attn_fwd_workspace_size(B, Hq, Hkv, Nq, Nk, D, dtype);
    if (need > 0) {
        if (!workspace) return ATTN_ERR_INVALID;
        if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
        if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    }
    CUtensorMap tmQ, tmK, tmV, tmV16;
    FwdParams p;
    rc = fwd_prepare(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, &tmQ, &tmK,
                     &tmV, &p);
    if (rc != ATTN_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t groups = static_cast<int64_t>(B) * Hkv;
    size_t off = 0;
    uint8_t* vflags = nullptr;
    if (bf16) {
        const size_t v_bytes = pad256(static_cast<size_t>(groups) * Nk * D * 2);
        if (make_map(&tmV16, ws, false, D, Nk, groups) != ATTN_OK) return ATTN_ERR_CUDA;
        vflags = ws + v_bytes;
        p.vflags = vflags;
        p.n_ktiles = static_cast<int>(key_tiles(Nk));
        off = v_bytes + pad256(static_cast<size_t>(groups) * key_tiles(Nk));
    }
    if (pl.splits == 1) p.n_half_pos = half_positions(B, Hq, Nq, Nk, causal, D, dtype, 0);
    if (pl.splits > 1) {
        p.n_splits = pl.splits;
        p.tiles_per_split = pl.tps;
        p.n_whole = static_cast<int>(pl.n_whole);
        plan_rows(pl, B, Hq, Hkv, Nq, &p.part_row0, &p.part_rows);
        p.o_part = reinterpret_cast<float*>(ws + off);
        p.lse_part = reinterpret_cast<float*>(
            ws + off + pad256(static_cast<size_t>(pl.splits) * p.part_rows * D * sizeof(float)));
    }
    cudaError_t e = cudaSuccess;
    if (bf16) e = launch_v_to_f16(D, v, ws, vflags, groups, Nk, st);
    if (e == cudaSuccess)
        e = launch_fwd(D, bf16, causal != ATTN_CAUSAL_NONE, tmQ, tmK, tmV, p, st,
                       bf16 ? &tmV16 : nullptr);
    if (e == cudaSuccess && pl.splits > 1) e = launch_splitkv_merge(D, bf16, p, st);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" int attn_fwd_half_positions(int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                       int causal, int dtype, int num_sms) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, dtype) != ATTN_OK) return -1;
    if (causal < ATTN_CAUSAL_NONE || causal > ATTN_CAUSAL_BOTTOM_RIGHT) return -1;
    return half_positions(B, Hq, Nq, Nk, causal, D, dtype, num_sms);
}

extern "C" int attn_fwd_ws_splits(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal,
                                  int num_sms) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, ATTN_F16) != ATTN_OK) return 0;
    return fwd_plan(B, Hq, Hkv, Nq, Nk, causal, D, num_sms).splits;
}

extern "C" int attn_fwd_masked(const void* q, const void* k, const void* v, void* out, float* lse,
                               const void* mask, int mask_kind, long long mask_stride_b,
                               long long mask_stride_h, long long mask_stride_q, int B, int Hq,
                               int Hkv, int Nq, int Nk, int D, float scale, int causal, int dtype,
                               void* stream) {
    int rc = check_mask(mask, mask_kind, mask_stride_b, mask_stride_h, mask_stride_q);
    if (rc != ATTN_OK) return rc;
    CUtensorMap tmQ, tmK, tmV;
    FwdParams p;
    rc = fwd_prepare(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype,
                               &tmQ, &tmK, &tmV, &p);
    if (rc != ATTN_OK) return rc;
    p.mask = mask;
    p.mask_kind = mask_kind;
    p.msb = mask_stride_b;
    p.msh = mask_stride_h;
    p.msq = mask_stride_q;
    const cudaError_t e = launch_fwd(D, dtype == ATTN_BF16, causal != ATTN_CAUSAL_NONE, tmQ, tmK,
                                     tmV, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" int attn_fwd_num_splits(int B, int Hq, int Hkv, int Nq, int Nk, int D, int num_sms) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, ATTN_F16) != ATTN_OK) return 1;
    if (num_sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            num_sms <= 0)
            return 1;
    }
    // One CTA per SM (shared memory and the 512 TMEM columns): fill one wave
    // of CTAs, keeping at least two key tiles per range.
    const int64_t rows = static_cast<int64_t>(Hq / Hkv) * Nq;
    const int64_t units = static_cast<int64_t>(B) * Hkv * ((rows + 255) / 256);
    if (units >= num_sms) return 1;
    int64_t want = num_sms / units;
    const int64_t by_len = key_tiles(Nk) / 2;
    if (want > by_len) want = by_len;
    if (want > kMaxSplits) want = kMaxSplits;
    return effective_splits(Nk, static_cast<int>(want < 1 ? 1 : want));
}

extern "C" size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                                  int num_splits) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, ATTN_F16) != ATTN_OK) return 0;
    if (num_splits < 1 || num_splits > kMaxSplits) return 0;
    const int splits = effective_splits(Nk, num_splits);
    if (splits == 1) return 0;
    const size_t rows = static_cast<size_t>(B) * Hq * Nq;
    const size_t o_bytes = (static_cast<size_t>(splits) * rows * D * sizeof(float) + 255) & ~size_t(255);
    const size_t l_bytes = (static_cast<size_t>(splits) * rows * sizeof(float) + 255) & ~size_t(255);
    return o_bytes + l_bytes;
}

extern "C" int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                                int Nq, int Nk, int D, float scale, int causal, int dtype,
                                int num_splits, void* stream) {
    if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID;
    int rc = check_shape(B, Hq, Hkv, Nq, Nk, D, scale, dtype);
    if (rc != ATTN_OK) return rc;
    const int splits = effective_splits(Nk, num_splits);
    if (splits > 1) {
        // Workspace checks come before any device call.
        if (!workspace) return ATTN_ERR_INVALID;
        if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
        if (workspace_bytes < attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, D, num_splits))
            return ATTN_ERR_WORKSPACE;
    }
    CUtensorMap tmQ, tmK, tmV;
    FwdParams p;
    rc = fwd_prepare(q, k, v, out, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, &tmQ, &tmK,
                     &tmV, &p);
    if (rc != ATTN_OK) return rc;
    const bool bf16 = dtype == ATTN_BF16;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (splits > 1) {
        if (static_cast<long long>(p.n_groups) * p.n_pairs * splits > 0x7fffffffll)
            return ATTN_ERR_UNSUPPORTED;
        const int64_t tiles = key_tiles(Nk);
        p.n_splits = splits;
        p.tiles_per_split = static_cast<int>((tiles + num_splits - 1) / num_splits);
        const size_t o_bytes =
            (static_cast<size_t>(splits) * p.total_rows * D * sizeof(float) + 255) & ~size_t(255);
        p.o_part = static_cast<float*>(workspace);
        p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes);
    }
    cudaError_t e = launch_fwd(D, bf16, causal != ATTN_CAUSAL_NONE, tmQ, tmK, tmV, p, st);
    if (e == cudaSuccess && splits > 1) e = launch_splitkv_merge(D, bf16, p, st);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

namespace tme {

// Two fp32 arrays (LSE * log2(e) and rowsum(dO * O)), each laid out per KV
// group with the group's rows padded to a multiple of 128.
size_t bwd_stats_bytes(int B, int Hq, int Hkv, int Nq) {
    const size_t groups = static_cast<size_t>(B) * Hkv;
    const size_t rows = static_cast<size_t>(Hq / Hkv) * Nq;
    const size_t rows_pad = (rows + 127) / 128 * 128;
    return (2 * groups * rows_pad * sizeof(float) + 255) & ~static_cast<size_t>(255);
}

// Partial dV and dK of `splits` query ranges: two fp32 arrays
// [splits][B * Hkv * Nk][D], each padded to 256 bytes.
size_t bwd_split_bytes(int B, int Hkv, int Nk, int D, int splits) {
    if (splits <= 1) return 0;
    const size_t one = static_cast<size_t>(splits) * B * Hkv * Nk * D * sizeof(float);
    return 2 * ((one + 255) & ~static_cast<size_t>(255));
}

namespace {

// Query ranges for the dK/dV kernel: enough CTAs (B * Hkv * key tiles *
// ranges) to give every SM of the current device one, keeping at least four
// query tiles per range and at most 32 ranges; 1 when the unsplit grid
// already fills the device or the SM count is unknown.  Every range is
// non-empty (the count is recomputed from the tiles per range).
// Query ranges the dK/dV work is cut into when the grid of B * Hkv *
// ceil(Nk/128) key tiles leaves SMs idle.  Without the causal mask every key
// tile meets every query tile: as many ranges as fill one wave.  With it key
// tile kt meets the Tq - kt query tiles of each head at or after it, so the
// CTAs of key tile 0 are the longest: enough ranges that the longest CTA does
// no more than the average work per SM (GQA 14:2, N = 4096: 5 ranges, 277 ->
// 381 TFLOP/s against the one-wave rule).  At least 4 query tiles per range,
// at most 32 ranges.
int bwd_splits(int B, int Hq, int Hkv, int Nq, int Nk, bool causal, int* tiles_per_split,
               int sms = 0) {
    const int64_t groups = static_cast<int64_t>(B) * Hkv;
    const int64_t n_qtiles = (static_cast<int64_t>(Hq / Hkv) * Nq + 127) / 128;
    *tiles_per_split = static_cast<int>(n_qtiles);
    if (sms <= 0) sms = device_sms();
    if (sms <= 0) return 1;
    const int64_t units = groups * key_tiles(Nk);
    if (units >= sms) return 1;
    int64_t want = (sms + units - 1) / units;
    if (causal) {
        const int64_t tq = (static_cast<int64_t>(Nq) + 127) / 128;   // query tiles per head
        int64_t total = 0;                                             // per head and group
        for (int64_t kt = 0; kt < key_tiles(Nk) && kt < tq; ++kt) total += tq - kt;
        if (total > 0) want = (tq * sms + groups * total - 1) / (groups * total);
    }
    if (want > n_qtiles / 4) want = n_qtiles / 4;
    if (want > 32) want = 32;
    if (want <= 1) return 1;
    const int64_t per = (n_qtiles + want - 1) / want;
    *tiles_per_split = static_cast<int>(per);
    return static_cast<int>((n_qtiles + per - 1) / per);
}

}  // namespace
}  // namespace tme

extern "C" int attn_bwd_splits(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal,
                               int num_sms) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, ATTN_F16) != ATTN_OK) return 0;
    int per = 0;
    return bwd_splits(B, Hq, Hkv, Nq, Nk, causal != ATTN_CAUSAL_NONE, &per, num_sms);
}

extern "C" size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                          int dtype) {
    if (check_shape(B, Hq, Hkv, Nq, Nk, D, 1.0f, dtype) != ATTN_OK) return 0;
    int per = 0;
    // the causal plan cuts at least as much as the plain one
    const int splits = bwd_splits(B, Hq, Hkv, Nq, Nk, true, &per);
    return bwd_stats_bytes(B, Hq, Hkv, Nq) + bwd_split_bytes(B, Hkv, Nk, D, splits);
}

namespace tme {
namespace {

int bwd_run(const void* q, const void* k, const void* v, const void* out, const void* dout,
            const float* lse, void* dq, void* dk, void* dv, void* workspace,
            size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
            int causal, int dtype, const void* mask, int mask_kind, long long msb, long long msh,
            long long msq, void* stream) {
    if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !workspace)
        return ATTN_ERR_INVALID;
    int rc = check_shape(B, Hq, Hkv, Nq, Nk, D, scale, dtype);
    if (rc != ATTN_OK) return rc;
    if (causal == ATTN_CAUSAL_BOTTOM_RIGHT) return ATTN_ERR_UNSUPPORTED;
    if (causal != ATTN_CAUSAL_NONE && causal != ATTN_CAUSAL_TOP_LEFT) return ATTN_ERR_INVALID;
    const void* ptrs[] = {q, k, v, out, dout, lse, dq, dk, dv, workspace};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return ATTN_ERR_ALIGN;
    const size_t stats_bytes = bwd_stats_bytes(B, Hq, Hkv, Nq);
    if (workspace_bytes < stats_bytes) return ATTN_ERR_WORKSPACE;
    unsigned int* status = nullptr;
    rc = device_setup(&status);
    if (rc != ATTN_OK) return rc;
    // Query ranges of the dK/dV kernel: as many as the device wants and the
    // workspace holds the partial sums of.
    int per = 0;
    int splits = bwd_splits(B, Hq, Hkv, Nq, Nk, causal != ATTN_CAUSAL_NONE, &per);
    if (splits > 1) {
        // the largest count whose partial sums the rest of the workspace holds
        const size_t room = workspace_bytes - stats_bytes;
        int fit = splits;
        while (fit > 1 && bwd_split_bytes(B, Hkv, Nk, D, fit) > room) --fit;
        if (fit < splits) {
            const int64_t nqt = (static_cast<int64_t>(Hq / Hkv) * Nq + 127) / 128;
            splits = fit;
            if (splits > 1) {
                per = static_cast<int>((nqt + splits - 1) / splits);
                splits = static_cast<int>((nqt + per - 1) / per);
            } else {
                per = static_cast<int>(nqt);
                splits = 1;
            }
        }
    }

    const bool bf16 = dtype == ATTN_BF16;
    const int64_t G = Hq / Hkv;
    const int64_t rows = G * Nq;
    const int64_t groups = static_cast<int64_t>(B) * Hkv;
    const int64_t n_qtiles = (rows + 127) / 128;
    CUtensorMap tmQ, tmK, tmV, tmDO;
    if (make_map(&tmQ, q, bf16, D, rows, groups) != ATTN_OK ||
        make_map(&tmDO, dout, bf16, D, rows, groups) != ATTN_OK ||
        make_map(&tmK, k, bf16, D, Nk, groups) != ATTN_OK ||
        make_map(&tmV, v, bf16, D, Nk, groups) != ATTN_OK)
        return ATTN_ERR_CUDA;
    BwdParams p{};
    p.out = out;
    p.dout = dout;
    p.lse = lse;
    p.nlse2 = static_cast<float*>(workspace);
    p.ndelta = p.nlse2 + groups * n_qtiles * 128;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.status = status;
    p.rows_per_group = rows;
    p.rows_pad = n_qtiles * 128;
    p.total_rows = rows * groups;
    p.Nq = Nq;
    p.Nk = Nk;
    p.n_groups = static_cast<int>(groups);
    p.n_qtiles = static_cast<int>(n_qtiles);
    p.n_ktiles = (Nk + 127) / 128;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.mask = mask;
    p.mask_kind = mask_kind;
    p.msb = msb;
    p.msh = msh;
    p.msq = msq;
    p.Hkv = Hkv;
    p.G = static_cast<int>(G);
    p.kv_splits = splits;
    p.qtiles_per_split = per;
    if (splits > 1) {
        const size_t one = bwd_split_bytes(B, Hkv, Nk, D, splits) / 2;
        p.dv_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + stats_bytes);
        p.dk_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + stats_bytes + one);
    }
    if (groups * p.n_ktiles * splits > 0x7fffffffll || groups * n_qtiles > 0x7fffffffll)
        return ATTN_ERR_UNSUPPORTED;
    const cudaError_t e = launch_bwd(D, bf16, causal != 0, tmQ, tmK, tmV, tmDO, p,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace tme

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq,
                        int Nk, int D, float scale, int causal, int dtype, void* stream) {
    return bwd_run(q, k, v, out, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nq,
                   Nk, D, scale, causal, dtype, nullptr, 0, 0, 0, 0, stream);
}

extern "C" int attn_bwd_masked(const void* q, const void* k, const void* v, const void* out,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               void* workspace, size_t workspace_bytes, const void* mask,
                               int mask_kind, long long mask_stride_b, long long mask_stride_h,
                               long long mask_stride_q, int B, int Hq, int Hkv, int Nq, int Nk,
                               int D, float scale, int causal, int dtype, void* stream) {
    const int rc = check_mask(mask, mask_kind, mask_stride_b, mask_stride_h, mask_stride_q);
    if (rc != ATTN_OK) return rc;
    return bwd_run(q, k, v, out, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nq,
                   Nk, D, scale, causal, dtype, mask, mask_kind, mask_stride_b, mask_stride_h,
                   mask_stride_q, stream);
}

extern "C" int attn_sync_status(void* stream) {
    unsigned int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != ATTN_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return (word & kStatusTimeout) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

extern "C" int attn_selftest_timeout(unsigned long long wait_ns, void* stream) {
    unsigned int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != ATTN_OK) return rc;
    if (wait_ns < 1000ull) wait_ns = 1000ull;
    if (wait_ns > 100000000ull) wait_ns = 100000000ull;
    return launch_kernel(selftest_timeout_kernel, dim3(1), dim3(32), 0,
                         static_cast<cudaStream_t>(stream), wait_ns, status) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

extern "C" const char* attn_strerror(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
        case ATTN_ERR_CUDA: return "CUDA runtime or driver error";
        case ATTN_ERR_TIMEOUT: return "a device-side wait timed out";
        case ATTN_ERR_WORKSPACE: return "workspace too small";
        case ATTN_ERR_MISMATCH: return "results that must agree differ";
        default: return "unknown status";
    }
}

extern "C" int attn_version(void) { return 100; }
