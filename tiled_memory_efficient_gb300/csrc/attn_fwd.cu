// attn_fwd.cu -- tiled scaled-dot-product attention forward for sm_103a.
//
// The method (noflash-attention forum post, ai-navigate-news, section "The DIY
// approach" and its "What worked" list): never form the N x N score matrix;
// tile Q along queries and K/V along keys, keep an online-softmax running max
// and sum per query row, flatten the query heads of a GQA group onto their
// shared KV head instead of broadcasting K/V, flush negligible softmax terms
// to zero, and optionally apply a causal mask.
//
// GB300 design (one CTA = 256 flattened query rows of one KV group, two
// 128-row Q tiles ping-ponging on the tensor core; warp numbers in FwdCfg):
//   producer    one thread: Q tiles once, then K_j / V_j tiles through two
//               mbarrier-guarded shared-memory rings (TMA, 128-byte swizzle).
//   MMA issuer  one elected lane: S_t = Q_t K_j^T with tcgen05.mma (both
//               operands in shared memory, fp32 accumulator in TMEM), then
//               O_t += P_t V_j with P_t read from TMEM.
//   softmax     one thread per query row at D = 128 and with a mask, one
//               per (row, 64-key half) otherwise: tcgen05.ld of the S row, masked
//               row max, lazy rescale of the running state, exp2 with a
//               flush-to-zero threshold, P packed to fp16/bf16 into TMEM; at
//               the end the epilogue divides O by the row sum and stores O
//               and the natural-log LSE.
// TMEM (512 columns): S_0 [0,128) S_1 [128,256) O_0 [256,256+D)
// O_1 [256+D,256+2D).  D = 128: P_t overwrites the first 64 columns of S_t
// (two 16-bit values per column).  D = 64: P_t has its own 64 columns at
// [384+64t, 448+64t), so S of the next key tile can be computed while the
// softmax still works on this one.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_internal.h"
#include "bias.cuh"
#include "ptx.cuh"

namespace tme {
namespace {

constexpr int kRows = 128;          // rows of a Q tile, keys of a K/V tile
constexpr float kLn2 = 0.6931471805599453f;
// Lazy rescale: the running max used for exponentiation is only moved when
// the true max exceeds it by more than this many powers of two.
constexpr float kRescaleThreshold = 8.0f;

// MK: 0 no mask; 1 a general attention bias (boolean or additive, any
// broadcast); 2 a boolean keep-mask that depends on the key alone (a padding
// mask, [B,1,1,Nk] or per head when G = 1), applied in the split layout.
// BF16: bf16 inputs, whose value tiles the PV product takes as fp16: converted
// in shared memory by converter warps, or (VPRE) read from an fp16 copy that
// the caller's workspace holds.
template <int D, int MK = 0, bool BF16 = false, bool VPRE = false>
struct FwdCfg {
    static constexpr int kTileBytes = kRows * D * 2;         // one 128 x D tile, 16-bit
    // D = 128: shared memory is full.  A general mask at D = 64 (fp16) gives
    // one K stage to its staged bias.
    static constexpr int kKStages = (D == 128) ? 2 : (MK == 1 && !BF16) ? 3 : 4;
    static constexpr int kVStages = (D == 128) ? 3 : 4;   // D = 128: 225.5 KB in all
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    static constexpr int kOCol = 256;                        // first O column in TMEM
    // With D=64 TMEM has room for P next to S and O, so S of the next key tile
    // can be computed while the softmax still works on this one.  With D=128
    // the four accumulators fill all 512 columns and P overwrites S.
    static constexpr bool kSepP = (D == 64);
    static constexpr int kPCol = 256 + 2 * D;                // P_t at kPCol + 64 t (kSepP)
    // Warp roles.  A softmax warp w reads TMEM lane quadrant w%4 and runs on
    // SM sub-partition w%4.
    //  D=128: warps 0-7 softmax, one thread per 128-key row; warp 8 only waits
    //         at the teardown, so the light roles land on sub-partitions 1-3:
    //         warps 9/10 issue the tensor-core work of Q tiles 0/1, warp 11 is
    //         the TMA producer.
    //  D=64:  the softmax is the bottleneck, so every row is split over two
    //         warps of 64 keys each: warps 0-15 softmax (Q tile (w/4)%2, key
    //         half w/8), warp 16 producer, warps 17/18 MMA issuers.
    // (Masks at D = 64 run split too: a key-only mask, MK = 2, with 16 keep
    // bytes per lane; a general bias, MK = 1, staged in shared memory.  bf16
    // inputs keep one thread per row: their value-tile converters take the
    // warps that layout leaves idle.)
    static constexpr bool kSplit = (D == 64 && !BF16);
    static constexpr int kSoftmaxWarps = kSplit ? 16 : 8;
    static constexpr int kProducerWarp = kSplit ? 16 : 11;
    static constexpr int kMmaWarp0 = kSplit ? 17 : 9;
    static constexpr int kThreads = kSplit ? 19 * 32 : 12 * 32;
    static constexpr int kTileThreads = kSplit ? 256 : 128;  // softmax threads per Q tile
    // bf16 inputs: warps that rewrite each value tile as fp16 in shared memory
    // so that P can be packed as fp16 (11 significant bits instead of 8):
    // warp 8 and, at D = 128 (one MMA issuer), warp 10.
    static constexpr int kConvWarps = (BF16 && !kSplit && !VPRE) ? (kSepP ? 1 : 2) : 0;
    static constexpr int kConvWarp0 = 8, kConvWarp1 = 10;
    // Split rows exchange partial maxima (double-buffered by key-tile parity)
    // and, at the end, partial sums: xm[2][2 tiles][128 rows][2 halves],
    // xl[2 tiles][128][2], xr[2 tiles][128][2] (floats).
    static constexpr int kXOff = kBarOff + 512;
    static constexpr int kXBytes = kSplit ? (4096 + 2048 + 2048) : 0;
    // A general mask at D = 64 stages the bias of the next key tile in shared
    // memory while the softmax works on this one: 32 rows x 256 bytes for
    // each of 8 warps (one thread per row), or 32 rows x 128 bytes (half a
    // row) for each of 16 (split); 16-bit additive, a boolean one uses half.
    // At D = 128 shared memory has no room for it and each row reads its
    // bias directly.
    static constexpr bool kBiasSmem = (MK == 1 && D == 64);
    static constexpr int kBOff = kXOff + kXBytes;
    static constexpr int kBiasBytes = kBiasSmem ? 8 * 32 * 256 : 0;
    static constexpr int kSmemBytes = kBarOff + 512 + kXBytes + kBiasBytes + 1024;
};

// Flush-to-zero threshold in the log2 domain: a softmax term p = 2^x with
// x = s*c - m is dropped when x < -T.  bf16 P: T = 126, which is exactly the
// flush of ex2.approx.ftz (results below 2^-126 are zero).  fp16 P: T = 24;
// the round-to-nearest conversion of P to fp16 is that flush (every p below
// 2^-25 becomes +0, the smallest fp16 subnormal is 2^-24), so no extra
// instruction is spent on it; the fp32 row sum still adds those terms, which
// changes it by less than Nk * 2^-25 (relative, since the sum is >= 1).
// The terms are computed two at a time by softmax_pair (ptx.cuh).

// Row maximum of 128 values with three-input max: a 5-level tree (65 ops),
// fully independent at the first level.
__device__ __forceinline__ float row_max128(const uint32_t (&s)[4][32]) {
    float t[43];
#pragma unroll
    for (int i = 0; i < 42; ++i) {
        const int a = 3 * i, b = 3 * i + 1, c = 3 * i + 2;
        t[i] = fmax3(__uint_as_float(s[a >> 5][a & 31]), __uint_as_float(s[b >> 5][b & 31]),
                     __uint_as_float(s[c >> 5][c & 31]));
    }
    t[42] = fmaxf(__uint_as_float(s[3][30]), __uint_as_float(s[3][31]));
    float u[15];
#pragma unroll
    for (int i = 0; i < 14; ++i) u[i] = fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[14] = t[42];
    float w[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = fmax3(u[3 * i], u[3 * i + 1], u[3 * i + 2]);
    return fmaxf(fmax3(w[0], w[1], w[2]), fmaxf(w[3], w[4]));
}

// Number of 128-key tiles a Q tile starting at flattened row `row0` needs.
__device__ __forceinline__ int kv_tiles_for(int64_t row0, const FwdParams& p, bool causal) {
    if (row0 >= p.rows_per_group) return 0;
    if (!causal) return (p.Nk + kRows - 1) / kRows;
    const int64_t last = min(row0 + kRows - 1, p.rows_per_group - 1);
    const int64_t max_pos = (row0 / p.Nq == last / p.Nq) ? (last % p.Nq) : (p.Nq - 1);
    // keys [0, max_pos + causal_off] are visible to the tile's last row
    int64_t keys = max_pos + p.causal_off + 1;
    if (keys > p.Nk) keys = p.Nk;
    if (keys <= 0) return 0;
    return static_cast<int>((keys + kRows - 1) / kRows);
}

// Key tiles of [kt0, kt0 + tps) below a tile's limit n_full.
__device__ __forceinline__ int tiles_in_range(int n_full, int kt0, int tps) {
    const int end = n_full < kt0 + tps ? n_full : kt0 + tps;
    return end > kt0 ? end - kt0 : 0;
}

// Epilogue stores.  Normal mode: 32 output columns of row `grow` rounded to
// the 16-bit dtype, as two 32-byte stores: each lane writes whole 32-byte
// sectors of its row (rows are D * 2 bytes apart and the 32 columns start at
// a multiple of 64 bytes, so they are 32-byte aligned whenever out is; an out
// that is only 16-byte aligned takes four 16-byte stores).  A key range of
// a split unit (split >= 0): the same values in fp32 to its partial arrays.
template <int D, bool BF16>
__device__ __forceinline__ void store_o32(const FwdParams& p, int split, int64_t grow, int c,
                                          const uint32_t (&o)[32], float inv_l) {
    if (split >= 0) {
        float4* dst = reinterpret_cast<float4*>(
            p.o_part + (static_cast<int64_t>(split) * p.part_rows + grow - p.part_row0) * D +
            c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                 __uint_as_float(o[4 * i + 2]) * inv_l,
                                 __uint_as_float(o[4 * i + 3]) * inv_l);
    } else {
        uint32_t w[2][8];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i >> 3][i & 7] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                                           __uint_as_float(o[2 * i + 1]) * inv_l);
        uint16_t* dst = static_cast<uint16_t*>(p.out) + grow * D + c * 32;
        if ((reinterpret_cast<uintptr_t>(p.out) & 31u) == 0) {
            st_global_v8(dst, w[0]);
            st_global_v8(dst + 16, w[1]);
        } else {   // out only 16-byte aligned: half sectors
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                d4[i] = make_uint4(w[i >> 1][4 * (i & 1)], w[i >> 1][4 * (i & 1) + 1],
                                   w[i >> 1][4 * (i & 1) + 2], w[i >> 1][4 * (i & 1) + 3]);
        }
    }
}

__device__ __forceinline__ void store_lse(const FwdParams& p, int split, int64_t grow, float v) {
    if (split >= 0)
        p.lse_part[static_cast<int64_t>(split) * p.part_rows + grow - p.part_row0] = v;
    else
        p.lse[grow] = v;
}

// Maximum of 64 values (three-input max tree).
__device__ __forceinline__ float row_max64(const uint32_t (&s)[2][32]) {
    float t[22];
#pragma unroll
    for (int i = 0; i < 21; ++i) {
        const int a = 3 * i, b = 3 * i + 1, c = 3 * i + 2;
        t[i] = fmax3(__uint_as_float(s[a >> 5][a & 31]), __uint_as_float(s[b >> 5][b & 31]),
                     __uint_as_float(s[c >> 5][c & 31]));
    }
    t[21] = __uint_as_float(s[1][31]);
    float u[8];
#pragma unroll
    for (int i = 0; i < 7; ++i) u[i] = fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[7] = t[21];
    return fmaxf(fmax3(u[0], u[1], u[2]), fmax3(u[3], u[4], fmax3(u[5], u[6], u[7])));
}

// The 128 softmax terms of one row (one thread per row): p = 2^(s * scale - m)
// pairwise, summed into acc2 (fp32 pairs), rounded to 16 bits (bf16 when
// OUT_BF16, else fp16) and stored to the row's P columns in TMEM, 32 keys
// (16 columns) at a time.
template <bool OUT_BF16>
__device__ __forceinline__ void pack_p128(const uint32_t (&sr)[4][32], uint32_t tP, uint64_t sl22,
                                          uint64_t nm2, uint64_t (&acc2)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2)
            pk[i >> 1] = softmax_pair<OUT_BF16>(sr[c][i], sr[c][i + 1], sl22, nm2, acc2[(i >> 1) & 3]);
        tmem_st16(tP + c * 16, pk);
    }
}

template <int D, bool BF16, bool CAUSAL, int MK, bool VPRE>
__global__ void __launch_bounds__(FwdCfg<D, MK, BF16, VPRE>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmV16, const FwdParams p) {
    using C = FwdCfg<D, MK, BF16, VPRE>;
    constexpr bool MASK = MK == 1;      // general bias
    constexpr bool KEYMASK = MK == 2;   // key-only keep-mask (split layout)
    constexpr int KS = C::kKStages, VS = C::kVStages;
    constexpr int kProducerWarp = C::kProducerWarp;
    constexpr int kMmaWarp0 = C::kMmaWarp0;
    constexpr int KB = D / 64;  // 64-element (128-byte) column blocks per row

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem + C::kQOff;
    uint8_t* sK = smem + C::kKOff;
    uint8_t* sV = smem + C::kVOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* q_full = bars;
    uint64_t* k_full = q_full + 1;       // [KS]
    uint64_t* k_empty = k_full + KS;     // [KS][2]: tile t is done with the K in slot s
    uint64_t* v_full = k_empty + 2 * KS; // [VS]
    uint64_t* v_empty = v_full + VS;     // [VS][2]
    uint64_t* s_full = v_empty + 2 * VS; // [2] S_t ready in TMEM
    uint64_t* p_full = s_full + 2;     // [2] P_t in TMEM and O_t rescaled
    uint64_t* o_full = p_full + 2;     // [2] last PV of tile t done
    uint64_t* s_free = o_full + 2;     // [2] softmax has read S_t (kSepP)
    uint64_t* pv_done = s_free + 2;    // [2] PV of tile t done (kSepP)
    uint64_t* mma_done = pv_done + 2;  // [2] every MMA of tile t done
    uint64_t* v_cvt = mma_done + 2;    // [VS] bf16: the slot's value tile is converted (or kept)
    uint64_t* cv_sync = v_cvt + VS;    // [2] the two converter warps have both read a tile
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cv_sync + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* v_keep16 = abort_flag + 1;  // [VS] 1: the slot's value tile stayed bf16
    volatile int* cv_wide = v_keep16 + VS;    // [2 buffers][2 converter warps] range flags
    volatile int* cta_v16 = cv_wide + 4;      // VPRE: 1 when every value tile of the CTA is fp16
    volatile int* key_lim = cta_v16 + 1;      // key-only masks: key tiles the CTA needs

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work unit (group, pair of Q tiles).  The heaviest units go first so the
    // last wave holds light ones: under the causal mask a pair's work grows
    // with the position of its rows in its head.  When every head is a whole
    // number m of pairs (Nq % 256 == 0) the order runs over the pair
    // position k = m-1 .. 0 and, within one position, over every (group,
    // head), which is heaviest-first across the whole grid.  A general mask
    // without the causal mask walks the pairs position-major (below).
    // Otherwise consecutive CTAs share a KV group (its K/V stay hot in L2):
    // without the causal mask pairs ascending (so the units of the last CTAs
    // cover the last rows of the output, contiguously), with it heaviest pair
    // first within the group.  Units [0, n_whole) run whole; after them the
    // CTAs of one split unit are adjacent and each takes the key tiles [kt0,
    // kt0 + tiles_per_split) (split < 0: the whole unit).
    int unit = static_cast<int>(blockIdx.x), split = -1;
    if (p.n_splits > 1 && unit >= p.n_whole) {
        const int c = unit - p.n_whole;
        unit = p.n_whole + c / p.n_splits;
        split = c % p.n_splits;
    }
    int group, pair;
    int only = -1;   // >= 0: the one Q tile of the pair this CTA runs
    if (CAUSAL && p.Nq % (2 * kRows) == 0) {
        const int m = p.Nq / (2 * kRows);        // pairs per head (n_pairs = G * m)
        const int heads = p.n_groups * p.G;      // (group, head) combinations
        // The n_half_pos heaviest positions run as two CTAs per pair, one per
        // Q tile (the later rows, which see one more key tile, first); the
        // other positions follow, one CTA per pair.
        const int n_half = 2 * heads * p.n_half_pos;
        int pos, r;                              // position from the top, (group, head)
        if (unit < n_half) {
            pos = unit / (2 * heads);
            r = (unit % (2 * heads)) >> 1;
            only = 1 - (unit & 1);
        } else {
            const int u = unit - n_half + heads * p.n_half_pos;
            pos = u / heads;
            r = u % heads;
        }
        group = r / p.G;
        pair = (r % p.G) * m + (m - 1 - pos);
    } else if (MASK && !CAUSAL) {
        // A general mask is often one bias for every head (and batch): with
        // the pairs walked position-major over the groups, the CTAs that read
        // one block of bias rows run together and share it through L2.
        group = unit % p.n_groups;
        pair = unit / p.n_groups;
    } else if (!CAUSAL) {
        group = unit / p.n_pairs;
        pair = unit % p.n_pairs;
    } else {
        group = unit / p.n_pairs;
        pair = p.n_pairs - 1 - unit % p.n_pairs;
    }
    const int64_t row_base = static_cast<int64_t>(pair) * (2 * kRows);
    const int kt0 = split >= 0 ? split * p.tiles_per_split : 0;
    const int tps = split >= 0 ? p.tiles_per_split : 0x7fffffff - kt0;
    int n0 = tiles_in_range(kv_tiles_for(row_base, p, CAUSAL), kt0, tps);
    int n1 = tiles_in_range(kv_tiles_for(row_base + kRows, p, CAUSAL), kt0, tps);
    if (only == 0) n1 = 0;
    if (only == 1) n0 = 0;
    int nmax = n0 > n1 ? n0 : n1;
    // A boolean mask that depends on the key alone (one row of keep bytes for
    // the whole CTA, as a padding mask is) removes every key tile past its
    // last kept key: the CTA stops there (keeping at least one tile, so rows
    // with no kept key still end with O = 0 and LSE = -inf).
    const bool key_only = MK != 0 && p.mask_kind == 1 && p.msq == 0 && (p.msh == 0 || p.G == 1);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[2 * i], 1);
            mbar_init(&k_empty[2 * i + 1], 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[2 * i], 1);
            mbar_init(&v_empty[2 * i + 1], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], C::kTileThreads);
            mbar_init(&o_full[t], 1);
            mbar_init(&s_free[t], C::kTileThreads);
            mbar_init(&pv_done[t], 1);
            mbar_init(&mma_done[t], 1);
        }
        if constexpr (C::kConvWarps > 0) {
            for (int i = 0; i < VS; ++i) mbar_init(&v_cvt[i], C::kConvWarps);
            mbar_init(&cv_sync[0], 2);
            mbar_init(&cv_sync[1], 2);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (VPRE) {
        // The CTA reads the fp16 copy of V only if the copy holds every one of
        // its key tiles (flag 0); otherwise all of them come from the bf16 V.
        if (warp == 0) {
            const uint8_t* fl = p.vflags + static_cast<int64_t>(group) * p.n_ktiles + kt0;
            bool wide = false;
            for (int i = lane; i < nmax; i += 32) wide |= fl[i] != 0;
            wide = __any_sync(0xffffffffu, wide);
            if (lane == 0) *cta_v16 = wide ? 0 : 1;
        }
    }
    if (key_only && warp == 0 && nmax > 0) {
        const uint8_t* krow_all = static_cast<const uint8_t*>(p.mask) +
                                  (group / p.Hkv) * p.msb + (group % p.Hkv) * p.msh;
        const int last = last_kept_key(krow_all, kt0 * kRows, min(p.Nk, (kt0 + nmax) * kRows), lane);
        if (lane == 0) *key_lim = last < 0 ? 1 : last / kRows + 1 - kt0;
    }
    if (warp == kMmaWarp0) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (key_only && nmax > 0) {
        const int lim = *key_lim;
        n0 = min(n0, lim);
        n1 = min(n1, lim);
        nmax = max(n0, n1);
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            if constexpr (VPRE) tma_prefetch_desc(&tmV16);
            mbar_arrive_expect_tx(q_full, 2 * C::kTileBytes);
            for (int t = 0; t < 2; ++t)
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d(&tmQ, q_full, sQ + t * C::kTileBytes + kb * (kRows * 128),
                                kb * 64, static_cast<int>(row_base + t * kRows), group);
            const int nt[2] = {n0, n1};
            int nk = 0, nv = 0;  // loads issued
            bool okp = true;
            for (int j = 0; okp && j < nmax; ++j) {
                // A slot is free once every tile that used its previous tile
                // (the one KS loads back) has released it.
                const int ks = j % KS;
                for (int t = 0; okp && t < 2; ++t)
                    if (j >= KS && j - KS < nt[t])
                        okp = mbar_wait(&k_empty[2 * ks + t], ((j - KS) / KS) & 1, abort_flag, p.status);
                if (!okp) break;
                mbar_arrive_expect_tx(&k_full[ks], C::kTileBytes);
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d(&tmK, &k_full[ks], sK + ks * C::kTileBytes + kb * (kRows * 128),
                                kb * 64, (kt0 + j) * kRows, group);
                ++nk;
                const int vs = j % VS;
                for (int t = 0; okp && t < 2; ++t)
                    if (j >= VS && j - VS < nt[t])
                        okp = mbar_wait(&v_empty[2 * vs + t], ((j - VS) / VS) & 1, abort_flag, p.status);
                if (!okp) break;
                mbar_arrive_expect_tx(&v_full[vs], C::kTileBytes);
                const CUtensorMap* mv = (VPRE && *cta_v16) ? &tmV16 : &tmV;
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d(mv, &v_full[vs], sV + vs * C::kTileBytes + kb * (kRows * 128),
                                kb * 64, (kt0 + j) * kRows, group);
                ++nv;
            }
            // Never leave a copy in flight into shared memory we are about to give up.
            mbar_wait_bounded(q_full, 0, p.status);
            for (int n = (nk > KS ? nk - KS : 0); n < nk; ++n)
                mbar_wait_bounded(&k_full[n % KS], (n / KS) & 1, p.status);
            for (int n = (nv > VS ? nv - VS : 0); n < nv; ++n)
                mbar_wait_bounded(&v_full[n % VS], (n / VS) & 1, p.status);
        }
    } else if (warp == kMmaWarp0 || (C::kSepP && warp == kMmaWarp0 + 1)) {
        // ------------------------------------------------------------ MMA issue
        // Converged warps; one elected lane issues each MMA group.  An issuing
        // thread waits while its previous group drains, so everything else it
        // does leaves the tensor pipe idle unless another issuer fills it.
        constexpr uint32_t idesc_s = idesc_f16(kRows, kRows, BF16, false);
        constexpr uint32_t idesc_o = idesc_f16(kRows, D, BF16, true);
        // bf16 inputs: P and the converted value tile are fp16
        constexpr uint32_t idesc_o16 = idesc_f16(kRows, D, false, true);
        // Descriptor start addresses are in 16-byte units: one tile is
        // kTileBytes/16, a 64-column block 1024.
        constexpr uint64_t kTileStep = C::kTileBytes >> 4;
        constexpr uint64_t kBlk = (kRows * 128) >> 4;
        const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), kRows * 128, 1024);
        auto nt = [&](int t) { return t == 0 ? n0 : n1; };

        // S_t = Q_t K_j^T (64 columns of D per call), then release K_j for tile t.
        auto issue_s = [&](int t, int j) {
            const int kslot = j % KS;
            warp_wait(&k_full[kslot], (j / KS) & 1, abort_flag, p.status);
            tc_fence_after();
            const uint64_t b0 = dk0 + kslot * kTileStep;
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                mma_ss_k64(tmem + t * kRows, dq0 + t * kTileStep + kb * kBlk, b0 + kb * kBlk,
                           idesc_s, kb > 0 ? 1u : 0u);
            mma_commit_elect(&s_full[t]);
            mma_commit_elect(&k_empty[2 * kslot + t]);
        };
        // O_t += P_t V_j with P_t from TMEM, then release V_j for tile t.
        auto issue_pv = [&](int t, int j) {
            const int vslot = j % VS;
            uint32_t idesc_pv = (VPRE && *cta_v16) ? idesc_o16 : idesc_o;
            if constexpr (C::kConvWarps > 0) {
                warp_wait(&v_cvt[vslot], (j / VS) & 1, abort_flag, p.status);
                if (v_keep16[vslot] == 0) idesc_pv = idesc_o16;
            } else {
                warp_wait(&v_full[vslot], (j / VS) & 1, abort_flag, p.status);
            }
            warp_wait(&p_full[t], j & 1, abort_flag, p.status);
            tc_fence_after();
            mma_ts_k128(tmem + C::kOCol + t * D,
                        tmem + (C::kSepP ? C::kPCol + t * 64 : t * kRows),
                        dv0 + vslot * kTileStep, idesc_pv, j > 0 ? 1u : 0u);
            if constexpr (C::kSepP) mma_commit_elect(&pv_done[t]);
            mma_commit_elect(&v_empty[2 * vslot + t]);
            if (j == nt(t) - 1) mma_commit_elect(&o_full[t]);
        };

        // A wait that times out sets the abort flag and later waits return at
        // once, so every loop below runs to its end without blocking.
        if constexpr (C::kSepP) {
            // Separate P: one issuer per Q tile.  S of key tile j+1 goes as soon
            // as the softmax has read S of tile j, then PV of tile j.
            const int t = warp - kMmaWarp0;
            const int n_t = nt(t);
            if (n_t > 0) {
                warp_wait(q_full, 0, abort_flag, p.status);
                issue_s(t, 0);
            }
            for (int j = 0; j < n_t; ++j) {
                if (j + 1 < n_t) {
                    warp_wait(&s_free[t], j & 1, abort_flag, p.status);
                    issue_s(t, j + 1);
                }
                issue_pv(t, j);
            }
            mma_commit_elect(&mma_done[t]);
            mbar_wait_bounded(&mma_done[t], 0, p.status);
        } else if (warp == kMmaWarp0) {
            // P over S: one issuer for both tiles in the order PV_0, S_0', PV_1,
            // S_1', which keeps the two tiles half a period apart so one tile's
            // softmax runs under the other tile's products.
            warp_wait(q_full, 0, abort_flag, p.status);
            if (n0 > 0) issue_s(0, 0);
            if (n1 > 0) issue_s(1, 0);
            for (int j = 0; j < nmax; ++j) {
                if (j < n0) issue_pv(0, j);
                if (j + 1 < n0) issue_s(0, j + 1);
                if (j < n1) issue_pv(1, j);
                if (j + 1 < n1) issue_s(1, j + 1);
            }
            mma_commit_elect(&mma_done[0]);
            mbar_wait_bounded(&mma_done[0], 0, p.status);
        }
    } else if (C::kConvWarps > 0 &&
               (warp == C::kConvWarp0 || (C::kConvWarps == 2 && warp == C::kConvWarp1))) {
        // ------------------------------------------------------------ value-tile converter (bf16)
        // Rewrites each bf16 value tile in place as fp16, so that the PV
        // product runs with fp16 P (its rounding error is 2^-11 relative
        // instead of bf16's 2^-8).  A tile is converted when its largest
        // magnitude lies in [2^-8, 2^16): fp16 holds every such bf16 value
        // exactly down to 2^-14, and the smaller ones (fp16 subnormals) are
        // off by at most 2^-25, under 2^-17 of the tile's largest value.  Any
        // other tile (a value of 2^16 or more, an inf or NaN, or only values
        // below 2^-8) is left as bf16 and flagged, and that key tile's P is
        // packed as bf16.  Two converter warps split a tile and agree on the
        // flag through shared memory before either writes.
        const int cw = warp == C::kConvWarp0 ? 0 : 1;
        constexpr int kChunks = C::kTileBytes / 16 / (C::kConvWarps > 0 ? C::kConvWarps : 1);
        for (int j = 0; j < nmax; ++j) {
            const int vs = j % VS;
            const bool okw = warp_wait(&v_full[vs], (j / VS) & 1, abort_flag, p.status);
            uint4* base = reinterpret_cast<uint4*>(sV + vs * C::kTileBytes) + cw * kChunks;
            // largest bf16 exponent field of the tile (both halves of each word)
            uint32_t ex = 0u;
            if (okw) {
#pragma unroll 4
                for (int i = lane; i < kChunks; i += 32) {
                    const uint4 w = base[i];
                    ex = __vmaxu2(ex, __vmaxu2(__vmaxu2(w.x & 0x7f807f80u, w.y & 0x7f807f80u),
                                               __vmaxu2(w.z & 0x7f807f80u, w.w & 0x7f807f80u)));
                }
            }
            uint32_t emax = __reduce_max_sync(0xffffffffu, max(ex & 0xffffu, ex >> 16) >> 7);
            if constexpr (C::kConvWarps == 2) {
                // Both warps publish their half's exponent and wait (bounded)
                // until both have, before either rewrites the tile.  Tiles j
                // and j+2 share a flag buffer and a barrier, whose phase for
                // tile j is j/2: a warp reaches tile j+2 only after the other
                // has arrived for tile j+1, i.e. after it read tile j's flags.
                volatile int* flags = cv_wide + 2 * (j & 1);
                if (lane == 0) {
                    flags[cw] = static_cast<int>(emax);
                    mbar_arrive(&cv_sync[j & 1]);
                }
                __syncwarp();
                warp_wait(&cv_sync[j & 1], (j >> 1) & 1, abort_flag, p.status);
                emax = max(static_cast<uint32_t>(flags[0]), static_cast<uint32_t>(flags[1]));
            }
            // exponent field 119..142: largest magnitude in [2^-8, 2^16)
            const int wide = (emax >= 143u || emax <= 118u) ? 1 : 0;
            if (okw && !wide) {
#pragma unroll 4
                for (int i = lane; i < kChunks; i += 32) {
                    uint4 w = base[i];
                    w.x = bf16x2_to_f16x2(w.x);
                    w.y = bf16x2_to_f16x2(w.y);
                    w.z = bf16x2_to_f16x2(w.z);
                    w.w = bf16x2_to_f16x2(w.w);
                    base[i] = w;
                }
            }
            // the tensor core reads these bytes after the arrival below
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (cw == 0) v_keep16[vs] = wide;
                mbar_arrive(&v_cvt[vs]);
            }
        }
    } else if (C::kSplit && warp < C::kSoftmaxWarps) {
        // ------------------------------------------------------------ split softmax (D=64)
        // Thread = (row, half of the key tile).  The two warps of a row pair
        // share the row max through shared memory; a wait that times out sets
        // the abort flag and later waits return at once, so both warps of a
        // pair always meet at every pair barrier.
        const int t = (warp >> 2) & 1;   // Q tile
        const int quad = warp & 3;       // TMEM lane quadrant = rows quad*32 .. +31
        const int h = warp >> 3;         // key half: keys [64h, 64h+64) of each key tile
        const int n_t = t == 0 ? n0 : n1;
        const int rl = quad * 32 + lane;              // row within the Q tile
        const int64_t row0 = row_base + t * kRows;
        const int64_t row = row0 + rl;
        const bool row_valid = row < p.rows_per_group;
        const int pos = static_cast<int>(row % p.Nq);
        const int64_t wr0 = row0 + quad * 32;
        const int64_t wr1 = min(wr0 + 31, p.rows_per_group - 1);
        const int warp_min_pos =
            (wr0 / p.Nq == wr1 / p.Nq) ? static_cast<int>(wr0 % p.Nq) : 0;
        // General bias (MK = 1): this row's bias row (query head hkv*G +
        // row/Nq of batch group/Hkv), staged one key tile ahead: this warp's
        // 32 rows x 64 keys, nvalid rows real.  A half-tile is staged when its
        // keys lie inside [0, Nk); the ragged one reads its bias directly.
        // An additive bias turns the scores into natural-log logits s * scale
        // + b, so the softmax scale below becomes log2(e).
        const uint8_t* mrow = nullptr;
        if constexpr (MASK) {
            const int64_t hq = static_cast<int64_t>(group % p.Hkv) * p.G + row / p.Nq;
            const int64_t bq = group / p.Hkv;
            mrow = static_cast<const uint8_t*>(p.mask) +
                   (bq * p.msb + hq * p.msh + pos * p.msq) * (p.mask_kind == 2 ? 2 : 1);
        }
        const int64_t wleft = p.rows_per_group - wr0;
        const int nvalid = wleft <= 0 ? 0 : wleft >= 32 ? 32 : static_cast<int>(wleft);
        const uint32_t bbuf = smem_u32(smem + C::kBOff) + warp * (32 * 128);
        auto staged = [&](int jj) {
            return nvalid > 0 && (kt0 + jj) * kRows + 64 * h + 64 <= p.Nk;
        };
        if constexpr (MASK)
            if (n_t > 0 && staged(0))
                bias_prefetch<64>(bbuf, mrow, p.mask_kind, kt0 * kRows + 64 * h, nvalid, lane);
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * kRows + 64 * h;
        const uint32_t tO = tmem + lane_base + C::kOCol + t * D;
        const uint32_t tP = tmem + lane_base + C::kPCol + t * 64 + 32 * h;
        // Shared-window byte addresses of this thread's exchange slots:
        // xm[2 buffers][2 tiles][128 rows][2 halves] (buffer stride 2048 B),
        // then xl[2][128][2] and xr[2][128][2].  The partner's slot is at
        // address ^ 4 (the half is the lowest index bit).
        const uint32_t x_slot = smem_u32(smem + C::kXOff) + ((t * 128 + rl) * 2 + h) * 4;
        const uint32_t xl_slot = x_slot + 4096;
        const uint32_t xr_slot = x_slot + 6144;
        const uint32_t pair_bar = 1 + t * 4 + quad;  // named barrier of the warp pair
        uint32_t xbuf = 0;                           // 0 / 2048: buffer of key tile j
        const float sl2 = (MASK && p.mask_kind == 2) ? 1.4426950408889634f : p.scale_log2;

        float m = -INFINITY;  // running max (log2 domain, scaled), same in both halves
        float l = 0.0f;       // this half's running sum of p
        float lres = 0.0f;    // running sum of the rounding residuals of the half-tile maxima
        // A warp whose 32 rows all lie past the group (a short group, e.g. a
        // decode step) has nothing to compute; it only keeps the barrier
        // counts, and waits for each p_full phase to complete before it can
        // arrive on the next one.  Both warps of a pair are alike.
        const bool warp_live = wr0 < p.rows_per_group;
        // Key-padding mask: one row of keep bytes for the whole CTA (batch
        // group / Hkv; head group % Hkv when a KV group is one query head).
        // Lane l holds 16 of this half's 64 keep bytes (chunk l & 3), loaded
        // before the wait for S (every warp of the CTA reads the same bytes,
        // so they come from L1); the four chunks meet by shuffles.  A tile
        // with no dropped key costs one minimum.
        const uint8_t* krow = nullptr;
        if constexpr (KEYMASK)
            krow = static_cast<const uint8_t*>(p.mask) + (group / p.Hkv) * p.msb +
                   (group % p.Hkv) * p.msh;
        // Keep bytes of key tile jj (zeros for a tile past the end or with
        // keys past Nk: those go key by key below).
        auto kload = [&](int jj) -> uint4 {
            const int k0 = (kt0 + jj) * kRows + 64 * h;
            if (jj < n_t && k0 + 64 <= p.Nk) return reinterpret_cast<const uint4*>(krow + k0)[lane & 3];
            return make_uint4(0u, 0u, 0u, 0u);
        };
        // First key tile j whose half-tile (keys key0(j) .. key0(j) + 63,
        // key0(j) = (kt0 + j) * 128 + 64 h) needs a per-key mask: it reaches
        // past Nk, or (causal) past what this warp's first row may see.  Both
        // conditions only grow with j.
        auto first_tile_past = [&](int64_t lim) -> int {   // first j with key0(j) + 63 >= lim
            const int64_t t = lim - 63 - 64 * h;            // need (kt0 + j) * 128 >= t
            if (t <= 0) return 0;
            const int64_t jj = (t + kRows - 1) / kRows - kt0;
            return jj < 0 ? 0 : static_cast<int>(jj);
        };
        int j_mask = first_tile_past(p.Nk);
        if (CAUSAL) j_mask = min(j_mask, first_tile_past(static_cast<int64_t>(warp_min_pos) +
                                                         p.causal_off + 1));
        for (int j = 0; j < n_t; ++j) {
            if (!warp_live) {
                warp_wait(&s_full[t], j & 1, abort_flag, p.status);
                mbar_arrive(&s_free[t]);
                mbar_arrive(&p_full[t]);
                warp_wait(&p_full[t], j & 1, abort_flag, p.status);
                continue;
            }
            const int key0 = (kt0 + j) * kRows + 64 * h;
            uint4 kcur = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (KEYMASK) kcur = kload(j);
            warp_wait(&s_full[t], j & 1, abort_flag, p.status);
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld64(tS, sr[0], sr[1]);
            tmem_wait_ld();
            reg_fence(sr[0]);
            reg_fence(sr[1]);
            // S_t is in registers: the MMA warp may compute the next S_t.
            tc_fence_before();
            mbar_arrive(&s_free[t]);

            if constexpr (MASK) {
                if (staged(j)) {
                    cp_async_wait_all();
                    __syncwarp();
                    bias_fold_smem64<BF16>(sr, bbuf, p.mask_kind, p.scale, lane);
                    __syncwarp();
                } else {
                    bias_fold_direct64<BF16>(sr, mrow, p.mask_kind, key0, p.Nk, p.scale, row_valid);
                }
                if (j + 1 < n_t && staged(j + 1))
                    bias_prefetch<64>(bbuf, mrow, p.mask_kind, key0 + kRows, nvalid, lane);
            }
            if constexpr (KEYMASK) {
                // does any of this lane's 16 keep bytes equal 0?  (w - 0x01..01) &
                // ~w & 0x80..80 is nonzero exactly when a byte of w is 0; the
                // lanes' chunks together cover the half-tile's 64 bytes
                auto zero_byte = [](uint32_t w) { return (w - 0x01010101u) & ~w & 0x80808080u; };
                const uint32_t z =
                    zero_byte(kcur.x) | zero_byte(kcur.y) | zero_byte(kcur.z) | zero_byte(kcur.w);
                if (__any_sync(0xffffffffu, z != 0u)) {   // the same in every lane
                    if (key0 + 64 <= p.Nk) {
#pragma unroll
                        for (int w = 0; w < 16; ++w) {
                            const uint32_t mine = (w & 3) == 0 ? kcur.x : (w & 3) == 1 ? kcur.y
                                                 : (w & 3) == 2 ? kcur.z : kcur.w;
                            const uint32_t word = __shfl_sync(0xffffffffu, mine, w >> 2);
#pragma unroll
                            for (int b = 0; b < 4; ++b)
                                if (((word >> (8 * b)) & 0xffu) == 0u)
                                    sr[w >> 3][(4 * w + b) & 31] = __float_as_uint(-INFINITY);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int key = key0 + 32 * c + i;
                                if (key < p.Nk && krow[key] == 0) sr[c][i] = __float_as_uint(-INFINITY);
                            }
                    }
                }
            }
            if (j >= j_mask) {
                // keys [0, lim) allowed
                const int lim = CAUSAL ? min(p.Nk, pos + p.causal_off + 1) : p.Nk;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (key0 + c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
            }
            const float pm = row_max64(sr);
            st_shared_f32(x_slot + xbuf, pm);
            named_bar_sync(pair_bar, 64);
            const float mx = fmaxf(pm, ld_shared_f32((x_slot ^ 4u) + xbuf));
            xbuf ^= 2048u;
            const float m_new = fmaxf(m, mx * sl2);
            const bool need = m_new > m + kRescaleThreshold;
            // Branch-free: alpha is only used when need (m = -inf gives 0).
            const float alpha = need ? ex2_ftz(m - m_new) : 1.0f;
            m = need ? m_new : m;
            const float m_sub = (m == -INFINITY) ? 0.0f : m;

            uint64_t acc2[4];
            const uint64_t sl22 = f2(sl2, sl2), nm2 = f2(-m_sub, -m_sub);
            // The largest term of this half-tile (the one that dominates a
            // one-hot row) is rounded like every term; its rounding residual
            // joins the normaliser, so such a row gets exactly its value row.
            const float rtop = round16_residual<BF16>(pm, sl2, -m_sub);
            // keys 64h + i -> P column 32h + i/2; four running sums of pairs,
            // each started by its first pair
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 8; i += 2)
                pk[i >> 1] = softmax_pair<BF16, false>(sr[0][i], sr[0][i + 1], sl22, nm2,
                                                       acc2[i >> 1]);
#pragma unroll
            for (int i = 8; i < 64; i += 2)
                pk[i >> 1] = softmax_pair<BF16>(sr[i >> 5][i & 31], sr[i >> 5][(i & 31) + 1], sl22,
                                                nm2, acc2[(i >> 1) & 3]);
            if (j > 0) {
                // P_t and O_t are still in use by the PV product of tile j-1.
                warp_wait(&pv_done[t], (j - 1) & 1, abort_flag, p.status);
                tc_fence_after();
            }
            tmem_st32(tP, pk);
            const uint64_t a2 = fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3]));
            const float rs = f2lo(a2) + f2hi(a2);
            lres = lres * alpha + rtop;
            // Each half rescales its half of O's columns (the decision is the
            // same in both halves).
            if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int c = h * (D / 64); c < (h + 1) * (D / 64); ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
                    reg_fence(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + c * 32, o);
                }
            }
            l = l * alpha + rs;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
        }
        // No bias copy may still be in flight when the CTA gives up its shared memory.
        if constexpr (MASK) cp_async_wait_all();

        if (n_t > 0 && warp_live) {
            warp_wait(&o_full[t], 0, abort_flag, p.status);
            tc_fence_after();
            st_shared_f32(xl_slot, l);
            st_shared_f32(xr_slot, lres);
            named_bar_sync(pair_bar, 64);
            const float lt = l + ld_shared_f32(xl_slot ^ 4u);
            const float lrest = lres + ld_shared_f32(xr_slot ^ 4u);
            const bool ok = *abort_flag == 0;
            // O is normalised by the sum of p plus the residuals of the tile
            // maxima; the LSE uses the sum of p alone.
            const float l_out = lt + lrest;
            const float inv_l = l_out > 0.0f ? 1.0f / l_out : 0.0f;
            const int64_t grow = static_cast<int64_t>(group) * p.rows_per_group + row;
#pragma unroll
            for (int c = h * (D / 64); c < (h + 1) * (D / 64); ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_wait_ld();
                reg_fence(o);
                if (ok && row_valid) store_o32<D, BF16>(p, split, grow, c, o, inv_l);
            }
            if (ok && row_valid && h == 0) {
                const float m_sub = (m == -INFINITY) ? 0.0f : m;
                store_lse(p, split, grow, lt > 0.0f ? (m_sub + lg2_approx(lt)) * kLn2 : -INFINITY);
            }
        } else if (split >= 0 && row_valid) {
            // No key of this range is visible to the tile: an empty partial.
            const int64_t grow = static_cast<int64_t>(group) * p.rows_per_group + row;
            const uint32_t z[32] = {};
#pragma unroll
            for (int c = h * (D / 64); c < (h + 1) * (D / 64); ++c)
                store_o32<D, BF16>(p, split, grow, c, z, 0.0f);
            if (h == 0) store_lse(p, split, grow, -INFINITY);
        }
    } else if (!C::kSplit && warp < C::kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = warp >> 2;         // Q tile of this warpgroup
        const int quad = warp & 3;       // TMEM lane quadrant = rows quad*32 .. +31
        const int n_t = t == 0 ? n0 : n1;
        const int64_t row0 = row_base + t * kRows;
        const int64_t row = row0 + quad * 32 + lane;
        const bool row_valid = row < p.rows_per_group;
        const int pos = static_cast<int>(row % p.Nq);
        // This row's bias: query head hkv*G + row/Nq of batch group/Hkv.
        const uint8_t* mrow = nullptr;
        if constexpr (MASK) {
            const int64_t h = static_cast<int64_t>(group % p.Hkv) * p.G + row / p.Nq;
            const int64_t b = group / p.Hkv;
            const int esz = p.mask_kind == 2 ? 2 : 1;
            mrow = static_cast<const uint8_t*>(p.mask) + (b * p.msb + h * p.msh + pos * p.msq) * esz;
        }
        // Smallest query position among this warp's rows: masking is needed on
        // key tiles that reach past it (or past Nk).
        const int64_t wr0 = row0 + quad * 32;
        const int64_t wr1 = min(wr0 + 31, p.rows_per_group - 1);
        const int warp_min_pos =
            (wr0 / p.Nq == wr1 / p.Nq) ? static_cast<int>(wr0 % p.Nq) : 0;
        // Staged bias (kBiasSmem): this warp's 32 rows, nvalid of them real.
        // A key tile is staged when it lies inside [0, Nk) and the warp has a
        // real row; the ragged last tile reads its bias directly.
        const int64_t left = p.rows_per_group - wr0;
        const int nvalid = left <= 0 ? 0 : left >= 32 ? 32 : static_cast<int>(left);
        const uint32_t bbuf = smem_u32(smem + C::kBOff) + warp * (32 * 256);
        auto staged = [&](int jj) { return nvalid > 0 && (kt0 + jj + 1) * kRows <= p.Nk; };
        if constexpr (C::kBiasSmem)
            if (n_t > 0 && staged(0)) bias_prefetch<128>(bbuf, mrow, p.mask_kind, kt0 * kRows, nvalid, lane);
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * kRows;
        const uint32_t tO = tmem + lane_base + C::kOCol + t * D;
        const uint32_t tP = C::kSepP ? tmem + lane_base + C::kPCol + t * 64 : tS;
        const float sl2 = p.scale_log2;

        float m = -INFINITY;  // running max (log2 domain, scaled) used for exponentiation
        float l = 0.0f;       // running sum of p (gives the LSE)
        float lres = 0.0f;    // running sum of the rounding residuals of the tile maxima
        bool ok = true;
        // A warp with no real row only keeps the barrier counts (as in the
        // split layout above).  (Not in the masked variant, whose registers
        // are already at the limit.)
        const bool warp_live = MASK || wr0 < p.rows_per_group;
        for (int j = 0; j < n_t; ++j) {
            if (!warp_live) {
                warp_wait(&s_full[t], j & 1, abort_flag, p.status);
                if constexpr (C::kSepP) mbar_arrive(&s_free[t]);
                mbar_arrive(&p_full[t]);
                warp_wait(&p_full[t], j & 1, abort_flag, p.status);
                continue;
            }
            const int key0 = (kt0 + j) * kRows;
            // D = 128 with a general mask: the first bias chunk is requested
            // before the wait for S, each later one a chunk ahead.
            const bool bfull = MASK && row_valid && key0 + kRows <= p.Nk;
            BiasChunk bn;
            if constexpr (MASK && !C::kBiasSmem) bias_load(bn, mrow, p.mask_kind, key0, bfull);
            if (!warp_wait(&s_full[t], j & 1, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            if constexpr (MASK && !C::kBiasSmem) {
                // Scores -> log2-domain logits with the bias, in place in TMEM
                // one 32-key chunk at a time (few live registers); the rest of
                // the tile then runs with scale 1 (sc below).
                const bool full = bfull;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const BiasChunk b = bn;
                    if (c < 3) bias_load(bn, mrow, p.mask_kind, key0 + 32 * (c + 1), full);
                    uint32_t x[32];
                    tmem_ld32(tS + c * 32, x);
                    tmem_wait_ld();
                    reg_fence(x);
                    bias_apply<BF16>(x, b, mrow, p.mask_kind, key0 + 32 * c, p.Nk, sl2, full,
                                     row_valid);
                    tmem_st32(tS + c * 32, x);
                }
                tmem_wait_st();
            }
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
            if constexpr (C::kSepP) {
                // S_t is in registers: the MMA warp may compute the next S_t.
                tc_fence_before();
                mbar_arrive(&s_free[t]);
            }
            if constexpr (C::kBiasSmem) {
                // Scores -> log2-domain logits with the staged bias; then the
                // next key tile's bias is requested into the same rows.
                if (staged(j)) {
                    cp_async_wait_all();
                    __syncwarp();
                    bias_fold_smem<BF16>(sr, bbuf, p.mask_kind, sl2, lane);
                    __syncwarp();
                } else {
                    const BiasChunk none{};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        bias_apply<BF16>(sr[c], none, mrow, p.mask_kind, key0 + 32 * c, p.Nk, sl2,
                                         false, row_valid);
                }
                if (j + 1 < n_t && staged(j + 1))
                    bias_prefetch<128>(bbuf, mrow, p.mask_kind, key0 + kRows, nvalid, lane);
            }

            const float sc = MASK ? 1.0f : sl2;   // scale still to apply to sr
            const bool need_mask =
                (key0 + kRows > p.Nk) || (CAUSAL && key0 + kRows - 1 > warp_min_pos + p.causal_off);
            if (need_mask) {
                // keys [0, lim) allowed
                const int lim = CAUSAL ? min(p.Nk, pos + p.causal_off + 1) : p.Nk;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (key0 + c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
            }
            const float mx = row_max128(sr);
            const float m_new = fmaxf(m, mx * sc);
            const bool need = m_new > m + kRescaleThreshold;
            // Branch-free: alpha is only used when need (m = -inf gives 0).
            const float alpha = need ? ex2_ftz(m - m_new) : 1.0f;
            m = need ? m_new : m;
            const float m_sub = (m == -INFINITY) ? 0.0f : m;

            if constexpr (C::kSepP) {
                // P_t and O_t are still in use by the PV product of tile j-1.
                if (j > 0) {
                    if (!warp_wait(&pv_done[t], (j - 1) & 1, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                }
            }
            // bf16 inputs: P is fp16 unless this key tile's values had to stay bf16
            bool p_bf16 = BF16 && !(VPRE && *cta_v16);
            if constexpr (C::kConvWarps > 0) {
                const int vs = j % VS;
                if (!warp_wait(&v_cvt[vs], (j / VS) & 1, abort_flag, p.status)) { ok = false; break; }
                p_bf16 = v_keep16[vs] != 0;
            }
            // partial row sums of p, as packed pairs; P of keys 32c..32c+31 goes
            // to TMEM columns 16c..16c+15 as soon as it is packed (with P over S
            // those scores are already read).  The largest term (the one that
            // dominates a one-hot row) is rounded like every term; its rounding
            // residual joins the normaliser, so such a row gets exactly its value row.
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
            const uint64_t sl22 = f2(sc, sc), nm2 = f2(-m_sub, -m_sub);
            float rtop;
            if (p_bf16) {
                rtop = round16_residual<true>(mx, sc, -m_sub);
                pack_p128<true>(sr, tP, sl22, nm2, acc2);
            } else {
                rtop = round16_residual<false>(mx, sc, -m_sub);
                pack_p128<false>(sr, tP, sl22, nm2, acc2);
            }
            const uint64_t a2 = fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3]));
            const float rs = f2lo(a2) + f2hi(a2);
            lres = lres * alpha + rtop;

            // O_t must be rescaled before the next PV accumulates into it.  PV
            // of key tile j-1 is complete: with P over S, S_t of tile j was
            // committed after it; with separate P, pv_done was waited above.
            if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
                    reg_fence(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + c * 32, o);
                }
            }
            l = l * alpha + rs;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
        }
        // No bias copy may still be in flight when the CTA gives up its shared memory.
        if constexpr (C::kBiasSmem) cp_async_wait_all();

        if (ok && warp_live && n_t > 0 && warp_wait(&o_full[t], 0, abort_flag, p.status)) {
            tc_fence_after();
            // O is normalised by the sum of p plus the residuals of the tile
            // maxima; the LSE uses the sum of p alone.
            const float l_out = l + lres;
            const float inv_l = l_out > 0.0f ? 1.0f / l_out : 0.0f;
            const int64_t grow = static_cast<int64_t>(group) * p.rows_per_group + row;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_wait_ld();
                reg_fence(o);
                if (row_valid) store_o32<D, BF16>(p, split, grow, c, o, inv_l);
            }
            if (row_valid) {
                const float m_sub = (m == -INFINITY) ? 0.0f : m;
                store_lse(p, split, grow, l > 0.0f ? (m_sub + lg2_approx(l)) * kLn2 : -INFINITY);
            }
        } else if (n_t == 0 && split >= 0 && row_valid) {
            // No key of this range is visible to the tile: an empty partial.
            const int64_t grow = static_cast<int64_t>(group) * p.rows_per_group + row;
            const uint32_t z[32] = {};
#pragma unroll
            for (int c = 0; c < D / 32; ++c) store_o32<D, BF16>(p, split, grow, c, z, 0.0f);
            store_lse(p, split, grow, -INFINITY);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool BF16, bool CAUSAL, int MK, bool VPRE>
cudaError_t launch_one(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmV16, const FwdParams& p, cudaStream_t stream) {
    auto kern = attn_fwd_kernel<D, BF16, CAUSAL, MK, VPRE>;
    constexpr int smem = FwdCfg<D, MK, BF16, VPRE>::kSmemBytes;
    constexpr int kThreads = FwdCfg<D, MK, BF16, VPRE>::kThreads;
    // Re-applied on every call: a cheap attribute write that is correct on
    // whichever device is current.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long units = static_cast<long long>(p.n_groups) * p.n_pairs;
    const long long ctas =
        (p.n_splits > 1 ? p.n_whole + (units - p.n_whole) * p.n_splits : units) +
        static_cast<long long>(p.n_groups) * p.G * p.n_half_pos;
    return launch_kernel(kern, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, stream,
                         tmQ, tmK, tmV, tmV16, p);
}

}  // namespace

cudaError_t launch_fwd(int D, bool bf16, bool causal, const CUtensorMap& tmQ,
                       const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                       cudaStream_t stream, const CUtensorMap* tmV16) {
    // A boolean mask that depends on the key alone (no query stride, and no
    // head stride unless every KV group is one query head) runs in the D=64
    // split layout (fp16 inputs; bf16 inputs never use that layout); every
    // other mask takes the general masked layout.
    int mk = 0;
    if (p.mask != nullptr) {
        const bool key_only = p.mask_kind == 1 && p.msq == 0 && (p.msh == 0 || p.G == 1);
        mk = (D == 64 && key_only && !bf16) ? 2 : 1;
    }
    // bf16 without a mask, given the fp16 copy of V (p.vflags and tmV16):
    // the instantiation without converter warps.
    if (tmV16 != nullptr) {
        if (!bf16 || mk != 0 || p.vflags == nullptr) return cudaErrorInvalidValue;
        if (D == 64 && !causal) return launch_one<64, true, false, 0, true>(tmQ, tmK, tmV, *tmV16, p, stream);
        if (D == 64 && causal) return launch_one<64, true, true, 0, true>(tmQ, tmK, tmV, *tmV16, p, stream);
        if (D == 128 && !causal) return launch_one<128, true, false, 0, true>(tmQ, tmK, tmV, *tmV16, p, stream);
        if (D == 128 && causal) return launch_one<128, true, true, 0, true>(tmQ, tmK, tmV, *tmV16, p, stream);
        return cudaErrorInvalidValue;
    }
#define TME_CASE(d, b, c, m)                                  \
    if (D == d && bf16 == b && causal == c && mk == m)        \
        return launch_one<d, b, c, m, false>(tmQ, tmK, tmV, tmV, p, stream);
#define TME_CASES(m)              \
    TME_CASE(64, false, false, m)  \
    TME_CASE(64, false, true, m)   \
    TME_CASE(64, true, false, m)   \
    TME_CASE(64, true, true, m)    \
    TME_CASE(128, false, false, m) \
    TME_CASE(128, false, true, m)  \
    TME_CASE(128, true, false, m)  \
    TME_CASE(128, true, true, m)
    TME_CASES(0)
    TME_CASES(1)
    TME_CASE(64, false, false, 2)
    TME_CASE(64, false, true, 2)
#undef TME_CASES
#undef TME_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tme
