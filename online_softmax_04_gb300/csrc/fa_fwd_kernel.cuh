// fa_fwd_kernel.cuh -- fused attention forward for sm_103a (GB300).
//
// A 128-row query tile of one (batch, head) stays resident while the key/value
// tiles stream past it ("Online Softmax: Tiling Across a Reduction", loop
// order: query blocks outer and resident, key/value blocks inner).  Per key
// tile j each query row updates its state with one correction factor
// ("Online softmax, and the register that can't move", section "Online
// softmax"):
//
//     m_new = max(m_old, rowmax(S_j))
//     l_new = l_old * exp(m_old - m_new) + rowsum(exp(S_j - m_new))
//     O_new = O_old * exp(m_old - m_new) + exp(S_j - m_new) V_j
//
// and after the last tile O /= l, LSE = m + ln l.  Scores are kept in the
// base-2 domain, t = s * scale * log2(e), so every exponential is one ex2.
//
// GB300 mapping:
//   * Persistent grid, one CTA per SM, each working through a sequence of query
//     tiles: causal tiles paired long with short and dealt out statically in
//     full rounds, the partial last round handed out one tile at a time from a
//     global counter.  The TMA ring, the S/P double buffers and every barrier phase
//     run on across tile boundaries, so the loads and first S products of the
//     next tile overlap the end of this one.
//   * S_j = Q K_j^T and O += P_j V_j run on tcgen05.mma (bf16 in, fp32
//     accumulate) with the accumulators in tensor memory (TMEM).  S is double
//     buffered and P has columns of its own, so S_{j+1} is computed while the
//     softmax works on S_j and nothing waits for a product to drain.
//   * Two MMA-issuing warps: one issues the S products as soon as a K tile
//     and an S buffer are free, the other the P V products as soon as P_j is
//     written.  A tcgen05.mma burst keeps its issuing thread busy until the
//     tensor pipe has taken it, so two issuers keep the pipe fed while either
//     one waits on a barrier.  Every instruction an issuer runs between
//     products costs feed rate, so the whole warp runs the loop (waits,
//     counters, descriptors built once per product and advanced by a 32-bit
//     add per K step) and an elect.sync lane issues the products and commits.
//   * P_j is written back to TMEM as bf16 and consumed from there as the A
//     operand of P V (no shared-memory round trip).
//   * Q, K_j and V_j are brought in by TMA (128-byte swizzle) into rings of
//     shared-memory stages guarded by mbarriers.
//   * Warp roles: warp 0 issues TMA loads, warp 1 owns TMEM and issues the S
//     products, warp 2 issues the P V products, warps 4-11 do the softmax, the
//     O rescale on TMEM and the epilogue (O/l -> bf16 -> global, LSE).  The
//     softmax warps form two groups of four (one warp per 32-row TMEM lane
//     quarter) that take alternate key tiles, a thread holding all 128 scores
//     of its row.  Only the reference maximum passes from one step to the
//     next; each group hands it to the other through shared memory (one
//     64-bit word per row tagged with the step) as soon as its row maximum is
//     known, so the exponentials of step j overlap the TMEM load and maximum of
//     step j+1.  Each group keeps its row sums
//     against the last reference it used; the two are combined at the end.
//   * The reference maximum of a row moves only when the row maximum has
//     grown past it by more than 64 in base-2 units; otherwise the old
//     reference is kept, exponentials up to 2^64 are accumulated in fp32 and
//     the O rescale on TMEM is skipped.  exp(x - m) / sum exp(x - m) does not
//     depend on m, so the result is unchanged.
//   * The P V product uses bf16-rounded weights.  O is divided by a sum that
//     accounts for that rounding where it matters most, the largest weight,
//     while LSE uses the fp32 sum of the unrounded exponentials.  At d = 64
//     the tensor core forms the exact sum of the rounded weights in extra
//     columns of the P V product (see FaSmem::kTcSum).  At d = 128 TMEM has
//     no room for them; there the sum is the fp32 sum plus, for every key
//     tile, bf16(p_max) - p_max of the tile's largest weight, recomputed from
//     the row maximum.  When one key dominates a row, that is the exact sum
//     of the rounded weights, and O / l returns that key's V row; elsewhere
//     the roundings of the many comparable weights average out.
//   * The row maximum of a step comes with the S read-out: the TMEM load's max
//     reduction over the 128 loaded columns.  Rows with masked keys in the
//     tile (diagonal, sequence end, windows, documents) reduce the masked
//     values instead.
//   * Epilogue: each group reads its half of O's columns out of TMEM in one
//     load, releases O to the next tile's first P V product at once, then
//     normalises and stores its half rows.
//   * Causal: key tiles wholly after the query tile are never visited; only
//     the diagonal tile is masked element by element ("Online Softmax: Tiling
//     Across a Reduction", causal section).  Keys >= N in the last tile are
//     masked the same way.
//
// Every barrier wait is bounded by a watchdog (global timer): on expiry the
// CTA records a status bit, tells its other warps to stop, lets its copies
// and MMAs drain, frees TMEM and exits.
#pragma once

#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;   // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 384;  // 12 warps
constexpr int kSoftmaxWarps = 8;  // two groups of four, one warp per TMEM lane quarter each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChunkBytes = 128u * 128u;  // one [128 rows][64 bf16] swizzled chunk
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kItemRing = 4;  // work items the producer may run ahead of the slowest role
// readers of each posted work item: the two MMA issuers and every softmax warp
constexpr int kItemReaders = 2 + 8;
// Base-2 growth of a row's maximum tolerated before its reference moves.  It
// bounds every exponential by 2^64, the row sums by N * 2^64 and |O| by
// N * 2^64 * max|V|: finite in fp32 for max|V| < 2^33 at any N < 2^31.
constexpr float kRescaleThreshold = 64.0f;

// device status bits (which wait ran out)
enum : unsigned int {
    kStatusLoadWait = 1u << 0,
    kStatusMmaWaitQ = 1u << 1,
    kStatusMmaWaitK = 1u << 2,
    kStatusMmaWaitP = 1u << 3,
    kStatusMmaWaitV = 1u << 4,
    kStatusSoftmaxWaitS = 1u << 5,
    kStatusSoftmaxWaitO = 1u << 6,
    kStatusDrain = 1u << 7,
    kStatusSelfTest = 1u << 8,
    kStatusMmaWaitSFree = 1u << 9,
    kStatusSoftmaxWaitPV = 1u << 10,
    kStatusSoftmaxWaitX = 1u << 11,
    kStatusItemWait = 1u << 12,
    kStatusSoftmaxRows = 1u << 13,
};

__device__ unsigned int g_fa_status = 0;

struct FaParams {
    void* o;     // bf16 [B*H][N][d]
    float* lse;  // fp32 [B*H][N]
    int BH;
    int H;                // heads per batch entry (b = bh / H)
    // key j is visible to query i iff j >= i - window_left (window_left >= 0),
    // j <= i + window_right (window_right >= 0) and, with doc, doc[b][j] ==
    // doc[b][i]; -1 leaves a side unbounded.  Causal attention: window_right = 0.
    int window_left, window_right;
    const int* doc;       // int32 [B][N] document ids, non-decreasing along each sequence, or nullptr
    // persistent schedule: rounds of tile pairs assigned statically per CTA, or -1
    // when the grid has one CTA per tile (CTA x takes tile x; no work counter)
    int static_rounds;
    unsigned int* queue;  // persistent schedule: {next dynamic item, CTAs finished}, zero on entry, reset on exit
    int N;
    int n_tiles;       // ceil(N / 128) query (= key) tiles
    int causal;
    float scale_log2;  // scale * log2(e)
    unsigned long long watchdog_ns;
    // watchdog self-test only: the S products are never issued, so the softmax
    // warps' first wait runs out (0 in every real launch)
    int withhold_s;
    // split-KV partial states (kSplit kernels only): [n_splits][B*H][N] rows
    int n_splits;
    float* ws_o;    // unnormalised O, fp32 [rows][d]
    float* ws_m;    // reference max, base-2 units
    float* ws_lbf;  // the sum that normalises O (rounded weights at d = 64; fp32 sum + max corrections at d = 128)
    float* ws_l32;  // fp32 sum of the exponentials
};

template <int D, int NK, int NV, bool kPair = false, bool kOStage = false>
struct FaSmem {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!kPair || D == 128, "CTA pairs at d = 128");
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = kBlockN * D * 2;
    // A CTA pair splits every K tile by keys (64 keys per CTA) and every V tile
    // by columns (64 of d per CTA): each CTA holds half of each.
    static constexpr uint32_t kKBytes = kPair ? kTileBytes / 2 : kTileBytes;
    static constexpr uint32_t kVBytes = kPair ? kTileBytes / 2 : kTileBytes;
    static constexpr uint32_t kKChunkBytes = kPair ? kChunkBytes / 2 : kChunkBytes;  // one 64-column chunk of a K stage
    static constexpr int kQBufs = 1;      // query tiles in flight: the next tile's Q lands early
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQBufs * kTileBytes;
    static constexpr uint32_t kOffV = kOffK + NK * kKBytes;
    // d = 64 leaves TMEM room for the row sums of P on the tensor core: the P V
    // product is widened to N = d + 16, and its B operand's second 64-column
    // block (reached through the descriptor's leading-byte offset) is a 2 KB
    // tile of ones, so columns d..d+15 of the accumulator receive the row sums
    // of the same bf16 P (16 key rows x 128 bytes; any swizzle of ones is ones)
    static constexpr bool kTcSum = D == 64;
    static constexpr uint32_t kOnesBytes = kTcSum ? 2048u : 0u;
    static constexpr uint32_t kOffOnes = kOffV + NV * kVBytes;
    static constexpr uint32_t kOffBar = kOffOnes + kOnesBytes;
    static constexpr int kBarQ = 0;  // per Q buffer: the tile landed
    static constexpr int kBarKFull = kBarQ + kQBufs;
    static constexpr int kBarKEmpty = kBarKFull + NK;
    // with two K stages, stage g % 2 is free once S_g (buffer g % 2) has finished:
    // the producer then waits on SFull and the S issuer commits one barrier a step
    static constexpr bool kKEmptyIsSFull = NK == 2;
    static constexpr int kBarVFull = kBarKEmpty + NK;
    static constexpr int kBarVEmpty = kBarVFull + NV;
    static constexpr int kBarSFull = kBarVEmpty + NV;  // per S buffer: S_j written
    static constexpr int kBarSFree = kBarSFull + 2;    // per S buffer: S_j read by the softmax
    static constexpr int kBarPFull = kBarSFree + 2;    // per P buffer: P_j written
    static constexpr int kBarPVDone = kBarPFull + 2;   // per P buffer: P_j V_j finished
    static constexpr int kBarOFinal = kBarPVDone + 2;  // per tile: its last P V product finished
    static constexpr int kBarQFree = kBarOFinal + 1;   // per Q buffer: the tile's last S product finished
    static constexpr int kBarOFree = kBarQFree + kQBufs;  // per tile: O read out of TMEM (accumulator reusable)
    static constexpr int kBarDrain = kBarOFree + 1;    // per MMA issuer
    static constexpr int kBarXSum = kBarDrain + 2;     // per lane quarter: both groups' row sums posted
    static constexpr int kBarItemFull = kBarXSum + 4;  // per item-ring slot: the producer posted an item
    static constexpr int kBarItemEmpty = kBarItemFull + kItemRing;  // per slot: every role has read it
    static constexpr int kNumBars = kBarItemEmpty + kItemRing;
    // reference hand-over slots [2 groups][128 rows] of (step << 32 | reference bits), then row
    // states [2 tile parities][2 groups][m, l, l32][128 rows]
    static constexpr uint32_t kOffXchg = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffXSum = kOffXchg + 2 * kBlockM * 8;
    // work-item ring: per entry {bh * n_tiles + qt, first key tile, key tiles, unused}
    static constexpr uint32_t kOffItems = kOffXSum + 2 * 2 * 3 * kBlockM * 4;
    static constexpr uint32_t kOffTmemSlot = kOffItems + kItemRing * 16;
    static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
    // kOStage: the epilogue writes O through shared memory and TMA stores, 2 KB per
    // softmax warp (16 rows of its 64-column half of O, 128-byte swizzle, 1024-byte aligned)
    static constexpr bool kOStaged = kOStage;
    static constexpr uint32_t kOStageWarpBytes = 16 * 128;
    static constexpr uint32_t kOffOStage = (kOffAbort + 4 + 1023) & ~1023u;
    static constexpr uint32_t kBytes = kOStage ? kOffOStage + 8 * kOStageWarpBytes : kOffAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    static_assert(kAlloc <= 232448u, "dynamic shared memory above the 227 KB a CTA may use");
    // TMEM columns: S0 S1 O [row sums] P0 P1
    __host__ __device__ static constexpr uint32_t col_s(int b) { return (uint32_t)b * 128u; }
    static constexpr uint32_t kColO = 256;
    static constexpr uint32_t kSumCols = kTcSum ? 16u : 0u;
    static constexpr uint32_t kColL = 256u + D;  // row sums of the bf16 P (kTcSum), column kColL
    __host__ __device__ static constexpr uint32_t col_p(int b) { return 256u + D + kSumCols + (uint32_t)b * 64u; }
    static_assert(256 + D + kSumCols + 128 <= kTmemCols, "TMEM budget");
};

// One poll of a barrier phase; kCl: with cluster-scope acquire (barriers the
// other CTA of a pair arrives on, directly or through a tensor-core commit).
template <bool kCl>
__device__ __forceinline__ bool fa_poll(uint32_t bar, uint32_t parity) {
    if constexpr (kCl)
        return mbar_try_wait_cluster(bar, parity);
    else
        return mbar_try_wait(bar, parity);
}

// The shared-memory layout of an instance: the epilogue stages O for TMA stores
// in the one-CTA kernels at d = 128 that write O (not split-KV, not pairs).
template <int D, int NK, int NV, bool kSplit, bool kPair>
using FwdSmem = FaSmem<D, NK, NV, kPair, D == 128 && !kSplit && !kPair>;

// Bounded wait on an mbarrier phase.  Gives up when another warp of the CTA
// has raised the abort flag, or after `limit_ns`, in which case it raises the
// flag and records `code` in the device status word.
template <bool kCl = false>
__device__ __forceinline__ bool fa_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns,
                                        unsigned int code) {
    if (fa_poll<kCl>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (fa_poll<kCl>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(&g_fa_status, code);
            return false;
        }
    }
}

// Same, with the verdict made uniform across the warp.
template <bool kCl = false>
__device__ __forceinline__ bool fa_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns, unsigned int code) {
    const bool ok = fa_wait<kCl>(bar, parity, abort_flag, limit_ns, code);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait used while tearing down after an abort: ignores the flag.
template <bool kCl = false>
__device__ __forceinline__ bool fa_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (fa_poll<kCl>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (fa_poll<kCl>(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(&g_fa_status, kStatusDrain);
            return false;
        }
    }
}

// The reference hand-over between the two softmax groups, one 64-bit shared-memory
// word per row: the step the reference belongs to in the high half, its bits in the
// low half.  A naturally aligned 64-bit store is single-copy atomic, so a reader that
// sees the step it expects also sees that step's reference, with no barrier between.
__device__ __forceinline__ void xref_put(uint32_t addr, uint32_t step, float m) {
    const uint64_t v = ((uint64_t)step << 32) | (uint64_t)__float_as_uint(m);
    asm volatile("st.volatile.shared.b64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// `x`, recomputed where it is used (an opaque copy the compiler cannot hoist out
// of a loop and hold in a register across it)
__device__ __forceinline__ uint32_t fa_here(uint32_t x) {
    uint32_t y;
    asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint64_t xref_ld(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.volatile.shared.b64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

// Bounded wait for step `step`'s reference in the slot at `addr` (watchdog as fa_wait).
__device__ __forceinline__ bool xref_get(uint32_t addr, uint32_t step, float& m, volatile int* abort_flag,
                                         uint64_t limit_ns) {
    uint64_t v = xref_ld(addr);
    if (__builtin_expect((uint32_t)(v >> 32) != step, 0)) {
        // elapsed SM cycles in 32 bits against the limit at 2 cycles per ns (at most 2^31)
        const uint32_t c0 = (uint32_t)clock();
        const uint32_t lim = limit_ns >= (1ull << 30) ? (1u << 31) : (uint32_t)limit_ns * 2u;
        for (;;) {
            v = xref_ld(addr);
            if ((uint32_t)(v >> 32) == step) break;
            if (*abort_flag) return false;
            if ((uint32_t)clock() - c0 > lim) {
                *abort_flag = 1;
                atomicOr(&g_fa_status, kStatusSoftmaxWaitX);
                return false;
            }
        }
    }
    m = __uint_as_float((uint32_t)v);
    return true;
}

// Exponentials of NE keys of a row against the reference -neg_m (base 2):
// P packed to bf16 pairs, and the fp32 sum of the unrounded values.
template <int NE>
__device__ __forceinline__ void exp_row_tile(const float (&s)[NE], float c2, float neg_m, uint32_t (&pk)[NE / 2],
                                             float& sum_f32) {
    const uint64_t c2x2 = f32x2_pack(c2, c2), negm2 = f32x2_pack(neg_m, neg_m);
    uint64_t r32[2] = {0ull, 0ull};  // packed (even, odd) fp32 partial sums
#pragma unroll
    for (int i = 0; i < NE / 2; ++i) {
        float x0, x1;
        f32x2_unpack(ffma2(f32x2_pack(s[2 * i], s[2 * i + 1]), c2x2, negm2), x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        pk[i] = pack_bf16x2(p0, p1);
        r32[i & 1] = fadd2(r32[i & 1], f32x2_pack(p0, p1));
    }
    float e0, e1, o0, o1;
    f32x2_unpack(r32[0], e0, o0);
    f32x2_unpack(r32[1], e1, o1);
    sum_f32 = (e0 + o0) + (e1 + o1);
}

// One unit of work: query tile qt of head bh against key tiles j0 .. j0+n_kv-1.
struct TileWork {
    int qt, bh, j0, n_kv;
};

// Persistent schedule.  The query tiles of a head are paired, (n_tiles-1-i, i):
// a long causal tile with a short one, so that every pair costs about the
// same; pairs are numbered head-major (the CTAs busy at any moment share the
// keys and values of a few heads in L2).  Each CTA first takes static_rounds
// pairs statically (pairs blockIdx.x, blockIdx.x + gridDim.x, ...; the host
// deals out every full round), which keeps a pair's two tiles, and the shared
// keys and values, on one SM.  The remaining pairs are split into single tiles
// that CTAs take one at a time from a global counter -- first all their long
// tiles, then the short ones -- so that CTAs that ran faster do more of the
// tail.
//
// A CTA pair schedules units of two adjacent query tiles (2u in the leading
// CTA, 2u + 1 in its peer) the same way, the pair counting as one worker.
__host__ __device__ inline int schedule_units(const FaParams& p, bool pair) {
    return pair ? (p.n_tiles + 1) / 2 : p.n_tiles;
}

__host__ __device__ inline long long persistent_pairs(const FaParams& p, bool pair = false) {
    return (long long)p.BH * ((schedule_units(p, pair) + 1) / 2);
}

__device__ inline void pair_tiles(int n_units, long long pair, int& bh, int& qt_long, int& qt_short) {
    const int per_head = (n_units + 1) / 2;
    bh = (int)(pair / per_head);
    const int i = (int)(pair % per_head);
    qt_long = n_units - 1 - i;
    qt_short = i;  // equal to qt_long for the middle unit of an odd count
}

// Document boundaries by binary search over non-decreasing ids (indices stay
// within [0, N) whatever the ids hold): the first and the last position of the
// document of position i.
__device__ inline int doc_first(const int* d, int i) {
    const int v = __ldg(d + i);
    int lo = 0, hi = i;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(d + mid) < v) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__device__ inline int doc_last(const int* d, int i, int N) {
    const int v = __ldg(d + i);
    int lo = i, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(d + mid) > v) hi = mid - 1; else lo = mid;
    }
    return lo;
}

// The key tiles query tile qt of head bh has to visit.  The first and last
// visible key of a row never decrease with the row (windows slide, documents
// are contiguous), so the tile's range runs from its first row's first key to
// its last row's last key; tiles outside it are never visited ("Online
// Softmax: Tiling Across a Reduction", causal section: masks become block-level
// skip decisions).
template <bool kMask>
__device__ inline void tile_work(const FaParams& p, int bh, int qt, TileWork& w) {
    w.qt = qt;
    w.bh = bh;
    if constexpr (!kMask) {  // full or causal attention
        w.j0 = 0;
        w.n_kv = p.causal ? min(qt + 1, p.n_tiles) : p.n_tiles;
        return;
    }
    const int r0 = qt * kBlockM, r1 = min(r0 + kBlockM, p.N) - 1;
    int lo = 0, hi = p.N - 1;
    if (p.window_left >= 0) lo = max(lo, r0 - p.window_left);
    if (p.window_right >= 0) hi = min(hi, r1 + p.window_right);
    if (p.doc) {
        const int* d = p.doc + (size_t)(bh / p.H) * (size_t)p.N;
        lo = max(lo, doc_first(d, r0));
        hi = min(hi, doc_last(d, r1, p.N));
    }
    w.j0 = lo / kBlockN;
    w.n_kv = hi >= lo ? hi / kBlockN - w.j0 + 1 : 0;
}

// The sequence of tiles one CTA processes; every role of the CTA walks its own
// copy and sees the same tiles in the same order.
//  * one-shot launch: the single tile (blockIdx.x from the last, longest
//    causal tile down; blockIdx.y = head), restricted to the key split
//    blockIdx.z when kSplit;
//  * persistent launch: the producer warp chooses the tiles (choose()),
//    works out their key ranges (tile_work()) and posts both in a
//    shared-memory ring (produce()); the other roles read them from there
//    (next()).  A negative entry ends the sequence.
//  * CTA pair: the leading CTA's producer chooses each unit and posts it in
//    both CTAs' rings; every reader of either CTA releases the slot on the
//    leading CTA's barrier.  Each CTA reads the unit as its own query tile.
//  * kTwo: units of two adjacent query tiles in one CTA (the two-tile kernel);
//    the item names the unit's first tile.
template <bool kSplit, bool kPersistent, bool kMask, bool kPair = false, bool kTwo = false>
struct TileSeq {
    static constexpr bool kUnits2 = kPair || kTwo;  // units of two query tiles
    int n = 0;               // items taken so far
    volatile int* ring;      // item ring in shared memory, 4 ints per entry
    uint32_t bar_full, bar_empty;
    volatile int* abort_flag;
    uint64_t limit;
    uint32_t rank;           // rank in the CTA pair (0 without pairs)
    __device__ TileSeq(volatile int* ring_, uint32_t full, uint32_t empty, volatile int* abort_, uint64_t limit_)
        : ring(ring_), bar_full(full), bar_empty(empty), abort_flag(abort_), limit(limit_),
          rank(kPair ? cluster_ctarank() : 0u) {}

    __device__ bool one_shot(const FaParams& p, TileWork& w) {
        if (n > 0) return false;
        n = 1;
        w.qt = (int)gridDim.x - 1 - (int)blockIdx.x;
        w.bh = (int)blockIdx.y;
        const int n_all = p.causal ? min(w.qt + 1, p.n_tiles) : p.n_tiles;
        w.j0 = 0;
        w.n_kv = n_all;
        if constexpr (kSplit) {
            const int chunk = (n_all + p.n_splits - 1) / p.n_splits;
            w.j0 = (int)blockIdx.z * chunk;
            w.n_kv = max(0, min(n_all - w.j0, chunk));
        }
        return true;
    }

    // producer (one thread): choose the next tile and post it
    int round = 0, sub = 0;  // static phase: pair round and tile within the pair
    __device__ bool choose(const FaParams& p, int& bh, int& qt) {
        const int nu = schedule_units(p, kUnits2);
        const unsigned worker = kPair ? blockIdx.x >> 1 : blockIdx.x;
        const unsigned workers = kPair ? gridDim.x >> 1 : gridDim.x;
        if (p.static_rounds < 0) {
            // one worker per unit: no pairing or counter needed
            if (round++ > 0) return false;
            bh = (int)(worker / (unsigned)nu);
            qt = nu - 1 - (int)(worker % (unsigned)nu);
            return true;
        }
        while (round < p.static_rounds) {
            int ql, qs;
            pair_tiles(nu, (long long)worker + (long long)round * workers, bh, ql, qs);
            if (sub == 0 || (sub == 1 && qs != ql)) {
                qt = sub == 0 ? ql : qs;
                ++sub;
                return true;
            }
            sub = 0;
            ++round;
        }
        const long long first = (long long)p.static_rounds * workers;  // first dynamic pair
        const long long n_dyn = persistent_pairs(p, kUnits2) - first;
        for (;;) {
            const long long k = (long long)atomicAdd(p.queue, 1u);
            if (k >= 2 * n_dyn) return false;
            int ql, qs;
            pair_tiles(nu, first + (k < n_dyn ? k : k - n_dyn), bh, ql, qs);
            if (k < n_dyn) {
                qt = ql;
                return true;
            }
            if (qs != ql) {
                qt = qs;
                return true;
            }
        }
    }

    __device__ bool produce(const FaParams& p, TileWork& w) {
        if constexpr (!kPersistent) {
            return one_shot(p, w);
        } else {
            const int s = n % kItemRing;
            if (n >= kItemRing &&
                !fa_wait<kPair>(bar_empty + 8u * s, (uint32_t)(((n - kItemRing) / kItemRing) & 1), abort_flag, limit,
                                kStatusItemWait))
                return false;
            int bh = 0, qt = 0;
            const bool more = choose(p, bh, qt);
            if (more) {
                if constexpr (kUnits2) {
                    // unit qt: query tiles 2 qt (here) and 2 qt + 1 (peer, or the second
                    // tile of this CTA) against every key tile either of them sees
                    w.qt = 2 * qt;
                    w.bh = bh;
                    w.j0 = 0;
                    w.n_kv = p.causal ? min(2 * qt + 2, p.n_tiles) : p.n_tiles;
                } else {
                    tile_work<kMask>(p, bh, qt, w);  // the key range is worked out once, here
                }
            }
            const int e0 = more ? bh * schedule_units(p, kUnits2) + qt : -1, e1 = more ? w.j0 : 0, e2 = more ? w.n_kv : 0;
            ring[4 * s + 0] = e0;
            ring[4 * s + 1] = e1;
            ring[4 * s + 2] = e2;
            if constexpr (kPair) {
                const uint32_t peer = mapa_shared(smem_u32(const_cast<int*>(ring + 4 * s)), 1);
                st_cluster_u32(peer + 0, (uint32_t)e0);
                st_cluster_u32(peer + 4, (uint32_t)e1);
                st_cluster_u32(peer + 8, (uint32_t)e2);
                mbar_arrive_cluster(mapa_shared(bar_full + 8u * s, 1));  // release: the peer's entry is visible
            }
            mbar_arrive(bar_full + 8u * s);  // release: the ring entry is visible to the readers
            ++n;
            return more;
        }
    }

    // reader: a single thread (kWarp = false) or a whole warp (kWarp = true)
    template <bool kWarp>
    __device__ bool next(const FaParams& p, TileWork& w) {
        if constexpr (!kPersistent) {
            return one_shot(p, w);
        } else {
            const int s = n % kItemRing;
            const uint32_t par = (uint32_t)((n / kItemRing) & 1);
            const bool ok = kWarp ? fa_wait_warp<kPair>(bar_full + 8u * s, par, abort_flag, limit, kStatusItemWait)
                                  : fa_wait<kPair>(bar_full + 8u * s, par, abort_flag, limit, kStatusItemWait);
            if (!ok) return false;
            const int item = ring[4 * s + 0], j0 = ring[4 * s + 1], n_kv = ring[4 * s + 2];
            if constexpr (kWarp) __syncwarp();  // every lane has read the entry
            if (!kWarp || (threadIdx.x & 31) == 0) {
                if constexpr (kPair)
                    mbar_arrive_cluster(mapa_shared(bar_empty + 8u * s, 0));  // the leading CTA's slot
                else
                    mbar_arrive(bar_empty + 8u * s);
            }
            ++n;
            if (item < 0) return false;
            const int nu = schedule_units(p, kUnits2);
            w.qt = kUnits2 ? 2 * (item % nu) + (int)rank : item % nu;
            w.bh = item / nu;
            w.j0 = j0;
            w.n_kv = n_kv;
            return true;
        }
    }
};

// kSplit: each CTA covers only the key tiles of split blockIdx.z and writes the
// partial row state (m, both sums, unnormalised O) instead of O and LSE; a
// merge kernel combines the splits ("5.2 CUDA Online Softmax", section 4.1:
// the (m, d) merge is associative, so partial results combine in any order).
// kPersistent: one CTA per SM walks a list of tiles; the TMA ring, the S and P
// double buffers and all barrier phases continue across tile boundaries, so
// the loads and first S products of the next tile overlap the end of this one.
// kPair: launched in clusters of two CTAs on two SMs that work on adjacent
// query tiles 2u and 2u + 1 against the same key tiles.  Both products are
// two-SM (cta_group::2, M = 256) products issued by the leading CTA (rank 0):
// each CTA loads its own Q tile and half of every K tile (64 keys) and V tile
// (64 of d), and the tensor cores of the pair exchange the halves, so each SM
// moves half the K/V bytes per step.  Each CTA keeps its own S, P and O in its
// own TMEM and runs its own softmax and epilogue; the barriers the leading
// CTA's issuers wait on collect arrivals from both CTAs, and the commits of
// the products arrive on both CTAs' barriers.  tm_k's box is 64 rows.
template <int D, int NK, int NV, bool kSplit, bool kPersistent, bool kMask = false, bool kPair = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const FaParams p) {
    static_assert(!kPair || (kPersistent && !kSplit && !kMask), "CTA pairs run the persistent unmasked kernel");
    using L = FwdSmem<D, NK, NV, kSplit, kPair>;
    using Seq = TileSeq<kSplit, kPersistent, kMask, kPair>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
    volatile int* items = reinterpret_cast<volatile int*>(smem + L::kOffItems);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = (int)(threadIdx.x & 31);
    const uint64_t limit = p.watchdog_ns;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0: this CTA issues the products
    // Arrivals the leading CTA's issuers wait for, on its barrier i (through its
    // shared::cluster address, looked up once).  These barriers, the ones the
    // products' commits arrive on and the waits on all of them are CTA-scope
    // operations even across the pair: what they order is tensor-memory and
    // operand traffic of the tcgen05 products, which the tcgen05 fences around
    // them order (a cluster-scope release or acquire on every step measured
    // 1.6x slower).  Data passed through shared memory between the CTAs (the
    // work-item ring) uses cluster-scope release and acquire.
    const uint32_t lead_bar0 = kPair ? mapa_shared(bar(0), 0) : 0u;
    auto arrive_lead = [&](int i) {
        if constexpr (kPair)
            mbar_arrive_remote(lead_bar0 + 8u * (uint32_t)i);
        else
            mbar_arrive(bar(i));
    };
    // commit of this thread's products to the barrier in both CTAs of a pair
    auto commit_all = [&](uint32_t b) {
        if constexpr (kPair)
            tc_commit_pair(b, (uint16_t)3);
        else
            tc_commit(b);
    };
    constexpr int kArrivers = kPair ? 2 : 1;  // CTAs whose warps arrive on the issuers' barriers

    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int qb = 0; qb < L::kQBufs; ++qb) {
            mbar_init(bar(L::kBarQ + qb), 1);
            mbar_init(bar(L::kBarQFree + qb), 1);
        }
#pragma unroll
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(L::kBarKFull + s), 1);
            mbar_init(bar(L::kBarKEmpty + s), 1);
        }
#pragma unroll
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(L::kBarVFull + s), 1);
            mbar_init(bar(L::kBarVEmpty + s), 1);
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::kBarSFull + b), 1);
            mbar_init(bar(L::kBarSFree + b), kArrivers * kSoftmaxWarps / 2);  // one arrival per warp of group b
            mbar_init(bar(L::kBarPFull + b), kArrivers * kSoftmaxWarps / 2);
            mbar_init(bar(L::kBarPVDone + b), 1);
            mbar_init(bar(L::kBarDrain + b), 1);
        }
        mbar_init(bar(L::kBarOFinal), 1);
        mbar_init(bar(L::kBarOFree), kArrivers * kSoftmaxWarps);
#pragma unroll
        for (int i = 0; i < 4; ++i) mbar_init(bar(L::kBarXSum + i), 2);
#pragma unroll
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(bar(L::kBarItemFull + i), 1);
            // a pair's peer reads with its producer warp and softmax warps (no issuers)
            mbar_init(bar(L::kBarItemEmpty + i), kItemReaders + (kPair ? kItemReaders - 1 : 0));
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
    }
    {
        // reference hand-over slots: no step yet
        volatile uint64_t* slots = reinterpret_cast<volatile uint64_t*>(smem + L::kOffXchg);
        for (uint32_t i = threadIdx.x; i < 2u * kBlockM; i += blockDim.x) slots[i] = ~0ull;
    }
    if constexpr (L::kTcSum) {
        // the tile of ones (bf16 1.0 pairs) that the row-sum products read
        uint32_t* ones = reinterpret_cast<uint32_t*>(smem + L::kOffOnes);
        for (uint32_t i = threadIdx.x; i < L::kOnesBytes / 4u; i += blockDim.x) ones[i] = 0x3F803F80u;
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    // a pair: the peer's barriers are initialised before anything arrives on them
    if constexpr (kPair) cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer.  Per tile t: K_0; Q into buffer t % 2 once tile t-2's
        // last S product has finished; K_1; then V_j and K_{j+2}: the order in
        // which the two MMA issuers consume them.
        // ------------------------------------------------------------------
        if (lane == 0) {
            int nk = 0, nv = 0, nq = 0;  // loads issued, over the whole tile sequence
            // A pair's loads all complete on the leading CTA's barriers, which its
            // producer arms with both CTAs' bytes.
            const bool arm = !kPair || rank == 0;
            auto full_bar = [&](uint32_t b) -> uint32_t { return kPair ? mapa_shared(b, 0) : b; };
            auto tma = [&](uint32_t dst, const CUtensorMap* m, uint32_t b, int c0, int c1, int c2) {
                if constexpr (kPair)
                    tma_load_3d_pair(dst, m, b, c0, c1, c2);
                else
                    tma_load_3d(dst, m, b, c0, c1, c2);
            };
            auto load_k = [&](const TileWork& w, int j) -> bool {
                const int s = nk % NK;
                const uint32_t r = (uint32_t)(nk / NK);
                const uint32_t empty = bar((L::kKEmptyIsSFull ? L::kBarSFull : L::kBarKEmpty) + s);
                if (!fa_wait(empty, (r & 1u) ^ 1u, abort_flag, limit, kStatusLoadWait)) return false;
                if (arm) mbar_arrive_expect_tx(bar(L::kBarKFull + s), kArrivers * L::kKBytes);
                const uint32_t fb = full_bar(bar(L::kBarKFull + s));
                // a pair: keys 64 rank .. 64 rank + 63 of the tile
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma(sbase + L::kOffK + s * L::kKBytes + c * L::kKChunkBytes, &tm_k, fb, c * 64,
                        (w.j0 + j) * kBlockN + (int)rank * (kBlockN / 2), w.bh);
                ++nk;
                return true;
            };
            auto load_v = [&](const TileWork& w, int j) -> bool {
                const int s = nv % NV;
                const uint32_t r = (uint32_t)(nv / NV);
                if (!fa_wait(bar(L::kBarVEmpty + s), (r & 1u) ^ 1u, abort_flag, limit, kStatusLoadWait))
                    return false;
                if (arm) mbar_arrive_expect_tx(bar(L::kBarVFull + s), kArrivers * L::kVBytes);
                const uint32_t fb = full_bar(bar(L::kBarVFull + s));
                if constexpr (kPair) {
                    // columns 64 rank .. 64 rank + 63 of d
                    tma(sbase + L::kOffV + s * L::kVBytes, &tm_v, fb, (int)rank * 64, (w.j0 + j) * kBlockN, w.bh);
                } else {
#pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
                        tma(sbase + L::kOffV + s * L::kVBytes + c * kChunkBytes, &tm_v, fb, c * 64,
                            (w.j0 + j) * kBlockN, w.bh);
                }
                ++nv;
                return true;
            };
            Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
            TileWork w;
            bool ok = true;
            // the leading CTA (or a lone CTA) chooses the work; a peer reads it
            while (ok && (arm ? seq.produce(p, w) : seq.template next<false>(p, w))) {
                if (w.n_kv == 0) continue;
                const int qb = nq % L::kQBufs;
                ok = load_k(w, 0);
                if (ok && nq >= L::kQBufs)
                    ok = fa_wait(bar(L::kBarQFree + qb), (uint32_t)(((nq - L::kQBufs) / L::kQBufs) & 1),
                                        abort_flag, limit, kStatusLoadWait);
                if (ok) {
                    if (arm) mbar_arrive_expect_tx(bar(L::kBarQ + qb), kArrivers * L::kTileBytes);
                    const uint32_t fb = full_bar(bar(L::kBarQ + qb));
                    // a pair's peer past the last tile loads a real tile; its rows are never stored
                    const int qrow = min(w.qt, p.n_tiles - 1) * kBlockM;
#pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
                        tma(sbase + L::kOffQ + qb * L::kTileBytes + c * kChunkBytes, &tm_q, fb, c * 64, qrow, w.bh);
                    ++nq;
                }
                if (ok && w.n_kv > 1) ok = load_k(w, 1);
                for (int j = 0; ok && j < w.n_kv; ++j) {
                    ok = load_v(w, j);
                    if (ok && j + 2 < w.n_kv) ok = load_k(w, j + 2);
                }
            }
            if (arm) {
                // let every copy already issued land before the CTA exits: after an
                // abort some are never consumed (in a normal run these waits succeed
                // at once).  A pair's peer cannot see its own copies land; they
                // complete on these barriers too.
                for (int qb = 0; qb < L::kQBufs; ++qb)
                    if (nq > qb)
                        fa_wait_drain(bar(L::kBarQ + qb), (uint32_t)(((nq - 1 - qb) / L::kQBufs) & 1), limit);
                for (int s = 0; s < NK; ++s)
                    if (nk > s) fa_wait_drain(bar(L::kBarKFull + s), (uint32_t)(((nk - 1 - s) / NK) & 1), limit);
                for (int s = 0; s < NV; ++s)
                    if (nv > s) fa_wait_drain(bar(L::kBarVFull + s), (uint32_t)(((nv - 1 - s) / NV) & 1), limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // S issuer: S_g = Q K_g^T into buffer g % 2 (g counts steps over the
        // whole tile sequence) once K_g has landed and the softmax has read
        // S_{g-2} out of that buffer.  After a tile's last S: commit QFree of
        // its Q buffer.
        // ------------------------------------------------------------------
        if (!kPair || rank == 0) {  // a pair's peer only allocates TMEM here
            // a pair: M = 256 (this CTA's 128 query rows, then the peer's)
            constexpr uint32_t kIdescS = idesc_bf16_f32(kPair ? 2 * kBlockM : kBlockM, kBlockN, false, false);
            int g = 0, t = 0;
            Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
            TileWork w;
            bool ok = true;
            while (ok && seq.template next<true>(p, w)) {
                if (w.n_kv == 0) continue;
                const int qb = t % L::kQBufs;
                const uint32_t qa = sbase + L::kOffQ + (uint32_t)qb * L::kTileBytes;
                ok = fa_wait_warp(bar(L::kBarQ + qb), (uint32_t)((t / L::kQBufs) & 1), abort_flag, limit,
                                         kStatusMmaWaitQ);
                if (p.withhold_s) break;
                for (int j = 0; ok && j < w.n_kv; ++j, ++g) {
                    const int b = g & 1;
                    const int ks = g % NK;
                    if (g >= 2)
                        ok = fa_wait_warp(bar(L::kBarSFree + b), (uint32_t)(((g - 2) >> 1) & 1), abort_flag,
                                                 limit, kStatusMmaWaitSFree);
                    ok = ok && fa_wait_warp(bar(L::kBarKFull + ks), (uint32_t)((g / NK) & 1), abort_flag, limit,
                                                   kStatusMmaWaitK);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t ka = sbase + L::kOffK + (uint32_t)ks * L::kKBytes;
                    // descriptors built once; K step kk moves the start address (16-byte
                    // units, the low field) by its byte offset
                    const uint64_t qd = sdesc_sw128(qa, 16, 1024), kd = sdesc_sw128(ka, 16, 1024);
                    if (elect_one_sync()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t in_row = (uint32_t)(kk & 3) * 32u;
                            const uint32_t offq = ((uint32_t)(kk >> 2) * kChunkBytes + in_row) >> 4;
                            const uint32_t offk = ((uint32_t)(kk >> 2) * L::kKChunkBytes + in_row) >> 4;
                            if constexpr (kPair)
                                mma_ss_pair(tmem + L::col_s(b), sdesc_add_lo(qd, offq), sdesc_add_lo(kd, offk), kIdescS,
                                            kk > 0 ? 1u : 0u);
                            else
                                mma_ss(tmem + L::col_s(b), sdesc_add_lo(qd, offq), sdesc_add_lo(kd, offk), kIdescS,
                                       kk > 0 ? 1u : 0u);
                        }
                        commit_all(bar(L::kBarSFull + b));
                        if constexpr (!L::kKEmptyIsSFull) commit_all(bar(L::kBarKEmpty + ks));
                    }
                    __syncwarp();
                }
                if (ok && elect_one_sync()) commit_all(bar(L::kBarQFree + qb));  // the Q buffer may be refilled once these finish
                __syncwarp();
                ++t;
            }
            if (elect_one_sync()) {
                // every MMA must finish before TMEM is released
                if constexpr (kPair)
                    tc_commit_pair(bar(L::kBarDrain + 0), (uint16_t)1);
                else
                    tc_commit(bar(L::kBarDrain + 0));
                fa_wait_drain(bar(L::kBarDrain + 0), 0, limit);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------------
        // P V issuer: O += P_g V_g once P_g is in TMEM and V_g has landed; the
        // first product of a tile (which overwrites O) also waits until the
        // softmax warps have read the previous tile's O out of TMEM.
        // ------------------------------------------------------------------
        if (!kPair || rank == 0) {
            // a pair: M = 256, and each CTA's V stage holds 64 of the N = d columns
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kPair ? 2 * kBlockM : kBlockM, D + L::kSumCols, false, true);
            int g = 0, t = 0;
            Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
            TileWork w;
            bool ok = true;
            while (ok && seq.template next<true>(p, w)) {
                if (w.n_kv == 0) continue;
                for (int j = 0; ok && j < w.n_kv; ++j, ++g) {
                    const int b = g & 1;
                    const int vs = g % NV;
                    ok = fa_wait_warp(bar(L::kBarPFull + b), (uint32_t)((g >> 1) & 1), abort_flag, limit,
                                             kStatusMmaWaitP) &&
                         fa_wait_warp(bar(L::kBarVFull + vs), (uint32_t)((g / NV) & 1), abort_flag, limit,
                                             kStatusMmaWaitV);
                    if (ok && j == 0 && t > 0)
                        ok = fa_wait_warp(bar(L::kBarOFree), (uint32_t)((t - 1) & 1), abort_flag, limit,
                                                 kStatusMmaWaitP);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t va = sbase + L::kOffV + (uint32_t)vs * L::kVBytes;
                    // second 64-column block of B: the next chunk of V (d = 128), or the
                    // ones tile for the row sums (d = 64), whose leading-byte offset from
                    // key rows 16 kk .. 16 kk + 15 shrinks as those rows advance (a pair:
                    // each CTA's 64 columns are a single block)
                    const uint64_t vd0 = sdesc_sw128(va, L::kTcSum ? sbase + L::kOffOnes - va : kChunkBytes, 1024);
                    constexpr uint32_t kStepDesc = L::kTcSum ? 128u - (128u << 16) : 128u;  // 2048 bytes per K step
                    if (elect_one_sync()) {
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk) {
                            if constexpr (kPair)
                                mma_ts_pair(tmem + L::kColO, tmem + L::col_p(b) + (uint32_t)kk * 8u,
                                            sdesc_add_lo(vd0, (uint32_t)kk * kStepDesc), kIdescPV,
                                            (j > 0 || kk > 0) ? 1u : 0u);
                            else
                                mma_ts(tmem + L::kColO, tmem + L::col_p(b) + (uint32_t)kk * 8u,
                                       sdesc_add_lo(vd0, (uint32_t)kk * kStepDesc), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        commit_all(bar(L::kBarVEmpty + vs));
                        commit_all(bar(L::kBarPVDone + b));
                        if (j + 1 == w.n_kv) commit_all(bar(L::kBarOFinal));
                    }
                    __syncwarp();
                }
                ++t;
            }
            if (elect_one_sync()) {
                if constexpr (kPair)
                    tc_commit_pair(bar(L::kBarDrain + 1), (uint16_t)1);
                else
                    tc_commit(bar(L::kBarDrain + 1));
                fa_wait_drain(bar(L::kBarDrain + 1), 0, limit);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------------
        // Softmax / correction / epilogue.  Thread = one query row (TMEM lane
        // `row`).  The two warpgroups take alternate steps: group wg handles
        // every step g with g % 2 == wg, all 128 keys of the row.  The online
        // recurrence only threads the reference maximum from one step to the
        // next, and that is handed over through shared memory right after the
        // row maximum is known, so one group's exponentials overlap the other
        // group's TMEM load and maximum of the following step.
        // ------------------------------------------------------------------
        const int quarter = warp & 3;    // TMEM lane quarter this warp may access
        const int wg = (warp - 4) >> 2;  // warps 4-7: even steps, warps 8-11: odd steps
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        // this row's hand-over slot of group gr (group 1's is 8 * 128 bytes after group 0's)
        auto xslot = [&](int gr) -> uint32_t {
            return fa_here(sbase) + L::kOffXchg + (uint32_t)(gr * kBlockM + row) * 8u;
        };
        float* xsum = reinterpret_cast<float*>(smem + L::kOffXSum);  // [2 tile parities][2 groups][3][128 rows]
        constexpr int kOCols = D / 2;  // O columns this thread stores in the epilogue
        const float c2 = p.scale_log2;
        int g = 0, t = 0;  // steps and non-empty tiles so far
        bool ok = true;
        bool in_tile = false;  // a tile has been started and its rows not yet written
        int q_idx = 0;
        bool valid = false;
        Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
        TileWork w;
        while (ok && seq.template next<true>(p, w)) {
            q_idx = w.qt * kBlockM + row;
            valid = q_idx < p.N;
            if constexpr (kSplit) {
                if (w.n_kv == 0) {
                    // no key of this split is visible: an empty partial state
                    if (valid) {
                        const size_t r = ((size_t)blockIdx.z * gridDim.y + (size_t)w.bh) * (size_t)p.N + (size_t)q_idx;
                        float4* dst = reinterpret_cast<float4*>(p.ws_o + r * D + wg * kOCols);
#pragma unroll
                        for (int u = 0; u < kOCols / 4; ++u) dst[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (wg == 0) {
                            p.ws_m[r] = -INFINITY;
                            p.ws_lbf[r] = 0.f;
                            p.ws_l32[r] = 0.f;
                        }
                    }
                    continue;
                }
            }
            // this row's visible keys, [row_lo, row_hi] (sequence positions): the window
            // intersected with the row's own document, which is one contiguous run because
            // the ids are non-decreasing (found once per tile, not per step); rows past N
            // see every key (they are never stored)
            int row_lo = 0, row_hi = p.N - 1;
            if (kMask && valid) {
                if (p.window_left >= 0) row_lo = max(0, q_idx - p.window_left);
                if (p.window_right >= 0) row_hi = min(row_hi, q_idx + p.window_right);
                if (p.doc) {
                    const int* dseq = p.doc + (size_t)(w.bh / p.H) * (size_t)p.N;
                    row_lo = max(row_lo, doc_first(dseq, q_idx));
                    row_hi = min(row_hi, doc_last(dseq, q_idx, p.N));
                }
            }
            in_tile = true;
            float m_own = -INFINITY;  // reference this group's sums are relative to (base-2 units)
            float l_run = 0.f;        // this group's sum that normalises O (d = 128; d = 64 reads TMEM)
            float l32_run = 0.f;      // this group's fp32 sum of 2^(t - m_own): gives LSE
            for (int j = 0; j < w.n_kv; ++j, ++g) {
                if ((g & 1) != wg) continue;
                const int b = wg;  // S and P buffer of this step
                if (!fa_wait_warp(bar(L::kBarSFull + b), (uint32_t)((g >> 1) & 1), abort_flag, limit,
                                         kStatusSoftmaxWaitS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                float s[kBlockN];
                float ld_max;  // the maximum of the 128 loaded scores, from the load itself
                {
                    uint32_t r[kBlockN];
                    tmem_ld128_max_wait(t_lane + L::col_s(b), r, ld_max);
#pragma unroll
                    for (int i = 0; i < kBlockN; ++i) s[i] = __uint_as_float(r[i]);
                }
                bool masked = false;  // some key of this row is masked in this tile
                // S_g is in registers: the buffer may take S_{g+2}
                tc_fence_before_sync();
                __syncwarp();
                if (elect_one_sync()) arrive_lead(L::kBarSFree + b);
                if constexpr (!kMask) {
                    // mask keys past the diagonal (causal) and past the end of the sequence
                    // (a pair's leading CTA also sees the key tile after its diagonal)
                    int lim = p.N - 1 - (w.j0 + j) * kBlockN;
                    if (p.causal && w.j0 + j >= w.qt) lim = min(lim, row + (w.qt - w.j0 - j) * kBlockN);
                    if (__builtin_expect(lim < kBlockN - 1, 0)) {
                        masked = true;
#pragma unroll
                        for (int i = 0; i < kBlockN; ++i) s[i] = (i > lim) ? -INFINITY : s[i];
                    }
                } else {
                    // keys this row may see in this tile: [first, last] (tile-relative);
                    // past the end of the sequence, outside the window (causal: past the
                    // diagonal) and outside the row's document are masked
                    const int k0 = (w.j0 + j) * kBlockN;
                    const int first = row_lo - k0;
                    const int last = min(row_hi, p.N - 1) - k0;
                    if (__builtin_expect(first > 0 || last < kBlockN - 1, 0)) {
                        masked = true;
#pragma unroll
                        for (int i = 0; i < kBlockN; ++i) s[i] = (i < first || i > last) ? -INFINITY : s[i];
                    }
                }
                // the row maximum: from the load, unless a key of the row is masked here
                float row_max = ld_max;
                if (__builtin_expect(__any_sync(0xffffffffu, masked), 0)) {
                    float mx[4] = {fmax3(s[0], s[1], s[2]), fmax3(s[3], s[4], s[5]), fmax3(s[6], s[7], s[8]),
                                   fmax3(s[9], s[10], s[11])};
#pragma unroll
                    for (int i = 12; i + 8 <= kBlockN; i += 8) {
                        mx[0] = fmax3(mx[0], s[i + 0], s[i + 1]);
                        mx[1] = fmax3(mx[1], s[i + 2], s[i + 3]);
                        mx[2] = fmax3(mx[2], s[i + 4], s[i + 5]);
                        mx[3] = fmax3(mx[3], s[i + 6], s[i + 7]);
                    }
                    mx[0] = fmax3(mx[0], s[124], s[125]);
                    mx[1] = fmax3(mx[1], s[126], s[127]);
                    if (masked) row_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                }
                // reference after step g-1, handed over by the other group (every step
                // after the first waits for it, so the hand-overs stay in lock step; a new
                // tile starts from -inf and ignores the value)
                float m_prev = -INFINITY;
                if (g > 0) {
                    const uint32_t other = xslot(wg ^ 1);
                    uint64_t xv = xref_ld(other);
                    if (__builtin_expect(__any_sync(0xffffffffu, (uint32_t)(xv >> 32) != (uint32_t)(g - 1)), 0)) {
                        float v = -INFINITY;
                        if (!__all_sync(0xffffffffu, xref_get(other, (uint32_t)(g - 1), v, abort_flag, limit))) {
                            ok = false;
                            break;
                        }
                        xv = (uint64_t)__float_as_uint(v);
                    }
                    if (j > 0) m_prev = __uint_as_float((uint32_t)xv);
                }
                // scale > 0, so max(s) * c2 == max(s * c2); the reference moves only
                // when the max grew past it by more than the threshold (always on
                // the first visible tile: -inf + 64 = -inf < any finite max)
                const float m_cand = fmaxf(m_prev, row_max * c2);
                const bool move = m_cand > m_prev + kRescaleThreshold;
                const float m_new = move ? m_cand : m_prev;
                xref_put(xslot(wg), (uint32_t)g, m_new);
                const bool any_move = __any_sync(0xffffffffu, move);
                // bring this group's sums to the new reference (its last step may be
                // two or more moves back)
                const float a_l = (m_own == m_new) ? 1.f : ex2_approx(m_own - m_new);  // 2^-inf = 0
                m_own = m_new;
                // a row with nothing visible yet keeps m = -inf and uses 0, so that its
                // -inf scores give 0 rather than NaN
                uint32_t pk[kBlockN / 2];
                float sum_f32;
                const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
                exp_row_tile<kBlockN>(s, c2, neg_m, pk, sum_f32);
                if constexpr (!L::kTcSum) {
                    // the sum that normalises O: the fp32 sum plus the bf16 rounding of
                    // this tile's largest weight, recomputed from the row maximum with
                    // the very operations the loop applied to it (fma, ex2, RN to bf16)
                    const float p_max = ex2_approx(fmaf(row_max, c2, neg_m));
                    const float r_max = __bfloat162float(__float2bfloat16_rn(p_max)) - p_max;
                    l_run = l_run * a_l + (sum_f32 + r_max);
                }
                l32_run = l32_run * a_l + sum_f32;
                if (g >= 2) {
                    // P buffer b last fed P_{g-2} V_{g-2}: that product must have read it
                    if (!fa_wait_warp(bar(L::kBarPVDone + b), (uint32_t)(((g - 2) >> 1) & 1), abort_flag, limit,
                                             kStatusSoftmaxWaitPV)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
                tmem_st64(t_lane + L::col_p(b), pk);
                if (__builtin_expect(j > 0 && any_move, 0)) {
                    // O must hold P_{g-1} V_{g-1} before it is rescaled; one load and
                    // one store of the whole row (P is already out of the registers)
                    if (!fa_wait_warp(bar(L::kBarPVDone + (b ^ 1)), (uint32_t)(((g - 1) >> 1) & 1), abort_flag,
                                             limit, kStatusSoftmaxWaitPV)) {
                        tmem_st_wait();  // the P store must complete before the CTA tears down
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const float a_o = move ? ex2_approx(m_prev - m_new) : 1.f;
                    uint32_t r[D];
                    if constexpr (D == 128)
                        tmem_ld128_wait(t_lane + L::kColO, r);
                    else
                        tmem_ld64_wait(t_lane + L::kColO, r);
                    {
                        const uint64_t a2 = f32x2_pack(a_o, a_o);
#pragma unroll
                        for (int i = 0; i < D / 2; ++i) {
                            float x0, x1;
                            f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), a2), x0,
                                         x1);
                            r[2 * i] = __float_as_uint(x0);
                            r[2 * i + 1] = __float_as_uint(x1);
                        }
                    }
                    if constexpr (D == 128)
                        tmem_st128(t_lane + L::kColO, r);
                    else
                        tmem_st64(t_lane + L::kColO, r);
                    if constexpr (L::kTcSum) {
                        // the row sums move to the new reference with O
                        const uint32_t lv = tmem_ld1_wait(t_lane + L::kColL);
                        tmem_st1(t_lane + L::kColL, __float_as_uint(__uint_as_float(lv) * a_o));
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (elect_one_sync()) arrive_lead(L::kBarPFull + b);
            }
            if (!ok) break;
            // whole-row state: both groups' sums brought to the later (larger) reference.
            // Both warps of the pair evaluate the same expression in the same order.
            float m_fin, l_fin, l32_fin;
            {
                float* xs = xsum + (size_t)(t & 1) * (2 * 3 * kBlockM);
                xs[(wg * 3 + 0) * kBlockM + row] = m_own;
                xs[(wg * 3 + 1) * kBlockM + row] = l_run;
                xs[(wg * 3 + 2) * kBlockM + row] = l32_run;
                __syncwarp();
                if (elect_one_sync()) mbar_arrive(bar(L::kBarXSum + quarter));
                ok = fa_wait_warp(bar(L::kBarXSum + quarter), (uint32_t)(t & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitX);
                if (!ok) break;
                const float m0 = xs[0 * kBlockM + row], m1 = xs[3 * kBlockM + row];
                m_fin = fmaxf(m0, m1);
                const float w0 = (m0 == m_fin) ? 1.f : ex2_approx(m0 - m_fin);
                const float w1 = (m1 == m_fin) ? 1.f : ex2_approx(m1 - m_fin);
                l_fin = xs[1 * kBlockM + row] * w0 + xs[4 * kBlockM + row] * w1;
                l32_fin = xs[2 * kBlockM + row] * w0 + xs[5 * kBlockM + row] * w1;
            }
            ok = fa_wait_warp(bar(L::kBarOFinal), (uint32_t)(t & 1), abort_flag, limit, kStatusSoftmaxWaitO);
            if (!ok) break;
            tc_fence_after_sync();
            // the tensor-core row sums are in the reference of the tile's last step,
            // the largest one, m_fin (references only grow), like O
            if constexpr (L::kTcSum) l_fin = __uint_as_float(tmem_ld1_wait(t_lane + L::kColL));
            const uint32_t o_col = t_lane + L::kColO + (uint32_t)(wg * kOCols);
            if constexpr (kSplit) {
                // partial state of this split: unnormalised O and (m, sums) per row.
                // The TMEM loads are warp-collective: every lane runs them, only rows
                // inside the sequence store.
                const size_t r = ((size_t)blockIdx.z * gridDim.y + (size_t)w.bh) * (size_t)p.N + (size_t)q_idx;
                float4* dst = reinterpret_cast<float4*>(p.ws_o + r * D + wg * kOCols);
#pragma unroll
                for (int c = 0; c < kOCols / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32_wait(o_col + 32u * c, v);
                    if (valid) {
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            dst[c * 8 + u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                                         __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
                    }
                }
                if (valid && wg == 0) {
                    p.ws_m[r] = m_fin;
                    p.ws_lbf[r] = l_fin;
                    p.ws_l32[r] = l32_fin;
                }
                // O has been read out of TMEM: the next tile's first P V may overwrite it
                tc_fence_before_sync();
                __syncwarp();
                if (elect_one_sync()) arrive_lead(L::kBarOFree);
            } else {
                // this thread's half row of O, 32 columns at a time, O/l -> bf16 as it
                // arrives (fewer registers live than one load of the half row); the next
                // tile's first P V may overwrite O as soon as it is all in registers
                const float inv_l = l_fin > 0.f ? 1.f / l_fin : 0.f;
                uint32_t wv[kOCols / 2];
#pragma unroll
                for (int h = 0; h < kOCols / 32; ++h) {
                    uint32_t r[32];
                    tmem_ld32_wait(o_col + 32u * (uint32_t)h, r);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        wv[16 * h + i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (elect_one_sync()) arrive_lead(L::kBarOFree);
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) +
                                      ((size_t)w.bh * (size_t)p.N + (size_t)q_idx) * D + wg * kOCols;
                if constexpr (L::kOStaged) {
                    // Through shared memory and the TMA unit, so that the warp goes on while
                    // the tile is written (row stores from registers kept the softmax warps
                    // ~1700 cycles a tile): two boxes of 16 rows x 64 columns per warp, each
                    // staged in the warp's 2 KB with the 128-byte swizzle (16-byte chunk u of
                    // row r at chunk u ^ (r % 8)); rows past N are dropped by the tensor map.
                    // The elected lane issues the stores and waits for its own earlier ones.
                    const uint32_t wst = fa_here(sbase) + L::kOffOStage + (uint32_t)(warp - 4) * L::kOStageWarpBytes;
                    const int row0 = w.qt * kBlockM + quarter * 32;  // sequence position of lane 0's row
#pragma unroll
                    for (int pass = 0; pass < 2; ++pass) {
                        // the staging area has been read by the previous box's store
                        if (elect_one_sync()) bulk_wait_read_all();
                        __syncwarp();
                        if ((lane >> 4) == pass) {
                            const uint32_t rowa = wst + (uint32_t)(lane & 15) * 128u;
#pragma unroll
                            for (int u = 0; u < kOCols / 8; ++u)
                                st_shared_v4(rowa + (uint32_t)((u ^ (lane & 7)) * 16), wv[4 * u], wv[4 * u + 1],
                                             wv[4 * u + 2], wv[4 * u + 3]);
                            fence_proxy_async_smem();  // visible to the TMA unit
                        }
                        __syncwarp();
                        if (elect_one_sync()) {
                            tma_store_3d(&tm_o, wst, wg * kOCols, row0 + 16 * pass, w.bh);
                            bulk_commit_group();
                        }
                        __syncwarp();
                    }
                } else if (valid) {
                    // straight from registers to the half row: 32-byte stores when O is
                    // 32-byte aligned (full L2 sectors), else 16-byte
                    if ((reinterpret_cast<uintptr_t>(p.o) & 31u) == 0) {
#pragma unroll
                        for (int u = 0; u < kOCols / 16; ++u) st_global_v8(orow + 16 * u, wv + 8 * u);
                    } else {
                        uint4* o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll
                        for (int u = 0; u < kOCols / 8; ++u)
                            o4[u] = make_uint4(wv[4 * u], wv[4 * u + 1], wv[4 * u + 2], wv[4 * u + 3]);
                    }
                }
                if (valid && wg == 0)
                    p.lse[(size_t)w.bh * (size_t)p.N + (size_t)q_idx] =
                        l32_fin > 0.f ? (m_fin + lg2_approx(l32_fin)) * kLn2 : -INFINITY;
            }
            in_tile = false;
            ++t;
        }
        if (!ok && in_tile && valid) {
            // the watchdog ended a wait inside this tile: its rows are never
            // finished, so their statistic is set to NaN (split-KV: the partial
            // maximum, which the merge turns into a NaN LSE and O)
            const float nan = __int_as_float(0x7fffffff);
            if constexpr (kSplit)
                p.ws_m[((size_t)blockIdx.z * gridDim.y + (size_t)w.bh) * (size_t)p.N + (size_t)q_idx] = nan;
            else
                p.lse[(size_t)w.bh * (size_t)p.N + (size_t)q_idx] = nan;
        }
        if constexpr (L::kOStaged) {
            // this warp's O stores have completed before the CTA exits
            if (elect_one_sync()) bulk_wait_all();
        }
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kPair) {
        // Neither CTA of a pair leaves while the other may still use it.  After an
        // abort the peer's copies may still be in flight with nothing left to wait
        // on: they are given a millisecond (copies take microseconds) first.
        if (threadIdx.x == 0 && *abort_flag) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 1000000ull) {
            }
        }
        cluster_sync_all();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem, kTmemCols);
        else
            tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (kPersistent) {
        // the last CTA out leaves the counter at zero for the next launch
        if (threadIdx.x == 0 && p.queue) {
            __threadfence();
            if (atomicAdd(p.queue + 1, 1u) == gridDim.x - 1) {
                atomicExch(p.queue + 0, 0u);
                atomicExch(p.queue + 1, 0u);
            }
        }
    }
}

// Split-KV merge: one warp per query row combines the partial states of all
// splits with the associative rule m = max_s m_s, w_s = 2^(m_s - m),
// l = sum_s w_s l_s, O = sum_s w_s O_s / l ("5.2 CUDA Online Softmax",
// section 4.1), then writes O (bf16) and LSE.  Splits that saw no key carry
// m = -inf and weigh nothing.
template <int D>
__global__ void __launch_bounds__(256)
    fa_splitkv_merge(const float* __restrict__ ws_o, const float* __restrict__ ws_m, const float* __restrict__ ws_lbf,
                     const float* __restrict__ ws_l32, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                     long long rows, int n_splits) {
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int s = 0; s < n_splits; ++s) m = fmaxf(m, ws_m[(size_t)s * rows + row]);
    float l = 0.f, l32 = 0.f, acc[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const size_t r = (size_t)s * rows + row;
        const float ms = ws_m[r];
        const float w = (ms == -INFINITY) ? 0.f : ex2_approx(ms - m);
        l += w * ws_lbf[r];
        l32 += w * ws_l32[r];
        const float* src = ws_o + r * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) acc[c] += w * src[c * 32 + lane];
    }
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* dst = o + (size_t)row * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) dst[c * 32 + lane] = __float2bfloat16_rn(acc[c] * inv_l);
    if (lane == 0) lse[row] = l32 > 0.f ? (m + lg2_approx(l32)) * kLn2 : -INFINITY;
}

// One CTA waits on a barrier nothing arrives on; the watchdog must end the
// wait, record kStatusSelfTest and let the kernel return normally.
__global__ void fa_watchdog_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_storage;
    const uint32_t b = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_storage = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) fa_wait(b, 0, reinterpret_cast<volatile int*>(&abort_storage), limit_ns, kStatusSelfTest);
    __syncthreads();
}

}  // namespace fa
