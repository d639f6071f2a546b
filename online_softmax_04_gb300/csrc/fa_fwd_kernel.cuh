// fa_fwd_kernel.cuh -- fused attention forward for sm_103a (GB300).
//
// One CTA owns one 128-row query tile of one (batch, head) and streams the
// key/value tiles past it ("Online Softmax: Tiling Across a Reduction", loop
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
//   * S_j = Q K_j^T and O += P_j V_j run on tcgen05.mma (bf16 in, fp32
//     accumulate) with the accumulators in tensor memory (TMEM).  S is double
//     buffered and P has columns of its own, so S_{j+1} is computed while the
//     softmax works on S_j and nothing waits for a product to drain.
//   * Two MMA-issuing warps: one issues the S products as soon as a K tile
//     and an S buffer are free, the other the P V products as soon as P_j is
//     written.  A tcgen05.mma burst keeps its issuing thread busy until the
//     tensor pipe has taken it, so two issuers keep the pipe fed while either
//     one waits on a barrier.
//   * P_j is written back to TMEM as bf16 and consumed from there as the A
//     operand of P V (no shared-memory round trip).
//   * Q, K_j and V_j are brought in by TMA (128-byte swizzle) into rings of
//     shared-memory stages guarded by mbarriers.
//   * Warp roles: warp 0 issues TMA loads, warp 1 owns TMEM and issues the S
//     products, warp 2 issues the P V products, warps 4-7 (one thread per
//     query row) do the softmax, the O rescale on TMEM and the epilogue
//     (O/l -> bf16 -> shared -> TMA store, LSE store).
//   * The reference maximum of a row moves only when the row maximum has
//     grown past it by more than 64 in base-2 units; otherwise the old
//     reference is kept, exponentials up to 2^64 are accumulated in fp32 and
//     the O rescale on TMEM is skipped.  exp(x - m) / sum exp(x - m) does not
//     depend on m, so the result is unchanged.
//   * O is divided by the sum of the bf16-rounded exponentials, the very
//     weights the P V product uses, so O / l is a convex combination of V
//     rows; LSE uses the fp32 sum of the unrounded exponentials.
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
constexpr int kThreads = 256;  // 8 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChunkBytes = 128u * 128u;  // one [128 rows][64 bf16] swizzled chunk
constexpr float kLn2 = 0.69314718055994530942f;
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
};

__device__ unsigned int g_fa_status = 0;

struct FaParams {
    float* lse;
    int N;
    int n_tiles;       // ceil(N / 128) query (= key) tiles
    int causal;
    float scale_log2;  // scale * log2(e)
    unsigned long long watchdog_ns;
    // split-KV partial states (kSplit kernels only): [n_splits][B*H][N] rows
    int n_splits;
    float* ws_o;    // unnormalised O, fp32 [rows][d]
    float* ws_m;    // reference max, base-2 units
    float* ws_lbf;  // sum of the bf16-rounded exponentials
    float* ws_l32;  // fp32 sum of the exponentials
};

template <int D, int NK, int NV>
struct FaSmem {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = kBlockN * D * 2;
    static constexpr uint32_t kOffQ = 0;  // the query tile, later the O staging
    static constexpr uint32_t kOffK = kOffQ + kTileBytes;
    static constexpr uint32_t kOffV = kOffK + NK * kTileBytes;
    static constexpr uint32_t kOffBar = kOffV + NV * kTileBytes;
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + NK;
    static constexpr int kBarVFull = kBarKEmpty + NK;
    static constexpr int kBarVEmpty = kBarVFull + NV;
    static constexpr int kBarSFull = kBarVEmpty + NV;  // per S buffer: S_j written
    static constexpr int kBarSFree = kBarSFull + 2;    // per S buffer: S_j read by the softmax
    static constexpr int kBarPFull = kBarSFree + 2;    // per P buffer: P_j written
    static constexpr int kBarPVDone = kBarPFull + 2;   // per P buffer: P_j V_j finished
    static constexpr int kBarOFinal = kBarPVDone + 2;  // the last P V product finished
    static constexpr int kBarDrain = kBarOFinal + 1;   // per MMA issuer
    static constexpr int kNumBars = kBarDrain + 2;
    static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
    static constexpr uint32_t kBytes = kOffAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    // TMEM columns: S0 S1 O P0 P1
    __host__ __device__ static constexpr uint32_t col_s(int b) { return (uint32_t)b * 128u; }
    static constexpr uint32_t kColO = 256;
    __host__ __device__ static constexpr uint32_t col_p(int b) { return 256u + D + (uint32_t)b * 64u; }
    static_assert(256 + D + 128 <= (int)kTmemCols, "TMEM budget");
};

// Bounded wait on an mbarrier phase.  Gives up when another warp of the CTA
// has raised the abort flag, or after `limit_ns`, in which case it raises the
// flag and records `code` in the device status word.
__device__ __forceinline__ bool fa_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns,
                                        unsigned int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(&g_fa_status, code);
            return false;
        }
    }
}

// Same, with the verdict made uniform across the warp.
__device__ __forceinline__ bool fa_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns, unsigned int code) {
    const bool ok = fa_wait(bar, parity, abort_flag, limit_ns, code);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait used while tearing down after an abort: ignores the flag.
__device__ __forceinline__ bool fa_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(&g_fa_status, kStatusDrain);
            return false;
        }
    }
}

// Exponentials of one 128-key row tile against the reference -neg_m (base 2):
// P packed to bf16 pairs, the sum of the bf16-rounded values and the fp32 sum.
__device__ __forceinline__ void exp_row_tile(const float (&s)[kBlockN], float c2, float neg_m,
                                             uint32_t (&pk)[kBlockN / 2], float& sum_bf, float& sum_f32) {
    const uint64_t c2x2 = f32x2_pack(c2, c2), negm2 = f32x2_pack(neg_m, neg_m);
    float rs[4] = {0.f, 0.f, 0.f, 0.f};
    uint64_t r32[2] = {0ull, 0ull};  // packed (even, odd) fp32 partial sums
#pragma unroll
    for (int i = 0; i < kBlockN / 2; ++i) {
        float x0, x1;
        f32x2_unpack(ffma2(f32x2_pack(s[2 * i], s[2 * i + 1]), c2x2, negm2), x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        pk[i] = pack_bf16x2(p0, p1);
        rs[i & 3] = add_bf16x2_f32(rs[i & 3], pk[i]);
        r32[i & 1] = fadd2(r32[i & 1], f32x2_pack(p0, p1));
    }
    float e0, e1, o0, o1;
    f32x2_unpack(r32[0], e0, o0);
    f32x2_unpack(r32[1], e1, o1);
    sum_bf = (rs[0] + rs[1]) + (rs[2] + rs[3]);
    sum_f32 = (e0 + o0) + (e1 + o1);
}

// kSplit: the CTA covers only the key tiles of split blockIdx.z and writes the
// partial row state (m, both sums, unnormalised O) instead of O and LSE; a
// merge kernel combines the splits ("5.2 CUDA Online Softmax", section 4.1:
// the (m, d) merge is associative, so partial results combine in any order).
template <int D, int NK, int NV, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const FaParams p) {
    using L = FaSmem<D, NK, NV>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = (int)(threadIdx.x & 31);
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest causal rows first
    const int bh = (int)blockIdx.y;
    const int n_all = p.causal ? min(qt + 1, p.n_tiles) : p.n_tiles;  // key tiles this query tile sees
    int j0 = 0, n_kv = n_all;  // this CTA's key tiles: j0 .. j0 + n_kv - 1
    if constexpr (kSplit) {
        const int chunk = (n_all + p.n_splits - 1) / p.n_splits;
        j0 = (int)blockIdx.z * chunk;
        n_kv = max(0, min(n_all - j0, chunk));
    }
    const uint64_t limit = p.watchdog_ns;

    if (warp == 0 && lane == 0) {
        mbar_init(bar(L::kBarQ), 1);
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
            mbar_init(bar(L::kBarSFree + b), 4);  // one arrival per softmax warp
            mbar_init(bar(L::kBarPFull + b), 4);
            mbar_init(bar(L::kBarPVDone + b), 1);
            mbar_init(bar(L::kBarDrain + b), 1);
        }
        mbar_init(bar(L::kBarOFinal), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_o);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer: Q once; K_0, K_1; then V_j and K_{j+2}, the order in
        // which the two MMA issuers consume them.
        // ------------------------------------------------------------------
        if (lane == 0 && n_kv > 0) {
            mbar_arrive_expect_tx(bar(L::kBarQ), L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
                tma_load_3d(sbase + L::kOffQ + c * kChunkBytes, &tm_q, bar(L::kBarQ), c * 64, qt * kBlockM, bh);
            int nk = 0, nv = 0;  // loads issued
            auto load_k = [&](int j) -> bool {
                const int s = j % NK;
                const uint32_t r = (uint32_t)(j / NK);
                if (!fa_wait(bar(L::kBarKEmpty + s), (r & 1u) ^ 1u, abort_flag, limit, kStatusLoadWait)) return false;
                mbar_arrive_expect_tx(bar(L::kBarKFull + s), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kOffK + s * L::kTileBytes + c * kChunkBytes, &tm_k, bar(L::kBarKFull + s),
                                c * 64, (j0 + j) * kBlockN, bh);
                ++nk;
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int s = j % NV;
                const uint32_t r = (uint32_t)(j / NV);
                if (!fa_wait(bar(L::kBarVEmpty + s), (r & 1u) ^ 1u, abort_flag, limit, kStatusLoadWait)) return false;
                mbar_arrive_expect_tx(bar(L::kBarVFull + s), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kOffV + s * L::kTileBytes + c * kChunkBytes, &tm_v, bar(L::kBarVFull + s),
                                c * 64, (j0 + j) * kBlockN, bh);
                ++nv;
                return true;
            };
            bool ok = load_k(0);
            if (ok && n_kv > 1) ok = load_k(1);
            for (int j = 0; ok && j < n_kv; ++j) {
                ok = load_v(j);
                if (ok && j + 2 < n_kv) ok = load_k(j + 2);
            }
            if (!ok) {
                // abort: let every copy already issued land before the CTA exits
                fa_wait_drain(bar(L::kBarQ), 0, limit);
                for (int s = 0; s < NK; ++s)
                    if (nk > s) fa_wait_drain(bar(L::kBarKFull + s), (uint32_t)(((nk - 1 - s) / NK) & 1), limit);
                for (int s = 0; s < NV; ++s)
                    if (nv > s) fa_wait_drain(bar(L::kBarVFull + s), (uint32_t)(((nv - 1 - s) / NV) & 1), limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // S issuer: S_j = Q K_j^T into buffer j % 2 once K_j has landed and
        // the softmax has read S_{j-2} out of that buffer.
        // ------------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
            const uint32_t qa = sbase + L::kOffQ;
            bool ok = n_kv > 0 && fa_wait(bar(L::kBarQ), 0, abort_flag, limit, kStatusMmaWaitQ);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int b = j & 1;
                const int ks = j % NK;
                if (j >= 2)
                    ok = fa_wait(bar(L::kBarSFree + b), (uint32_t)(((j - 2) >> 1) & 1), abort_flag, limit,
                                 kStatusMmaWaitSFree);
                ok = ok && fa_wait(bar(L::kBarKFull + ks), (uint32_t)((j / NK) & 1), abort_flag, limit,
                                   kStatusMmaWaitK);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t ka = sbase + L::kOffK + (uint32_t)ks * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kChunkBytes + (uint32_t)(kk & 3) * 32u;
                    mma_ss(tmem + L::col_s(b), sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                           kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(L::kBarSFull + b));
                tc_commit(bar(L::kBarKEmpty + ks));
            }
            tc_commit(bar(L::kBarDrain + 0));  // every MMA must finish before TMEM is released
            fa_wait_drain(bar(L::kBarDrain + 0), 0, limit);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------------
        // P V issuer: O += P_j V_j once P_j is in TMEM and V_j has landed.
        // ------------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, false, true);
            bool ok = true;
            for (int j = 0; ok && j < n_kv; ++j) {
                const int b = j & 1;
                const int vs = j % NV;
                ok = fa_wait(bar(L::kBarPFull + b), (uint32_t)((j >> 1) & 1), abort_flag, limit, kStatusMmaWaitP) &&
                     fa_wait(bar(L::kBarVFull + vs), (uint32_t)((j / NV) & 1), abort_flag, limit, kStatusMmaWaitV);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t va = sbase + L::kOffV + (uint32_t)vs * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts(tmem + L::kColO, tmem + L::col_p(b) + (uint32_t)kk * 8u,
                           sdesc_sw128(va + (uint32_t)kk * 2048u, kChunkBytes, 1024), kIdescPV,
                           (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(L::kBarVEmpty + vs));
                tc_commit(bar(L::kBarPVDone + b));
                if (j + 1 == n_kv) tc_commit(bar(L::kBarOFinal));
            }
            tc_commit(bar(L::kBarDrain + 1));
            fa_wait_drain(bar(L::kBarDrain + 1), 0, limit);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------------
        // Softmax / correction / epilogue: thread = one query row = TMEM lane.
        // ------------------------------------------------------------------
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int q_idx = qt * kBlockM + row;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const float c2 = p.scale_log2;
        float m_run = -INFINITY;  // reference max, base-2 scaled units
        float l_run = 0.f;        // sum of bf16(2^(t - m_run)): normalises O
        float l32_run = 0.f;      // sum of 2^(t - m_run) in fp32: gives LSE
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            if (!fa_wait_warp(bar(L::kBarSFull + b), (uint32_t)((j >> 1) & 1), abort_flag, limit,
                              kStatusSoftmaxWaitS)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float s[kBlockN];
            {
                uint32_t r[kBlockN];
                tmem_ld128_wait(t_lane + L::col_s(b), r);
#pragma unroll
                for (int i = 0; i < kBlockN; ++i) s[i] = __uint_as_float(r[i]);
            }
            // S_j is in registers: the buffer may take S_{j+2}
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kBarSFree + b));
            // mask keys past the diagonal (causal) and past the end of the sequence
            int lim = p.N - 1 - (j0 + j) * kBlockN;
            if (p.causal && j0 + j == qt) lim = min(lim, row);
            if (lim < kBlockN - 1) {
#pragma unroll
                for (int i = 0; i < kBlockN; ++i) s[i] = (i > lim) ? -INFINITY : s[i];
            }
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
            // scale > 0, so max(s) * c2 == max(s * c2)
            const float m_cand = fmaxf(m_run, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2);
            // move the reference only when the max grew past the threshold
            // (always on the first visible tile: -inf + 64 = -inf < any finite max)
            const bool move = m_cand > m_run + kRescaleThreshold;
            const float alpha = move ? ex2_approx(m_run - m_cand) : 1.f;  // exp2(-inf) = 0 wipes the empty state
            const bool any_move = __any_sync(0xffffffffu, move);
            if (move) m_run = m_cand;
            // a row with nothing visible yet keeps m = -inf and uses 0, so that its
            // -inf scores give 0 rather than NaN
            uint32_t pk[kBlockN / 2];
            float sum_bf, sum_f32;
            exp_row_tile(s, c2, (m_run == -INFINITY) ? 0.f : -m_run, pk, sum_bf, sum_f32);
            l_run = l_run * alpha + sum_bf;
            l32_run = l32_run * alpha + sum_f32;
            if (j > 0 && any_move) {
                // O must hold P_{j-1} V_{j-1} before it is rescaled
                if (!fa_wait_warp(bar(L::kBarPVDone + (b ^ 1)), (uint32_t)(((j - 1) >> 1) & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitPV)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32_wait(t_lane + L::kColO + 32u * c, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                    tmem_st32(t_lane + L::kColO + 32u * c, r);
                }
            }
            if (j >= 2) {
                // P buffer b last fed P_{j-2} V_{j-2}: that product must have read it
                if (!fa_wait_warp(bar(L::kBarPVDone + b), (uint32_t)(((j - 2) >> 1) & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitPV)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
            }
            const uint32_t pcol = t_lane + L::col_p(b);
            tmem_st32(pcol, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
            tmem_st32(pcol + 32u, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kBarPFull + b));
        }
        if (ok && n_kv > 0) ok = fa_wait_warp(bar(L::kBarOFinal), 0, abort_flag, limit, kStatusSoftmaxWaitO);
        if constexpr (kSplit) {
            // partial state of this split: unnormalised O and (m, sums) per row.
            // The TMEM loads are warp-collective, so every lane runs them and
            // only rows inside the sequence store.
            const bool valid = q_idx < p.N;
            const size_t r = ((size_t)blockIdx.z * gridDim.y + (size_t)bh) * (size_t)p.N + (size_t)q_idx;
            float4* dst = reinterpret_cast<float4*>(p.ws_o + r * D);
            if (ok && n_kv > 0) {
                tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32_wait(t_lane + L::kColO + 32u * c, v);
                    if (valid) {
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            dst[c * 8 + u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                                         __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
                    }
                }
            } else if (ok && valid) {
#pragma unroll
                for (int u = 0; u < D / 4; ++u) dst[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (ok && valid) {
                p.ws_m[r] = m_run;
                p.ws_lbf[r] = l_run;
                p.ws_l32[r] = l32_run;
            }
            tc_fence_before_sync();
        } else {
        // Q is dead once the last S product has finished (the softmax read it): stage O there
        const uint32_t stage = sbase + L::kOffQ;
        if (ok) {
            tc_fence_after_sync();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32_wait(t_lane + L::kColO + 32u * c, r);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
                const uint32_t chunk = stage + (uint32_t)(c >> 1) * kChunkBytes + (uint32_t)row * 128u;
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) {
                    const uint32_t u = (uint32_t)((c & 1) * 4 + u4);  // 16-byte unit within the 128-byte row
                    st_shared_v4(chunk + ((u ^ (uint32_t)(row & 7)) << 4), w[4 * u4], w[4 * u4 + 1], w[4 * u4 + 2],
                                 w[4 * u4 + 3]);
                }
            }
            if (q_idx < p.N)
                p.lse[(size_t)bh * (size_t)p.N + (size_t)q_idx] =
                    l32_run > 0.f ? (m_run + lg2_approx(l32_run)) * kLn2 : -INFINITY;
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_barrier_sync(1, 128);
        if (warp == 4 && lane == 0 && *abort_flag == 0) {
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) tma_store_3d(&tm_o, stage + c * kChunkBytes, c * 64, qt * kBlockM, bh);
            bulk_commit_group();
            bulk_wait_group_all();
        }
        }  // kSplit
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
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
