// fa_fwd_two_kernel.cuh -- the d = 64 forward with two query tiles per CTA.
//
// Same method as fa_fwd_sm103 (the online recurrence of "Online softmax, and
// the register that can't move", section "Online softmax", with the query
// tile resident and the key/value tiles streaming past it as in "Online
// Softmax: Tiling Across a Reduction", loop order), arranged differently on
// the SM.  A unit of work is two adjacent query tiles of one head, A = 2u and
// B = 2u + 1, against every key tile either sees; the key and value tiles are
// loaded once for both.  Each tile has its own softmax warpgroup, its own MMA
// issuer, its own S, P and O in TMEM and its own row state:
//
//   TMEM columns: S_A 0-127, S_B 128-255, O_A 256-319, O_B 320-383,
//                 P_A 384-447, P_B 448-511.
//
// The two tiles' chains share nothing but the loads, so neither group waits
// for the other: a group hands no reference maximum across, and its P V
// product waits only for its own previous one.  The one-tile kernel instead
// splits one tile's steps between its two groups, which then wait on each
// other every step; at d = 64, where a step's products (12 tensor-core
// instructions of ~64 cycles: an N = 64 instruction costs what an N = 128 one
// does) are not much longer than its 512 cycles of exponentials, those waits
// set the step.
//
// Per tile and key step g (counted over the CTA's whole sequence):
//   issuer:  S_g = Q K_g^T once the group has read S_{g-1} out of TMEM, then
//            O += P_{g-1} V_{g-1} once P_{g-1} is written (the first product
//            of a tile also waits until the previous tile's O has been read);
//   softmax: read S_g (with the row maximum), release S, exponentials against
//            the reference maximum, P_g into TMEM once P_{g-1} V_{g-1} has
//            finished, O rescaled on TMEM when the reference moved.
// The reference moves only past the threshold of the one-tile kernel, so the
// rescale is as rare there.  TMEM has no room for the tensor-core row sums, so
// O is normalised as at d = 128: the fp32 sum of the exponentials plus, per key
// tile, the bf16 rounding of the tile's largest weight.
//
// Causal units: tile A does not see key tile 2u + 1; its step there is fully
// masked (weights 0), one wasted step in 4u + 4.  A unit past the last query
// tile's partner (odd tile count) loads a real tile for B and never stores
// its rows.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

template <int NK, int NV>
struct TwoSmem {
    static constexpr int D = 64;
    static constexpr uint32_t kTileBytes = kBlockN * D * 2;  // 16 KB: [128 rows][64 bf16], 128-byte swizzle
    static constexpr uint32_t kOffQ = 0;                      // Q_A, Q_B
    static constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;
    static constexpr uint32_t kOffV = kOffK + NK * kTileBytes;
    static constexpr uint32_t kOffBar = kOffV + NV * kTileBytes;
    // per tile x = 0 (A), 1 (B)
    static constexpr int kBarQ = 0;                      // Q_x landed
    static constexpr int kBarQFree = kBarQ + 2;          // the unit's last S_x finished
    static constexpr int kBarKFull = kBarQFree + 2;
    static constexpr int kBarKEmpty = kBarKFull + NK;    // both tiles' S products of the stage finished
    static constexpr int kBarVFull = kBarKEmpty + NK;
    static constexpr int kBarVEmpty = kBarVFull + NV;    // both tiles' P V products of the stage finished
    static constexpr int kBarSFull = kBarVEmpty + NV;    // S_x written
    static constexpr int kBarSFree = kBarSFull + 2;      // S_x read by its group
    static constexpr int kBarPFull = kBarSFree + 2;      // P_x written
    static constexpr int kBarPVDone = kBarPFull + 2;     // P_x V finished
    static constexpr int kBarOFinal = kBarPVDone + 2;    // the unit's last P_x V finished
    static constexpr int kBarOFree = kBarOFinal + 2;     // O_x read out of TMEM
    static constexpr int kBarDrain = kBarOFree + 2;      // per issuer
    static constexpr int kBarItemFull = kBarDrain + 2;
    static constexpr int kBarItemEmpty = kBarItemFull + kItemRing;
    static constexpr int kNumBars = kBarItemEmpty + kItemRing;
    static constexpr uint32_t kOffItems = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffTmemSlot = kOffItems + kItemRing * 16;
    static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
    static constexpr uint32_t kBytes = kOffAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    static_assert(kAlloc <= 232448u, "dynamic shared memory above the 227 KB a CTA may use");
    __host__ __device__ static constexpr uint32_t col_s(int x) { return (uint32_t)x * 128u; }
    __host__ __device__ static constexpr uint32_t col_o(int x) { return 256u + (uint32_t)x * 64u; }
    __host__ __device__ static constexpr uint32_t col_p(int x) { return 384u + (uint32_t)x * 64u; }
    static_assert(384 + 2 * 64 <= kTmemCols, "TMEM budget");
};

template <int NK, int NV>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd2_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FaParams p) {
    constexpr int D = 64;
    using L = TwoSmem<NK, NV>;
    using Seq = TileSeq<false, true, false, false, true>;
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

    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(L::kBarQ + x), 1);
            mbar_init(bar(L::kBarQFree + x), 1);
            mbar_init(bar(L::kBarSFull + x), 1);
            mbar_init(bar(L::kBarSFree + x), kSoftmaxWarps / 2);  // one arrival per warp of group x
            mbar_init(bar(L::kBarPFull + x), kSoftmaxWarps / 2);
            mbar_init(bar(L::kBarPVDone + x), 1);
            mbar_init(bar(L::kBarOFinal + x), 1);
            mbar_init(bar(L::kBarOFree + x), kSoftmaxWarps / 2);
            mbar_init(bar(L::kBarDrain + x), 1);
        }
#pragma unroll
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(L::kBarKFull + s), 1);
            mbar_init(bar(L::kBarKEmpty + s), 2);  // a commit from each issuer
        }
#pragma unroll
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(L::kBarVFull + s), 1);
            mbar_init(bar(L::kBarVEmpty + s), 2);
        }
#pragma unroll
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(bar(L::kBarItemFull + i), 1);
            mbar_init(bar(L::kBarItemEmpty + i), kItemReaders);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
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
        // TMA producer.  Per unit: K_0, Q_A and Q_B (each once the previous
        // unit's last S product of that tile has finished), K_1, then V_j and
        // K_{j+2}.
        // ------------------------------------------------------------------
        if (lane == 0) {
            int nk = 0, nv = 0, nq[2] = {0, 0};  // loads issued over the whole sequence
            auto load_k = [&](const TileWork& w, int j) -> bool {
                const int s = nk % NK;
                const uint32_t r = (uint32_t)(nk / NK);
                if (!fa_wait(bar(L::kBarKEmpty + s), (r & 1u) ^ 1u, abort_flag, limit, kStatusLoadWait)) return false;
                mbar_arrive_expect_tx(bar(L::kBarKFull + s), L::kTileBytes);
                tma_load_3d(sbase + L::kOffK + s * L::kTileBytes, &tm_k, bar(L::kBarKFull + s), 0,
                            (w.j0 + j) * kBlockN, w.bh);
                ++nk;
                return true;
            };
            auto load_v = [&](const TileWork& w, int j) -> bool {
                const int s = nv % NV;
                const uint32_t r = (uint32_t)(nv / NV);
                if (!fa_wait(bar(L::kBarVEmpty + s), (r & 1u) ^ 1u, abort_flag, limit, kStatusLoadWait)) return false;
                mbar_arrive_expect_tx(bar(L::kBarVFull + s), L::kTileBytes);
                tma_load_3d(sbase + L::kOffV + s * L::kTileBytes, &tm_v, bar(L::kBarVFull + s), 0,
                            (w.j0 + j) * kBlockN, w.bh);
                ++nv;
                return true;
            };
            Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
            TileWork w;
            bool ok = true;
            while (ok && seq.produce(p, w)) {
                if (w.n_kv == 0) continue;
                ok = load_k(w, 0);
                for (int x = 0; ok && x < 2; ++x) {
                    if (nq[x] > 0)
                        ok = fa_wait(bar(L::kBarQFree + x), (uint32_t)((nq[x] - 1) & 1), abort_flag, limit,
                                     kStatusLoadWait);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(L::kBarQ + x), L::kTileBytes);
                    // tile B past the last tile (odd count) loads a real tile; its rows are never stored
                    const int qrow = min(w.qt + x, p.n_tiles - 1) * kBlockM;
                    tma_load_3d(sbase + L::kOffQ + (uint32_t)x * L::kTileBytes, &tm_q, bar(L::kBarQ + x), 0, qrow,
                                w.bh);
                    ++nq[x];
                }
                if (ok && w.n_kv > 1) ok = load_k(w, 1);
                for (int j = 0; ok && j < w.n_kv; ++j) {
                    ok = load_v(w, j);
                    if (ok && j + 2 < w.n_kv) ok = load_k(w, j + 2);
                }
            }
            // every copy already issued lands before the CTA exits (after an abort
            // some are never consumed; in a normal run these waits succeed at once)
            for (int x = 0; x < 2; ++x)
                if (nq[x] > 0) fa_wait_drain(bar(L::kBarQ + x), (uint32_t)((nq[x] - 1) & 1), limit);
            for (int s = 0; s < NK; ++s)
                if (nk > s) fa_wait_drain(bar(L::kBarKFull + s), (uint32_t)(((nk - 1 - s) / NK) & 1), limit);
            for (int s = 0; s < NV; ++s)
                if (nv > s) fa_wait_drain(bar(L::kBarVFull + s), (uint32_t)(((nv - 1 - s) / NV) & 1), limit);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------------
        // MMA issuer of tile x: S_g, then the P V product of the step before.
        // ------------------------------------------------------------------
        const int x = warp - 1;
        constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, false, true);
        const uint32_t qa = sbase + L::kOffQ + (uint32_t)x * L::kTileBytes;
        int g = 0, t = 0;  // steps and units of this tile so far
        bool ok = true;
        // O_x += P_x V of step gg, the tile's step j of n_kv
        auto pv = [&](int gg, int j, int n_kv) -> bool {
            const int vs = gg % NV;
            bool good = fa_wait_warp(bar(L::kBarPFull + x), (uint32_t)(gg & 1), abort_flag, limit, kStatusMmaWaitP) &&
                        fa_wait_warp(bar(L::kBarVFull + vs), (uint32_t)((gg / NV) & 1), abort_flag, limit,
                                     kStatusMmaWaitV);
            if (good && j == 0 && t > 0)
                good = fa_wait_warp(bar(L::kBarOFree + x), (uint32_t)((t - 1) & 1), abort_flag, limit,
                                    kStatusMmaWaitP);
            if (!good) return false;
            tc_fence_after_sync();
            const uint32_t va = sbase + L::kOffV + (uint32_t)vs * L::kTileBytes;
            const uint64_t vd = sdesc_sw128(va, kChunkBytes, 1024);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)  // 16 keys (2048 bytes of V) per product
                    mma_ts(tmem + L::col_o(x), tmem + L::col_p(x) + (uint32_t)kk * 8u,
                           sdesc_add_lo(vd, (uint32_t)kk * 128u), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(L::kBarVEmpty + vs));
                tc_commit(bar(L::kBarPVDone + x));
                if (j + 1 == n_kv) tc_commit(bar(L::kBarOFinal + x));
            }
            __syncwarp();
            return true;
        };
        Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
        TileWork w;
        while (ok && seq.template next<true>(p, w)) {
            if (w.n_kv == 0) continue;
            ok = fa_wait_warp(bar(L::kBarQ + x), (uint32_t)(t & 1), abort_flag, limit, kStatusMmaWaitQ);
            if (p.withhold_s) break;
            for (int j = 0; ok && j < w.n_kv; ++j, ++g) {
                const int ks = g % NK;
                if (g >= 1)
                    ok = fa_wait_warp(bar(L::kBarSFree + x), (uint32_t)((g - 1) & 1), abort_flag, limit,
                                      kStatusMmaWaitSFree);
                ok = ok && fa_wait_warp(bar(L::kBarKFull + ks), (uint32_t)((g / NK) & 1), abort_flag, limit,
                                        kStatusMmaWaitK);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t ka = sbase + L::kOffK + (uint32_t)ks * L::kTileBytes;
                const uint64_t qd = sdesc_sw128(qa, 16, 1024), kd = sdesc_sw128(ka, 16, 1024);
                if (elect_one_sync()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // 16 of d (32 bytes of the swizzled row) per product
                        const uint32_t off = ((uint32_t)kk * 32u) >> 4;
                        mma_ss(tmem + L::col_s(x), sdesc_add_lo(qd, off), sdesc_add_lo(kd, off), kIdescS,
                               kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(L::kBarSFull + x));
                    tc_commit(bar(L::kBarKEmpty + ks));
                    if (j + 1 == w.n_kv) tc_commit(bar(L::kBarQFree + x));  // Q_x may be refilled
                }
                __syncwarp();
                if (j > 0) ok = pv(g - 1, j - 1, w.n_kv);
            }
            if (ok) ok = pv(g - 1, w.n_kv - 1, w.n_kv);
            ++t;
        }
        if (elect_one_sync()) {
            // every MMA must finish before TMEM is released
            tc_commit(bar(L::kBarDrain + x));
            fa_wait_drain(bar(L::kBarDrain + x), 0, limit);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------------
        // Softmax, O rescale and epilogue of tile x.  Thread = one query row
        // (TMEM lane `row`), all 128 keys of every step.
        // ------------------------------------------------------------------
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int x = (warp - 4) >> 2;  // warps 4-7: tile A, warps 8-11: tile B
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const float c2 = p.scale_log2;
        // this group's barrier i, its address recomputed where it is used rather than
        // held in a register across the loop
        auto xbar = [&](int i) -> uint32_t { return fa_here(sbase) + L::kOffBar + 8u * (uint32_t)(i + x); };
        int g = 0, t = 0;
        bool ok = true;
        bool in_tile = false;
        int q_idx = 0;
        bool valid = false;
        Seq seq(items, bar(L::kBarItemFull), bar(L::kBarItemEmpty), abort_flag, limit);
        TileWork w;
        while (ok && seq.template next<true>(p, w)) {
            if (w.n_kv == 0) continue;
            const int qt = w.qt + x;
            q_idx = qt * kBlockM + row;
            valid = q_idx < p.N;
            in_tile = true;
            float m_ref = -INFINITY;  // reference maximum (base-2 units) the sums and O are relative to
            float l_run = 0.f;        // sum that normalises O: fp32 sum + per-tile largest-weight rounding
            float l32_run = 0.f;      // fp32 sum of 2^(t - m_ref): gives LSE
            for (int j = 0; j < w.n_kv; ++j, ++g) {
                if (!fa_wait_warp(xbar(L::kBarSFull), (uint32_t)(g & 1), abort_flag, limit, kStatusSoftmaxWaitS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                float s[kBlockN];
                float ld_max;
                {
                    uint32_t r[kBlockN];
                    tmem_ld128_max_wait(t_lane + L::col_s(x), r, ld_max);
#pragma unroll
                    for (int i = 0; i < kBlockN; ++i) s[i] = __uint_as_float(r[i]);
                }
                // S_g is in registers: the buffer may take S_{g+1}
                tc_fence_before_sync();
                __syncwarp();
                if (elect_one_sync()) mbar_arrive(xbar(L::kBarSFree));
                // mask keys past the diagonal (causal; tile A's step on key tile 2u + 1 is
                // wholly masked) and past the end of the sequence
                bool masked = false;
                {
                    int lim = p.N - 1 - (w.j0 + j) * kBlockN;
                    if (p.causal && w.j0 + j >= qt) lim = min(lim, row + (qt - w.j0 - j) * kBlockN);
                    if (__builtin_expect(lim < kBlockN - 1, 0)) {
                        masked = true;
#pragma unroll
                        for (int i = 0; i < kBlockN; ++i) s[i] = (i > lim) ? -INFINITY : s[i];
                    }
                }
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
                // the reference moves only when the maximum grew past it by more than the
                // threshold (always on the first visible key: -inf + 64 = -inf)
                const float m_prev = m_ref;
                const float m_cand = fmaxf(m_prev, row_max * c2);
                const bool move = m_cand > m_prev + kRescaleThreshold;
                const float m_new = move ? m_cand : m_prev;
                const bool any_move = __any_sync(0xffffffffu, move);
                const float a_l = (m_prev == m_new) ? 1.f : ex2_approx(m_prev - m_new);  // 2^-inf = 0
                m_ref = m_new;
                uint32_t pk[kBlockN / 2];
                float sum_f32;
                const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
                exp_row_tile<kBlockN>(s, c2, neg_m, pk, sum_f32);
                {
                    // the rounding of this tile's largest weight, recomputed from the row
                    // maximum with the operations the loop applied to it (fma, ex2, RN to bf16)
                    const float p_max = ex2_approx(fmaf(row_max, c2, neg_m));
                    const float r_max = __bfloat162float(__float2bfloat16_rn(p_max)) - p_max;
                    l_run = l_run * a_l + (sum_f32 + r_max);
                }
                l32_run = l32_run * a_l + sum_f32;
                if (g >= 1) {
                    // P_x last fed P_{g-1} V_{g-1}: that product must have read it (and O holds it)
                    if (!fa_wait_warp(xbar(L::kBarPVDone), (uint32_t)((g - 1) & 1), abort_flag, limit,
                                      kStatusSoftmaxWaitPV)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
                tmem_st64(t_lane + L::col_p(x), pk);
                if (__builtin_expect(j > 0 && any_move, 0)) {
                    // O to the new reference, on TMEM (rows whose reference stayed scale by 1)
                    const float a_o = move ? ex2_approx(m_prev - m_new) : 1.f;
                    uint32_t r[D];
                    tmem_ld64_wait(t_lane + L::col_o(x), r);
                    const uint64_t a2 = f32x2_pack(a_o, a_o);
#pragma unroll
                    for (int i = 0; i < D / 2; ++i) {
                        float x0, x1;
                        f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), a2),
                                     x0, x1);
                        r[2 * i] = __float_as_uint(x0);
                        r[2 * i + 1] = __float_as_uint(x1);
                    }
                    tmem_st64(t_lane + L::col_o(x), r);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (elect_one_sync()) mbar_arrive(xbar(L::kBarPFull));
            }
            if (!ok) break;
            ok = fa_wait_warp(xbar(L::kBarOFinal), (uint32_t)(t & 1), abort_flag, limit, kStatusSoftmaxWaitO);
            if (!ok) break;
            tc_fence_after_sync();
            // the row of O, 32 columns at a time, O/l -> bf16; O is released to the
            // next unit's first P V product as soon as it is all in registers
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            uint32_t wv[D / 2];
#pragma unroll
            for (int h = 0; h < D / 32; ++h) {
                uint32_t r[32];
                tmem_ld32_wait(t_lane + L::col_o(x) + 32u * (uint32_t)h, r);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    wv[16 * h + i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (elect_one_sync()) mbar_arrive(xbar(L::kBarOFree));
            if (valid) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + ((size_t)w.bh * (size_t)p.N + (size_t)q_idx) * D;
                if ((reinterpret_cast<uintptr_t>(p.o) & 31u) == 0) {
#pragma unroll
                    for (int u = 0; u < D / 16; ++u) st_global_v8(orow + 16 * u, wv + 8 * u);
                } else {
                    uint4* o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll
                    for (int u = 0; u < D / 8; ++u) o4[u] = make_uint4(wv[4 * u], wv[4 * u + 1], wv[4 * u + 2], wv[4 * u + 3]);
                }
                p.lse[(size_t)w.bh * (size_t)p.N + (size_t)q_idx] =
                    l32_run > 0.f ? (m_ref + lg2_approx(l32_run)) * kLn2 : -INFINITY;
            }
            in_tile = false;
            ++t;
        }
        if (!ok && in_tile && valid) {
            // the watchdog ended a wait inside this tile: its rows are never
            // finished, so their statistic is set to NaN
            p.lse[(size_t)w.bh * (size_t)p.N + (size_t)q_idx] = __int_as_float(0x7fffffff);
        }
        __syncwarp();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
    // the last CTA out leaves the work counter at zero for the next launch
    if (threadIdx.x == 0 && p.queue) {
        __threadfence();
        if (atomicAdd(p.queue + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.queue + 0, 0u);
            atomicExch(p.queue + 1, 0u);
        }
    }
}

}  // namespace fa
