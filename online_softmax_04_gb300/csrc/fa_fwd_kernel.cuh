// fa_fwd_kernel.cuh -- fused attention forward for sm_103a (GB300).
//
// One CTA owns one 128-row query tile of one (batch, head) and streams the
// key/value tiles past it ("Online Softmax: Tiling Across a Reduction", loop
// order: query blocks outer and resident, key/value blocks inner).  Per key
// tile j the running row state is updated with one correction factor
// ("Online softmax, and the register that can't move", section "Online
// softmax"):
//
//     m_new = max(m_old, rowmax(S_j))
//     l_new = l_old * exp(m_old - m_new) + rowsum(exp(S_j - m_new))
//     O_new = O_old * exp(m_old - m_new) + exp(S_j - m_new) V_j
//
// and after the last tile O /= l, LSE = m + ln l.  Scores are kept in the
// base-2 domain: t = s * scale * log2(e), so every exponential is one ex2.
//
// GB300 mapping:
//   * S_j = Q K_j^T and O += P_j V_j run on tcgen05.mma (bf16 in, fp32
//     accumulate) with the accumulators in tensor memory (TMEM): S is double
//     buffered so S_{j+1} is computed while the softmax works on S_j.
//   * P_j is written back to TMEM as bf16 and consumed from there as the A
//     operand of the P V product (no shared-memory round trip).
//   * Q, K_j and V_j are brought in by TMA (128-byte swizzle) into a ring of
//     shared-memory stages guarded by mbarriers.
//   * Warp roles: warp 0 issues TMA loads, warp 1 owns TMEM and issues the
//     MMAs, warps 2-5 (one thread per query row) do the softmax, the O
//     rescale on TMEM and the epilogue (O/l -> bf16 -> shared -> TMA store,
//     LSE store).
//   * Causal: key tiles wholly after the query tile are never visited; only
//     the diagonal tile is masked element by element ("Online Softmax: Tiling
//     Across a Reduction", causal section).  Keys >= N in the last tile are
//     masked the same way.
//
// Every barrier wait is bounded by a watchdog (global timer): on expiry the
// CTA records a status bit, tells its other warps to stop, lets its copies
// and MMAs drain, frees TMEM and exits.
#pragma once

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;   // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 192;  // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChunkBytes = 128u * 128u;  // one [128 rows][64 bf16] swizzled chunk
constexpr float kLn2 = 0.69314718055994530942f;

// device status bits (which wait ran out)
enum : unsigned int {
    kStatusLoadWait = 1u << 0,
    kStatusMmaWaitQ = 1u << 1,
    kStatusMmaWaitK = 1u << 2,
    kStatusMmaWaitP = 1u << 3,
    kStatusMmaWaitV = 1u << 4,
    kStatusSoftmaxWaitS = 1u << 5,
    kStatusSoftmaxWaitPV = 1u << 6,
    kStatusDrain = 1u << 7,
    kStatusSelfTest = 1u << 8,
};

__device__ unsigned int g_fa_status = 0;

struct FaParams {
    float* lse;
    int N;
    int n_tiles;       // ceil(N / 128)
    int causal;
    float scale_log2;  // scale * log2(e)
    unsigned long long watchdog_ns;
};

template <int D, int NK, int NV>
struct FaSmem {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = kBlockN * D * 2;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kTileBytes;
    static constexpr uint32_t kOffV = kOffK + NK * kTileBytes;
    static constexpr uint32_t kOffBar = kOffV + NV * kTileBytes;
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + NK;
    static constexpr int kBarVFull = kBarKEmpty + NK;
    static constexpr int kBarVEmpty = kBarVFull + NV;
    static constexpr int kBarSFull = kBarVEmpty + NV;  // 2 buffers
    static constexpr int kBarPFull = kBarSFull + 2;    // 2 buffers
    static constexpr int kBarPV = kBarPFull + 2;
    static constexpr int kBarDrain = kBarPV + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
    static constexpr uint32_t kBytes = kOffAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    // TMEM columns
    static constexpr uint32_t kColS0 = 0;
    static constexpr uint32_t kColS1 = 128;
    static constexpr uint32_t kColO = 256;
    static constexpr uint32_t kColP0 = 256 + D;
    static constexpr uint32_t kColP1 = 256 + D + 64;
    static_assert(kColP1 + 64 <= kTmemCols, "TMEM budget");
    static_assert(D == 64 || D == 128, "head dim");
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

template <int D, int NK, int NV>
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
    const int n_kv = p.causal ? (qt + 1) : p.n_tiles;
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
            mbar_init(bar(L::kBarPFull + b), 4);  // one arrival per softmax warp
        }
        mbar_init(bar(L::kBarPV), 1);
        mbar_init(bar(L::kBarDrain), 1);
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
        // TMA producer: Q once, then K_0, and K_{j+1} ahead of V_j, which is
        // the order the MMA warp consumes them in.
        // ------------------------------------------------------------------
        if (lane == 0) {
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
                                c * 64, j * kBlockN, bh);
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
                                c * 64, j * kBlockN, bh);
                ++nv;
                return true;
            };
            bool ok = load_k(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) ok = load_k(j + 1);
                if (ok) ok = load_v(j);
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
        // MMA issuer (one thread).  Order: S_0, S_1, then per j:
        // [P_j ready] O += P_j V_j, S_{j+2}.
        // ------------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, false, true);
            bool ok = fa_wait(bar(L::kBarQ), 0, abort_flag, limit, kStatusMmaWaitQ);
            auto issue_s = [&](int j) -> bool {
                const int s = j % NK;
                const uint32_t r = (uint32_t)(j / NK);
                if (!fa_wait(bar(L::kBarKFull + s), r & 1u, abort_flag, limit, kStatusMmaWaitK)) return false;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem + ((j & 1) ? L::kColS1 : L::kColS0);
                const uint32_t qa = sbase + L::kOffQ;
                const uint32_t ka = sbase + L::kOffK + s * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kChunkBytes + (uint32_t)(kk & 3) * 32u;
                    mma_ss(d_tmem, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), kIdescS,
                           kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(L::kBarKEmpty + s));
                tc_commit(bar(L::kBarSFull + (j & 1)));
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n_kv > 1) ok = issue_s(1);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int b = j & 1;
                if (!fa_wait(bar(L::kBarPFull + b), (uint32_t)((j >> 1) & 1), abort_flag, limit, kStatusMmaWaitP)) {
                    ok = false;
                    break;
                }
                const int s = j % NV;
                const uint32_t r = (uint32_t)(j / NV);
                if (!fa_wait(bar(L::kBarVFull + s), r & 1u, abort_flag, limit, kStatusMmaWaitV)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t va = sbase + L::kOffV + s * L::kTileBytes;
                const uint32_t pa = tmem + (b ? L::kColP1 : L::kColP0);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts(tmem + L::kColO, pa + (uint32_t)kk * 8u, sdesc_sw128(va + (uint32_t)kk * 2048u, kChunkBytes, 1024),
                           kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(L::kBarVEmpty + s));
                tc_commit(bar(L::kBarPV));
                if (j + 2 < n_kv) ok = issue_s(j + 2);
            }
            // every MMA must finish before TMEM is released
            tc_commit(bar(L::kBarDrain));
            fa_wait_drain(bar(L::kBarDrain), 0, limit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------
        // Softmax / correction / epilogue: thread = one query row = TMEM lane.
        // ------------------------------------------------------------------
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int q_idx = qt * kBlockM + row;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const float c2 = p.scale_log2;
        float m_run = -INFINITY;  // running max, base-2 scaled units
        float l_run = 0.f;        // running sum of 2^(t - m_run)
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
                const uint32_t scol = t_lane + (b ? L::kColS1 : L::kColS0);
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32_wait(scol + 32u * c, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(r[i]);
                }
            }
            // mask keys past the diagonal (causal) and past the end of the sequence
            int lim = p.N - 1 - j * kBlockN;
            if (p.causal && j == qt) lim = min(lim, row);
            if (lim < kBlockN - 1) {
#pragma unroll
                for (int i = 0; i < kBlockN; ++i) s[i] = (i > lim) ? -INFINITY : s[i];
            }
            // tile row max (scale > 0, so max(s) * c2 == max(s * c2))
            float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int i = 4; i < kBlockN; i += 4) {
                mx[0] = fmaxf(mx[0], s[i + 0]);
                mx[1] = fmaxf(mx[1], s[i + 1]);
                mx[2] = fmaxf(mx[2], s[i + 2]);
                mx[3] = fmaxf(mx[3], s[i + 3]);
            }
            const float tile_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const float m_new = fmaxf(m_run, tile_max * c2);
            // correction factor; exp2(-inf) = 0 wipes the empty initial state,
            // and a row with nothing visible yet keeps factor 1 (no -inf - -inf)
            const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m_run - m_new);
            const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
            uint32_t pk[kBlockN / 2];
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < kBlockN / 2; ++i) {
                const float p0 = ex2_approx(fmaf(s[2 * i], c2, neg_m));
                const float p1 = ex2_approx(fmaf(s[2 * i + 1], c2, neg_m));
                rs[(2 * i) & 3] += p0;
                rs[(2 * i + 1) & 3] += p1;
                pk[i] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
            m_run = m_new;
            if (j > 0) {
                // O holds P_{j-1} V_{j-1} once that product has finished; rescale it
                if (!fa_wait_warp(bar(L::kBarPV), (uint32_t)((j - 1) & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitPV)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32_wait(t_lane + L::kColO + 32u * c, r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(t_lane + L::kColO + 32u * c, r);
                    }
                }
            }
            const uint32_t pcol = t_lane + (b ? L::kColP1 : L::kColP0);
            tmem_st32(pcol, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
            tmem_st32(pcol + 32u, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kBarPFull + b));
        }
        if (ok)
            ok = fa_wait_warp(bar(L::kBarPV), (uint32_t)((n_kv - 1) & 1), abort_flag, limit, kStatusSoftmaxWaitPV);
        const uint32_t stage = sbase + L::kOffQ;  // Q is dead once the last S product has finished
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
                for (int t = 0; t < 4; ++t) {
                    const uint32_t u = (uint32_t)((c & 1) * 4 + t);  // 16-byte unit within the 128-byte row
                    st_shared_v4(chunk + ((u ^ (uint32_t)(row & 7)) << 4), w[4 * t], w[4 * t + 1], w[4 * t + 2],
                                 w[4 * t + 3]);
                }
            }
            if (q_idx < p.N)
                p.lse[(size_t)bh * (size_t)p.N + (size_t)q_idx] =
                    l_run > 0.f ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_barrier_sync(1, 128);
        if (warp == 2 && lane == 0 && *abort_flag == 0) {
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) tma_store_3d(&tm_o, stage + c * kChunkBytes, c * 64, qt * kBlockM, bh);
            bulk_commit_group();
            bulk_wait_group_all();
        }
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
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
