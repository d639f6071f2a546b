// fa_bwd_kernel.cuh -- attention backward pass for sm_103a (GB300).
//
// Gradients of L = sum(O * dO) through O = softmax(scale Q K^T) V.  Nothing of
// the forward's N x N weights is stored: the scores are recomputed tile by
// tile from Q and K and normalised with the saved per-row statistic LSE, so
// each tile is final in one pass -- no running max or rescaling on the way
// back ("Online Softmax: Tiling Across a Reduction", backward-pass section).
// For a visible pair (i, j):
//
//     P_ij  = exp(S_ij - LSE_i)                     S_ij = scale q_i . k_j
//     D_i   = sum_c dO_ic O_ic
//     dV_j  = sum_i P_ij dO_i
//     dS_ij = P_ij (dO_i . v_j - D_i)
//     dQ_i  = scale sum_j dS_ij k_j,      dK_j = scale sum_i dS_ij q_i
//
// Three kernels, enqueued in this order:
//   * fa_bwd_delta: D_i, one warp per row, into a caller workspace.
//   * fa_bwd_dq_sm103: one CTA per query tile (Q, dO resident in shared
//     memory; K_j, V_j streamed by TMA).  Per key tile: S = Q K_j^T and
//     dP = dO V_j^T on tcgen05.mma into TMEM; the compute warps (thread =
//     query row = TMEM lane) turn them into dS in bf16, written back to TMEM;
//     dQ += dS K_j is a TMEM-A (TS) product.  dQ never leaves TMEM until the
//     epilogue, so no atomics are needed.
//   * fa_bwd_dkdv_sm103: one CTA per key tile (K, V resident; Q_i, dO_i
//     streamed).  Per query tile: S^T = K Q_i^T and dP^T = V dO_i^T into TMEM;
//     the compute warps (thread = key row) write P^T and dS^T in bf16 (over
//     the columns they have just read at d = 128, into spare columns at
//     d = 64); dV += P^T dO_i and dK += dS^T Q_i are TS products accumulating
//     in TMEM.
// Splitting dQ from dK/dV costs two extra products per tile pair (S and dP
// are formed twice) and buys kernels with no cross-CTA reduction.
//
// Warp roles (384 threads): warp 0 issues TMA loads, warp 1 owns TMEM, and
// warps 1 and 3 issue the MMAs (dQ kernel: S and dP on warp 1, dQ on warp 3;
// dK/dV kernel: S^T then dV on warp 1, dP^T then dK on warp 3), each running
// its loop on the whole warp and issuing from an elect.sync lane.  Warps 4-11
// compute: two warps per 32-row TMEM lane quarter, each taking half of the
// 128 columns of a step and half of the epilogue.
// Every barrier wait is bounded by the same watchdog as the forward kernel.
#pragma once

#include <cuda_bf16.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kBwdThreads = 384;  // 12 warps: 8 of them compute, two per TMEM lane quarter

// D_i = sum_c dO_ic O_ic in fp32, one warp per row; rows = B*H*N
template <int D>
__global__ void __launch_bounds__(256)
    fa_bwd_delta(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout, float* __restrict__ delta,
                 long long rows) {
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(o + (size_t)row * D);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(dout + (size_t)row * D);
    float acc = 0.f;
#pragma unroll
    for (int c = lane; c < D / 2; c += 32) {
        const float2 a = __bfloat1622float2(o2[c]), b = __bfloat1622float2(d2[c]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[row] = acc;
}

struct BwdParams {
    void* grad;             // dq kernel: dQ; dkdv kernel: dK (bf16 [B*H][N][d])
    void* grad2;            // dkdv kernel: dV
    const float* lse;       // fp32 [B*H][N], natural log
    const float* delta;     // fp32 [B*H][N]
    int N, n_tiles, causal;
    float scale, scale_log2;
    unsigned long long watchdog_ns;
};

// shared memory of the dK/dV kernel: two resident tiles, a ring of NS stages of
// two streamed tiles, barriers, per-warp LSE/D staging
template <int D, int NS>
struct BwdSmem {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = 128u * D * 2u;
    static constexpr uint32_t kOffRes = 0;                            // resident tiles A, B
    static constexpr uint32_t kOffRing = 2 * kTileBytes;              // [NS][2] streamed tiles
    static constexpr uint32_t kOffBar = kOffRing + NS * 2 * kTileBytes;
    static constexpr int kBarRes = 0;                   // resident tiles landed
    static constexpr int kBarFull = 1;                  // [NS] stage landed
    static constexpr int kBarEmpty = kBarFull + NS;     // [NS] stage consumed by the MMAs
    // [2] each: SFull per score-like product (S, dP); DSFull and Used per dK/dV issuer in
    // the dK/dV kernel, Used per dS buffer in the dQ kernel
    static constexpr int kBarSFull = kBarEmpty + NS;    // score-like product of a step finished
    static constexpr int kBarDSFull = kBarSFull + 2;    // compute warps wrote the bf16 operand(s)
    static constexpr int kBarUsed = kBarDSFull + 2;     // the products reading those operands finished
    static constexpr int kBarFinal = kBarUsed + 2;      // the accumulators are complete
    static constexpr int kBarDrain = kBarFinal + 1;     // [2] per MMA issuer
    static constexpr int kBarSRead = kBarDrain + 2;     // [2] dQ kernel: the compute warps hold S / dP in registers
    static constexpr int kBarPHalf = kBarSRead + 2;     // dK/dV kernel, d = 128: half of each warp's P^T written
    static constexpr int kNumBars = kBarPHalf + 1;
    static constexpr uint32_t kOffStage = kOffBar + kNumBars * 8;     // [8 warps][2][LSE 128, D 128] floats
    static constexpr uint32_t kOffTmemSlot = kOffStage + 8 * 2 * 256 * 4;
    static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
    static constexpr uint32_t kBytes = kOffAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448u, "shared memory");
};

// shared memory of the dQ kernel: Q and dO resident, then separate rings of NK
// key and NV value tiles.  K_j is read by S_j and, a whole step later, by the dQ
// product; V_j only by dP_j.  So K needs the deeper ring: with one ring of K and V
// stages the next K_{j+2} could only load once dQ_j had finished, and S_{j+2}
// waited for that load.
template <int D, int NK, int NV>
struct DqSmem {
    static constexpr uint32_t kTileBytes = 128u * D * 2u;
    static constexpr uint32_t kOffRes = 0;                       // Q, dO
    static constexpr uint32_t kOffK = 2 * kTileBytes;            // [NK] key tiles
    static constexpr uint32_t kOffV = kOffK + NK * kTileBytes;   // [NV] value tiles
    static constexpr uint32_t kOffBar = kOffV + NV * kTileBytes;
    static constexpr int kBarRes = 0;                    // resident tiles landed
    static constexpr int kBarKFull = 1;                  // [NK] key stage landed
    static constexpr int kBarKEmpty = kBarKFull + NK;    // [NK] key stage read by S_j and dQ_j
    static constexpr int kBarVFull = kBarKEmpty + NK;    // [NV]
    static constexpr int kBarVEmpty = kBarVFull + NV;    // [NV] value stage read by dP_j
    static constexpr int kBarSFull = kBarVEmpty + NV;    // [2] S_j / dP_j finished
    static constexpr int kBarDSFull = kBarSFull + 2;     // dS_j written
    static constexpr int kBarUsed = kBarDSFull + 1;      // [2] per dS buffer: its dQ product finished
    static constexpr int kBarFinal = kBarUsed + 2;       // dQ complete
    static constexpr int kBarDrain = kBarFinal + 1;      // [2] per MMA issuer
    static constexpr int kBarSRead = kBarDrain + 2;      // [2] the compute warps hold S / dP in registers
    static constexpr int kNumBars = kBarSRead + 2;
    static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
    static constexpr uint32_t kBytes = kOffAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448u, "shared memory");
};

// loads of the 64-column chunks of a [128 rows][D] tile
template <int D>
__device__ __forceinline__ void bwd_load_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar, int row0, int bh) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * kChunkBytes, m, bar, c * 64, row0, bh);
}

// ---------------------------------------------------------------------------
// dQ: one CTA per (query tile, head).  TMEM: S [0,128), dP [128,256),
// dQ [256, 256+D), dS bf16 in two buffers [256+D, 256+D+64) and
// [256+D+64, 256+D+128), alternating by step, so that dS(j) is formed while
// the dQ product of dS(j-1) still reads the other buffer.
// ---------------------------------------------------------------------------
template <int D, int NK, int NV>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
    using L = DqSmem<D, NK, NV>;
    constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 256 + D;
    static_assert(256 + D + 128 <= kTmemCols, "TMEM budget");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = (int)(threadIdx.x & 31);
    const uint64_t limit = p.watchdog_ns;
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest causal tiles first
    const int bh = (int)blockIdx.y;
    const int n_kv = p.causal ? min(qt + 1, p.n_tiles) : p.n_tiles;

    if (warp == 0 && lane == 0) {
        mbar_init(bar(L::kBarRes), 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(L::kBarKFull + s), 1);
            mbar_init(bar(L::kBarKEmpty + s), 1);  // the dQ product's commit
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(L::kBarVFull + s), 1);
            mbar_init(bar(L::kBarVEmpty + s), 1);  // the dP product's commit
        }
        mbar_init(bar(L::kBarSFull + 0), 1);  // S
        mbar_init(bar(L::kBarSFull + 1), 1);  // dP
        mbar_init(bar(L::kBarDSFull), 8);
        mbar_init(bar(L::kBarUsed + 0), 1);  // per dS buffer: its dQ product finished
        mbar_init(bar(L::kBarUsed + 1), 1);
        mbar_init(bar(L::kBarFinal), 1);
        mbar_init(bar(L::kBarDrain), 1);
        mbar_init(bar(L::kBarDrain + 1), 1);
        mbar_init(bar(L::kBarSRead + 0), 8);  // S in registers
        mbar_init(bar(L::kBarSRead + 1), 8);  // dP in registers
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t res_q = sbase + L::kOffRes, res_do = sbase + L::kOffRes + L::kTileBytes;
    auto ring_k = [&](int s) { return sbase + L::kOffK + (uint32_t)s * L::kTileBytes; };
    auto ring_v = [&](int s) { return sbase + L::kOffV + (uint32_t)s * L::kTileBytes; };

    if (warp == 0) {
        // the whole warp walks the loop; one elected lane issues the copies
        {
            bool ok = true;
            if (elect_one_sync()) {
                mbar_arrive_expect_tx(bar(L::kBarRes), 2 * L::kTileBytes);
                bwd_load_tile<D>(res_q, &tm_q, bar(L::kBarRes), qt * 128, bh);
                bwd_load_tile<D>(res_do, &tm_do, bar(L::kBarRes), qt * 128, bh);
            }
            __syncwarp();
            int nk = 0, nv = 0;  // key and value tiles loaded
            while (ok && nk < n_kv) {
                const int j = nk;
                const int sk = j % NK, sv = j % NV;
                if (j >= NK)
                    ok = fa_wait_warp(bar(L::kBarKEmpty + sk), (uint32_t)(((j - NK) / NK) & 1), abort_flag, limit,
                                      kStatusLoadWait);
                if (!ok) break;
                if (elect_one_sync()) {
                    mbar_arrive_expect_tx(bar(L::kBarKFull + sk), L::kTileBytes);
                    bwd_load_tile<D>(ring_k(sk), &tm_k, bar(L::kBarKFull + sk), j * 128, bh);
                }
                __syncwarp();
                ++nk;
                if (j >= NV)
                    ok = fa_wait_warp(bar(L::kBarVEmpty + sv), (uint32_t)(((j - NV) / NV) & 1), abort_flag, limit,
                                      kStatusLoadWait);
                if (!ok) break;
                if (elect_one_sync()) {
                    mbar_arrive_expect_tx(bar(L::kBarVFull + sv), L::kTileBytes);
                    bwd_load_tile<D>(ring_v(sv), &tm_v, bar(L::kBarVFull + sv), j * 128, bh);
                }
                __syncwarp();
                ++nv;
            }
            if (lane == 0 && (!ok || *abort_flag)) {  // let every issued copy land before the CTA exits
                fa_wait_drain(bar(L::kBarRes), 0, limit);
                for (int s = 0; s < NK; ++s)
                    if (nk > s) fa_wait_drain(bar(L::kBarKFull + s), (uint32_t)(((nk - 1 - s) / NK) & 1), limit);
                for (int s = 0; s < NV; ++s)
                    if (nv > s) fa_wait_drain(bar(L::kBarVFull + s), (uint32_t)(((nv - 1 - s) / NV) & 1), limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // score products: S_j = Q K_j^T and then dP_j = dO V_j^T, each as soon as
        // K_j, V_j have landed and the compute warps hold S_{j-1} (resp. dP_{j-1}) in
        // registers; each is signalled on its own, so the compute warps start on S_j
        // while dP_j is still being formed
        {
            constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
            const uint64_t qd = sdesc_sw128(res_q, 16, 1024), dod = sdesc_sw128(res_do, 16, 1024);
            bool ok = fa_wait_warp(bar(L::kBarRes), 0, abort_flag, limit, kStatusMmaWaitQ);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int sk = j % NK, sv = j % NV;
                ok = fa_wait_warp(bar(L::kBarKFull + sk), (uint32_t)((j / NK) & 1), abort_flag, limit, kStatusMmaWaitK);
                if (ok && j > 0)
                    ok = fa_wait_warp(bar(L::kBarSRead + 0), (uint32_t)((j - 1) & 1), abort_flag, limit,
                                      kStatusMmaWaitSFree);
                if (!ok) break;
                tc_fence_after_sync();
                const uint64_t kd = sdesc_sw128(ring_k(sk), 16, 1024), vd = sdesc_sw128(ring_v(sv), 16, 1024);
                if (elect_one_sync()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((uint32_t)(kk >> 2) * kChunkBytes + (uint32_t)(kk & 3) * 32u) >> 4;
                        mma_ss(tmem + kColS, sdesc_add_lo(qd, off), sdesc_add_lo(kd, off), kIdescS, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(L::kBarSFull + 0));
                }
                __syncwarp();
                ok = fa_wait_warp(bar(L::kBarVFull + sv), (uint32_t)((j / NV) & 1), abort_flag, limit, kStatusMmaWaitV);
                if (ok && j > 0)
                    ok = fa_wait_warp(bar(L::kBarSRead + 1), (uint32_t)((j - 1) & 1), abort_flag, limit,
                                      kStatusMmaWaitSFree);
                if (!ok) break;
                tc_fence_after_sync();
                if (elect_one_sync()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((uint32_t)(kk >> 2) * kChunkBytes + (uint32_t)(kk & 3) * 32u) >> 4;
                        mma_ss(tmem + kColDP, sdesc_add_lo(dod, off), sdesc_add_lo(vd, off), kIdescS,
                               kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(L::kBarSFull + 1));
                    tc_commit(bar(L::kBarVEmpty + sv));  // V_j is read by dP_j only
                }
                __syncwarp();
            }
            if (elect_one_sync()) {
                tc_commit(bar(L::kBarDrain));
                fa_wait_drain(bar(L::kBarDrain), 0, limit);
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // gradient products, on a second issuing thread so that they overlap the
        // next step's score products: dQ += dS_j K_j once dS_j is in TMEM
        {
            constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, false, true);
            bool ok = fa_wait_warp(bar(L::kBarRes), 0, abort_flag, limit, kStatusMmaWaitQ);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j % NK;
                ok = fa_wait_warp(bar(L::kBarKFull + s), (uint32_t)((j / NK) & 1), abort_flag, limit,
                                  kStatusMmaWaitK) &&
                     fa_wait_warp(bar(L::kBarDSFull), (uint32_t)(j & 1), abort_flag, limit, kStatusMmaWaitP);
                if (!ok) break;
                tc_fence_after_sync();
                const uint64_t kd = sdesc_sw128(ring_k(s), kChunkBytes, 1024);  // + 2048 bytes per 16 keys
                if (elect_one_sync()) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kColDQ, tmem + kColDS + 64u * (uint32_t)(j & 1) + (uint32_t)kk * 8u,
                               sdesc_add_lo(kd, (uint32_t)kk * 128u), kIdescDQ, (j > 0 || kk > 0) ? 1u : 0u);
                    // S_j finished before dS_j was written, so this covers both products
                    // that read K_j
                    tc_commit(bar(L::kBarKEmpty + s));
                    tc_commit(bar(L::kBarUsed + (j & 1)));
                }
                __syncwarp();
            }
            if (elect_one_sync()) {
                if (ok && n_kv > 0) tc_commit(bar(L::kBarFinal));
                tc_commit(bar(L::kBarDrain + 1));
                fa_wait_drain(bar(L::kBarDrain + 1), 0, limit);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const int half = (warp - 4) >> 2;  // columns [64 half, 64 half + 64) of every step
        const int row = quarter * 32 + lane;
        const int q_idx = qt * 128 + row;
        const bool valid = q_idx < p.N;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const size_t r = (size_t)bh * p.N + (size_t)q_idx;
        // rows past N: P = 0 (LSE = +inf), nothing stored
        const float lse2 = valid ? p.lse[r] * kLog2e : INFINITY;
        const float drow = valid ? p.delta[r] : 0.f;
        const float c2 = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            // Phase 1, as soon as S_j is in: P in place of S (fp32 bits), while dP_j
            // is still being formed
            ok = fa_wait_warp(bar(L::kBarSFull + 0), (uint32_t)(j & 1), abort_flag, limit, kStatusSoftmaxWaitS);
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t sv[64], dv[64];
            tmem_ld64_wait(t_lane + kColS + 64u * half, sv);
            tc_fence_before_sync();
            __syncwarp();
            if (elect_one_sync()) mbar_arrive(bar(L::kBarSRead + 0));  // S columns free for S_{j+1}
            // keys visible to this row in this tile: c <= last
            int last = p.N - 1 - j * 128;
            if (p.causal && j == qt) last = min(last, row);
            if (__all_sync(0xffffffffu, last >= 127)) {
                // every key of the tile visible to every row of the warp: packed
                // fp32x2 arithmetic, no masks
                const uint64_t c2x2 = f32x2_pack(c2, c2), nl2 = f32x2_pack(-lse2, -lse2);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x0, x1;
                    f32x2_unpack(ffma2(f32x2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), c2x2, nl2),
                                 x0, x1);
                    sv[2 * i] = __float_as_uint(ex2_approx(x0));
                    sv[2 * i + 1] = __float_as_uint(ex2_approx(x1));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const int c = 64 * half + e;
                    sv[e] = __float_as_uint((c <= last) ? ex2_approx(fmaf(__uint_as_float(sv[e]), c2, -lse2)) : 0.f);
                }
            }
            // Phase 2, once dP_j is in: dS = P (dP - D) into dS buffer j & 1
            ok = fa_wait_warp(bar(L::kBarSFull + 1), (uint32_t)(j & 1), abort_flag, limit, kStatusSoftmaxWaitS);
            if (!ok) break;
            tc_fence_after_sync();
            tmem_ld64_wait(t_lane + kColDP + 64u * half, dv);
            tc_fence_before_sync();
            __syncwarp();
            if (elect_one_sync()) mbar_arrive(bar(L::kBarSRead + 1));  // dP columns free for dP_{j+1}
            // dS buffer j & 1 last held dS(j-2): its dQ product must have read it
            if (j >= 2)
                ok = fa_wait_warp(bar(L::kBarUsed + (j & 1)), (uint32_t)(((j - 2) >> 1) & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitPV);
            if (!ok) break;
            tc_fence_after_sync();
            {
                const uint64_t nd2 = f32x2_pack(-drow, -drow);
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    const int ch = 2 * half + hc;
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 32 * hc + 2 * i;
                        float d0, d1;
                        f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                           fadd2(f32x2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd2)),
                                     d0, d1);
                        pk[i] = pack_bf16x2(d0, d1);
                    }
                    tmem_st16(t_lane + kColDS + 64u * (uint32_t)(j & 1) + 16u * ch, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (elect_one_sync()) mbar_arrive(bar(L::kBarDSFull));
        }
        if (ok && n_kv > 0) ok = fa_wait_warp(bar(L::kBarFinal), 0, abort_flag, limit, kStatusSoftmaxWaitO);
        if (ok) {
            tc_fence_after_sync();
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.grad) + r * D);
#pragma unroll
            for (int hc = 0; hc < D / 64; ++hc) {  // this warp's half of the columns
                const int c = half * (D / 64) + hc;
                uint32_t v[32];
                tmem_ld32_wait(t_lane + kColDQ + 32u * c, v);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack_bf16x2(n_kv > 0 ? __uint_as_float(v[2 * i]) * p.scale : 0.f,
                                       n_kv > 0 ? __uint_as_float(v[2 * i + 1]) * p.scale : 0.f);
                if (valid) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) dst[c * 4 + u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
            }
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

// ---------------------------------------------------------------------------
// dK, dV: one CTA per (key tile, head).  TMEM: S^T [0,128), dP^T [128,256),
// dV [256, 256+D), dK [256+D, 256+2D).  The bf16 operands P^T and dS^T:
//  * D = 128 (TMEM full): over the columns they are formed from, [0,32) and
//    [64,96) of S^T (resp. dP^T), so a score product waits until the gradient
//    product of the step before has read them;
//  * D = 64: in columns of their own, P^T [384,448), dS^T [448,512), so the
//    next score product starts as soon as the compute warps hold the scores
//    in registers, and only the operand store waits for the gradient product.
// ---------------------------------------------------------------------------
template <int D, int NS>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const BwdParams p) {
    using L = BwdSmem<D, NS>;
    constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    constexpr bool kSepOp = 256 + 2 * D + 128 <= kTmemCols;  // operands in columns of their own
    constexpr uint32_t kColOp0 = kSepOp ? 256 + 2 * D : kColS, kColOp1 = kSepOp ? 256 + 2 * D + 64 : kColDP;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = (int)(threadIdx.x & 31);
    const uint64_t limit = p.watchdog_ns;
    const int kt = (int)blockIdx.x;  // causal: the lowest key tiles see the most query tiles and go first
    const int bh = (int)blockIdx.y;
    const int i0 = p.causal ? kt : 0;
    const int n_q = p.n_tiles - i0;

    if (warp == 0 && lane == 0) {
        mbar_init(bar(L::kBarRes), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(L::kBarFull + s), 1);
            mbar_init(bar(L::kBarEmpty + s), 2);  // both issuers' products read the stage
        }
        mbar_init(bar(L::kBarSFull + 0), 1);   // S^T (warp 1)
        mbar_init(bar(L::kBarSFull + 1), 1);   // dP^T (warp 3)
        mbar_init(bar(L::kBarDSFull + 0), 8);  // P^T written
        mbar_init(bar(L::kBarDSFull + 1), 8);  // dS^T written
        mbar_init(bar(L::kBarUsed + 0), 1);  // dV products (warp 1)
        mbar_init(bar(L::kBarUsed + 1), 1);  // dK products (warp 3)
        mbar_init(bar(L::kBarFinal), 2);
        mbar_init(bar(L::kBarDrain), 1);
        mbar_init(bar(L::kBarDrain + 1), 1);
        mbar_init(bar(L::kBarSRead + 0), 8);  // S^T in registers (separate operand columns only)
        mbar_init(bar(L::kBarSRead + 1), 8);  // dP^T in registers
        mbar_init(bar(L::kBarPHalf), 8);      // the first 32 queries of each warp's P^T written (d = 128)
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t res_k = sbase + L::kOffRes, res_v = sbase + L::kOffRes + L::kTileBytes;
    auto ring_q = [&](int s) { return sbase + L::kOffRing + (uint32_t)(2 * s) * L::kTileBytes; };
    auto ring_do = [&](int s) { return sbase + L::kOffRing + (uint32_t)(2 * s + 1) * L::kTileBytes; };

    if (warp == 0) {
        {
            bool ok = true;
            if (elect_one_sync()) {
                mbar_arrive_expect_tx(bar(L::kBarRes), 2 * L::kTileBytes);
                bwd_load_tile<D>(res_k, &tm_k, bar(L::kBarRes), kt * 128, bh);
                bwd_load_tile<D>(res_v, &tm_v, bar(L::kBarRes), kt * 128, bh);
            }
            __syncwarp();
            int i = 0;
            for (; ok && i < n_q; ++i) {
                const int s = i % NS;
                if (i >= NS)
                    ok = fa_wait_warp(bar(L::kBarEmpty + s), (uint32_t)(((i - NS) / NS) & 1), abort_flag, limit,
                                      kStatusLoadWait);
                if (!ok) break;
                if (elect_one_sync()) {
                    mbar_arrive_expect_tx(bar(L::kBarFull + s), 2 * L::kTileBytes);
                    bwd_load_tile<D>(ring_q(s), &tm_q, bar(L::kBarFull + s), (i0 + i) * 128, bh);
                    bwd_load_tile<D>(ring_do(s), &tm_do, bar(L::kBarFull + s), (i0 + i) * 128, bh);
                }
                __syncwarp();
            }
            if (lane == 0 && (!ok || *abort_flag)) {
                fa_wait_drain(bar(L::kBarRes), 0, limit);
                for (int s = 0; s < NS; ++s)
                    if (i > s) fa_wait_drain(bar(L::kBarFull + s), (uint32_t)(((i - 1 - s) / NS) & 1), limit);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // Two issuing threads, so that two MMA streams run at once: warp 1 issues
        // S^T = K Q_i^T and then dV += P^T dO_i, warp 3 issues dP^T = V dO_i^T and
        // then dK += dS^T Q_i.  Each thread's score product overwrites the columns
        // its own gradient product of step i-1 read, so it waits for that product.
        {
            const int u = warp == 1 ? 0 : 1;  // 0: S / dV, 1: dP / dK
            constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, false, true);
            const uint32_t res_a = u == 0 ? res_k : res_v;  // K for S^T, V for dP^T
            const uint32_t col_sc = u == 0 ? kColS : kColDP;
            const uint32_t col_acc = u == 0 ? kColDV : kColDK;
            const uint64_t ad = sdesc_sw128(res_a, 16, 1024);
            bool ok = fa_wait_warp(bar(L::kBarRes), 0, abort_flag, limit, kStatusMmaWaitQ);
            if constexpr (kSepOp) {
                const uint32_t col_op = u == 0 ? kColOp0 : kColOp1;  // its bf16 operand
                // the score product of step i, once Q_i / dO_i have landed and the compute
                // warps hold the scores of step i-1 in registers
                auto score = [&](int i) -> bool {
                    const int s = i % NS;
                    bool k = fa_wait_warp(bar(L::kBarFull + s), (uint32_t)((i / NS) & 1), abort_flag, limit,
                                          kStatusMmaWaitK);
                    if (k && i > 0)
                        k = fa_wait_warp(bar(L::kBarSRead + u), (uint32_t)((i - 1) & 1), abort_flag, limit,
                                         kStatusMmaWaitSFree);
                    if (!k) return false;
                    tc_fence_after_sync();
                    const uint64_t bd = sdesc_sw128(u == 0 ? ring_q(s) : ring_do(s), 16, 1024);
                    if (elect_one_sync()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((uint32_t)(kk >> 2) * kChunkBytes + (uint32_t)(kk & 3) * 32u) >> 4;
                            mma_ss(tmem + col_sc, sdesc_add_lo(ad, off), sdesc_add_lo(bd, off), kIdescS, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(L::kBarSFull + u));
                    }
                    __syncwarp();
                    return true;
                };
                // the gradient product of step i, once its bf16 operand (P^T, written
                // first, or dS^T) is in TMEM
                auto gradient = [&](int i) -> bool {
                    const int s = i % NS;
                    if (!fa_wait_warp(bar(L::kBarDSFull + u), (uint32_t)(i & 1), abort_flag, limit, kStatusMmaWaitP))
                        return false;
                    tc_fence_after_sync();
                    // the operands of queries 16 kk .. 16 kk + 15 sit at column 8 kk; the B rows
                    // advance 2048 bytes per 16 queries
                    const uint64_t gd = sdesc_sw128(u == 0 ? ring_do(s) : ring_q(s), kChunkBytes, 1024);
                    if (elect_one_sync()) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tmem + col_acc, tmem + col_op + (uint32_t)kk * 8u,
                                   sdesc_add_lo(gd, (uint32_t)kk * 128u), kIdescG, (i > 0 || kk > 0) ? 1u : 0u);
                        // covers every earlier product of this thread that read stage s
                        tc_commit(bar(L::kBarEmpty + s));
                        tc_commit(bar(L::kBarUsed + u));
                    }
                    __syncwarp();
                    return true;
                };
                // the score product of step i+1 goes ahead of the gradient product of step i
                if (ok && n_q > 0) ok = score(0);
                for (int i = 0; ok && i < n_q; ++i) {
                    if (i + 1 < n_q) ok = score(i + 1);
                    ok = ok && gradient(i);
                }
            } else {
                for (int i = 0; ok && i < n_q; ++i) {
                    const int s = i % NS;
                    const uint32_t b_sc = u == 0 ? ring_q(s) : ring_do(s);   // B of the score product
                    const uint32_t b_acc = u == 0 ? ring_do(s) : ring_q(s);  // B of the gradient product
                    ok = fa_wait_warp(bar(L::kBarFull + s), (uint32_t)((i / NS) & 1), abort_flag, limit,
                                      kStatusMmaWaitK);
                    // the score columns hold this thread's bf16 operand of step i-1 until its
                    // gradient product has finished
                    if (ok && i > 0)
                        ok = fa_wait_warp(bar(L::kBarUsed + u), (uint32_t)((i - 1) & 1), abort_flag, limit,
                                          kStatusMmaWaitSFree);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint64_t bd = sdesc_sw128(b_sc, 16, 1024);
                    if (elect_one_sync()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((uint32_t)(kk >> 2) * kChunkBytes + (uint32_t)(kk & 3) * 32u) >> 4;
                            mma_ss(tmem + col_sc, sdesc_add_lo(ad, off), sdesc_add_lo(bd, off), kIdescS,
                                   kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(L::kBarSFull + u));
                    }
                    __syncwarp();
                    // the bf16 operands of queries 16 kk .. 16 kk + 15 sit at column 8 kk (first
                    // half of the queries) or 32 + 8 kk (second half); the B rows advance 2048
                    // bytes per 16 queries
                    const uint64_t gd = sdesc_sw128(b_acc, kChunkBytes, 1024);
                    auto grad_mma = [&](int kk) {
                        mma_ts(tmem + col_acc, tmem + col_sc + (uint32_t)kk * 8u + (kk >= 4 ? 32u : 0u),
                               sdesc_add_lo(gd, (uint32_t)kk * 128u), kIdescG, (i > 0 || kk > 0) ? 1u : 0u);
                    };
                    if (u == 0) {
                        // dV in two halves: queries 0-31 and 64-95 (each warp's first 32 columns
                        // of P^T) as soon as those are written, while the rest is formed
                        ok = fa_wait_warp(bar(L::kBarPHalf), (uint32_t)(i & 1), abort_flag, limit, kStatusMmaWaitP);
                        if (!ok) break;
                        tc_fence_after_sync();
                        if (elect_one_sync()) {
                            grad_mma(0);
                            grad_mma(1);
                            grad_mma(4);
                            grad_mma(5);
                        }
                        __syncwarp();
                    }
                    // its bf16 operand: P^T (written first) or dS^T
                    ok = fa_wait_warp(bar(L::kBarDSFull + u), (uint32_t)(i & 1), abort_flag, limit, kStatusMmaWaitP);
                    // dK(i) after S^T(i+1) has finished: the pipe interleaves the two issuers'
                    // products, so issued beside S^T(i+1) it would double the latency of the
                    // product the compute warps wait for next
                    if (ok && u == 1 && i + 1 < n_q)
                        ok = fa_wait_warp(bar(L::kBarSFull + 0), (uint32_t)((i + 1) & 1), abort_flag, limit,
                                          kStatusMmaWaitP);
                    if (!ok) break;
                    tc_fence_after_sync();
                    if (elect_one_sync()) {
                        if (u == 0) {
                            grad_mma(2);
                            grad_mma(3);
                            grad_mma(6);
                            grad_mma(7);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) grad_mma(kk);
                        }
                        tc_commit(bar(L::kBarEmpty + s));
                        tc_commit(bar(L::kBarUsed + u));
                    }
                    __syncwarp();
                }
            }
            if (elect_one_sync()) {
                if (ok && n_q > 0) tc_commit(bar(L::kBarFinal));
                tc_commit(bar(L::kBarDrain + u));
                fa_wait_drain(bar(L::kBarDrain + u), 0, limit);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const int half = (warp - 4) >> 2;      // query columns [64 half, 64 half + 64) of every step
        const int row = quarter * 32 + lane;  // key row of this thread
        const int k_idx = kt * 128 + row;
        const bool valid = k_idx < p.N;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        float* stage = reinterpret_cast<float*>(smem + L::kOffStage) + (warp - 4) * 2 * 256;  // [2][LSE 128, D 128]
        const float c2 = p.scale_log2;
        bool ok = true;
        // LSE and D of query tile i0 + i into staging buffer i & 1, one step ahead,
        // with cp.async (no registers held, no stall on the loads); queries past N
        // read nothing
        auto prefetch = [&](int i) {
            const uint32_t sb = smem_u32(stage + (i & 1) * 256);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = u * 32 + lane;
                const int q = (i0 + i) * 128 + c;
                const bool in = q < p.N;
                const size_t r = (size_t)bh * p.N + (size_t)(in ? q : 0);
                cp_async_4(sb + 4u * (uint32_t)c, p.lse + r, in ? 4u : 0u);
                cp_async_4(sb + 4u * (uint32_t)(128 + c), p.delta + r, in ? 4u : 0u);
            }
        };
        if (n_q > 0) prefetch(0);
        for (int i = 0; i < n_q; ++i) {
            const int qi = i0 + i;
            // this query tile's -LSE (log2 units) and -D: each lane converts the entries
            // it copied; queries past N get -LSE = -inf, so their weights are 0
            float* st = stage + (i & 1) * 256;
            cp_async_wait_all();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = u * 32 + lane;
                const bool in = qi * 128 + c < p.N;
                st[c] = in ? -(st[c] * kLog2e) : -INFINITY;
                st[128 + c] = in ? -st[128 + c] : 0.f;
            }
            __syncwarp();
            if (i + 1 < n_q) prefetch(i + 1);
            // causal: query q sees key k_idx iff k_idx <= q, i.e. column c >= first
            // (only the diagonal tile masks; queries past N weigh 0 through -LSE)
            const bool diag = p.causal && qi == kt;
            const int first = diag ? row : 0;
            const uint64_t c2x2 = f32x2_pack(c2, c2);
            // P^T and dS^T of query columns [64 half, +64) go to operand columns
            // [32 half, 32 half + 32) of their own (separate operand columns), or over
            // the scores to [64 half, 64 half + 32): inside what this warp has already
            // read (64 half + 16 hc + 16 <= 64 half + 32 hc + 32), never into the other
            // half's columns.
            const uint32_t op_off = kSepOp ? 32u * (uint32_t)half : 64u * (uint32_t)half;
            // Phase 1, as soon as S^T is in: P, stored as bf16 for the dV product
            // (which starts at once) and kept in fp32 for dS.
            ok = fa_wait_warp(bar(L::kBarSFull + 0), (uint32_t)(i & 1), abort_flag, limit, kStatusSoftmaxWaitS);
            // separate operand columns: P^T of step i-1 must have been read by its dV product
            if (kSepOp && ok && i > 0)
                ok = fa_wait_warp(bar(L::kBarUsed + 0), (uint32_t)((i - 1) & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitPV);
            if (!ok) break;
            tc_fence_after_sync();
            float pf[64];
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                const int ch = 2 * half + hc;
                uint32_t sv[32], pk[16];
                tmem_ld32_wait(t_lane + kColS + 32u * ch, sv);
                if (kSepOp && hc == 1) {  // S^T is in registers: its columns may take S^T(i+1)
                    tc_fence_before_sync();
                    __syncwarp();
                    if (elect_one_sync()) mbar_arrive(bar(L::kBarSRead + 0));
                }
                if (!diag) {
                    // packed fp32x2 arithmetic; -LSE of two queries per load
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2) {
                        const int c0 = 32 * ch + 2 * i2;
                        const float2 nl = *reinterpret_cast<const float2*>(st + c0);
                        float x0, x1;
                        f32x2_unpack(ffma2(f32x2_pack(__uint_as_float(sv[2 * i2]), __uint_as_float(sv[2 * i2 + 1])),
                                           c2x2, f32x2_pack(nl.x, nl.y)),
                                     x0, x1);
                        pf[32 * hc + 2 * i2] = ex2_approx(x0);
                        pf[32 * hc + 2 * i2 + 1] = ex2_approx(x1);
                    }
                } else {
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2) {
                        const int c0 = 32 * ch + 2 * i2;
                        pf[32 * hc + 2 * i2] =
                            (c0 >= first) ? ex2_approx(fmaf(__uint_as_float(sv[2 * i2]), c2, st[c0])) : 0.f;
                        pf[32 * hc + 2 * i2 + 1] =
                            (c0 + 1 >= first) ? ex2_approx(fmaf(__uint_as_float(sv[2 * i2 + 1]), c2, st[c0 + 1])) : 0.f;
                    }
                }
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2) pk[i2] = pack_bf16x2(pf[32 * hc + 2 * i2], pf[32 * hc + 2 * i2 + 1]);
                tmem_st16(t_lane + kColOp0 + op_off + 16u * hc, pk);
                if (!kSepOp && hc == 0) {  // the first half of the dV product may start
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (elect_one_sync()) mbar_arrive(bar(L::kBarPHalf));
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (elect_one_sync()) mbar_arrive(bar(L::kBarDSFull + 0));
            // Phase 2, once dP^T is in: dS = P (dP - D), for the dK product
            ok = fa_wait_warp(bar(L::kBarSFull + 1), (uint32_t)(i & 1), abort_flag, limit, kStatusSoftmaxWaitS);
            if (kSepOp && ok && i > 0)  // dS^T of step i-1 read by its dK product
                ok = fa_wait_warp(bar(L::kBarUsed + 1), (uint32_t)((i - 1) & 1), abort_flag, limit,
                                  kStatusSoftmaxWaitPV);
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                const int ch = 2 * half + hc;
                uint32_t dv[32], dk[16];
                tmem_ld32_wait(t_lane + kColDP + 32u * ch, dv);
                if (kSepOp && hc == 1) {  // dP^T is in registers: its columns may take dP^T(i+1)
                    tc_fence_before_sync();
                    __syncwarp();
                    if (elect_one_sync()) mbar_arrive(bar(L::kBarSRead + 1));
                }
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2) {
                    const int c0 = 32 * ch + 2 * i2;
                    const float2 nd = *reinterpret_cast<const float2*>(st + 128 + c0);
                    float d0, d1;
                    f32x2_unpack(fmul2(f32x2_pack(pf[32 * hc + 2 * i2], pf[32 * hc + 2 * i2 + 1]),
                                       fadd2(f32x2_pack(__uint_as_float(dv[2 * i2]), __uint_as_float(dv[2 * i2 + 1])),
                                             f32x2_pack(nd.x, nd.y))),
                                 d0, d1);
                    dk[i2] = pack_bf16x2(d0, d1);
                }
                tmem_st16(t_lane + kColOp1 + op_off + 16u * hc, dk);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (elect_one_sync()) mbar_arrive(bar(L::kBarDSFull + 1));
        }
        cp_async_wait_all();  // after an abort a prefetch may still be in flight
        if (ok && n_q > 0) ok = fa_wait_warp(bar(L::kBarFinal), 0, abort_flag, limit, kStatusSoftmaxWaitO);
        if (ok) {
            tc_fence_after_sync();
            const size_t r = (size_t)bh * p.N + (size_t)k_idx;
#pragma unroll
            for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (times scale)
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which ? p.grad : p.grad2) + r * D);
                const float f = which ? p.scale : 1.f;
                const uint32_t col = which ? kColDK : kColDV;
#pragma unroll
                for (int hc = 0; hc < D / 64; ++hc) {  // this warp's half of the columns
                    const int c = half * (D / 64) + hc;
                    uint32_t v[32];
                    tmem_ld32_wait(t_lane + col + 32u * c, v);
                    uint32_t w[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        w[u] = pack_bf16x2(n_q > 0 ? __uint_as_float(v[2 * u]) * f : 0.f,
                                           n_q > 0 ? __uint_as_float(v[2 * u + 1]) * f : 0.f);
                    if (valid) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) dst[c * 4 + u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
            }
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

}  // namespace fa
