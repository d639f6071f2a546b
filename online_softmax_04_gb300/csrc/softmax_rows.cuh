// softmax_rows.cuh -- row-wise softmax of an fp32 matrix with the online
// normaliser, for sm_103a (GB300).
//
// For every row x of length N ("5.2 CUDA Online Softmax", section 2; "Online
// softmax, and the register that can't move", section "Online softmax"):
//
//     (m, d) = running max and running sum of exp(x_j - m), one element at a
//              time: m' = max(m, x_j), d = d * exp(m - m') + exp(x_j - m')
//     y_j    = exp(x_j - m) / d,        lse = m + ln d
//
// Partial states of disjoint pieces of a row combine with the associative rule
// of the same page, section 4.1: m = max(m1, m2),
// d = d1 exp(m1 - m) + d2 exp(m2 - m).
//
// GB300 mapping.  The job is HBM-bound (one read and one write of every
// element), so the point is to touch HBM exactly once per element:
//   * kernel softmax_rows_smem: one CTA per row (rows blockIdx.x,
//     blockIdx.x + gridDim.x, ... when M exceeds the grid limit).  The row is
//     brought into shared memory by one bulk TMA copy; the block scheduler
//     keeps up to 8 such CTAs per SM in flight, which measured faster than a
//     persistent grid that prefetches the next row.  Each thread runs the online
//     recurrence over float4 chunks of the row in shared memory; the 256 partial states
//     are merged with warp shuffles and then across warps; a second sweep of
//     shared memory writes y with coalesced float4 stores.  HBM traffic: 8
//     bytes per element plus 4 per row for lse.
//   * kernel softmax_rows_warp: short rows (N <= 2048): one warp per chunk of
//     consecutive rows (up to 8 KB, one bulk copy), reduced with shuffles only.
//   * kernel softmax_rows_stream: rows too long for shared memory, or not
//     16-byte aligned: the same recurrence straight from global memory, then a
//     second read for the normalisation (12 bytes per element).
// Exponentials are ex2 of (x - m) * log2(e); a row with no finite element has
// d = 0 and gives y = 0, lse = -inf.
#pragma once

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kSmThreads = 256;
constexpr int kSmWarps = kSmThreads / 32;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2f = 0.69314718055994530942f;
// largest row held in shared memory (two buffers of this many bytes per CTA)
constexpr uint32_t kSmMaxRowBytes = 100u * 1024u;

// online state of part of a row: running max m (x units) and sum d of exp(x - m)
struct RowState {
    float m, d;
};

// exp(x - m) as ex2((x - m) log2 e): the difference first, so that the
// argument is small and accurate where the result is large (x near m), also
// when |m| itself is large.  exp(-inf - m) = 0.
__device__ __forceinline__ float exp_from(float x, float m) { return ex2_approx((x - m) * kLog2e); }

// fold four more elements into (m, d): one correction and four exponentials
__device__ __forceinline__ void fold4(RowState& s, float4 v) {
    const float m_new = fmaxf(fmaxf(s.m, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
    if (m_new == -INFINITY) return;  // nothing finite yet: the state stays empty
    s.d = s.d * exp_from(s.m, m_new) +  // exp(m - m'), 0 when m = -inf
          ((exp_from(v.x, m_new) + exp_from(v.y, m_new)) + (exp_from(v.z, m_new) + exp_from(v.w, m_new)));
    s.m = m_new;
}

__device__ __forceinline__ void fold1(RowState& s, float x) {
    const float m_new = fmaxf(s.m, x);
    if (m_new == -INFINITY) return;
    s.d = s.d * exp_from(s.m, m_new) + exp_from(x, m_new);
    s.m = m_new;
}

// the associative merge; commutative bit for bit, so every lane of a butterfly
// ends with the same state
__device__ __forceinline__ RowState merge(RowState a, RowState b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return RowState{m, 0.f};
    return RowState{m, a.d * exp_from(a.m, m) + b.d * exp_from(b.m, m)};
}

// whole-CTA merge of every thread's state; `scratch` holds 2 * kSmWarps floats.
// Every thread returns the same state.  Ends with a __syncthreads.
__device__ __forceinline__ RowState block_merge(RowState s, float* scratch) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        RowState o{__shfl_xor_sync(0xffffffffu, s.m, off), __shfl_xor_sync(0xffffffffu, s.d, off)};
        s = merge(s, o);
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        scratch[2 * warp] = s.m;
        scratch[2 * warp + 1] = s.d;
    }
    __syncthreads();
    RowState t{scratch[0], scratch[1]};
#pragma unroll
    for (int w = 1; w < kSmWarps; ++w) t = merge(t, RowState{scratch[2 * w], scratch[2 * w + 1]});
    __syncthreads();  // scratch may be reused by the next row
    return t;
}

__device__ __forceinline__ float row_lse(RowState s) {
    return s.d > 0.f ? s.m + lg2_approx(s.d) * kLn2f : -INFINITY;
}

// Rows of N floats (N % 4 == 0, x and y 16-byte aligned, 4N <= kSmMaxRowBytes)
// through shared memory, one row buffer.  Dynamic shared memory:
// softmax_rows_smem_bytes(N).
__host__ __device__ constexpr size_t softmax_rows_smem_bytes(int N) {
    return (size_t)N * 4u + 16u + 2u * kSmWarps * 4u;
}

__global__ void __launch_bounds__(kSmThreads)
    softmax_rows_smem(const float* __restrict__ x, float* y, float* lse, long long M, int N,
                      unsigned long long limit_ns) {
    extern __shared__ __align__(128) uint8_t sm_raw[];
    const uint32_t row_bytes = (uint32_t)N * 4u;
    const float* row = reinterpret_cast<const float*>(sm_raw);            // [N]
    uint64_t* bar_p = reinterpret_cast<uint64_t*>(sm_raw + row_bytes);      // the row's mbarrier
    float* scratch = reinterpret_cast<float*>(bar_p + 2);                   // [2 * kSmWarps]
    __shared__ int give_up;
    const uint32_t bar = smem_u32(bar_p);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        give_up = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    auto issue = [&](long long r) {
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_load_1d(smem_u32(row), x + (size_t)r * N, row_bytes, bar);
    };
    long long r = blockIdx.x;
    if (threadIdx.x == 0 && r < M) issue(r);
    const int n4 = N / 4;
    for (int i = 0; r < M; ++i, r += gridDim.x) {
        // wait for this row (bounded: a copy that never lands ends the kernel,
        // after the copy itself has been given the same time to land)
        if (threadIdx.x == 0) {
            const uint32_t par = (uint32_t)(i & 1);
            if (!mbar_try_wait(bar, par)) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar, par)) {
                    if (global_timer_ns() - t0 > limit_ns) {
                        atomicOr(&g_fa_status, kStatusSoftmaxRows);
                        give_up = 1;
                        const uint64_t t1 = global_timer_ns();
                        while (!mbar_try_wait(bar, par) && global_timer_ns() - t1 <= limit_ns) {
                        }
                        break;
                    }
                }
            }
        }
        __syncthreads();
        if (give_up) break;
        const float4* row4 = reinterpret_cast<const float4*>(row);
        RowState s{-INFINITY, 0.f};
        for (int c = threadIdx.x; c < n4; c += kSmThreads) fold4(s, row4[c]);
        const RowState t = block_merge(s, scratch);
        const float inv_d = t.d > 0.f ? 1.f / t.d : 0.f;
        const float m = t.m == -INFINITY ? 0.f : t.m;  // an empty row: every exp is 0 and y = 0
        float4* out = reinterpret_cast<float4*>(y + (size_t)r * N);
        for (int c = threadIdx.x; c < n4; c += kSmThreads) {
            const float4 v = row4[c];
            out[c] = make_float4(exp_from(v.x, m) * inv_d, exp_from(v.y, m) * inv_d, exp_from(v.z, m) * inv_d,
                                 exp_from(v.w, m) * inv_d);
        }
        if (lse && threadIdx.x == 0) lse[r] = row_lse(t);
        __syncthreads();  // the buffer is free again
        if (threadIdx.x == 0 && r + gridDim.x < M) issue(r + gridDim.x);
    }
}

// Short rows (N % 4 == 0, x and y 16-byte aligned, N <= kWarpMaxN): one warp per
// chunk of up to kWarpChunkRows(N) consecutive rows, copied into the warp's own
// shared-memory slot by one bulk TMA copy; each row is reduced with shuffles
// only (no block barrier), so many rows are in flight per SM.  Chunk c of the
// launch belongs to warp (blockIdx.x * kSmWarps + warp); dynamic shared memory:
// kSmWarps * (kWarpChunkBytes + 16).
constexpr int kWarpMaxN = 2048;
constexpr uint32_t kWarpChunkBytes = 8192;
__host__ __device__ constexpr int warp_chunk_rows(int N) {
    return (int)(kWarpChunkBytes / 4u) / N > 0 ? (int)(kWarpChunkBytes / 4u) / N : 1;
}

__global__ void __launch_bounds__(kSmThreads)
    softmax_rows_warp(const float* __restrict__ x, float* y, float* lse, long long M, int N,
                      unsigned long long limit_ns) {
    extern __shared__ __align__(128) uint8_t sm_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* slot = reinterpret_cast<float*>(sm_raw + (size_t)warp * (kWarpChunkBytes + 16u));
    uint64_t* bar_p = reinterpret_cast<uint64_t*>(sm_raw + (size_t)warp * (kWarpChunkBytes + 16u) + kWarpChunkBytes);
    const uint32_t bar = smem_u32(bar_p);
    const int R = warp_chunk_rows(N);
    const long long row0 = ((long long)blockIdx.x * kSmWarps + warp) * R;
    if (row0 >= M) return;
    const int rows = (int)(M - row0 < R ? M - row0 : R);
    bool landed = true;
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbarrier_init();
        const uint32_t bytes = (uint32_t)rows * (uint32_t)N * 4u;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load_1d(smem_u32(slot), x + (size_t)row0 * N, bytes, bar);
        if (!mbar_try_wait(bar, 0)) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar, 0)) {
                if (global_timer_ns() - t0 > limit_ns) {
                    atomicOr(&g_fa_status, kStatusSoftmaxRows);
                    landed = false;
                    const uint64_t t1 = global_timer_ns();  // give the copy the same time before leaving
                    while (!mbar_try_wait(bar, 0) && global_timer_ns() - t1 <= limit_ns) {
                    }
                    break;
                }
            }
        }
    }
    if (!__shfl_sync(0xffffffffu, landed, 0)) return;
    __syncwarp();
    const int n4 = N / 4;
    for (int rr = 0; rr < rows; ++rr) {
        const float4* row4 = reinterpret_cast<const float4*>(slot + (size_t)rr * N);
        RowState s{-INFINITY, 0.f};
        for (int c = lane; c < n4; c += 32) fold4(s, row4[c]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            s = merge(s, RowState{__shfl_xor_sync(0xffffffffu, s.m, off), __shfl_xor_sync(0xffffffffu, s.d, off)});
        const float inv_d = s.d > 0.f ? 1.f / s.d : 0.f;
        const float m = s.m == -INFINITY ? 0.f : s.m;
        float4* out = reinterpret_cast<float4*>(y + (size_t)(row0 + rr) * N);
        for (int c = lane; c < n4; c += 32) {
            const float4 v = row4[c];
            out[c] = make_float4(exp_from(v.x, m) * inv_d, exp_from(v.y, m) * inv_d, exp_from(v.z, m) * inv_d,
                                 exp_from(v.w, m) * inv_d);
        }
        if (lse && lane == 0) lse[row0 + rr] = row_lse(s);
    }
}

// Any N, any 4-byte alignment: one CTA per row at a time, two sweeps of global
// memory (the online recurrence, then the normalisation).
__global__ void __launch_bounds__(kSmThreads)
    softmax_rows_stream(const float* x, float* y, float* lse, long long M, int N) {
    __shared__ float scratch[2 * kSmWarps];
    for (long long r = blockIdx.x; r < M; r += gridDim.x) {
        const float* xr = x + (size_t)r * N;
        float* yr = y + (size_t)r * N;
        RowState s{-INFINITY, 0.f};
        const bool vec = ((reinterpret_cast<uintptr_t>(xr) | reinterpret_cast<uintptr_t>(yr)) & 15u) == 0;
        const int n4 = vec ? N / 4 : 0;
        for (int c = threadIdx.x; c < n4; c += kSmThreads) fold4(s, reinterpret_cast<const float4*>(xr)[c]);
        for (int j = 4 * n4 + threadIdx.x; j < N; j += kSmThreads) fold1(s, xr[j]);
        const RowState t = block_merge(s, scratch);
        const float inv_d = t.d > 0.f ? 1.f / t.d : 0.f;
        const float m = t.m == -INFINITY ? 0.f : t.m;
        for (int c = threadIdx.x; c < n4; c += kSmThreads) {
            const float4 v = reinterpret_cast<const float4*>(xr)[c];
            reinterpret_cast<float4*>(yr)[c] = make_float4(exp_from(v.x, m) * inv_d, exp_from(v.y, m) * inv_d,
                                                           exp_from(v.z, m) * inv_d, exp_from(v.w, m) * inv_d);
        }
        for (int j = 4 * n4 + threadIdx.x; j < N; j += kSmThreads) yr[j] = exp_from(xr[j], m) * inv_d;
        if (lse && threadIdx.x == 0) lse[r] = row_lse(t);
    }
}

}  // namespace fa
