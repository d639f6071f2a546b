// fa_fwd.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, TMA descriptor encoding and the kernel launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_fwd_kernel.cuh"
#include "fa_fwd_two_kernel.cuh"
#include "softmax_rows.cuh"
#include "fa_bwd_kernel.cuh"

namespace {

constexpr int kVersion = 1 * 10000 + 2 * 100 + 0;
constexpr int kMaxDevices = 64;

uint64_t g_watchdog_ns = 1000000000ull;  // 1 s
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_device_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_device_ok[dev] == 1 ? FA_OK : FA_ERR_DEVICE;
}

// [B*H][N][d] bf16 viewed as a 3-D tensor (d, N, B*H); box = one 128-row (or
// box_rows-row) x 64-column chunk, 128-byte swizzle.  Rows past N read as zero
// (loads) and are dropped (stores), per head.
bool encode_bhnd(CUtensorMap* m, const void* base, int d, int N, int BH, unsigned box_rows = 128u) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2u, (cuuint64_t)N * (cuuint64_t)d * 2u};
    cuuint32_t box[3] = {64u, box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int sm_count();
int queue_slot(unsigned int** out);

// kSplit: one CTA per (query tile, head, key split).  Otherwise a persistent
// grid of at most one CTA per SM walks the work items (see fa::TileSeq).
template <int D, int NK, int NV, bool kSplit, bool kMask = false>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
           fa::FaParams p, int BH, cudaStream_t stream) {
    using L = fa::FwdSmem<D, NK, NV, kSplit, false>;
    constexpr bool kPersistent = !kSplit;
    auto kern = fa::fa_fwd_sm103<D, NK, NV, kSplit, kPersistent, kMask>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc) != cudaSuccess)
        return FA_ERR_CUDA;
    dim3 grid;
    if constexpr (kSplit) {
        // blockIdx.x runs from the last (longest causal) tile down: heaviest first
        grid = dim3((unsigned)p.n_tiles, (unsigned)BH, (unsigned)p.n_splits);
    } else {
        const int sms = sm_count() > 0 ? sm_count() : 148;
        const long long pairs = fa::persistent_pairs(p);
        const long long tiles = (long long)BH * p.n_tiles;
        if (tiles <= sms) {
            // one CTA per tile, each CTA's tile fixed by its index: no work counter
            grid = dim3((unsigned)tiles, 1, 1);
            p.static_rounds = -1;
            p.queue = nullptr;
        } else {
            // every persistent launch takes its own work counter (the dynamic tail)
            const int qrc = queue_slot(&p.queue);
            if (qrc != FA_OK) return qrc;
            grid = dim3((unsigned)sms, 1, 1);
            // every full round of pairs is dealt out statically; the partial last
            // round goes to the dynamic tail as single tiles, long ones first
            // (measured best against 70-95% static)
            p.static_rounds = (int)(pairs / sms);
        }
    }
    kern<<<grid, fa::kThreads, L::kAlloc, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Clusters of two CTAs of `kern` (one per SM) that fit on the device at once,
// per device, looked up on first use.
int g_pair_clusters[kMaxDevices];

template <typename K>
int pair_clusters(K kern, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_pair_clusters[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * 256, 1, 1);
        cfg.blockDim = dim3(fa::kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return 0;
        g_pair_clusters[dev] = n;
    }
    return g_pair_clusters[dev];
}

// The d = 128 persistent kernel in CTA pairs (see fa::fa_fwd_sm103, kPair):
// clusters of two CTAs; tk_half is K's map with a 64-row box.
template <int D, int NK, int NV>
int launch_pair(const CUtensorMap& tq, const CUtensorMap& tk_half, const CUtensorMap& tv, fa::FaParams p,
                cudaStream_t stream) {
    using L = fa::FwdSmem<D, NK, NV, false, true>;
    auto kern = fa::fa_fwd_sm103<D, NK, NV, false, true, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc) != cudaSuccess)
        return FA_ERR_CUDA;
    const int clusters = pair_clusters(kern, L::kAlloc);
    if (clusters < 1) return FA_ERR_CUDA;
    const long long units = (long long)p.BH * fa::schedule_units(p, true);
    unsigned grid;
    if (units <= clusters) {
        // one pair per unit, fixed by its index: no work counter
        grid = (unsigned)(2 * units);
        p.static_rounds = -1;
        p.queue = nullptr;
    } else {
        const int qrc = queue_slot(&p.queue);
        if (qrc != FA_OK) return qrc;
        grid = (unsigned)(2 * clusters);
        p.static_rounds = (int)(fa::persistent_pairs(p, true) / clusters);
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(fa::kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // the pair kernel writes O from registers: its tm_o parameter is unused
    if (cudaLaunchKernelEx(&cfg, kern, tq, tk_half, tv, tq, p) != cudaSuccess) return FA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The d = 64 persistent kernel with two query tiles per CTA (see fa::fa_fwd2_sm103).
template <int NK, int NV>
int launch_two(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, fa::FaParams p,
               cudaStream_t stream) {
    using L = fa::TwoSmem<NK, NV>;
    auto kern = fa::fa_fwd2_sm103<NK, NV>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc) != cudaSuccess)
        return FA_ERR_CUDA;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const long long units = (long long)p.BH * fa::schedule_units(p, true);
    unsigned grid;
    if (units <= sms) {
        // one CTA per unit, fixed by its index: no work counter
        grid = (unsigned)units;
        p.static_rounds = -1;
        p.queue = nullptr;
    } else {
        const int qrc = queue_slot(&p.queue);
        if (qrc != FA_OK) return qrc;
        grid = (unsigned)sms;
        p.static_rounds = (int)(fa::persistent_pairs(p, true) / sms);
    }
    kern<<<grid, fa::kThreads, L::kAlloc, stream>>>(tq, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

struct Prepared {
    CUtensorMap tq, tk, tv;
    CUtensorMap tk_half;  // K with a 64-row box (d = 128: the CTA-pair kernel)
    CUtensorMap to;       // O with a 16-row box (d = 128: the one-CTA kernels' TMA stores)
    fa::FaParams p;
    int BH;
};

// K and V stages (16 KB each) of the CTA-pair kernel: measured best against
// 4+6, 6+4, 6+5, 7+3, 7+4, 8+2 and 9+2 on causal and full shapes
constexpr int kPairNK = 8, kPairNV = 3;
// Causal attention takes CTA pairs from this many query tiles on: the pair
// computes one fully masked key tile per two query tiles, 1 / (n_tiles / 2 + 1)
// of the work, against ~3% faster steps (measured break-even at 64 tiles).
constexpr int kPairMinCausalTiles = 96;

std::atomic<int> g_pairing{FA_PAIR_AUTO};

bool use_pair(int d, int causal, int n_tiles) {
    if (d != 128) return false;
    const int mode = g_pairing.load();
    if (mode == FA_PAIR_OFF) return false;
    if (mode == FA_PAIR_ON) return true;
    return !causal || n_tiles >= kPairMinCausalTiles;
}

// K and V stages (16 KB each) of the two-tile kernel
constexpr int kTwoNK = 6, kTwoNV = 5;

// The d = 64 kernel with two query tiles per CTA runs a tile step in ~0.9 of
// the one-tile kernel's time (0.88-0.95 measured over causal and full shapes),
// but it has half as many work units, and a causal unit also computes the key
// tile after its first tile's diagonal.  Under FA_PAIR_AUTO it is taken when a
// model of both schedules on a 152-SM GB300 says it finishes first: full
// attention runs ceil(units / SMs) rounds of equal units; causal attention is
// balanced by the long+short schedule, so its time is the steps per SM or the
// longest unit, whichever is larger.  (Host-only: no device is queried.)
constexpr long long kPolicySms = 152;

bool use_two(int d, int causal, int n_tiles, long long BH) {
    if (d != 64) return false;
    const int mode = g_pairing.load();
    if (mode == FA_PAIR_OFF) return false;
    if (mode == FA_PAIR_ON) return true;
    const long long n = n_tiles, units = (n + 1) / 2;
    const double r = 0.9;  // a two-tile step against a one-tile step
    double one, two;
    if (!causal) {
        one = (double)((BH * n + kPolicySms - 1) / kPolicySms) * (double)n;
        two = r * (double)((BH * units + kPolicySms - 1) / kPolicySms) * 2.0 * (double)n;
    } else {
        // steps per head: query tile t sees t + 1 key tiles; unit u runs both its
        // tiles over min(2u + 2, n) key tiles
        const long long steps_one = n * (n + 1) / 2;
        long long steps_two = 0;
        for (long long u = 0; u < units; ++u) steps_two += 2 * std::min(2 * u + 2, n);
        one = std::max((double)(BH * steps_one) / (double)kPolicySms, (double)n);
        two = r * std::max((double)(BH * steps_two) / (double)kPolicySms, 2.0 * (double)n);
    }
    return two < one;
}

// two: -1 lets the policy choose the d = 64 kernel for these sizes; 0 or 1 forces
// one tile or two tiles per CTA (a caller that splits one problem into several
// launches decides once, for the whole problem)
template <bool kSplit, bool kMask = false>
int launch_d(int d, const Prepared& pr, cudaStream_t s, int two = -1) {
    // (tm_o is read only by the kernels that stage O, at d = 128; the others get tq)
    if constexpr (!kSplit && !kMask)
        if (d == 64 && (two >= 0 ? two == 1 : use_two(d, pr.p.causal, pr.p.n_tiles, pr.BH)))
            return launch_two<kTwoNK, kTwoNV>(pr.tq, pr.tk, pr.tv, pr.p, s);
    if (d == 64) return launch<64, 6, 6, kSplit, kMask>(pr.tq, pr.tk, pr.tv, pr.tq, pr.p, pr.BH, s);
    if constexpr (!kSplit && !kMask)
        if (use_pair(d, pr.p.causal, pr.p.n_tiles))
            return launch_pair<128, kPairNK, kPairNV>(pr.tq, pr.tk_half, pr.tv, pr.p, s);
    return launch<128, 2, 3, kSplit, kMask>(pr.tq, pr.tk, pr.tv, kSplit ? pr.tq : pr.to, pr.p, pr.BH, s);
}

// Host-side argument validation shared by the entry points (no CUDA calls).
int validate(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             float scale) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_POINTER;
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
    const long long BH = (long long)B * (long long)H;
    if (BH > 65535) return FA_ERR_SHAPE;
    // the persistent schedule numbers the (head, query tile) pairs in 32 bits
    if (BH * (((long long)N + fa::kBlockN - 1) / fa::kBlockN) >= (1ll << 31)) return FA_ERR_SHAPE;
    auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
    if (mis16(q) || mis16(k) || mis16(v) || mis16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return FA_ERR_ALIGNMENT;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
    const size_t tensor_bytes = (size_t)BH * (size_t)N * (size_t)d * 2u;
    const size_t lse_bytes = (size_t)BH * (size_t)N * 4u;
    if (overlaps(o, tensor_bytes, q, tensor_bytes) || overlaps(o, tensor_bytes, k, tensor_bytes) ||
        overlaps(o, tensor_bytes, v, tensor_bytes) || overlaps(lse, lse_bytes, q, tensor_bytes) ||
        overlaps(lse, lse_bytes, k, tensor_bytes) || overlaps(lse, lse_bytes, v, tensor_bytes) ||
        overlaps(lse, lse_bytes, o, tensor_bytes))
        return FA_ERR_ALIAS;
    return FA_OK;
}

// The device check and the TMA descriptors, after validate() passed.
int prepare(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, int causal,
            float scale, Prepared* out) {
    const long long BH = (long long)B * (long long)H;
    const int dev_rc = check_device();
    if (dev_rc != FA_OK) return dev_rc;
    if (!encode_bhnd(&out->tq, q, d, N, (int)BH) || !encode_bhnd(&out->tk, k, d, N, (int)BH) ||
        !encode_bhnd(&out->tv, v, d, N, (int)BH) ||
        (d == 128 && (!encode_bhnd(&out->tk_half, k, d, N, (int)BH, 64u) || !encode_bhnd(&out->to, o, d, N, (int)BH, 16u))))
        return FA_ERR_TENSOR_MAP;
    fa::FaParams& p = out->p;
    p = fa::FaParams{};
    p.o = o;
    p.lse = lse;
    p.BH = (int)BH;
    p.H = H;
    p.window_left = -1;
    p.window_right = causal ? 0 : -1;
    p.doc = nullptr;
    p.N = N;
    p.n_tiles = (N + fa::kBlockN - 1) / fa::kBlockN;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.44269504088896340736f;
    p.n_splits = 1;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        p.watchdog_ns = g_watchdog_ns;
    }
    out->BH = (int)BH;
    return FA_OK;
}

constexpr int kMaxSplits = 64;

size_t splitkv_bytes(long long BH, long long N, int d, int n_splits) {
    return (size_t)n_splits * (size_t)BH * (size_t)N * (size_t)(d + 3) * sizeof(float);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// ----------------------------------------------------------------------------
// Static scratch for fa_fwd_splitkv_noalloc.  It lives in the module image, so
// every device that loads this library holds FA_NOALLOC_SCRATCH_BYTES of it
// until the process exits.  Host code only ever names it to ask the runtime
// for its device address (once per device); the kernels get that address.
// ----------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

void* g_noalloc_addr[kMaxDevices];  // device address of the scratch, per device (nullptr: not looked up yet)

// Device address of the scratch on the current device, looked up on first use.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_fa_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return FA_OK;
}

// ----------------------------------------------------------------------------
// Work-queue counters of the persistent kernel: {next item, CTAs finished} per
// slot, zero at load time and left at zero by the last CTA of every launch.
// Each fa_fwd call takes the next slot round-robin, so that calls running at
// the same time on different streams do not share a counter (unless more than
// kQueueSlots - 1 launches are in flight at once).
// ----------------------------------------------------------------------------
constexpr unsigned kQueueSlots = 1024;
static __device__ unsigned int g_fa_queue[2 * kQueueSlots];

unsigned int* g_queue_addr[kMaxDevices];
std::atomic<unsigned> g_queue_seq{0};

int queue_slot(unsigned int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_queue_addr[dev]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_fa_queue) != cudaSuccess || !ptr) return FA_ERR_CUDA;
            g_queue_addr[dev] = static_cast<unsigned int*>(ptr);
        }
    }
    *out = g_queue_addr[dev] + 2u * (g_queue_seq.fetch_add(1u) % kQueueSlots);
    return FA_OK;
}

// The backward's second stream and its two events, per device, made on first
// use and kept; the enqueue of concurrent fa_bwd calls on one device is
// serialised because they share them.
struct BwdPipe {
    bool ready = false;
    cudaStream_t side = nullptr;
    cudaEvent_t delta_done = nullptr, kv_done = nullptr;
};
BwdPipe g_bwd_pipe[kMaxDevices];
std::mutex g_bwd_mu;

int bwd_pipe(BwdPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    BwdPipe& bp = g_bwd_pipe[dev];
    if (!bp.ready) {
        if (cudaStreamCreateWithFlags(&bp.side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&bp.delta_done, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&bp.kv_done, cudaEventDisableTiming) != cudaSuccess)
            return FA_ERR_CUDA;
        bp.ready = true;
    }
    *out = &bp;
    return FA_OK;
}

// key and value stages of the dQ kernel: at d = 128, 3 K + 2 V stages of 32 KB
// (K is read again by the dQ product a step after S); at d = 64, 4 + 4 of 16 KB
template <int D>
struct DqStages {
    static constexpr int NK = D == 64 ? 4 : 3, NV = D == 64 ? 4 : 2;
};

template <int D, int NS>
int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
               const void* o, const void* dout, float* delta, void* dq, void* dk, void* dv, fa::BwdParams p, int BH,
               cudaStream_t st) {
    using L = fa::BwdSmem<D, NS>;
    const long long rows = (long long)BH * p.N;
    fa::fa_bwd_delta<D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                                                      static_cast<const __nv_bfloat16*>(dout), delta,
                                                                      rows);
    using LQ = fa::DqSmem<D, DqStages<D>::NK, DqStages<D>::NV>;
    auto kq = fa::fa_bwd_dq_sm103<D, DqStages<D>::NK, DqStages<D>::NV>;
    auto kkv = fa::fa_bwd_dkdv_sm103<D, NS>;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LQ::kAlloc) != cudaSuccess ||
        cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc) != cudaSuccess)
        return FA_ERR_CUDA;
    const dim3 grid((unsigned)p.n_tiles, (unsigned)BH);
    // dQ and dK/dV are independent once D is known: dK/dV runs on a second
    // stream, so that each kernel's CTAs fill the other's last, partial wave
    BwdPipe* bp = nullptr;
    std::lock_guard<std::mutex> lk(g_bwd_mu);
    const int prc = bwd_pipe(&bp);
    if (prc != FA_OK) return prc;
    if (cudaEventRecord(bp->delta_done, st) != cudaSuccess || cudaStreamWaitEvent(bp->side, bp->delta_done, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    p.delta = delta;
    p.grad = dk;
    p.grad2 = dv;
    kkv<<<grid, fa::kBwdThreads, L::kAlloc, bp->side>>>(tq, tk, tv, tdo, p);
    p.grad = dq;
    p.grad2 = nullptr;
    kq<<<grid, fa::kBwdThreads, LQ::kAlloc, st>>>(tq, tk, tv, tdo, p);
    // the caller's stream continues once both have finished
    if (cudaEventRecord(bp->kv_done, bp->side) != cudaSuccess || cudaStreamWaitEvent(st, bp->kv_done, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// fa_fwd_host: host-resident tensors streamed through three device slots
// ---------------------------------------------------------------------------
constexpr size_t kHostAlign = 256;
// Chunk c's inputs wait for the read-back of the chunk that used its slot
// before, c - kHostSlots.  With two slots that read-back (chunk c - 2: its
// kernel and copy-out) ends after chunk c - 1's input copy, and the input
// stream, which the host link limits, stalls on every chunk; with three it
// ends long before.
constexpr int kHostSlots = 3;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int host_chunk_heads(long long BH, int heads_per_chunk) {
    return heads_per_chunk > 0 ? heads_per_chunk : (int)((BH + 7) / 8);
}

// one slot: q, k, v, o (bf16) and lse (fp32) of `hc` heads, each 256-byte aligned
size_t host_slot_bytes(int hc, int N, int d) {
    const size_t t = align_up((size_t)hc * (size_t)N * (size_t)d * 2u, kHostAlign);
    return 4 * t + align_up((size_t)hc * (size_t)N * 4u, kHostAlign);
}

// The two copy streams and the events of the pipeline, per device, made on
// first use and kept for the life of the process.  (Separate input streams
// for q, k and v measured slower: the host link, not the copy engines, limits.)
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kHostSlots] = {}, compute_done[kHostSlots] = {}, out_done[kHostSlots] = {};
};
HostPipe g_host_pipe[kMaxDevices];
std::mutex g_host_mu;  // serialises the enqueue of fa_fwd_host calls (shared streams and events)

int host_pipe(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    HostPipe& hp = g_host_pipe[dev];
    if (!hp.ready) {
        const unsigned ev = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.start, ev) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.end, ev) == cudaSuccess;
        for (int i = 0; ok && i < kHostSlots; ++i)
            ok = cudaEventCreateWithFlags(&hp.in_done[i], ev) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.compute_done[i], ev) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.out_done[i], ev) == cudaSuccess;
        if (!ok) return FA_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return FA_OK;
}

// Resources of one kernel as the runtime reports them, with the dynamic shared
// memory it is launched with.
template <typename K>
int kernel_resources(K kern, int threads, size_t dyn_smem, int tmem_cols, fa_kernel_resources_t* out) {
    cudaFuncAttributes a{};
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem) != cudaSuccess ||
        cudaFuncGetAttributes(&a, kern) != cudaSuccess)
        return FA_ERR_CUDA;
    int ctas = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, kern, threads, dyn_smem) != cudaSuccess) return FA_ERR_CUDA;
    out->registers_per_thread = a.numRegs;
    out->threads_per_cta = threads;
    out->dynamic_smem_bytes = (int)dyn_smem;
    out->static_smem_bytes = (int)a.sharedSizeBytes;
    out->local_bytes_per_thread = (int)a.localSizeBytes;
    out->ctas_per_sm = ctas;
    out->tmem_columns = tmem_cols;
    return FA_OK;
}

template <int D, int NK, int NV>
int fwd_resources(int kernel, fa_kernel_resources_t* out) {
    switch (kernel) {
        case FA_KERNEL_FWD:
            return kernel_resources(fa::fa_fwd_sm103<D, NK, NV, false, true, false>, fa::kThreads,
                                    fa::FwdSmem<D, NK, NV, false, false>::kAlloc, (int)fa::kTmemCols, out);
        case FA_KERNEL_FWD_PAIR:
            if constexpr (D == 128) {
                using LP = fa::FwdSmem<D, kPairNK, kPairNV, false, true>;
                return kernel_resources(fa::fa_fwd_sm103<D, kPairNK, kPairNV, false, true, false, true>, fa::kThreads,
                                        LP::kAlloc, (int)fa::kTmemCols, out);
            } else {
                return FA_ERR_HEAD_DIM;
            }
        case FA_KERNEL_FWD_TWO:
            if constexpr (D == 64) {
                return kernel_resources(fa::fa_fwd2_sm103<kTwoNK, kTwoNV>, fa::kThreads,
                                        fa::TwoSmem<kTwoNK, kTwoNV>::kAlloc, (int)fa::kTmemCols, out);
            } else {
                return FA_ERR_HEAD_DIM;
            }
        case FA_KERNEL_FWD_MASKED:
            return kernel_resources(fa::fa_fwd_sm103<D, NK, NV, false, true, true>, fa::kThreads,
                                    fa::FwdSmem<D, NK, NV, false, false>::kAlloc, (int)fa::kTmemCols, out);
        case FA_KERNEL_FWD_SPLITKV:
            return kernel_resources(fa::fa_fwd_sm103<D, NK, NV, true, false, false>, fa::kThreads,
                                    fa::FwdSmem<D, NK, NV, true, false>::kAlloc, (int)fa::kTmemCols, out);
        case FA_KERNEL_BWD_DQ:
            return kernel_resources(fa::fa_bwd_dq_sm103<D, DqStages<D>::NK, DqStages<D>::NV>, fa::kBwdThreads,
                                    fa::DqSmem<D, DqStages<D>::NK, DqStages<D>::NV>::kAlloc, (int)fa::kTmemCols, out);
        case FA_KERNEL_BWD_DKDV:
            return kernel_resources(fa::fa_bwd_dkdv_sm103<D, D == 64 ? 4 : 2>, fa::kBwdThreads,
                                    fa::BwdSmem<D, D == 64 ? 4 : 2>::kAlloc, (int)fa::kTmemCols, out);
        default: return FA_ERR_SHAPE;
    }
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, int causal,
           float scale, fa_stream_t stream) {
    int rc = validate(q, k, v, o, lse, B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    Prepared pr;
    rc = prepare(q, k, v, o, lse, B, H, N, d, causal, scale, &pr);
    if (rc != FA_OK) return rc;
    return launch_d<false>(d, pr, reinterpret_cast<cudaStream_t>(stream));
}

int fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  int window_left, int window_right, const int32_t* doc_ids, float scale, fa_stream_t stream) {
    int rc = validate(q, k, v, o, lse, B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    if (window_left < -1 || window_right < -1) return FA_ERR_MASK;
    if (doc_ids) {
        if ((reinterpret_cast<uintptr_t>(doc_ids) & 3u) != 0) return FA_ERR_ALIGNMENT;
        const size_t doc_bytes = (size_t)B * (size_t)N * 4u;
        const size_t tensor_bytes = (size_t)B * H * (size_t)N * (size_t)d * 2u;
        if (overlaps(doc_ids, doc_bytes, o, tensor_bytes) || overlaps(doc_ids, doc_bytes, lse, (size_t)B * H * N * 4u))
            return FA_ERR_ALIAS;
    }
    Prepared pr;
    rc = prepare(q, k, v, o, lse, B, H, N, d, window_right == 0 ? 1 : 0, scale, &pr);
    if (rc != FA_OK) return rc;
    pr.p.window_left = window_left;
    pr.p.window_right = window_right;
    pr.p.doc = doc_ids;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // full or causal attention without documents takes the unmasked kernel
    if (window_left < 0 && (window_right < 0 || window_right == 0) && !doc_ids)
        return launch_d<false, false>(d, pr, st);
    return launch_d<false, true>(d, pr, st);
}

size_t fa_splitkv_workspace_bytes(int B, int H, int N, int d, int n_splits) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || n_splits < 1 || n_splits > kMaxSplits) return 0;
    return splitkv_bytes((long long)B * H, N, d, n_splits);
}

int fa_splitkv_auto_splits(int B, int H, int N, int d, int causal) {
    (void)d;
    (void)causal;
    if (B < 1 || H < 1 || N < 1) return 1;
    const long long tiles = (N + fa::kBlockN - 1) / fa::kBlockN;
    const long long ctas = tiles * (long long)B * H;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    if (ctas >= sms) return 1;
    long long s = sms / ctas;  // fill at most one wave of one-CTA-per-SM blocks
    if (s > tiles) s = tiles;
    if (s > kMaxSplits) s = kMaxSplits;
    return s < 1 ? 1 : (int)s;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   int causal, float scale, int n_splits, void* workspace, size_t workspace_bytes,
                   fa_stream_t stream) {
    int rc = validate(q, k, v, o, lse, B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    if (n_splits < 0 || n_splits > kMaxSplits) return FA_ERR_SPLITS;
    if (!workspace) return FA_ERR_NULL_POINTER;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FA_ERR_ALIGNMENT;
    const long long BH = (long long)B * (long long)H;
    // the automatic count needs the device; size checks use the worst case first
    const size_t tensor_bytes = (size_t)BH * (size_t)N * (size_t)d * 2u;
    const size_t lse_bytes = (size_t)BH * (size_t)N * 4u;
    if (n_splits > 0) {
        const size_t need = splitkv_bytes(BH, N, d, n_splits);
        if (workspace_bytes < need) return FA_ERR_WORKSPACE;
        if (overlaps(workspace, need, q, tensor_bytes) || overlaps(workspace, need, k, tensor_bytes) ||
            overlaps(workspace, need, v, tensor_bytes) || overlaps(workspace, need, o, tensor_bytes) ||
            overlaps(workspace, need, lse, lse_bytes))
            return FA_ERR_ALIAS;
    }
    Prepared pr;
    rc = prepare(q, k, v, o, lse, B, H, N, d, causal, scale, &pr);
    if (rc != FA_OK) return rc;
    if (n_splits == 0) {
        n_splits = fa_splitkv_auto_splits(B, H, N, d, causal);
        const size_t need = splitkv_bytes(BH, N, d, n_splits);
        if (workspace_bytes < need) return FA_ERR_WORKSPACE;
        if (overlaps(workspace, need, q, tensor_bytes) || overlaps(workspace, need, k, tensor_bytes) ||
            overlaps(workspace, need, v, tensor_bytes) || overlaps(workspace, need, o, tensor_bytes) ||
            overlaps(workspace, need, lse, lse_bytes))
            return FA_ERR_ALIAS;
    }
    const long long rows = (long long)pr.BH * N;
    float* ws = static_cast<float*>(workspace);
    pr.p.n_splits = n_splits;
    pr.p.ws_o = ws;
    pr.p.ws_m = ws + (size_t)n_splits * rows * d;
    pr.p.ws_lbf = pr.p.ws_m + (size_t)n_splits * rows;
    pr.p.ws_l32 = pr.p.ws_lbf + (size_t)n_splits * rows;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int lrc = launch_d<true>(d, pr, s);
    if (lrc != FA_OK) return lrc;
    const unsigned blocks = (unsigned)((rows + 7) / 8);  // 8 warps per block, one row per warp
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
    if (d == 64)
        fa::fa_splitkv_merge<64><<<blocks, 256, 0, s>>>(pr.p.ws_o, pr.p.ws_m, pr.p.ws_lbf, pr.p.ws_l32, ob, lse, rows,
                                                        n_splits);
    else
        fa::fa_splitkv_merge<128><<<blocks, 256, 0, s>>>(pr.p.ws_o, pr.p.ws_m, pr.p.ws_lbf, pr.p.ws_l32, ob, lse,
                                                         rows, n_splits);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                           int d, int causal, float scale, int n_splits, fa_stream_t stream) {
    int rc = validate(q, k, v, o, lse, B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    if (n_splits < 0 || n_splits > kMaxSplits) return FA_ERR_SPLITS;
    const long long BH = (long long)B * (long long)H;
    if (n_splits > 0 && splitkv_bytes(BH, N, d, n_splits) > (size_t)FA_NOALLOC_SCRATCH_BYTES)
        return FA_ERR_SCRATCH_LIMIT;
    Prepared pr;
    rc = prepare(q, k, v, o, lse, B, H, N, d, causal, scale, &pr);
    if (rc != FA_OK) return rc;
    if (n_splits == 0) {
        // the automatic count, reduced until the partial states fit the scratch
        n_splits = fa_splitkv_auto_splits(B, H, N, d, causal);
        while (n_splits > 1 && splitkv_bytes(BH, N, d, n_splits) > (size_t)FA_NOALLOC_SCRATCH_BYTES) --n_splits;
        if (splitkv_bytes(BH, N, d, n_splits) > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
    }
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != FA_OK) return rc;
    // Every partial state the merge reads is written by the split kernel of the
    // same call (empty chunks write m = -inf and zeros), so whatever an earlier
    // call left in the scratch never needs clearing.
    const long long rows = BH * N;
    float* ws = static_cast<float*>(scratch);
    pr.p.n_splits = n_splits;
    pr.p.ws_o = ws;
    pr.p.ws_m = ws + (size_t)n_splits * rows * d;
    pr.p.ws_lbf = pr.p.ws_m + (size_t)n_splits * rows;
    pr.p.ws_l32 = pr.p.ws_lbf + (size_t)n_splits * rows;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int lrc = launch_d<true>(d, pr, s);
    if (lrc != FA_OK) return lrc;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
    if (d == 64)
        fa::fa_splitkv_merge<64><<<blocks, 256, 0, s>>>(pr.p.ws_o, pr.p.ws_m, pr.p.ws_lbf, pr.p.ws_l32, ob, lse, rows,
                                                        n_splits);
    else
        fa::fa_splitkv_merge<128><<<blocks, 256, 0, s>>>(pr.p.ws_o, pr.p.ws_m, pr.p.ws_lbf, pr.p.ws_l32, ob, lse,
                                                         rows, n_splits);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d, int heads_per_chunk) {
    if ((d != 64 && d != 128) || B < 1 || H < 1 || N < 1) return 0;
    const long long BH = (long long)B * (long long)H;
    if (heads_per_chunk < 0 || heads_per_chunk > BH) return 0;
    return kHostSlots * host_slot_bytes(host_chunk_heads(BH, heads_per_chunk), N, d);
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                int causal, float scale, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                fa_stream_t stream) {
    int rc = validate(q, k, v, o, lse, B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    const long long BH = (long long)B * (long long)H;
    if (heads_per_chunk < 0 || heads_per_chunk > BH) return FA_ERR_SHAPE;
    if (!workspace) return FA_ERR_NULL_POINTER;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kHostAlign - 1)) != 0) return FA_ERR_ALIGNMENT;
    const int hc = host_chunk_heads(BH, heads_per_chunk);
    const size_t slot = host_slot_bytes(hc, N, d);
    if (workspace_bytes < kHostSlots * slot) return FA_ERR_WORKSPACE;
    rc = check_device();
    if (rc != FA_OK) return rc;

    std::lock_guard<std::mutex> lk(g_host_mu);
    HostPipe* hp = nullptr;
    rc = host_pipe(&hp);
    if (rc != FA_OK) return rc;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t head_elems = (size_t)N * (size_t)d;
    const size_t tbytes = align_up((size_t)hc * head_elems * 2u, kHostAlign);
    bool ok = cudaEventRecord(hp->start, cs) == cudaSuccess && cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hp->d2h, hp->start, 0) == cudaSuccess;
    const long long n_chunks = (BH + hc - 1) / hc;
    // every chunk runs the kernel fa_fwd would choose for all B*H heads: same bits
    const int two = use_two(d, causal ? 1 : 0, (N + fa::kBlockN - 1) / fa::kBlockN, BH) ? 1 : 0;
    for (long long c = 0; ok && c < n_chunks; ++c) {
        const int sl = (int)(c % kHostSlots);
        const long long h0 = c * hc;
        const int nh = (int)std::min<long long>(hc, BH - h0);
        uint8_t* base = static_cast<uint8_t*>(workspace) + (size_t)sl * slot;
        void* dq = base;
        void* dk = base + tbytes;
        void* dv = base + 2 * tbytes;
        void* dout = base + 3 * tbytes;
        float* dlse = reinterpret_cast<float*>(base + 4 * tbytes);
        const size_t off = (size_t)h0 * head_elems * 2u;  // byte offset of the chunk's first head
        const size_t bytes = (size_t)nh * head_elems * 2u;
        // inputs: once the slot's previous chunk has been read back
        if (c >= kHostSlots) ok = cudaStreamWaitEvent(hp->h2d, hp->out_done[sl], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + off, bytes, cudaMemcpyDefault, hp->h2d) == cudaSuccess &&
             cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + off, bytes, cudaMemcpyDefault, hp->h2d) == cudaSuccess &&
             cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + off, bytes, cudaMemcpyDefault, hp->h2d) == cudaSuccess &&
             cudaEventRecord(hp->in_done[sl], hp->h2d) == cudaSuccess &&
             cudaStreamWaitEvent(cs, hp->in_done[sl], 0) == cudaSuccess;
        if (!ok) break;
        // the kernel, on the caller's stream: the chunk's heads as one batch
        Prepared pr;
        rc = prepare(dq, dk, dv, dout, dlse, 1, nh, N, d, causal, scale, &pr);
        if (rc != FA_OK) return rc;
        rc = launch_d<false>(d, pr, cs, two);
        if (rc != FA_OK) return rc;
        // outputs
        ok = cudaEventRecord(hp->compute_done[sl], cs) == cudaSuccess &&
             cudaStreamWaitEvent(hp->d2h, hp->compute_done[sl], 0) == cudaSuccess &&
             cudaMemcpyAsync(static_cast<uint8_t*>(o) + off, dout, bytes, cudaMemcpyDefault, hp->d2h) == cudaSuccess &&
             cudaMemcpyAsync(lse + (size_t)h0 * (size_t)N, dlse, (size_t)nh * (size_t)N * 4u, cudaMemcpyDefault,
                             hp->d2h) == cudaSuccess &&
             cudaEventRecord(hp->out_done[sl], hp->d2h) == cudaSuccess;
    }
    // the caller's stream continues after the last read-back
    ok = ok && cudaEventRecord(hp->end, hp->d2h) == cudaSuccess && cudaStreamWaitEvent(cs, hp->end, 0) == cudaSuccess;
    return ok ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    return (size_t)B * (size_t)H * (size_t)N * sizeof(float);
}


int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
           size_t workspace_bytes, fa_stream_t stream) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_NULL_POINTER;
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
    const long long BH = (long long)B * (long long)H;
    if (BH > 65535) return FA_ERR_SHAPE;
    auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
    if (mis16(q) || mis16(k) || mis16(v) || mis16(o) || mis16(dout) || mis16(dq) || mis16(dk) || mis16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
        return FA_ERR_ALIGNMENT;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
    if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_WORKSPACE;
    const size_t tb = (size_t)BH * (size_t)N * (size_t)d * 2u, lb = (size_t)BH * (size_t)N * 4u;
    const void* ins[6] = {q, k, v, o, dout, lse};
    const size_t in_bytes[6] = {tb, tb, tb, tb, tb, lb};
    void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_bytes[4] = {tb, tb, tb, lb};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return FA_ERR_ALIAS;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA_ERR_ALIAS;
    }
    const int dev_rc = check_device();
    if (dev_rc != FA_OK) return dev_rc;
    CUtensorMap tq, tk, tv, tdo;
    if (!encode_bhnd(&tq, q, d, N, (int)BH) || !encode_bhnd(&tk, k, d, N, (int)BH) ||
        !encode_bhnd(&tv, v, d, N, (int)BH) || !encode_bhnd(&tdo, dout, d, N, (int)BH))
        return FA_ERR_TENSOR_MAP;
    fa::BwdParams p{};
    p.lse = lse;
    p.N = N;
    p.n_tiles = (N + 127) / 128;
    p.causal = causal ? 1 : 0;
    p.scale = scale;
    p.scale_log2 = scale * 1.44269504088896340736f;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        p.watchdog_ns = g_watchdog_ns;
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* delta = static_cast<float*>(workspace);
    if (d == 64) return launch_bwd<64, 4>(tq, tk, tv, tdo, o, dout, delta, dq, dk, dv, p, (int)BH, st);
    return launch_bwd<128, 2>(tq, tk, tv, tdo, o, dout, delta, dq, dk, dv, p, (int)BH, st);
}

int fa_softmax_rows(const float* x, float* y, float* lse, long long M, int N, fa_stream_t stream) {
    if (!x || !y) return FA_ERR_NULL_POINTER;
    if (M < 1 || N < 1 || M > (1ll << 40)) return FA_ERR_SHAPE;
    const uintptr_t ax = reinterpret_cast<uintptr_t>(x), ay = reinterpret_cast<uintptr_t>(y),
                    al = reinterpret_cast<uintptr_t>(lse);
    if (((ax | ay) & 3u) != 0 || (lse && (al & 3u) != 0)) return FA_ERR_ALIGNMENT;
    const size_t bytes = (size_t)M * (size_t)N * 4u;
    if (ax != ay && overlaps(x, bytes, y, bytes)) return FA_ERR_ALIAS;  // in place is fine, a shift is not
    if (lse && (overlaps(lse, (size_t)M * 4u, x, bytes) || overlaps(lse, (size_t)M * 4u, y, bytes)))
        return FA_ERR_ALIAS;
    const int dev_rc = check_device();
    if (dev_rc != FA_OK) return dev_rc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    unsigned long long limit;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        limit = g_watchdog_ns;
    }
    const bool aligned = (N % 4 == 0) && ((ax | ay) & 15u) == 0;
    if (aligned && N <= fa::kWarpMaxN) {
        // short rows: one warp per chunk of rows
        const long long chunks = (M + fa::warp_chunk_rows(N) - 1) / fa::warp_chunk_rows(N);
        const long long ctas = (chunks + fa::kSmWarps - 1) / fa::kSmWarps;
        if (ctas > 0x7fffffffll) return FA_ERR_SHAPE;
        const size_t smem = (size_t)fa::kSmWarps * (fa::kWarpChunkBytes + 16u);
        if (cudaFuncSetAttribute(fa::softmax_rows_warp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return FA_ERR_CUDA;
        fa::softmax_rows_warp<<<(unsigned)ctas, fa::kSmThreads, smem, st>>>(x, y, lse, M, N, limit);
    } else if (aligned && (size_t)N * 4u <= fa::kSmMaxRowBytes) {
        // one CTA per row: the block scheduler keeps every SM full
        const size_t smem = fa::softmax_rows_smem_bytes(N);
        if (cudaFuncSetAttribute(fa::softmax_rows_smem, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return FA_ERR_CUDA;
        const long long ctas = std::min<long long>(M, 0x7fffffffll);
        fa::softmax_rows_smem<<<(unsigned)ctas, fa::kSmThreads, smem, st>>>(x, y, lse, M, N, limit);
    } else {
        const long long ctas = std::min<long long>(M, (long long)sms * 8);
        fa::softmax_rows_stream<<<(unsigned)ctas, fa::kSmThreads, 0, st>>>(x, y, lse, M, N);
    }
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

const char* fa_strerror(int code) {
    switch (code) {
        case FA_OK: return "ok";
        case FA_ERR_NULL_POINTER: return "a tensor pointer is NULL";
        case FA_ERR_HEAD_DIM: return "head dimension must be 64 or 128";
        case FA_ERR_SHAPE: return "B, H and N must be >= 1 and B*H <= 65535";
        case FA_ERR_ALIGNMENT: return "q, k, v, o must be 16-byte aligned and lse 4-byte aligned";
        case FA_ERR_SCALE: return "scale must be positive and finite";
        case FA_ERR_ALIAS: return "o or lse overlaps an input or each other";
        case FA_ERR_TENSOR_MAP: return "the driver rejected a TMA tensor map";
        case FA_ERR_CUDA: return "a CUDA runtime call failed";
        case FA_ERR_DEVICE: return "the current device is not an sm_103 GPU";
        case FA_ERR_SPLITS: return "n_splits must be 0 (automatic) or 1..64";
        case FA_ERR_WORKSPACE: return "the split-KV workspace is smaller than fa_splitkv_workspace_bytes()";
        case FA_ERR_SCRATCH_LIMIT:
            return "the partial states need more than FA_NOALLOC_SCRATCH_BYTES; call fa_fwd_splitkv with a workspace";
        case FA_ERR_MASK: return "window_left and window_right must be -1 (unbounded) or >= 0";
        default: return "unknown error code";
    }
}

int fa_get_device_status(unsigned int* status) {
    if (!status) return FA_ERR_NULL_POINTER;
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(status, fa::g_fa_status, sizeof(unsigned int)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

int fa_clear_device_status(void) {
    const unsigned int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

uint64_t fa_set_watchdog_ns(uint64_t ns) {
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t old = g_watchdog_ns;
    g_watchdog_ns = ns < 1000000ull ? 1000000ull : ns;
    return old;
}

int fa_watchdog_selftest(uint64_t ns, fa_stream_t stream, unsigned int* status) {
    if (!status) return FA_ERR_NULL_POINTER;
    const int dev_rc = check_device();
    if (dev_rc != FA_OK) return dev_rc;
    if (fa_clear_device_status() != FA_OK) return FA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    fa::fa_watchdog_selftest_kernel<<<1, 32, 0, s>>>((unsigned long long)ns);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    return fa_get_device_status(status);
}

int fa_watchdog_selftest_fwd(uint64_t ns, const void* q, const void* k, const void* v, void* o, float* lse, int N,
                             int d, fa_stream_t stream, unsigned int* status) {
    if (!status) return FA_ERR_NULL_POINTER;
    if (N > fa::kBlockM) return FA_ERR_SHAPE;  // one query tile, so the one CTA starts every row
    int rc = validate(q, k, v, o, lse, 1, 1, N, d, 1.0f);
    if (rc != FA_OK) return rc;
    Prepared pr;
    rc = prepare(q, k, v, o, lse, 1, 1, N, d, 0, 1.0f / std::sqrt((float)d), &pr);
    if (rc != FA_OK) return rc;
    if (fa_clear_device_status() != FA_OK) return FA_ERR_CUDA;
    pr.p.watchdog_ns = ns < 1000000ull ? 1000000ull : ns;
    pr.p.withhold_s = 1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rc = launch_d<false>(d, pr, s);
    if (rc != FA_OK) return rc;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    return fa_get_device_status(status);
}

int fa_get_last_error(void) {
    unsigned int st = 0;
    const int rc = fa_get_device_status(&st);
    if (rc != FA_OK) return rc;
    return (int)(st & 0x7fffffffu);
}

int fa_kernel_resources(int d, int kernel, fa_kernel_resources_t* out) {
    if (!out) return FA_ERR_NULL_POINTER;
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    const int dev_rc = check_device();
    if (dev_rc != FA_OK) return dev_rc;
    return d == 64 ? fwd_resources<64, 6, 6>(kernel, out) : fwd_resources<128, 2, 3>(kernel, out);
}

int fa_set_fwd_pairing(int mode) {
    if (mode != FA_PAIR_AUTO && mode != FA_PAIR_OFF && mode != FA_PAIR_ON) return FA_ERR_SHAPE;
    return g_pairing.exchange(mode);
}

int fa_fwd_kernel_for(int B, int H, int N, int d, int causal) {
    if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
    if (B < 1 || H < 1 || N < 1 || (long long)B * H > 65535) return FA_ERR_SHAPE;
    const int n_tiles = (N + fa::kBlockN - 1) / fa::kBlockN;
    if (use_two(d, causal ? 1 : 0, n_tiles, (long long)B * H)) return FA_KERNEL_FWD_TWO;
    return use_pair(d, causal ? 1 : 0, n_tiles) ? FA_KERNEL_FWD_PAIR : FA_KERNEL_FWD;
}

int fa_version(void) { return kVersion; }

}  // extern "C"
