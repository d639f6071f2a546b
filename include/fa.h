/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * The operation ("Online softmax, and the register that can't move",
 * section "Online softmax"; "Online Softmax: Tiling Across a Reduction",
 * loop-order and statistics sections):
 *
 *     O   = softmax(Q K^T * scale) V          row by row, in one pass
 *     LSE = m + ln(l)                          per query row
 *
 * computed key tile by key tile with a running row maximum m, a running sum
 * of exponentials l and an output accumulator, each corrected by
 * exp(m_old - m_new) when the maximum moves, and O divided by l once at the
 * end.  The N x N score matrix never reaches device memory.  LSE (the
 * natural-log normaliser) is the per-row statistic the backward pass needs
 * ("Online Softmax: Tiling Across a Reduction", backward-pass section).
 *
 * Causal attention (key j visible to query i iff j <= i) skips key tiles
 * that lie wholly after the query tile and masks element by element only on
 * the diagonal tile ("Online Softmax: Tiling Across a Reduction", causal
 * section).
 *
 * Layout (all contiguous, row-major, no padding):
 *     q, k, v, o : bf16  [B][H][N][d]      (element (b,h,i,c) at ((b*H+h)*N+i)*d+c)
 *     lse        : fp32  [B][H][N]
 * Query and key sequences have the same length N.
 *
 * Ownership: every pointer is a DEVICE pointer owned by the caller (except the
 * tensors of fa_fwd_host, which are host pointers).  The library allocates no
 * memory per call, keeps no reference after returning, and never synchronises
 * the host: the work is enqueued on `stream` (0 = the legacy default stream)
 * and completes asynchronously.  fa_fwd_host and fa_bwd also use internal
 * per-device streams, made once and kept.  Events order that work with
 * `stream` in both directions.
 *
 * Errors: each entry point returns FA_OK (0) or a negative FA_ERR_* code;
 * argument errors are detected on the host before anything is enqueued.
 * fa_strerror() names a code.  A kernel that waits longer than its
 * watchdog limit on an internal barrier abandons its tile, records a bit in
 * a device status word and exits; fa_get_last_error() and
 * fa_get_device_status() read that word.  The forward kernels (fa_fwd,
 * fa_fwd_masked, fa_fwd_splitkv, fa_fwd_splitkv_noalloc, fa_fwd_host) also
 * write NaN into the lse of every row of the tile they abandon, so that an
 * abort shows in the outputs; tiles a CTA had not started keep whatever the
 * output buffers held, so the status word is the authoritative signal.
 *
 * Per-device state (the device addresses of the library's static arrays, and
 * the internal streams and events of fa_fwd_host and fa_bwd) is set up by the
 * first call on each device and kept for the life of the process.  After
 * cudaDeviceReset() on a device, do not call this library on that device
 * again in the same process: the cached addresses and handles belong to the
 * destroyed context.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers */
typedef struct CUstream_st* fa_stream_t;

enum {
    FA_OK = 0,
    FA_ERR_NULL_POINTER = -1,   /* q, k, v, o or lse is NULL */
    FA_ERR_HEAD_DIM = -2,       /* d is not 64 or 128 */
    FA_ERR_SHAPE = -3,          /* B, H or N < 1, B*H > 65535, or B*H*ceil(N/128) >= 2^31 */
    FA_ERR_ALIGNMENT = -4,      /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
    FA_ERR_SCALE = -5,          /* scale not finite or not > 0 */
    FA_ERR_ALIAS = -6,          /* o or lse overlaps q, k or v, or each other */
    FA_ERR_TENSOR_MAP = -7,     /* the driver rejected a TMA descriptor */
    FA_ERR_CUDA = -8,           /* a CUDA runtime call failed (launch, attribute, driver entry point) */
    FA_ERR_DEVICE = -9,         /* the current device is not an sm_103 GPU */
    FA_ERR_SPLITS = -10,        /* n_splits outside 0..64 */
    FA_ERR_WORKSPACE = -11,     /* split-KV workspace smaller than fa_splitkv_workspace_bytes() */
    FA_ERR_SCRATCH_LIMIT = -12, /* fa_fwd_splitkv_noalloc: partial states exceed FA_NOALLOC_SCRATCH_BYTES */
    FA_ERR_MASK = -13           /* fa_fwd_masked: a window bound below -1 */
};

/* Size of the library's static split-KV scratch used by fa_fwd_splitkv_noalloc (32 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * fa_fwd -- fused attention forward.
 *
 *   q, k, v : device bf16 [B][H][N][d], 16-byte aligned, read only.
 *   o       : device bf16 [B][H][N][d], 16-byte aligned, written.
 *   lse     : device fp32 [B][H][N], written: ln(sum_j exp(scale * q_i . k_j))
 *             over the visible keys j.
 *   B, H    : batch and heads, >= 1, B*H <= 65535.
 *   N       : sequence length >= 1 (any value; the last tile is masked).
 *   d       : head dimension, 64 or 128.
 *   causal  : nonzero masks key j > query i.
 *   scale   : positive finite multiplier of the scores (1/sqrt(d) usually).
 *   stream  : CUDA stream the work is enqueued on.
 *
 * Inputs are not modified.  o and lse must not overlap q, k, v or each other.
 * Returns FA_OK once the kernel is enqueued.
 *
 * The kernel is persistent (at most one CTA per SM) and takes its query tiles
 * from a work counter in the library's static device memory; each call uses
 * the next of 1024 counters in turn, so calls may run concurrently on several
 * streams as long as fewer than 1024 of them are in flight at once.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           int causal, float scale, fa_stream_t stream);

/*
 * fa_fwd_masked -- fa_fwd under a structured mask: a sliding window and/or
 * document boundaries ("Online Softmax: Tiling Across a Reduction", causal
 * section: sliding windows and document-boundary masks become block-level
 * skip decisions).  Key j is visible to query i of batch entry b iff
 *
 *     (window_left  < 0  or  j >= i - window_left)    and
 *     (window_right < 0  or  j <= i + window_right)   and
 *     (doc_ids == NULL   or  doc_ids[b][j] == doc_ids[b][i]).
 *
 * window_right = 0 is causal attention, window_left = W - 1 with it a causal
 * sliding window of W keys; window_left = window_right = -1 with doc_ids NULL
 * is fa_fwd non-causal.  Key tiles no row of a query tile can see are never
 * loaded or multiplied; only tiles a boundary crosses are masked element by
 * element.
 *
 *   window_left, window_right : -1 (unbounded) or >= 0.
 *   doc_ids : device int32 [B][N], 4-byte aligned, or NULL.  The ids must not
 *             decrease along a sequence (each document is one contiguous run of
 *             positions); other ids give undefined results, never an
 *             out-of-bounds access.
 *   other arguments : as fa_fwd (there is no causal flag: use window_right).
 *
 * Every row sees at least itself.  Returns FA_OK, an fa_fwd argument error,
 * FA_ERR_MASK for a window bound below -1, FA_ERR_ALIGNMENT for doc_ids, or
 * FA_ERR_ALIAS when doc_ids overlaps o or lse.
 */
int fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  int window_left, int window_right, const int32_t* doc_ids, float scale, fa_stream_t stream);

/*
 * fa_fwd_splitkv -- the same forward for problems with few query tiles.
 *
 * The key range of every query tile is cut into n_splits contiguous chunks
 * of key tiles, each handled by its own CTA, so that small B*H*N still fills
 * the GPU.  Each CTA leaves a partial row state -- reference max m, the sum of
 * exponentials against it, and the unnormalised output -- in `workspace`; a
 * merge kernel then combines the chunks with the associative rule of
 * "5.2 CUDA Online Softmax", section 4.1 (m = max(m1, m2);
 * d = d1 e^(m1 - m) + d2 e^(m2 - m), applied to the output as well) and writes
 * o and lse exactly as fa_fwd does.
 *
 *   n_splits        : 1..64, or 0 to use fa_splitkv_auto_splits().  Chunks past
 *                     a causal tile's diagonal are empty and weigh nothing.
 *   workspace       : device memory owned by the caller, 16-byte aligned, at
 *                     least fa_splitkv_workspace_bytes(B, H, N, d, n_splits)
 *                     bytes, not overlapping any tensor; its contents on entry
 *                     do not matter and are overwritten.
 *   other arguments : as fa_fwd.
 *
 * Two kernels are enqueued on `stream`; calls sharing a workspace must not
 * overlap on the GPU.  Returns FA_OK, an fa_fwd argument error, FA_ERR_SPLITS,
 * FA_ERR_WORKSPACE, FA_ERR_ALIGNMENT or FA_ERR_NULL_POINTER for the workspace.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   int causal, float scale, int n_splits, void* workspace, size_t workspace_bytes,
                   fa_stream_t stream);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv without a caller workspace and
 * without allocating anything.  (An addition of this library; the pages have
 * no counterpart.)
 *
 * For callers that cannot allocate device memory when they run attention:
 * code whose device memory is owned by a host framework or an engine with a
 * fixed budget, or a latency-critical path that must not pay for cudaMalloc
 * and the device-wide synchronisation it may imply.  Instead of a workspace,
 * the partial states live in one static device array inside this library,
 * FA_NOALLOC_SCRATCH_BYTES (32 MiB) large, which every GPU that loads the
 * library keeps until the process exits.
 *
 *   arguments       : as fa_fwd_splitkv, minus workspace and workspace_bytes.
 *   n_splits        : 1..64, or 0 for the automatic count, lowered as needed
 *                     until n_splits * B*H*N * (d + 3) * 4 bytes fit.
 *
 * Returns FA_ERR_SCRATCH_LIMIT, enqueueing nothing, when the partial states
 * do not fit in FA_NOALLOC_SCRATCH_BYTES; other codes as fa_fwd_splitkv.
 *
 * The first call on a device looks up the array's device address (a
 * cudaGetSymbolAddress with that device current) and caches it; make that
 * first call before any stream capture.  The array is shared by every call
 * and keeps whatever the last call left in it, none of which is read by the
 * next call.  Calls that may run at the same time on the GPU (two streams,
 * two host threads) race on it and must be serialised by the caller.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                           int d, int causal, float scale, int n_splits, fa_stream_t stream);

/* Workspace bytes fa_fwd_splitkv needs: n_splits * B*H*N * (d + 3) * 4; 0 for invalid arguments. */
size_t fa_splitkv_workspace_bytes(int B, int H, int N, int d, int n_splits);

/*
 * A split count that fills about one wave of the current device (one CTA per
 * SM): floor(SMs / (query tiles * B*H)), at most the number of key tiles and
 * 64, at least 1.  Returns 1 when the plain fa_fwd already fills the GPU.
 */
int fa_splitkv_auto_splits(int B, int H, int N, int d, int causal);

/*
 * fa_fwd_host -- fa_fwd on HOST-resident tensors, streamed through the GPU.
 *
 * Arguments as for fa_fwd, except that q, k, v, o and lse are host pointers.
 * They must be pinned (page-locked, e.g. cudaHostAlloc) for the copies to
 * overlap the compute; pageable memory works but serialises.  Layouts are
 * unchanged ([B][H][N][d] bf16, lse [B][H][N] fp32), because the heads are
 * independent problems ("Online Softmax: Tiling Across a Reduction": each
 * query row's softmax needs only its own scores).  The call walks the B*H
 * heads in chunks of heads_per_chunk through three device slots in `workspace`,
 * on three streams.  While the forward kernel runs on chunk c, later chunks are
 * copied to the device (chunk c+k waits only for the read-back of chunk
 * c+k-3, whose slot it takes) and chunk c-1's o and lse are copied back.
 *
 *   heads_per_chunk  1 .. B*H, or 0 for ceil(B*H / 8)
 *   workspace        device memory, 256-byte aligned, at least
 *                    fa_fwd_host_workspace_bytes(B, H, N, d, heads_per_chunk)
 *                    bytes; owned by the caller, reusable once the call's work
 *                    on `stream` has completed
 *   stream           the caller's stream: the kernels run on it, and every copy
 *                    is ordered after the work already on it and before the work
 *                    enqueued on it afterwards (the call returns after enqueueing
 *                    and does not synchronise)
 *
 * Two internal copy streams per device are created on first use and kept.  The
 * enqueue of concurrent calls on one device is serialised by a lock.  Results
 * are identical to fa_fwd's, bit for bit.  Returns FA_OK, an fa_fwd argument
 * error, FA_ERR_SHAPE for heads_per_chunk outside 0..B*H, FA_ERR_NULL_POINTER or
 * FA_ERR_ALIGNMENT for the workspace, FA_ERR_WORKSPACE, FA_ERR_DEVICE,
 * FA_ERR_TENSOR_MAP or FA_ERR_CUDA.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                int causal, float scale, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                fa_stream_t stream);

/* Device workspace fa_fwd_host needs (three slots of one chunk's q, k, v, o and lse); 0 for bad arguments. */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d, int heads_per_chunk);

/*
 * fa_bwd -- attention backward pass: the gradients of L = sum(O * dO) with
 * respect to q, k and v, for the forward of fa_fwd.  Nothing of the N x N
 * weights is read back: the scores are recomputed tile by tile from q and k
 * and normalised with the saved per-row statistic lse, so every tile is
 * final in one pass ("Online Softmax: Tiling Across a Reduction",
 * backward-pass section).  With P = exp(scale q k^T - lse) and
 * D_i = sum_c dO_ic o_ic (visible pairs only):
 *
 *     dv = P^T dO,   ds = P * (dO v^T - D),   dq = scale ds k,   dk = scale ds^T q
 *
 *   q, k, v    : device bf16 [B][H][N][d], the forward's inputs.
 *   o, lse     : device bf16 [B][H][N][d] and fp32 [B][H][N], the forward's
 *                outputs (lse is the natural-log statistic fa_fwd writes).
 *   dout       : device bf16 [B][H][N][d], the gradient of L with respect to o.
 *   dq, dk, dv : device bf16 [B][H][N][d], written.
 *   causal, scale, B, H, N, d : as fa_fwd.
 *   workspace  : device memory owned by the caller, 4-byte aligned, at least
 *                fa_bwd_workspace_bytes() bytes (D, fp32 per row); contents on
 *                entry do not matter.
 *
 * Bf16 tensors 16-byte aligned; outputs and workspace must not overlap any
 * input or each other.  Three kernels: D on `stream`, then dq on `stream` and,
 * at the same time, dk and dv on an internal per-device stream (made on first
 * use and kept).  Events order the dk/dv kernel after D, and the work enqueued
 * on `stream` afterwards after both.  The enqueue of concurrent fa_bwd calls on
 * one device is serialised by a lock.  Returns FA_OK, or FA_ERR_NULL_POINTER, FA_ERR_HEAD_DIM,
 * FA_ERR_SHAPE, FA_ERR_ALIGNMENT, FA_ERR_SCALE, FA_ERR_WORKSPACE,
 * FA_ERR_ALIAS, FA_ERR_DEVICE, FA_ERR_TENSOR_MAP, FA_ERR_CUDA.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
           size_t workspace_bytes, fa_stream_t stream);

/* Workspace bytes fa_bwd needs: B*H*N*4; 0 for invalid arguments. */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_softmax_rows -- row-wise softmax of an fp32 matrix with the online
 * normaliser ("5.2 CUDA Online Softmax", sections 2 and 4.1; "Online softmax,
 * and the register that can't move", section "Online softmax"):
 *
 *     y[i][j] = exp(x[i][j] - m_i) / d_i,     lse[i] = m_i + ln(d_i)
 *
 * with (m_i, d_i) the running max and running sum of exp(x - m) of row i,
 * built in one pass and merged across threads with the associative rule.
 *
 *   x    : device fp32 [M][N], row-major, 4-byte aligned, read only.
 *   y    : device fp32 [M][N], written.  May be x itself (in place); must not
 *          overlap x otherwise.
 *   lse  : device fp32 [M], written, or NULL.
 *   M, N : rows and row length, >= 1 (M <= 2^40).
 *
 * Rows with N % 4 == 0, x and y 16-byte aligned and 4N <= 100 KiB are read
 * from HBM once (bulk copies into shared memory: one warp per chunk of rows up
 * to N = 2048, one CTA per row above); others are read twice.
 * A row with no finite element gives y = 0 and lse = -inf; +inf or NaN in a row
 * give NaN.  Returns FA_OK once the kernel is enqueued on `stream`, or
 * FA_ERR_NULL_POINTER, FA_ERR_SHAPE, FA_ERR_ALIGNMENT, FA_ERR_ALIAS,
 * FA_ERR_DEVICE, FA_ERR_CUDA.
 */
int fa_softmax_rows(const float* x, float* y, float* lse, long long M, int N, fa_stream_t stream);

/* Human-readable name of an FA_* code; never NULL. */
const char* fa_strerror(int code);

/*
 * Device status word of the current device: 0 when no kernel has given up
 * on a barrier since the last fa_clear_device_status(); otherwise bit flags
 * naming the wait that timed out.  Synchronises with the device.  Returns 0
 * and stores the word in *status, or FA_ERR_CUDA.
 */
int fa_get_device_status(unsigned int* status);

/*
 * fa_get_last_error -- the device-side timeout flag of the current device as
 * an int: 0 when no kernel has given up on a barrier since the last
 * fa_clear_device_status(), otherwise the (positive) status word of
 * fa_get_device_status(), whose bits name the wait that ran out; FA_ERR_CUDA
 * (negative) when the device could not be read.  It reports, it does not
 * clear.  Synchronises with the device, so it is a debugging call, not one for
 * the hot path.
 */
int fa_get_last_error(void);

/* Reset the device status word of the current device to 0 (synchronous). */
int fa_clear_device_status(void);

/*
 * Watchdog limit in nanoseconds applied to every barrier wait of later
 * launches from this process (default 1e9).  Values below 1e6 are raised
 * to 1e6.  Returns the previous value.
 */
uint64_t fa_set_watchdog_ns(uint64_t ns);

/*
 * Watchdog self-test: launches one CTA that waits on a shared-memory
 * barrier no one arrives on, with a limit of `ns` nanoseconds, so the wait
 * runs out.  The kernel records the timeout bit and returns; nothing faults
 * or hangs.  Synchronises `stream` and stores the kernel's report in
 * *status.  Returns FA_OK or FA_ERR_CUDA.
 */
int fa_watchdog_selftest(uint64_t ns, fa_stream_t stream, unsigned int* status);

/*
 * Watchdog self-test of the forward kernel itself: fa_fwd on one query tile
 * (B = H = 1, 1 <= N <= 128) with its S products withheld, so that the softmax
 * warps' first wait on S runs out after `ns` nanoseconds (at least 1e6).  The
 * kernel then takes its abort path: it records the timeout bit, writes NaN into
 * lse[0 .. N-1], leaves o untouched, lets its copies land, frees its tensor
 * memory and returns; nothing faults or hangs.  Clears the status word first,
 * synchronises `stream` and stores the word in *status.  Arguments as fa_fwd.
 * Returns FA_OK, FA_ERR_SHAPE for N > 128, an fa_fwd argument error or
 * FA_ERR_CUDA.
 */
int fa_watchdog_selftest_fwd(uint64_t ns, const void* q, const void* k, const void* v, void* o, float* lse, int N,
                             int d, fa_stream_t stream, unsigned int* status);

/*
 * fa_kernel_resources -- what the runtime reports for one of the library's
 * kernels at head dimension d (64 or 128), as launched: registers per thread,
 * threads per CTA, dynamic and static shared memory, local memory per thread,
 * resident CTAs per SM (cudaOccupancyMaxActiveBlocksPerMultiprocessor) and the
 * tensor-memory columns it allocates.  A resource report, not part of the
 * computation (the pages' "LLM kernels 3: attention and online softmax"
 * reports the same figures for its kernels).
 *
 *   kernel : FA_KERNEL_FWD (fa_fwd, fa_fwd_host: one CTA per query tile),
 *            FA_KERNEL_FWD_PAIR (the same at d = 128 in CTA pairs; see
 *            fa_set_fwd_pairing; d = 64 gives FA_ERR_HEAD_DIM),
 *            FA_KERNEL_FWD_TWO (the same at d = 64 with two query tiles
 *            per CTA; d = 128 gives FA_ERR_HEAD_DIM),
 *            FA_KERNEL_FWD_MASKED, FA_KERNEL_FWD_SPLITKV, FA_KERNEL_BWD_DQ,
 *            FA_KERNEL_BWD_DKDV.
 *
 * Returns FA_OK, FA_ERR_NULL_POINTER, FA_ERR_HEAD_DIM, FA_ERR_SHAPE for an
 * unknown kernel, FA_ERR_DEVICE or FA_ERR_CUDA.
 */
enum {
    FA_KERNEL_FWD = 0,
    FA_KERNEL_FWD_MASKED = 1,
    FA_KERNEL_FWD_SPLITKV = 2,
    FA_KERNEL_BWD_DQ = 3,
    FA_KERNEL_BWD_DKDV = 4,
    FA_KERNEL_FWD_PAIR = 5,
    FA_KERNEL_FWD_TWO = 6
};
typedef struct {
    int registers_per_thread;
    int threads_per_cta;
    int dynamic_smem_bytes;
    int static_smem_bytes;
    int local_bytes_per_thread;
    int ctas_per_sm;
    int tmem_columns;
} fa_kernel_resources_t;
int fa_kernel_resources(int d, int kernel, fa_kernel_resources_t* out);

/*
 * Forward kernel choice for full and causal attention (fa_fwd, fa_fwd_host,
 * and fa_fwd_masked without windows or documents): one query tile per CTA, or
 * units of two adjacent query tiles.  Same results either way, up to rounding
 * order; the choice is a matter of speed.
 *
 *   d = 128: units are CTA pairs (FA_KERNEL_FWD_PAIR): two CTAs on two SMs
 *       take the two tiles against the same key tiles with two-SM tensor-core
 *       products, each SM loading half of every K and V tile.
 *   d = 64: units are two tiles in one CTA (FA_KERNEL_FWD_TWO), each tile with
 *       its own softmax warpgroup, S, P and O, the K and V tiles loaded once
 *       for both.
 *
 *   FA_PAIR_AUTO (default): at d = 128, CTA pairs for full attention and for
 *       causal attention with at least 96 query tiles (N > 12160); at d = 64,
 *       two tiles per CTA when a model of both schedules on a 152-SM GB300
 *       (the two-tile kernel's step at 0.9 of the one-tile kernel's, half as
 *       many units) says it finishes first, which holds once there are about
 *       as many units as SMs (not for one head of N = 4096); one query tile
 *       per CTA (FA_KERNEL_FWD) otherwise.
 *   FA_PAIR_OFF, FA_PAIR_ON: always the one, always the other.
 *
 * In causal attention a unit also computes the key tile after its first
 * tile's diagonal, fully masked for that tile, which costs 1 / (key tiles + 1)
 * of the work and is why short causal sequences keep one tile per CTA.
 * Applies to launches enqueued after the call, process-wide.  Returns the
 * previous mode, or FA_ERR_SHAPE for an unknown one.
 */
enum { FA_PAIR_AUTO = 0, FA_PAIR_OFF = 1, FA_PAIR_ON = 2 };
int fa_set_fwd_pairing(int mode);

/*
 * The forward kernel fa_fwd launches for these sizes under the current mode:
 * FA_KERNEL_FWD, FA_KERNEL_FWD_PAIR (d = 128) or FA_KERNEL_FWD_TWO (d = 64);
 * FA_ERR_HEAD_DIM or FA_ERR_SHAPE for sizes fa_fwd rejects.  No device is
 * touched.
 */
int fa_fwd_kernel_for(int B, int H, int N, int d, int causal);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
