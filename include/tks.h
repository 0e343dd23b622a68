/*
 * tks.h - C ABI of libtks, a GB300 (sm_103a) top-k index selector for
 * DeepSeek-Sparse-Attention-style indexer logits.
 *
 * The operation ("Technical Deep Dive | How to Use FlagOS's New Triton-TLE
 * Language to Build a TopK Selector Faster Than FlashInfer", section
 * "01. Why the TopK Selector Needs Optimization", step 2 of the three-step
 * workflow): for every row of logits, return the positions of the k largest
 * values; indices only, no sorted output.  It is computed by radix selection
 * (same page, section "02. Traditional GPU Approach: Radix Selection"):
 * logits are mapped to order-preserving unsigned keys, keys are binned by
 * digits from the most significant bits down, a histogram of each digit
 * locates the bin holding the k-th element, the rest are discarded, and the
 * elements above the final threshold are collected.
 *
 * Result order and ties.  Positions are ranked by value, largest first; +0.0
 * ranks above -0.0; equal values rank by position, lowest first (the page's
 * collection step appends equal values in scan order).  -inf is an ordinary
 * (lowest) value.  Subnormals keep their exact order.  NaN inside a row's
 * valid length is outside the contract (no error is raised; the result is
 * unspecified).  The selected set is unique; its order within the output row
 * is unspecified.
 *
 * Everything here is plain C: pointers, sizes and a CUDA stream passed as
 * void* (a cudaStream_t; NULL is the legacy default stream).
 */
#ifndef TKS_H
#define TKS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Logit element types. */
typedef enum {
    TKS_F32 = 0,  /* IEEE binary32 */
    TKS_BF16 = 1  /* bfloat16, stored as its 16 raw bits */
} tks_dtype;

/* Status codes returned by every entry point. */
typedef enum {
    TKS_OK = 0,
    TKS_E_INVAL = 1,       /* a bad argument; nothing was launched */
    TKS_E_UNSUPPORTED = 2, /* no usable device (not sm_100-class or no CUDA device) */
    TKS_E_CUDA = 3,        /* a CUDA runtime call failed (allocation, launch) */
    TKS_E_TIMEOUT = 4,     /* a device-side wait between thread blocks gave up */
    TKS_E_INTERNAL = 5,    /* a device-side consistency check failed */
    TKS_E_ROW_LEN = 6,     /* a device row length was < 0 or > row_stride (clamped) */
    TKS_E_TOO_LARGE = 7    /* more rows than tks_topk_indices_noalloc's fixed scratch holds */
} tks_status;

/* Largest k accepted. */
#define TKS_K_MAX (1 << 24)

/*
 * tks_topk_indices - enqueue the top-k selection of `batch` rows on `stream`.
 *
 *   logits      device pointer, `batch` rows of `row_stride` elements of type
 *               `dtype`, row r starting at element r * row_stride.  Must be
 *               aligned to the element size.  Only the first row_len[r]
 *               elements of row r are read, each exactly once from HBM.
 *   row_len     device pointer to `batch` int32 valid lengths, or NULL (every
 *               row has row_stride valid elements).  A length outside
 *               [0, row_stride] is clamped into it and reported as
 *               TKS_E_ROW_LEN by tks_device_status().
 *   batch       number of rows, >= 0 (0 enqueues nothing).
 *   row_stride  elements between row starts, 0 <= row_stride < 2^31.
 *   k           number of positions to select per row, 1 <= k <= TKS_K_MAX.
 *   dtype       a tks_dtype.
 *   out_idx     device pointer, int32 [batch][k] with row stride k.  Slots
 *               0 .. min(k, len)-1 of row r receive the selected positions
 *               (0-based within the row) in unspecified order; slots
 *               min(k, len) .. k-1 receive -1.
 *   stream      a cudaStream_t (NULL: the legacy default stream).
 *
 * Ownership: the caller owns logits, row_len and out_idx, which must stay
 * valid until the enqueued work completes; the library keeps no reference to
 * them.  The library owns a per-(device, stream) workspace, allocated and
 * zeroed on the first call made on that stream (so make that first call
 * before any CUDA-graph capture on the stream); later calls allocate nothing
 * and never synchronise, so they can be captured.  Calls on one stream run in
 * order; calls on different streams use different workspaces.
 *
 * Scheduling: the kernel is launched with programmatic stream serialisation,
 * so it may be made resident while the previous kernel of the stream is still
 * finishing; it waits for that kernel to complete (and for its writes to be
 * visible) before it reads or writes any global memory.
 *
 * Errors: argument errors return TKS_E_INVAL and launch nothing; CUDA errors
 * during setup or launch return TKS_E_CUDA.  Errors detected on the device
 * are recorded in the stream's workspace; read them with tks_device_status().
 * Returns TKS_OK once the work is enqueued.
 */
int tks_topk_indices(const void *logits, const int32_t *row_len, int32_t batch,
                     int64_t row_stride, int32_t k, int32_t dtype, int32_t *out_idx,
                     void *stream);

/*
 * tks_topk_indices_host - tks_topk_indices (the operation defined at the top
 * of this file) on buffers in page-locked host memory, for callers whose
 * logits are on the host: `logits`, `row_len` (or NULL) and `out_idx` have the layouts of
 * tks_topk_indices but are host addresses of memory allocated with
 * cudaHostAlloc / cudaMallocHost or registered with cudaHostRegister on the
 * current device's context.  The kernel reads the logits and row lengths
 * across the host link itself (plain loads, each logit once) and writes the
 * indices straight into `out_idx`; no copy through device memory is made.
 *
 * Asynchronous like tks_topk_indices: the indices are in `out_idx` once
 * `stream` has synchronised (tks_device_status(stream) does both).  The
 * caller must not write `logits` or `row_len`, nor read `out_idx`, until then.
 * Returns TKS_E_INVAL, launching nothing, when a non-empty buffer is not
 * page-locked host memory (device memory included), or on the argument
 * errors of tks_topk_indices; otherwise as tks_topk_indices.
 */
int tks_topk_indices_host(const void *logits, const int32_t *row_len, int32_t batch,
                          int64_t row_stride, int32_t k, int32_t dtype, int32_t *out_idx,
                          void *stream);

/*
 * tks_topk_indices_sorted - tks_topk_indices followed by the rank ordering of
 * each row's result: slots 0 .. min(k, len)-1 of row r hold the selected
 * positions ordered by value, largest first (+0.0 before -0.0), equal values
 * by lower position first, i.e. the selector's own order; slots min(k, len)
 * .. k-1 hold -1.  This is the optional sorted output of the radix_topk
 * pseudocode's final step ("Technical Deep Dive | ... Triton-TLE ... TopK
 * Selector", section "02. Traditional GPU Approach: Radix Selection").
 *
 * Arguments, ownership, workspace and device-side errors are those of
 * tks_topk_indices, with 1 <= k <= TKS_SORTED_K_MAX (a larger k returns
 * TKS_E_INVAL and launches nothing).  Two kernels are enqueued on `stream`,
 * the second waiting for the first.  For up to 8 rows with k <= 4096 the
 * selection is written to a scratch area of the stream's workspace, and the
 * second kernel places every slot over many blocks (each counts, for a tile
 * of slots, the row's selected values below each one); otherwise the
 * selection is written to out_idx and the second kernel sorts each row in
 * place, one block per row.  Returns TKS_E_CUDA if the second launch fails
 * (the first is enqueued).
 */
#define TKS_SORTED_K_MAX 16384
int tks_topk_indices_sorted(const void *logits, const int32_t *row_len, int32_t batch,
                            int64_t row_stride, int32_t k, int32_t dtype, int32_t *out_idx,
                            void *stream);

/*
 * tks_device_status - synchronise `stream`, then return and clear the first
 * device-side error recorded by calls on it (TKS_OK if none, or if no call
 * was ever made on it).  After an error the stream's workspace is re-zeroed,
 * so the next call starts clean.  Returns TKS_E_CUDA if synchronising fails.
 */
int tks_device_status(void *stream);

/* A static English description of a status code (never NULL). */
const char *tks_status_string(int status);

/* Version of the library as major * 10000 + minor * 100 + patch. */
int tks_version(void);

/* Frees every workspace the library holds (call with no work in flight). */
int tks_release(void);

/*
 * Tuning and test options (process-wide; take effect at the next call).
 *   TKS_OPT_FORCE_GROUP      thread blocks per row: 0 = automatic, else the
 *                            value, clamped to what the device can co-schedule
 *   TKS_OPT_SPIN_LIMIT_NS    how long a block waits for the others of its row
 *                            before giving up with TKS_E_TIMEOUT (default 1 s)
 *   TKS_OPT_MIN_PER_BLOCK    automatic split: rows of at most 4096 elements
 *                            stay on one block; longer rows get one block per
 *                            this many elements (default 4096, chosen by
 *                            measurement), leaving one block slot of the
 *                            device free when the row count allows
 *   TKS_OPT_TEST_SKIP_ARRIVE test only: 1 makes the first block of each row
 *                            skip its first arrival, so the others' waits run
 *                            out and report TKS_E_TIMEOUT; 0 = off
 *   TKS_OPT_FORCE_THREADS    threads per block: 0 = automatic (512 for rows
 *                            split into slices of 96 KiB or more, else 256),
 *                            or 256 or 512
 *   TKS_OPT_CLUSTER          rows split over one thread-block cluster, whose
 *                            blocks merge through distributed shared memory:
 *                            0 = automatic and 1 = never (split rows merge
 *                            through L2, measured faster), n >= 2 = clusters
 *                            of n blocks (at most what the device schedules)
 *                            for every row they fit
 * Returns TKS_E_INVAL for an unknown option, a negative value or (for
 * TKS_OPT_FORCE_THREADS) a block size other than 0, 256 or 512.
 */
typedef enum {
    TKS_OPT_FORCE_GROUP = 1,
    TKS_OPT_SPIN_LIMIT_NS = 2,
    TKS_OPT_MIN_PER_BLOCK = 3,
    TKS_OPT_TEST_SKIP_ARRIVE = 4,
    TKS_OPT_FORCE_THREADS = 5,
    TKS_OPT_CLUSTER = 6
} tks_option;
int tks_set_option(int option, int64_t value);

/*
 * tks_plan - the launch the next tks_topk_indices call with these sizes would
 * use on the current device: thread blocks per row (`group`) and grid size.
 * Either output pointer may be NULL.  Returns TKS_E_UNSUPPORTED without a
 * usable device.
 */
int tks_plan(int32_t batch, int64_t row_stride, int32_t k, int32_t dtype, int32_t *group,
             int32_t *grid);

/*
 * tks_topk_indices_noalloc - the same selection as tks_topk_indices, for
 * callers that cannot allocate device memory: code that runs where a
 * cudaMalloc is not allowed or not wanted (inside a pre-planned memory pool,
 * under an allocator that must not grow, or from a runtime that forbids
 * allocation after start-up).  The papers this library follows have no
 * counterpart to it; it exists only for such callers.
 *
 * Arguments, result layout and argument errors are those of
 * tks_topk_indices; the caller still provides logits, row_len and out_idx.
 * Instead of a workspace, the call uses a fixed scratch array compiled into
 * the library (about 2.9 MB, present on every device that loads the library
 * until the process exits).  That array holds at most TKS_NOALLOC_MAX_ROWS
 * rows: a larger batch returns TKS_E_TOO_LARGE and launches nothing.  The call
 * makes no cudaMalloc, cudaFree or other allocating call.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any CUDA-graph capture.  Every
 * call clears the part of the array it uses before its kernel runs, on
 * `stream`.  All calls share the one array, so calls that overlap on the GPU
 * (on different streams, or from several threads) race and give wrong
 * results: serialise them.
 *
 * Device-side errors of this entry point are not reported: tks_device_status
 * covers only the allocating entry points, and the next call clears the
 * array's status word.  A row length outside [0, row_stride] is clamped to
 * that range without notice (the result is that of the clamped length).
 * After a wait between thread blocks that timed out (a block held back for
 * longer than TKS_OPT_SPIN_LIMIT_NS) or a failed internal consistency check,
 * the affected row of out_idx may hold any mix of positions written before
 * the failure and the values it held before the call; no error code tells
 * this apart from a good result.  Callers that must detect such failures use
 * tks_topk_indices and tks_device_status instead.
 */
#define TKS_NOALLOC_MAX_ROWS 8
int tks_topk_indices_noalloc(const void *logits, const int32_t *row_len, int32_t batch,
                             int64_t row_stride, int32_t k, int32_t dtype, int32_t *out_idx,
                             void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TKS_H */
