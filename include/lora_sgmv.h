/*
 * lora_sgmv.h -- C ABI of the GB300 multi-LoRA delta path (Punica-style
 * segmented gather matrix-vector / matrix multiplication, "SGMV").
 *
 * The path computes, for a batch of M token rows where row i carries an
 * adapter slot ids[i] in a contiguous adapter pool,
 *
 *     y[i, :] += s_a * (x[i, :] . A[a]^T) . B[a]^T        a = ids[i]
 *
 * (unmerged LoRA delta with its alpha/r scaling: "vLLM-Ascend LoRA"
 * article, section 1.1; the per-token routing through a weight pool:
 * "09. Triton Fused LoRA", Steps 1-3; the segmented form
 * Y = X W + (x1 A1 B1, ..., xn An Bn): "III.Punica: Multi-Tenant LoRA
 * Serving", section SGMV).  The base product X W is not part of this
 * library; y holds it on entry.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument named as "device" is a CUDA device pointer; the
 *    library never allocates, frees or synchronises.  All work is enqueued
 *    on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *    stream) and runs asynchronously.  The caller owns every buffer and
 *    must keep it alive until the stream has finished the call.
 *  - Element types: LORA_F32 or LORA_BF16.  x, the pools and y share one
 *    type; the intermediate h is always fp32; accumulation is always fp32.
 *    fp32 inputs are computed with fp32 FMA only (no reduced-precision
 *    tensor math).
 *  - Layouts (element strides; the innermost dimension is contiguous):
 *      x       [M][ldx]                      row i = token i
 *      A pool  [n_adapters][r_max][d_in]     rows of A[a] at a_stride_r,
 *                                            adapters at a_stride_adapter
 *      B pool  [n_adapters][d_out][r_max]    per output slice
 *      y       [M][ldy]                      updated in place (+=)
 *      h       [M][ldh]  fp32                indexed by token row
 *    ("09. Triton Fused LoRA", Step 1: lora_a_pool is (num_loras, r,
 *    in_features); its test builds lora_b_pool as (num_loras, out, r).)
 *  - Alignment: every base pointer 16-byte aligned; every row stride a
 *    multiple of 16 bytes; d_in, every slice's d_out and y column offset
 *    multiples of 8 (bf16) or 4 (fp32) elements.
 *  - Rows whose id is -1 carry no adapter and are left bit-identical.  Ids
 *    outside [-1, n_adapters) are treated the same way and counted on the
 *    device (LORA_COUNT_INVALID).  Nothing traps.
 *  - Mixed ranks: with a rank table ranks[a] (device, may be NULL = every
 *    adapter has rank r_max), adapter a uses rows [0, ranks[a]) of A[a] and
 *    columns [0, ranks[a]) of B[a]; the padding up to r_max is never read
 *    into a result ("vLLM-Ascend LoRA" article, section 3.4).  A rank
 *    outside [0, r_max] skips that adapter's rows and sets
 *    LORA_DEVERR_RANK in the batch counters.
 *  - Scale: s_a = adapter_scale[a] when adapter_scale (device, fp32,
 *    n_adapters entries) is non-NULL, else `scale`.  It is applied exactly
 *    once, to the fp32 intermediate ("vLLM-Ascend LoRA" article, sections
 *    2.1 and 3.3: alpha/r is kept apart from the weights and multiplied in
 *    once, as (tmp * scale) . B^T).
 *  - y is rounded once: fp32(y) + delta, converted to y's type (round to
 *    nearest even).
 *
 * Device state: the library keeps per-device set-up (kernel attributes,
 * occupancy figures, the static workspace's device address) for the life
 * of the process; it assumes no cudaDeviceReset while it is in use.
 *
 * Errors: every call returns lora_status_t.  Host-side argument checks
 * return LORA_ERR_INVALID / LORA_ERR_UNSUPPORTED / LORA_ERR_WORKSPACE
 * before anything is enqueued; a failed kernel launch returns
 * LORA_ERR_CUDA.  lora_last_error_string() describes the last failure on
 * the calling thread.  Conditions only the device can see are reported
 * through the batch's device counters (see LORA_COUNT_*), never by a trap.
 */
#ifndef LORA_SGMV_H
#define LORA_SGMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int lora_status_t;

#define LORA_OK 0
#define LORA_ERR_INVALID (-1)     /* a null pointer, negative size, bad stride */
#define LORA_ERR_UNSUPPORTED (-2) /* dtype, alignment or size outside the support */
#define LORA_ERR_WORKSPACE (-3)   /* workspace smaller than lora_workspace_size() */
#define LORA_ERR_CUDA (-4)        /* a CUDA call or kernel launch failed */

#define LORA_F32 0
#define LORA_BF16 1

/* Path selection for lora_delta / lora_shrink / lora_expand. */
#define LORA_PATH_AUTO 0      /* fused bf16: batches of at most 256 rows on the small-batch kernel,
                                 of at most 2048 on the streaming kernel (see lora_delta); larger
                                 batches: groups with >= tc_min_rows rows on the tcgen05 kernel,
                                 the others on the small-segment kernel */
#define LORA_PATH_CUDA_CORE 1 /* no tcgen05 kernel: the small-batch or streaming kernel where they
                                 take the batch, else the small-segment kernel (clusters of CTAs,
                                 warp-level bf16 tensor-core tiles; fp32: CUDA-core FMAs) */
#define LORA_PATH_TENSOR 2    /* every segment on the tcgen05 kernel (bf16 only; lora_delta,
                                 lora_shrink and lora_expand) */

/* Largest supported sizes. */
#define LORA_MAX_TOKENS (1 << 24)
#define LORA_MAX_RANK 128
#define LORA_MAX_SLICES 4
#define LORA_DESC_INLINE_ROWS 28 /* token rows held inline in a segment descriptor */

/* Device counters written by lora_prepare_batch (int32 each, in order). */
#define LORA_COUNT_SEGS 0       /* number of segments S */
#define LORA_COUNT_ACTIVE 1     /* rows with a valid adapter */
#define LORA_COUNT_INVALID 2    /* rows whose id is outside [-1, n_adapters) */
#define LORA_COUNT_SMALL_SEGS 3 /* segments of groups with fewer than tc_min_rows rows */
#define LORA_COUNT_TC_SEGS 4    /* segments of groups with at least tc_min_rows rows */
#define LORA_COUNT_TC_ROWS 5    /* rows inside those segments */
#define LORA_COUNT_DEVERR 6     /* bit set of LORA_DEVERR_* raised by later calls */
#define LORA_COUNT_GROUPS 7     /* distinct adapters in the batch */
#define LORA_NUM_COUNTS 8

/* Bit of a descriptor's segment-index field: the segment is in tc_segs. */
#define LORA_DESC_TC_FLAG 0x40000000

#define LORA_DEVERR_RANK 1 /* an adapter's rank was outside [0, r_max] */
#define LORA_DEVERR_WAIT 2 /* a bounded device wait gave up (result incomplete) */
#define LORA_DEVERR_ROW 4  /* lora_batch_update named a row outside [0, M) (skipped) */

/*
 * Segment metadata of one batch, built on the device by lora_prepare_batch
 * (token regrouping of "III.Punica: Multi-Tenant LoRA Serving", section
 * 代码: weight_indices, seg_lens, seg_indptr, sorted_token_ids).
 *
 * Device arrays (all int32, inside the caller's workspace):
 *   sorted_token_ids[M]     token rows grouped by adapter; the first
 *                           counts[LORA_COUNT_ACTIVE] entries are valid
 *   seg_indptr[max_segs+1]  start of segment s in sorted_token_ids
 *   seg_lens[max_segs]      rows in segment s (> 0)
 *   weight_indices[max_segs] adapter slot of segment s
 *   seg_records[max_segs][32] per segment s a 128-byte descriptor
 *                             {start, len, adapter, s | flag, rows[28]}:
 *                             flag is LORA_DESC_TC_FLAG when the segment
 *                             is in tc_segs; rows holds the segment's
 *                             first min(len, 28) token rows; entries
 *                             s >= num_segs have len 0
 *   small_segs[max_segs][4]   records {start, len, adapter, s} of the
 *                             segments whose adapter group has fewer than
 *                             tc_min_rows rows, in segment order
 *   tc_segs[max_segs][4]      records of the segments whose adapter group
 *                             has at least tc_min_rows rows (all chunks of
 *                             such a group), in segment order
 *   tc_indptr[max_segs+1]   prefix sum of rows over tc_segs
 *   counts[LORA_NUM_COUNTS] see LORA_COUNT_*
 * Host fields describe the batch the metadata was built for.
 */
typedef struct lora_batch {
    int32_t *sorted_token_ids;
    int32_t *seg_indptr;
    int32_t *seg_lens;
    int32_t *weight_indices;
    int32_t *seg_records;
    int32_t *small_segs;
    int32_t *tc_segs;
    int32_t *tc_indptr;
    int32_t *counts;
    int32_t M;           /* token rows */
    int32_t n_adapters;  /* pool size the ids index into */
    int32_t chunk_size;  /* 0 = one segment per adapter group */
    int32_t max_segs;    /* capacity of the segment arrays */
    int32_t tc_min_rows; /* tensor-core row threshold used for the split */
    uint32_t magic;      /* set by lora_prepare_batch */
    const int32_t *ids;  /* the ids the batch stands for (device; the caller's
                            array until lora_batch_update, then ids_store);
                            read again by the small-batch and streaming kernels */
    int32_t *ids_store;  /* the batch's own copy of the ids (in the workspace),
                            written by lora_batch_update */
    int32_t order;       /* LORA_ORDER_* the batch was built with */
    int32_t stale;       /* 1: ids changed since the segment metadata was built
                            (lora_batch_update); lora_batch_refresh rebuilds it */
} lora_batch_t;

/* One output slice of the expand step: B pool and the y columns it writes
 * (a fused projection such as QKV keeps one B pool per slice). */
typedef struct lora_b_slice {
    const void *B_pool;     /* device; element (adapter a, output n, rank k) at
                               a * stride_adapter + n * stride_n + k * stride_r */
    int64_t stride_adapter; /* elements between adapters */
    int64_t stride_n;       /* elements between outputs: >= r_max when stride_r <= 1
                               ([n_adapters][d_out][>= r_max], rank-contiguous rows);
                               1 when rank-major */
    int32_t d_out;          /* rows of this slice */
    int32_t y_col;          /* first y column written by this slice */
    const void *A_pool;     /* lora_delta only: this slice's own A pool (a fused
                               projection whose slices each have their A), laid
                               out like the call's A_pool (same strides); NULL:
                               the call's A_pool */
    int64_t stride_r;       /* elements between ranks: 0 or 1 (rank-contiguous rows,
                               the default), or >= d_out with stride_n = 1: the
                               rank-major layout [n_adapters][>= r_max][d_out], in
                               which an adapter of rank r reads r whole rows and
                               no padding ("vLLM-Ascend LoRA" article, section
                               4.2: adapter-major, rank-secondary weight blocks).
                               All slices of a call share one layout; rank-major
                               pools run on the streaming kernel only (bf16
                               lora_delta; a batch above its 2048 rows runs as
                               consecutive launches over 2048-row ranges), other
                               calls return LORA_ERR_UNSUPPORTED. */
} lora_b_slice_t;

/*
 * Workspace bytes lora_prepare_batch needs for a batch of M rows over a
 * pool of n_adapters with the given chunk size (0 = no chunking).  Returns
 * 0 when an argument is out of range.
 */
size_t lora_workspace_size(int32_t M, int32_t n_adapters, int32_t chunk_size);

/*
 * Build segment metadata on the device, with no host synchronisation.
 *
 * ids          device int32[M]: adapter slot per token row, -1 = none.
 * M            rows, 0 <= M <= LORA_MAX_TOKENS.
 * n_adapters   pool size, >= 1.
 * chunk_size   0: one segment per adapter group; > 0: every group is cut
 *              into segments of chunk_size rows, the last one shorter
 *              ("III.Punica: Multi-Tenant LoRA Serving", section 代码:
 *              the regrouped token stream is cut into fixed-size chunks,
 *              each a logical segment with its own adapter).
 * tc_min_rows  the segments of adapter groups with at least this many rows
 *              go to the tensor-core kernel under LORA_PATH_AUTO
 *              ("vLLM-Ascend LoRA" article, section 4.1: blocks below a row
 *              threshold use vector dot products; with chunking, every chunk
 *              of a long group counts as part of its group); <= 0 selects
 *              the library default, 32 rows (on GB300, for batches of 8192
 *              rows with every group of L rows, the CUDA-core kernel is ahead
 *              for L <= 24, the tensor-core kernel for L = 32, 64, 128 and
 *              256, the two even at 48).  Batches of at most 2048 rows do not
 *              use the split: the streaming kernel takes them whole.
 * workspace    device buffer of >= lora_workspace_size(M, n_adapters,
 *              chunk_size) bytes, 256-byte aligned; owned by the caller and
 *              referenced by *batch until the batch is no longer used.
 * batch        host struct filled with pointers into workspace.
 *
 * Grouping rule: adapter groups appear in the order in which their adapter
 * first occurs among the rows; rows inside a group keep ascending row
 * order (the Punica page's example: ids 2 2 2 5 5 1 1 give
 * seg_indptr = [0, 3, 5, 7]).  Rows with id -1 or an out-of-range id are
 * in no segment.
 *
 * Ordering: the kernel is launched with programmatic dependent launch and
 * reads ids while the previous kernel in the stream may still be running
 * (the workspace is written only after that kernel has completed).  ids
 * must therefore be final before that previous kernel starts, which holds
 * whenever ids come from a copy or from any kernel enqueued before it, and
 * when that previous kernel is one of this library's (they never write ids).
 * The batch keeps the ids pointer: calls that use the batch may group the
 * rows again from it, so ids must keep these values while the batch is used.
 */
lora_status_t lora_prepare_batch(const int32_t *ids, int32_t M, int32_t n_adapters,
                                 int32_t chunk_size, int32_t tc_min_rows,
                                 void *workspace, size_t workspace_bytes,
                                 lora_batch_t *batch, void *stream);

/* Group orders for lora_prepare_batch_ordered. */
#define LORA_ORDER_FIRST_APPEARANCE 0 /* the default: groups as their adapter first occurs */
#define LORA_ORDER_ASCENDING 1        /* groups by increasing adapter id */

/*
 * lora_prepare_batch with a choice of group order.  "III.Punica:
 * Multi-Tenant LoRA Serving", section 代码, says only that prepare_lora_batch
 * regroups the tokens by adapter; LORA_ORDER_ASCENDING reads that as a sort
 * by adapter id (ids 2 2 2 5 5 1 1 give seg_indptr = [0, 2, 5, 7] and
 * weight_indices = [1, 2, 5]).  Rows inside a group keep ascending row
 * order either way, and the segments, chunks and every other output are
 * those of the same groups in the other order.  An order other than the two
 * returns LORA_ERR_INVALID; everything else as for lora_prepare_batch.
 */
lora_status_t lora_prepare_batch_ordered(const int32_t *ids, int32_t M, int32_t n_adapters,
                                         int32_t chunk_size, int32_t tc_min_rows, int32_t order,
                                         void *workspace, size_t workspace_bytes,
                                         lora_batch_t *batch, void *stream);

/*
 * lora_prepare_batch with no caller workspace and no allocation: the
 * metadata goes to a device array that this library owns
 * (LORA_STATIC_WORKSPACE_BYTES on every GPU that loads the library, held
 * until the process exits).  The pages have no counterpart of this call; it
 * is for callers that cannot allocate device memory at the point where they
 * build a batch: code running inside another framework that owns the
 * device's memory through its own allocator and forbids direct cudaMalloc,
 * or a serving loop that must not pay cudaMalloc's device-wide
 * synchronisation on its step path.
 *
 * Arguments and result are those of lora_prepare_batch, without workspace
 * and workspace_bytes.  The batch needs lora_workspace_size(M, n_adapters,
 * chunk_size) <= LORA_STATIC_WORKSPACE_BYTES (4 MiB: about 8 bytes per
 * row plus a fixed part that grows with n_adapters, so for example up to
 * about 355000 rows with 4096 adapters unchunked, 264000 with 64-row
 * chunks); a larger batch returns
 * LORA_ERR_WORKSPACE and launches nothing.  The call allocates no memory:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Set-up: the first call on a device (the current device) looks up the
 * array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.  A failed look-up returns LORA_ERR_CUDA.
 *
 * Sharing: every call on a device writes the same array, and the array
 * keeps the last call's contents.  A batch returned by this call stays
 * valid only until the next lora_prepare_batch_static on that device has
 * run; calls whose kernels can overlap on the GPU (different streams
 * without ordering, or a later call before the previous batch's
 * lora_shrink / lora_expand / lora_delta have run) race.  The kernel
 * rewrites every value the batch reads, so nothing has to be cleared
 * between calls.
 */
#define LORA_STATIC_WORKSPACE_BYTES (4u << 20)
lora_status_t lora_prepare_batch_static(const int32_t *ids, int32_t M, int32_t n_adapters,
                                        int32_t chunk_size, int32_t tc_min_rows, lora_batch_t *batch,
                                        void *stream);

/*
 * Incremental update of a prepared batch: the grouping is kept across decode
 * steps and patched when sequences join or leave ("vLLM-Ascend LoRA"
 * article, sections 4.2 and 5.3: the index preparation is cached rather
 * than rebuilt every step).
 *
 * lora_batch_update sets, for k < n, the adapter of row rows[k] to
 * new_ids[k] (-1: the row leaves; an id: the row joins or switches), in the
 * batch's own copy of the ids (ids_store, in the workspace; the first update
 * copies the batch's ids there).  rows and new_ids are device int32[n];
 * rows must lie in [0, M) (others are skipped and raise LORA_DEVERR_ROW in
 * the counters, which report it until the metadata is rebuilt);
 * when a row appears twice, the later entry wins.  No host
 * synchronisation.  The segment metadata (sorted_token_ids, seg_indptr, ...)
 * and the counters then describe the old ids (batch->stale = 1): the
 * small-batch and streaming kernels, which group the rows themselves, use
 * the patched ids directly, so a decode step needs no rebuild; every other
 * path rebuilds the metadata into the workspace before it runs (each call,
 * while the batch is stale), and lora_batch_refresh rebuilds it once and
 * clears stale.  After lora_batch_refresh the batch equals the one
 * lora_prepare_batch_ordered builds from the patched ids.  The update
 * enqueues one kernel, which waits for the kernels ahead of it before it
 * writes; the kernels of later calls on an updated batch read its ids only
 * after their own wait on the kernels ahead (the ordering contract of
 * lora_delta does not apply to them).
 * Not in the pages' interface: an addition for serving loops.
 */
lora_status_t lora_batch_update(lora_batch_t *batch, const int32_t *rows, const int32_t *new_ids, int32_t n,
                                void *stream);
lora_status_t lora_batch_refresh(lora_batch_t *batch, void *stream);

/*
 * Shrink: h[i, j] = sum_k x[i, k] * A[a, j, k] for j < r_a, and 0 for
 * r_a <= j < r_max, for every row i in a segment (unscaled; "vLLM-Ascend
 * LoRA" article, section 3.2: first project d_in down to r).  Rows in no
 * segment keep their h contents.  h: device fp32 [M][ldh], ldh >= r_max.
 * Kernels (bf16): under LORA_PATH_AUTO the segments of groups with at least
 * tc_min_rows rows and a tensor-core rank (a multiple of 8, at most 32) run
 * on the tcgen05 kernel (x jobs only, h written from its fp32 accumulator),
 * the others on the small-segment kernel, side by side; LORA_PATH_TENSOR puts
 * every segment on the tcgen05 kernel, LORA_PATH_CUDA_CORE (and fp32) every
 * segment on the small-segment kernel.
 */
lora_status_t lora_shrink(const lora_batch_t *batch, int32_t dtype,
                          const void *x, int64_t ldx, int32_t d_in,
                          const void *A_pool, int64_t a_stride_adapter,
                          int64_t a_stride_r, int32_t r_max,
                          const int32_t *ranks, float *h, int64_t ldh,
                          int32_t path, void *stream);

/*
 * Expand: y[i, y_col_t + n] += s_a * sum_{j < r_a} h[i, j] * B_t[a, n, j]
 * for every row i in a segment and every slice t ("vLLM-Ascend LoRA"
 * article, section 3.3: delta = (tmp * scale) . B^T added into out).
 * slices: host array of n_slices (1..LORA_MAX_SLICES) descriptors.
 * Kernels as for lora_shrink (the tcgen05 kernel runs y jobs only).  On the
 * tcgen05 kernel s_a * h is rounded once to bf16 for the tensor cores, as in
 * lora_delta; y + delta is formed in fp32 and rounded to y's type once.
 */
lora_status_t lora_expand(const lora_batch_t *batch, int32_t dtype,
                          const float *h, int64_t ldh, int32_t r_max,
                          const lora_b_slice_t *slices, int32_t n_slices,
                          const int32_t *ranks, float scale,
                          const float *adapter_scale, void *y, int64_t ldy,
                          int32_t path, void *stream);

/*
 * Fused delta: shrink, scale and expand in one pass; the M x r
 * intermediate stays in registers, shared memory or tensor memory and is
 * never written to global memory ("vLLM-Ascend LoRA" article, section 4.3).
 * Arguments as for lora_shrink and lora_expand.  Each y element is read,
 * y + delta is formed in fp32 and rounded to y's type once.
 * Batches of up to 2048 rows (bf16, LORA_PATH_AUTO or LORA_PATH_CUDA_CORE):
 * a kernel that groups the rows itself from the batch's ids (the same groups
 * as lora_prepare_batch) runs the whole batch, so that it does not wait for
 * the batch metadata: up to 256 rows (a decode step) the single-pass
 * small-batch kernel (r_max <= 64, d_in a multiple of 16 per cluster CTA),
 * above that the streaming kernel (r_max 16, 32 or 64, d_in a multiple of
 * 64 per cluster CTA, min(M, n_adapters) <= 2048), whose
 * tiles stream through a ring of TMA copies.  A batch neither takes runs on
 * the kernels of larger batches.  Rank-major B pools run on the streaming
 * kernel at every batch size: above 2048 rows as consecutive launches over
 * 2048-row ranges, each grouping its own rows.  These kernels read ids, the A and B pools,
 * ranks and adapter_scale before they wait for the kernels ahead of them in
 * the stream (programmatic dependent launch): those must be final before the
 * kernel preceding this call starts (adapter weights loaded earlier, ids from
 * a copy or an earlier kernel).  x and y are read only after that wait.
 * Non-finite y: every path adds y per element, so a NaN or infinity in
 * y[i, n] gives a non-finite result there and nowhere else.
 */
lora_status_t lora_delta(const lora_batch_t *batch, int32_t dtype,
                         const void *x, int64_t ldx, int32_t d_in,
                         const void *A_pool, int64_t a_stride_adapter,
                         int64_t a_stride_r, int32_t r_max,
                         const lora_b_slice_t *slices, int32_t n_slices,
                         const int32_t *ranks, float scale,
                         const float *adapter_scale, void *y, int64_t ldy,
                         int32_t path, void *stream);

/* Description of the last failure on the calling thread ("" if none). */
const char *lora_last_error_string(void);

/* ABI version of this library (major * 100 + minor). */
int32_t lora_abi_version(void);

/* Number of kernel launches this library has enqueued in this process (a
 * diagnostic; launches captured into a CUDA graph are counted once, at
 * capture). */
int64_t lora_launch_count(void);

/* Kernels of the library (bits of lora_last_kernels). */
#define LORA_KERNEL_PREPARE 1   /* segment metadata (lora_prepare_batch*) */
#define LORA_KERNEL_SMALL 2     /* small-batch fused kernel: rows grouped on chip */
#define LORA_KERNEL_CUDA_CORE 4 /* small-segment kernel (clusters, warp-level tiles) */
#define LORA_KERNEL_TENSOR 8    /* tcgen05 kernel for long segments */
#define LORA_KERNEL_STREAM 16   /* streaming fused kernel: rows grouped on chip, chunks through a TMA ring */

/* The kernels the calling thread's last call of this library enqueued, as a
 * bit set of LORA_KERNEL_* (0 if it enqueued none; a diagnostic). */
int32_t lora_last_kernels(void);

/*
 * Diagnostic of the bounded device waits.  Enqueues one CTA that waits, with
 * the same bounded wait the kernels use on their mbarriers, on a barrier that
 * nothing completes (no copy is in flight); the wait gives up after its limit
 * (about 0.1 s) and the CTA sets LORA_DEVERR_WAIT in counts[LORA_COUNT_DEVERR]
 * and returns.  counts: device int32[LORA_NUM_COUNTS] (the caller's; a batch's
 * counts work).  The context stays usable afterwards.
 */
lora_status_t lora_selftest_wait(int32_t *counts, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_SGMV_H */
