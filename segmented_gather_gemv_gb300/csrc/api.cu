// api.cu -- the extern "C" boundary of the library: argument checks,
// workspace carving and kernel dispatch.  Declarations and the contract of
// every entry point are in include/lora_sgmv.h.
#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace lora {
cudaError_t launch_prepare(const int32_t *ids, int32_t M, int32_t n, int32_t chunk, int32_t tc_min, bool ascending,
                           int32_t share_grid, char *ws, const WsLayout &L, lora_batch_t *b, cudaStream_t stream);
cudaError_t launch_cc(const DeltaArgs &p, int dtype, int mode, int cluster, int sms, cudaStream_t stream);
int cc_cluster_size(int d_in, int d_out);
cudaError_t launch_tc(const DeltaArgs &p, int mode, int sms, cudaStream_t stream);
bool tc_available();
bool try_launch_small(const DeltaArgs &p, int sms, cudaStream_t stream, cudaError_t *err);
bool try_launch_stream(const DeltaArgs &p, int sms, cudaStream_t stream, cudaError_t *err);
}  // namespace lora

namespace lora {
std::atomic<int64_t> &launch_counter() {
    static std::atomic<int64_t> count{0};
    return count;
}
}  // namespace lora

using namespace lora;

// A wait that cannot end: the barrier expects one arrival that never comes
// and no copy targets it.  The bounded wait gives up, the error bit is set.
__global__ void selftest_wait_kernel(int32_t *counts) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) raise_deverr(counts, LORA_DEVERR_WAIT);
}

// lora_batch_update: for k < n in order, store[rows[k]] = new_ids[k].  The
// warp takes 32 entries at a time; an entry whose row comes again later in
// the same 32 is dropped, so the later entry wins.  The grid before may
// still read the store: the writes wait for it.  The grid after may start at
// once: it reads the ids only after its own wait, which covers this grid.
__global__ void batch_update_kernel(int32_t *__restrict__ store, int32_t M, const int32_t *__restrict__ rows,
                                    const int32_t *__restrict__ new_ids, int32_t n, int32_t *counts) {
    const int lane = threadIdx.x;
    griddep_launch_dependents();
    griddep_wait();
    int bad = 0;
    for (int base = 0; base < n; base += 32) {
        const int k = base + lane;
        const bool valid = k < n;
        const int r = valid ? __ldg(rows + k) : INT_MIN + lane;  // distinct for the lanes past n
        const int v = valid ? __ldg(new_ids + k) : 0;
        const unsigned same = __match_any_sync(0xffffffffu, r);
        const bool later = (same >> lane) > 1u;  // a later lane of this 32 has the same row
        if (valid && !later) {
            if (r >= 0 && r < M) store[r] = v;
            else bad = 1;
        }
        __syncwarp();
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_deverr(counts, LORA_DEVERR_ROW);
}

// Starts the kernels after it at once; launched without programmatic
// serialization, it starts only after the kernel before it has finished.
__global__ void order_kernel() { griddep_launch_dependents(); }

namespace {

thread_local char g_err[512];
thread_local int32_t g_last_kernels = 0;  // LORA_KERNEL_* bits of the last call

lora_status_t fail(lora_status_t code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int dtype) { return dtype == LORA_BF16 ? 2 : 4; }

// Number of SMs of the current device (cached per device).
int sm_count() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cache[dev] = v;
    }
    return cache[dev];
}

// Grid of the tensor-core kernel for a batch of M rows: one CTA per 64 rows,
// at most one per SM, and one SM always left free.  A tensor-core job costs a
// CTA about the same for 8 rows as for 64 (its epilogue works per warp, not
// per row), so a small batch gains nothing from more CTAs and leaves the
// other SMs to the CUDA-core kernel, which then runs beside it.  The free SM
// takes the next prepare in the stream (the tensor-core CTAs fill whole SMs):
// it then runs beside this grid instead of after it.
int tc_grid(int M) {
    const int sms = sm_count() > 1 ? sm_count() - 1 : 1;
    const int g = (M + 63) / 64;
    return g < 1 ? 1 : (g < sms ? g : sms);
}

lora_status_t check_batch(const lora_batch_t *b) {
    if (!b) return fail(LORA_ERR_INVALID, "batch is NULL");
    if (b->magic != kBatchMagic || !b->counts || !b->sorted_token_ids)
        return fail(LORA_ERR_INVALID, "batch was not filled by lora_prepare_batch");
    return LORA_OK;
}

lora_status_t check_dtype_path(int32_t dtype, int32_t path) {
    if (dtype != LORA_F32 && dtype != LORA_BF16) return fail(LORA_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
    if (path != LORA_PATH_AUTO && path != LORA_PATH_CUDA_CORE && path != LORA_PATH_TENSOR)
        return fail(LORA_ERR_INVALID, "unknown path %d", path);
    if (path == LORA_PATH_TENSOR && dtype != LORA_BF16)
        return fail(LORA_ERR_UNSUPPORTED, "the tensor-core path computes bf16 inputs only");
    return LORA_OK;
}

lora_status_t check_rank(int32_t r_max) {
    if (r_max < 1 || r_max > LORA_MAX_RANK) return fail(LORA_ERR_UNSUPPORTED, "r_max %d outside [1, %d]", r_max, LORA_MAX_RANK);
    return LORA_OK;
}

lora_status_t check_x_a(const lora_batch_t *b, int32_t dtype, const void *x, int64_t ldx, int32_t d_in,
                        const void *A, int64_t sa, int64_t sr, int32_t r_max) {
    const int es = elem_size(dtype), V = 16 / es;
    if (d_in < 1 || d_in % V) return fail(LORA_ERR_UNSUPPORTED, "d_in %d must be a positive multiple of %d", d_in, V);
    if (b->M > 0 && (!x || !A)) return fail(LORA_ERR_INVALID, "x or A_pool is NULL");
    if (!aligned16(x) || !aligned16(A)) return fail(LORA_ERR_UNSUPPORTED, "x and A_pool must be 16-byte aligned");
    if (ldx < d_in || (ldx * es) % 16) return fail(LORA_ERR_UNSUPPORTED, "ldx %lld invalid", (long long)ldx);
    if (sr < d_in || (sr * es) % 16) return fail(LORA_ERR_UNSUPPORTED, "a_stride_r %lld invalid", (long long)sr);
    if (sa < (int64_t)r_max * sr || (sa * es) % 16)
        return fail(LORA_ERR_UNSUPPORTED, "a_stride_adapter %lld invalid", (long long)sa);
    return LORA_OK;
}

lora_status_t check_slices(const lora_batch_t *b, int32_t dtype, const lora_b_slice_t *slices, int32_t n_slices,
                           int32_t r_max, const void *y, int64_t ldy, DeltaArgs &p) {
    const int es = elem_size(dtype), V = 16 / es;
    if (!slices || n_slices < 1 || n_slices > LORA_MAX_SLICES)
        return fail(LORA_ERR_INVALID, "n_slices %d outside [1, %d] or slices NULL", n_slices, LORA_MAX_SLICES);
    if (b->M > 0 && !y) return fail(LORA_ERR_INVALID, "y is NULL");
    if (!aligned16(y) || ldy < 1 || (ldy * es) % 16) return fail(LORA_ERR_UNSUPPORTED, "y alignment or ldy invalid");
    int col = 0;
    for (int t = 0; t < n_slices; ++t) {
        const lora_b_slice_t &s = slices[t];
        if (b->M > 0 && !s.B_pool) return fail(LORA_ERR_INVALID, "slice %d: B_pool is NULL", t);
        if (!aligned16(s.B_pool)) return fail(LORA_ERR_UNSUPPORTED, "slice %d: B_pool not 16-byte aligned", t);
        if (s.d_out < 1 || s.d_out % V) return fail(LORA_ERR_UNSUPPORTED, "slice %d: d_out %d not a multiple of %d", t, s.d_out, V);
        const bool rank_major = s.stride_r > 1;
        if (t > 0 && rank_major != (p.b_rank_major != 0))
            return fail(LORA_ERR_UNSUPPORTED, "slices %d and 0 have different B layouts", t);
        p.b_rank_major = rank_major ? 1 : 0;
        if (rank_major) {
            if (s.stride_n != 1 || s.stride_r < s.d_out || (s.stride_r * es) % 16)
                return fail(LORA_ERR_UNSUPPORTED, "slice %d: rank-major B needs stride_n 1 and stride_r >= d_out", t);
            if (s.stride_adapter < (int64_t)r_max * s.stride_r || (s.stride_adapter * es) % 16)
                return fail(LORA_ERR_UNSUPPORTED, "slice %d: stride_adapter invalid", t);
        } else {
            if (s.stride_n < r_max || (s.stride_n * es) % 16)
                return fail(LORA_ERR_UNSUPPORTED, "slice %d: stride_n invalid", t);
            if (s.stride_adapter < (int64_t)s.d_out * s.stride_n || (s.stride_adapter * es) % 16)
                return fail(LORA_ERR_UNSUPPORTED, "slice %d: stride_adapter invalid", t);
        }
        if (s.y_col < 0 || s.y_col % V || (int64_t)s.y_col + s.d_out > ldy)
            return fail(LORA_ERR_UNSUPPORTED, "slice %d: y_col %d invalid", t, s.y_col);
        for (int u = 0; u < t; ++u) {
            const lora_b_slice_t &o = slices[u];
            if (s.y_col < o.y_col + o.d_out && o.y_col < s.y_col + s.d_out)
                return fail(LORA_ERR_INVALID, "slices %d and %d write overlapping y columns", u, t);
        }
        p.slices[t].A = s.A_pool;
        p.slices[t].B = s.B_pool;
        p.slices[t].stride_adapter = s.stride_adapter;
        p.slices[t].stride_n = s.stride_n;
        p.slices[t].stride_r = rank_major ? s.stride_r : 1;
        p.slices[t].d_out = s.d_out;
        p.slices[t].y_col = s.y_col;
        p.slices[t].col_begin = col;
        col += s.d_out;
    }
    p.n_slices = n_slices;
    p.d_out_total = col;
    p.y = const_cast<void *>(y);
    p.ldy = ldy;
    return LORA_OK;
}

void fill_batch(const lora_batch_t *b, DeltaArgs &p) {
    p.ids = b->ids;
    p.ids_after_wait = b->ids_store != nullptr && b->ids == b->ids_store ? 1 : 0;
    p.sorted = b->sorted_token_ids;
    p.tc_indptr = b->tc_indptr;
    p.counts = b->counts;
}

// Rebuilds a batch's segment metadata from its ids into its workspace.
// prepare reads the ids before it waits on the grid before it, and an
// update's kernel may be that grid: the ordering kernel (launched without
// programmatic serialization, so it starts once the grid before it has
// finished) goes first.
cudaError_t refresh_metadata(const lora_batch_t *b, cudaStream_t stream) {
    order_kernel<<<1, 32, 0, stream>>>();
    cudaError_t oe = cudaGetLastError();
    if (oe != cudaSuccess) return oe;
    launch_counter().fetch_add(1, std::memory_order_relaxed);
    const WsLayout L = ws_layout(b->M, b->n_adapters, b->chunk_size);
    char *base = reinterpret_cast<char *>(b->seg_records) - L.rec;
    lora_batch_t tmp{};
    const int grid = tc_grid(b->M);
    return launch_prepare(b->ids, b->M, b->n_adapters, b->chunk_size, b->tc_min_rows,
                          b->order == LORA_ORDER_ASCENDING, grid <= kMaxShareGrid ? grid : 0, base, L, &tmp, stream);
}

// Rows one streaming launch groups on chip.
constexpr int kStreamRangeRows = 2048;

// The streaming kernel over a batch of any size: consecutive launches over
// row ranges of at most kStreamRangeRows (ids, x and y offset by the range's
// first row).  Each launch groups its own rows and writes only them, so the
// ranges are independent; an adapter seen by several ranges has its weights
// read once per range.  The kernel's launch geometry only shrinks with the
// rows, so when the first (fullest) range is taken every later one is too;
// when it is declined nothing was launched and this returns false.  Sets
// *n_launched to the launches made.
static bool try_launch_stream_ranges(const DeltaArgs &p, int sms, cudaStream_t stream, cudaError_t *err,
                                     int *n_launched) {
    *n_launched = 0;
    const size_t es = 2;  // bf16
    for (int lo = 0; lo < p.M_rows; lo += kStreamRangeRows) {
        DeltaArgs q = p;
        q.M_rows = std::min(kStreamRangeRows, p.M_rows - lo);
        q.ids = p.ids + lo;
        q.x = static_cast<const char *>(p.x) + (size_t)lo * (size_t)p.ldx * es;
        q.y = static_cast<char *>(p.y) + (size_t)lo * (size_t)p.ldy * es;
        if (!try_launch_stream(q, sms, stream, err)) {
            if (lo == 0) return false;
            *err = cudaErrorNotSupported;  // not reached: a smaller range fits where the first did
            return true;
        }
        if (*err != cudaSuccess) return true;
        ++*n_launched;
    }
    return true;
}

// Launches the kernels of one call according to the path.
lora_status_t dispatch_one(const lora_batch_t *b, int32_t dtype, int mode, int32_t path, int d_in, DeltaArgs &p,
                           cudaStream_t stream) {
    g_last_kernels = 0;
    fill_batch(b, p);
    if (b->M == 0) return LORA_OK;
    const int sms = sm_count();
    const int cluster = cc_cluster_size(mode == kExpand ? 1 : d_in, p.d_out_total ? p.d_out_total : 1);
    cudaError_t e = cudaSuccess;
    const bool tensor_ok = dtype == LORA_BF16 && tc_available();
    p.desc = reinterpret_cast<const SegDesc *>(b->seg_records);
    p.max_list = b->max_segs;
    p.M_rows = b->M;
    p.n_adapters = b->n_adapters;
    // Batches of up to a few thousand rows: kernels that group the rows
    // themselves from the ids, so nothing on their path waits for prepare's
    // metadata.  Up to kSmallAutoRows rows (a decode step): the single-pass
    // small-batch kernel.  Larger ones: the streaming kernel, which keeps
    // every SM busy however the rows fall into groups (on a mixed serving
    // step of 2048 rows it takes 59 us alone against 110 us beside a
    // tensor-core grid of one CTA per 64 rows that takes the long groups).
    // With kStreamSplitTc set, LORA_PATH_AUTO gives the long groups to the
    // tensor-core kernel instead.
    if (p.b_rank_major) {
        // rank-major B pools: the streaming kernel only (batches above its
        // row limit as consecutive launches over row ranges)
        int n_launched = 0;
        if (mode == kFused && dtype == LORA_BF16 && (path == LORA_PATH_AUTO || path == LORA_PATH_CUDA_CORE) &&
            try_launch_stream_ranges(p, sms, stream, &e, &n_launched)) {
            launch_counter().fetch_add(n_launched, std::memory_order_relaxed);
            if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
            g_last_kernels = LORA_KERNEL_STREAM;
            return LORA_OK;
        }
        return fail(LORA_ERR_UNSUPPORTED,
                    "rank-major B pools run on the streaming kernel only (bf16 lora_delta, r_max 16, 32 or 64)");
    }
    if (mode == kFused && dtype == LORA_BF16 && (path == LORA_PATH_AUTO || path == LORA_PATH_CUDA_CORE)) {
        if (b->M <= kSmallAutoRows) {
            if (try_launch_small(p, sms, stream, &e)) {
                if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
                launch_counter().fetch_add(1, std::memory_order_relaxed);
                g_last_kernels = LORA_KERNEL_SMALL;
                return LORA_OK;
            }
        }
        const bool split = kStreamSplitTc && path == LORA_PATH_AUTO && tensor_ok && b->M > kSmallAutoRows &&
                           b->M >= b->tc_min_rows;
        const int g = split ? tc_grid(b->M) : 0;
        DeltaArgs ps = p;
        ps.split_tc = split ? 1 : 0;
        ps.max_len = split ? b->tc_min_rows : 0x7fffffff;
        ps.trigger_after_wait = split ? 1 : 0;
        if (try_launch_stream(ps, sms - g, stream, &e)) {
            if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
            launch_counter().fetch_add(1, std::memory_order_relaxed);
            g_last_kernels = LORA_KERNEL_STREAM;
            if (split) {
                // after the streaming grid's wait on prepare: the metadata is
                // final; waits for that grid before it exits
                DeltaArgs q = p;
                q.after_cc = 1;
                q.tc_ptr = b->tc_indptr;
                q.tc_start = b->tc_segs;
                q.tc_adapter = b->tc_segs + 2;
                q.tc_rec_stride = 4;
                q.tc_count_index = LORA_COUNT_TC_SEGS;
                q.tc_rows_index = LORA_COUNT_TC_ROWS;
                q.tc_only = 0;
                q.tc_share = share_table(b->counts);
                q.tc_share_grid = g <= kMaxShareGrid ? g : -1;
                e = launch_tc(q, mode, g, stream);
                if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
                launch_counter().fetch_add(1, std::memory_order_relaxed);
                g_last_kernels |= LORA_KERNEL_TENSOR;
            }
            return LORA_OK;
        }
    }
    if (b->stale) {
        // the ids changed since the metadata was built (lora_batch_update):
        // rebuild it for the kernels below
        e = refresh_metadata(b, stream);
        if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "prepare launch failed: %s", cudaGetErrorString(e));
        launch_counter().fetch_add(1, std::memory_order_relaxed);
        g_last_kernels |= LORA_KERNEL_PREPARE;
    }
    if (path == LORA_PATH_TENSOR) {
        if (!tensor_ok) return fail(LORA_ERR_UNSUPPORTED, "the tensor-core path computes bf16 only");
        if (p.r_max > kTcMaxRankCommon && !p.ranks)
            return fail(LORA_ERR_UNSUPPORTED, "the tensor-core path takes ranks up to %d", kTcMaxRankCommon);
        // every segment: the row space is the sorted rows themselves
        p.tc_ptr = b->seg_indptr;
        p.tc_start = b->seg_indptr;
        p.tc_adapter = b->weight_indices;
        p.tc_rec_stride = 1;
        p.tc_count_index = LORA_COUNT_SEGS;
        p.tc_rows_index = LORA_COUNT_ACTIVE;
        p.tc_only = 1;
        const int g = tc_grid(b->M);
        // prepare's shares, which the kernel takes when every segment is on
        // the tensor-core list
        p.tc_share = share_table(b->counts);
        p.tc_share_grid = g <= kMaxShareGrid ? g : -1;
        e = launch_tc(p, mode, g, stream);
        if (e == cudaSuccess) {
            launch_counter().fetch_add(1, std::memory_order_relaxed);
            g_last_kernels |= LORA_KERNEL_TENSOR;
        }
    } else {
        const bool split = path == LORA_PATH_AUTO && tensor_ok;
        p.min_len = 0;
        p.max_len = split ? b->tc_min_rows : 0x7fffffff;
        p.split_tc = split ? 1 : 0;
        // every adapter at a rank the tensor cores take: the CUDA-core
        // kernel's segments are prepare's small-segment list
        p.small_list = split && !p.ranks && tc_rank_ok(p.r_max) ? reinterpret_cast<const int4 *>(b->small_segs)
                                                                 : nullptr;
        // The two kernels write disjoint rows of y and run side by side.  The
        // CUDA-core kernel starts first: it waits on prepare, then lets the
        // tensor-core grid launch, which starts at once and waits for it only
        // before it exits (so that its completion implies the CUDA-core
        // kernel's).  With the tensor-core grid launched first, the CUDA-core
        // CTAs (and behind them the next prepare) found no free SM until the
        // tensor-core CTAs left: on a prefill step of 9962 rows, 84 us per
        // step against 68 us in this order.
        const bool with_tc = split && b->M >= b->tc_min_rows;
        const int g = with_tc ? tc_grid(b->M) : 0;
        // beside a tensor-core grid: the SMs that grid and the next prepare leave
        e = launch_cc(p, dtype, mode, cluster, with_tc ? sms - g - 1 : sms, stream);
        if (e == cudaSuccess) {
            launch_counter().fetch_add(1, std::memory_order_relaxed);
            g_last_kernels |= LORA_KERNEL_CUDA_CORE;
        }
        if (with_tc && e == cudaSuccess) {
            DeltaArgs q = p;
            q.after_cc = 1;
            q.tc_ptr = b->tc_indptr;
            q.tc_start = b->tc_segs;
            q.tc_adapter = b->tc_segs + 2;
            q.tc_rec_stride = 4;
            q.tc_count_index = LORA_COUNT_TC_SEGS;
            q.tc_rows_index = LORA_COUNT_TC_ROWS;
            q.tc_only = 0;
            q.tc_share = share_table(b->counts);
            q.tc_share_grid = g <= kMaxShareGrid ? g : -1;
            e = launch_tc(q, mode, g, stream);
            if (e == cudaSuccess) {
                launch_counter().fetch_add(1, std::memory_order_relaxed);
                g_last_kernels |= LORA_KERNEL_TENSOR;
            }
        }
    }
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return LORA_OK;
}

// A fused call whose slices have their own A pools: the streaming kernel
// stacks the slices' rank blocks into one shrink where they fit (at most 64
// stacked ranks); otherwise every slice runs as a call of its own.
lora_status_t dispatch(const lora_batch_t *b, int32_t dtype, int mode, int32_t path, int d_in, DeltaArgs &p,
                       cudaStream_t stream) {
    bool per_slice_a = false;
    for (int t = 0; t < p.n_slices; ++t) {
        if (!p.slices[t].A) p.slices[t].A = p.A;
        if (p.slices[t].A != p.A) per_slice_a = true;
    }
    if (!per_slice_a || mode != kFused) return dispatch_one(b, dtype, mode, path, d_in, p, stream);
    const int rs = p.r_max <= 16 ? 16 : (p.r_max <= 32 ? 32 : 64);
    if (dtype == LORA_BF16 && (path == LORA_PATH_AUTO || path == LORA_PATH_CUDA_CORE) && p.n_slices * rs <= 64 &&
        (p.r_max == 16 || p.r_max == 32 || p.r_max == 64) && b->M > 0) {
        g_last_kernels = 0;
        fill_batch(b, p);
        p.desc = reinterpret_cast<const SegDesc *>(b->seg_records);
        p.max_list = b->max_segs;
        p.M_rows = b->M;
        p.n_adapters = b->n_adapters;
        p.stacked = 1;
        p.max_len = 0x7fffffff;
        cudaError_t e = cudaSuccess;
        // rank-major pools run on the streaming kernel alone, so a larger
        // batch takes it over row ranges (one stacked shrink per range)
        // rather than one pass per slice
        int n_launched = 0;
        bool taken;
        if (p.b_rank_major) {
            taken = try_launch_stream_ranges(p, sm_count(), stream, &e, &n_launched);
        } else {
            taken = try_launch_stream(p, sm_count(), stream, &e);
            n_launched = taken && e == cudaSuccess ? 1 : 0;
        }
        if (taken) {
            launch_counter().fetch_add(n_launched, std::memory_order_relaxed);
            if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
            g_last_kernels = LORA_KERNEL_STREAM;
            return LORA_OK;
        }
        p.stacked = 0;
    }
    int32_t bits = 0;
    for (int t = 0; t < p.n_slices; ++t) {
        DeltaArgs q = p;
        q.A = p.slices[t].A;
        q.slices[0] = p.slices[t];
        q.slices[0].col_begin = 0;
        q.n_slices = 1;
        q.d_out_total = p.slices[t].d_out;
        const lora_status_t st = dispatch_one(b, dtype, mode, path, d_in, q, stream);
        if (st != LORA_OK) return st;
        bits |= g_last_kernels;
    }
    g_last_kernels = bits;
    return LORA_OK;
}

}  // namespace

extern "C" {

size_t lora_workspace_size(int32_t M, int32_t n_adapters, int32_t chunk_size) {
    if (M < 0 || M > LORA_MAX_TOKENS || n_adapters < 1 || chunk_size < 0) return 0;
    return ws_layout(M, n_adapters, chunk_size).total;
}

lora_status_t lora_prepare_batch(const int32_t *ids, int32_t M, int32_t n_adapters, int32_t chunk_size,
                                 int32_t tc_min_rows, void *workspace, size_t workspace_bytes,
                                 lora_batch_t *batch, void *stream) {
    return lora_prepare_batch_ordered(ids, M, n_adapters, chunk_size, tc_min_rows, LORA_ORDER_FIRST_APPEARANCE,
                                      workspace, workspace_bytes, batch, stream);
}

lora_status_t lora_prepare_batch_ordered(const int32_t *ids, int32_t M, int32_t n_adapters, int32_t chunk_size,
                                         int32_t tc_min_rows, int32_t order, void *workspace,
                                         size_t workspace_bytes, lora_batch_t *batch, void *stream) {
    g_err[0] = 0;
    g_last_kernels = 0;
    if (order != LORA_ORDER_FIRST_APPEARANCE && order != LORA_ORDER_ASCENDING)
        return fail(LORA_ERR_INVALID, "order %d is not a LORA_ORDER_* value", order);
    if (!batch) return fail(LORA_ERR_INVALID, "batch is NULL");
    if (M < 0 || M > LORA_MAX_TOKENS) return fail(LORA_ERR_INVALID, "M %d outside [0, %d]", M, LORA_MAX_TOKENS);
    if (n_adapters < 1) return fail(LORA_ERR_INVALID, "n_adapters %d < 1", n_adapters);
    if (chunk_size < 0) return fail(LORA_ERR_INVALID, "chunk_size %d < 0", chunk_size);
    if (M > 0 && !ids) return fail(LORA_ERR_INVALID, "ids is NULL");
    if (!workspace) return fail(LORA_ERR_INVALID, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(LORA_ERR_UNSUPPORTED, "workspace not 256-byte aligned");
    const WsLayout L = ws_layout(M, n_adapters, chunk_size);
    if (workspace_bytes < L.total)
        return fail(LORA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, L.total);
    const int32_t tc_min = tc_min_rows > 0 ? tc_min_rows : kDefaultTcMinRows;
    lora_batch_t b{};
    const int grid = tc_grid(M);
    cudaError_t e = launch_prepare(ids, M, n_adapters, chunk_size, tc_min, order == LORA_ORDER_ASCENDING,
                                   grid <= kMaxShareGrid ? grid : 0,
                                   static_cast<char *>(workspace), L, &b,
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "prepare launch failed: %s", cudaGetErrorString(e));
    launch_counter().fetch_add(1, std::memory_order_relaxed);
    g_last_kernels = LORA_KERNEL_PREPARE;
    b.M = M;
    b.n_adapters = n_adapters;
    b.chunk_size = chunk_size;
    b.max_segs = L.max_segs;
    b.tc_min_rows = tc_min;
    b.magic = kBatchMagic;
    b.ids = ids;
    b.ids_store = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + L.ids_store);
    b.order = order;
    b.stale = 0;
    *batch = b;
    return LORA_OK;
}

lora_status_t lora_batch_update(lora_batch_t *batch, const int32_t *rows, const int32_t *new_ids, int32_t n,
                                void *stream) {
    g_err[0] = 0;
    g_last_kernels = 0;
    lora_status_t st;
    if ((st = check_batch(batch))) return st;
    if (n < 0) return fail(LORA_ERR_INVALID, "n %d < 0", n);
    if (n > 0 && (!rows || !new_ids)) return fail(LORA_ERR_INVALID, "rows or new_ids is NULL");
    if (n == 0 || batch->M == 0) return LORA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (batch->ids != batch->ids_store)
        e = cudaMemcpyAsync(batch->ids_store, batch->ids, (size_t)batch->M * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(32);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, batch_update_kernel, batch->ids_store, batch->M, rows, new_ids, n,
                               batch->counts);
    }
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "update launch failed: %s", cudaGetErrorString(e));
    launch_counter().fetch_add(1, std::memory_order_relaxed);
    batch->ids = batch->ids_store;
    batch->stale = 1;
    return LORA_OK;
}

lora_status_t lora_batch_refresh(lora_batch_t *batch, void *stream) {
    g_err[0] = 0;
    g_last_kernels = 0;
    lora_status_t st;
    if ((st = check_batch(batch))) return st;
    if (!batch->stale) return LORA_OK;
    const cudaError_t e = refresh_metadata(batch, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "prepare launch failed: %s", cudaGetErrorString(e));
    launch_counter().fetch_add(1, std::memory_order_relaxed);
    g_last_kernels = LORA_KERNEL_PREPARE;
    batch->stale = 0;
    return LORA_OK;
}

lora_status_t lora_shrink(const lora_batch_t *batch, int32_t dtype, const void *x, int64_t ldx, int32_t d_in,
                          const void *A_pool, int64_t a_stride_adapter, int64_t a_stride_r, int32_t r_max,
                          const int32_t *ranks, float *h, int64_t ldh, int32_t path, void *stream) {
    g_err[0] = 0;
    lora_status_t st;
    if ((st = check_batch(batch)) || (st = check_dtype_path(dtype, path)) || (st = check_rank(r_max))) return st;
    if ((st = check_x_a(batch, dtype, x, ldx, d_in, A_pool, a_stride_adapter, a_stride_r, r_max))) return st;
    if (batch->M > 0 && !h) return fail(LORA_ERR_INVALID, "h is NULL");
    if (ldh < r_max) return fail(LORA_ERR_INVALID, "ldh %lld < r_max", (long long)ldh);
    DeltaArgs p{};
    p.x = x;
    p.ldx = ldx;
    p.d_in = d_in;
    p.A = A_pool;
    p.a_stride_adapter = a_stride_adapter;
    p.a_stride_r = a_stride_r;
    p.r_max = r_max;
    p.ranks = ranks;
    p.scale = 1.f;
    p.h = h;
    p.ldh = ldh;
    p.n_slices = 0;
    p.d_out_total = 0;
    return dispatch(batch, dtype, kShrink, path, d_in, p, static_cast<cudaStream_t>(stream));
}

lora_status_t lora_expand(const lora_batch_t *batch, int32_t dtype, const float *h, int64_t ldh, int32_t r_max,
                          const lora_b_slice_t *slices, int32_t n_slices, const int32_t *ranks, float scale,
                          const float *adapter_scale, void *y, int64_t ldy, int32_t path, void *stream) {
    g_err[0] = 0;
    lora_status_t st;
    if ((st = check_batch(batch)) || (st = check_dtype_path(dtype, path)) || (st = check_rank(r_max))) return st;
    if (batch->M > 0 && !h) return fail(LORA_ERR_INVALID, "h is NULL");
    if (ldh < r_max) return fail(LORA_ERR_INVALID, "ldh %lld < r_max", (long long)ldh);
    DeltaArgs p{};
    if ((st = check_slices(batch, dtype, slices, n_slices, r_max, y, ldy, p))) return st;
    p.r_max = r_max;
    p.ranks = ranks;
    p.scale = scale;
    p.adapter_scale = adapter_scale;
    p.h = const_cast<float *>(h);
    p.ldh = ldh;
    return dispatch(batch, dtype, kExpand, path, 0, p, static_cast<cudaStream_t>(stream));
}

lora_status_t lora_delta(const lora_batch_t *batch, int32_t dtype, const void *x, int64_t ldx, int32_t d_in,
                         const void *A_pool, int64_t a_stride_adapter, int64_t a_stride_r, int32_t r_max,
                         const lora_b_slice_t *slices, int32_t n_slices, const int32_t *ranks, float scale,
                         const float *adapter_scale, void *y, int64_t ldy, int32_t path, void *stream) {
    g_err[0] = 0;
    lora_status_t st;
    if ((st = check_batch(batch)) || (st = check_dtype_path(dtype, path)) || (st = check_rank(r_max))) return st;
    if ((st = check_x_a(batch, dtype, x, ldx, d_in, A_pool, a_stride_adapter, a_stride_r, r_max))) return st;
    DeltaArgs p{};
    if ((st = check_slices(batch, dtype, slices, n_slices, r_max, y, ldy, p))) return st;
    for (int t = 0; t < n_slices; ++t)
        if (!aligned16(slices[t].A_pool)) return fail(LORA_ERR_UNSUPPORTED, "slice %d: A_pool not 16-byte aligned", t);
    p.x = x;
    p.ldx = ldx;
    p.d_in = d_in;
    p.A = A_pool;
    p.a_stride_adapter = a_stride_adapter;
    p.a_stride_r = a_stride_r;
    p.r_max = r_max;
    p.ranks = ranks;
    p.scale = scale;
    p.adapter_scale = adapter_scale;
    return dispatch(batch, dtype, kFused, path, d_in, p, static_cast<cudaStream_t>(stream));
}

const char *lora_last_error_string(void) { return g_err; }

int32_t lora_abi_version(void) { return 200; }

int64_t lora_launch_count(void) { return launch_counter().load(std::memory_order_relaxed); }

int32_t lora_last_kernels(void) { return g_last_kernels; }

lora_status_t lora_selftest_wait(int32_t *counts, void *stream) {
    g_err[0] = 0;
    g_last_kernels = 0;
    if (!counts) return fail(LORA_ERR_INVALID, "counts is NULL");
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(counts);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "self-test launch failed: %s", cudaGetErrorString(e));
    return LORA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// lora_prepare_batch_static: the workspace is a device array of this library.
// ---------------------------------------------------------------------------
// One copy per GPU that loads the library, alive until the process exits;
// every call on a device shares it.  In host code the name stands for the
// symbol only: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_workspace[LORA_STATIC_WORKSPACE_BYTES];

namespace {

std::mutex g_static_mu;
void *g_static_addr[64];  // device address of g_static_workspace, per device

// Device address of the array on the current device, looked up once per
// device (the first call on a device, which should precede any capture).
lora_status_t static_workspace(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(LORA_ERR_UNSUPPORTED, "device %d: at most 64 devices", dev);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_workspace);
        if (e != cudaSuccess || !ptr)
            return fail(LORA_ERR_CUDA, "cudaGetSymbolAddress of the static workspace failed: %s",
                        cudaGetErrorString(e));
        g_static_addr[dev] = ptr;
    }
    *out = g_static_addr[dev];
    return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_prepare_batch_static(const int32_t *ids, int32_t M, int32_t n_adapters,
                                                   int32_t chunk_size, int32_t tc_min_rows, lora_batch_t *batch,
                                                   void *stream) {
    g_err[0] = 0;
    if (M < 0 || M > LORA_MAX_TOKENS || n_adapters < 1 || chunk_size < 0)
        return fail(LORA_ERR_INVALID, "M %d, n_adapters %d or chunk_size %d out of range", M, n_adapters, chunk_size);
    const size_t need = ws_layout(M, n_adapters, chunk_size).total;
    if (need > LORA_STATIC_WORKSPACE_BYTES)
        return fail(LORA_ERR_WORKSPACE,
                    "batch needs %zu workspace bytes; the static workspace holds %u (LORA_STATIC_WORKSPACE_BYTES)",
                    need, (unsigned)LORA_STATIC_WORKSPACE_BYTES);
    void *ws = nullptr;
    const lora_status_t st = static_workspace(&ws);
    if (st != LORA_OK) return st;
    return lora_prepare_batch(ids, M, n_adapters, chunk_size, tc_min_rows, ws, LORA_STATIC_WORKSPACE_BYTES, batch,
                              stream);
}
