// common.cuh -- shared definitions of the sm_103a multi-LoRA delta kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/lora_sgmv.h"

namespace lora {

// ---------------------------------------------------------------------------
// Workspace layout of a prepared batch.  Every array starts on a 256-byte
// boundary so that the device arrays are aligned for vector access.
// ---------------------------------------------------------------------------
// Largest tensor-core grid whose CTA shares prepare computes in advance.
constexpr int kMaxShareGrid = 1024;

struct WsLayout {
    size_t sorted, indptr, lens, widx, rec, small, tc, tcptr, counts;
    size_t shares;                                   // right after counts: [kMaxShareGrid + 1] int2
    size_t first_pos, adapter_cnt, adapter_group;   // per adapter [n]
    size_t group_adapter, group_row, group_seg;      // per group [g_max]
    size_t warp_hist;                                // [32][g_max]
    size_t ids_store;                                // [M]: the batch's own copy of the ids
    size_t total;
    int32_t max_segs, g_max;
};

static inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

static inline int64_t max_segments(int64_t M, int64_t n, int64_t chunk) {
    int64_t g = M < n ? M : n;              // distinct groups
    if (chunk <= 0) return g;
    int64_t s = M / chunk + g;              // sum ceil(L_g / C) <= M / C + G
    return s < M ? s : M;                   // and never more than the rows
}

// The share table of a batch, from its counts pointer (ws_layout puts it
// right after the counts).
static inline const int2 *share_table(const int32_t *counts) {
    return reinterpret_cast<const int2 *>(reinterpret_cast<const char *>(counts) + align256(LORA_NUM_COUNTS * 4));
}

// prepare's outputs (descriptors, small and tensor-core lists, indptr,
// lengths, adapters, tensor-core indptr, sorted rows) lie in one block whose
// byte layout is the same in the workspace and in prepare's shared-memory
// staging, so that the staged outputs leave in one contiguous copy.
struct OutLayout {
    size_t rec, small, tc, indptr, lens, widx, tcptr, sorted, total;  // bytes, multiples of 16
};
__host__ __device__ inline OutLayout out_layout(int64_t ms, int64_t M) {
    OutLayout O{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += (bytes + 15) & ~size_t(15); return at; };
    O.rec = take((size_t)ms * 128);
    O.small = take((size_t)ms * 16);
    O.tc = take((size_t)ms * 16);
    O.indptr = take(((size_t)ms + 1) * 4);
    O.lens = take((size_t)ms * 4);
    O.widx = take((size_t)ms * 4);
    O.tcptr = take(((size_t)ms + 1) * 4);
    O.sorted = take((M > 0 ? (size_t)M : 1) * 4);
    O.total = o;
    return O;
}

static inline WsLayout ws_layout(int32_t M, int32_t n, int32_t chunk) {
    WsLayout L{};
    int64_t ms = max_segments(M, n, chunk);
    int64_t gm = M < n ? M : n;
    if (ms < 1) ms = 1;
    if (gm < 1) gm = 1;
    L.max_segs = (int32_t)ms;
    L.g_max = (int32_t)gm;
    const OutLayout O = out_layout(ms, M);
    L.rec = O.rec;
    L.small = O.small;
    L.tc = O.tc;
    L.indptr = O.indptr;
    L.lens = O.lens;
    L.widx = O.widx;
    L.tcptr = O.tcptr;
    L.sorted = O.sorted;
    size_t o = align256(O.total);
    auto take = [&](size_t ints) { size_t at = o; o = align256(o + ints * 4); return at; };
    L.counts = take(LORA_NUM_COUNTS);
    L.shares = take(2 * ((size_t)kMaxShareGrid + 1));
    L.first_pos = take((size_t)n);
    L.adapter_cnt = take((size_t)n);
    L.adapter_group = take((size_t)n);
    L.group_adapter = take((size_t)gm);
    L.group_row = take((size_t)gm + 1);
    L.group_seg = take((size_t)gm + 1);
    L.warp_hist = take((size_t)gm * 32);
    L.ids_store = take(M > 0 ? (size_t)M : 1);
    L.total = o;
    return L;
}

// Runs a set-up step once per device (kernel attributes are per device).
struct DeviceOnce {
    static constexpr int kMaxDevices = 64;
    volatile bool done[kMaxDevices] = {};
    template <typename F>
    cudaError_t run(F &&f) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (done[dev]) return cudaSuccess;
        e = f();
        if (e == cudaSuccess) done[dev] = true;
        return e;
    }
};

// Process-wide count of kernel launches made by the library.
std::atomic<int64_t> &launch_counter();

constexpr uint32_t kBatchMagic = 0x4C6F5241u;  // "LoRA"
// Adapter groups of at least this many rows go to the tensor-core kernel
// (measured crossover on GB300: the CUDA-core kernel is ahead for groups of
// up to 24 rows, the tensor-core kernel from 32).
constexpr int kDefaultTcMinRows = 32;
// Batches of at most this many rows run whole on the single-pass small-batch
// kernel under LORA_PATH_AUTO; larger ones that the streaming kernel takes
// run on it (see the dispatch in api.cu).
constexpr int kSmallAutoRows = 256;
// Whether LORA_PATH_AUTO gives the long groups of a streaming-kernel batch to
// the tensor-core kernel (false: the streaming kernel takes the whole batch).
constexpr bool kStreamSplitTc = false;
constexpr int kTcMaxRankCommon = 32;
// Ranks the tensor-core kernel computes (exact 8-column masking, <= 32).
__host__ __device__ __forceinline__ bool tc_rank_ok(int r) { return r > 0 && r <= kTcMaxRankCommon && (r & 7) == 0; }

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy through the async-copy unit.  `src_bytes`
// (0..16) bytes are read; the rest of the 16 are zero-filled.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Thread-block cluster helpers.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Programmatic dependent launch: let the next grid in the stream start its
// prologue early / wait until the previous grid has completed and its
// memory is visible.  Both are no-ops when the launch did not opt in.
// The delta kernels of this library wait before they trigger; prepare
// triggers at its start (it writes its workspace only after its wait).  So
// a grid that starts early finds complete every grid before the last delta
// kernel ahead of it: at most that delta kernel and a prepare after it are
// still running.  Before its own wait a grid reads only what none of them
// writes: ids, adapter pools, ranks and scales.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Brings a tensor map (a kernel parameter) into the copy unit's descriptor
// cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const void *map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// mbarrier helpers (shared::cta barriers, transaction-count based).
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// One test of phase `parity`; the thread may sleep up to kSuspendNs in it
// until the phase completes (so waiting warps do not keep the shared-memory
// pipe busy with polls while other warps issue copies).
constexpr uint32_t kSuspendNs = 1000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// Longest a kernel waits on one barrier before it gives up, in SM clock
// cycles (about 0.1 s at 2 GHz).  Real waits last microseconds; the limit only
// ends a wait that can no longer complete.  The SM-local cycle counter is
// read every 64 tests.
constexpr long long kWaitLimitCycles = 200ll * 1000 * 1000;
// Bounded wait for phase `parity` of `bar`.  Returns false if the barrier did
// not complete in time (the caller flags an error; it never spins forever).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long deadline = clock64() + kWaitLimitCycles;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (clock64() > deadline) return false;
    }
}
// As mbar_wait, but also gives up as soon as another role of the CTA has
// set `*abort`, and sets it on its own timeout.
__device__ __forceinline__ bool mbar_wait_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long deadline = clock64() + kWaitLimitCycles;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() > deadline) {
            *abort = 1;
            return false;
        }
    }
}

// Bulk (non-tensor) async copy global -> shared, completing on `bar`.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Store to the same shared-memory location in another CTA of the cluster.
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Element helpers: a 16-byte vector holds 8 bf16 or 4 fp32 values.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kVec = 4;
    using PairT = float2;  // two consecutive elements
    __device__ __forceinline__ static float2 pair_to_f32(const float2 &v) { return v; }
    __device__ __forceinline__ static void store_pair(float *p, const float2 &v) {
        *reinterpret_cast<float2 *>(p) = v;
    }
    __device__ __forceinline__ static void to_f32(const uint4 &v, float *o) {
        o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
        o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static float load1(const float *p) { return *p; }
    __device__ __forceinline__ static void store1(float *p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    using PairT = uint32_t;  // two consecutive elements
    __device__ __forceinline__ static float2 pair_to_f32(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
    __device__ __forceinline__ static void store_pair(__nv_bfloat16 *p, const float2 &v) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(v.x, v.y);
    }
    __device__ __forceinline__ static void to_f32(const uint4 &v, float *o) {
        // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32.
        o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
        o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
        o[4] = __uint_as_float(v.z << 16); o[5] = __uint_as_float(v.z & 0xFFFF0000u);
        o[6] = __uint_as_float(v.w << 16); o[7] = __uint_as_float(v.w & 0xFFFF0000u);
    }
    __device__ __forceinline__ static float load1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ __forceinline__ static void store1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
};

// Two consecutive elements of a 16-byte vector as a float2 (word q holds
// elements 2q and 2q+1 for bf16; for fp32 the pair is elements 2q, 2q+1).
template <typename T> __device__ __forceinline__ float2 pair_of(const uint4 &v, int q);
template <> __device__ __forceinline__ float2 pair_of<__nv_bfloat16>(const uint4 &v, int q) {
    const uint32_t w = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <> __device__ __forceinline__ float2 pair_of<float>(const uint4 &v, int q) {
    return q == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
}

__device__ __forceinline__ void raise_deverr(int32_t *counts, int bit) {
    if (counts) atomicOr(reinterpret_cast<unsigned int *>(counts + LORA_COUNT_DEVERR), (unsigned)bit);
}

// ---------------------------------------------------------------------------
// Host-side launch descriptors (internal).
// ---------------------------------------------------------------------------
struct SliceDesc {
    const void *A;  // this slice's A pool (the call's A pool when it has none of its own)
    const void *B;
    int64_t stride_adapter, stride_n, stride_r;  // stride_r 1: rank-contiguous rows; > 1: rank-major
    int32_t d_out, y_col, col_begin;  // col_begin: first column in the concatenated N range
};

// 128-byte segment descriptor written by prepare: header + inline rows.
constexpr int kInlineRows = LORA_DESC_INLINE_ROWS;
struct SegDesc {
    int32_t start, len, adapter, seg;
    int32_t rows[kInlineRows];
};
static_assert(sizeof(SegDesc) == 128, "segment descriptor is 128 bytes");

struct DeltaArgs {
    // batch
    const int32_t *ids;      // the batch's ids (the small-batch kernel groups rows from them)
    const int32_t *sorted;   // sorted_token_ids
    const SegDesc *desc;     // all segment descriptors (len 0 past the last)
    // small-segment list {start, len, adapter, s} (counts[LORA_COUNT_SMALL_SEGS]
    // of them): with it, the CUDA-core kernel walks these segments only
    const int4 *small_list;
    const int32_t *tc_indptr;
    int32_t *counts;
    int32_t max_list;        // host-side capacity of desc / recs
    int32_t min_len, max_len;  // the CUDA-core kernel takes segments with min_len <= len < max_len
    int32_t split_tc;          // 1: segments >= max_len with a tensor-core rank go to the tensor-core kernel
    int32_t after_cc;          // 1: tensor-core kernel launched right after the CUDA-core kernel, which waited on prepare
    int32_t trigger_after_wait;  // small-batch kernel: trigger the next grid only after its own wait
    int32_t stacked;             // streaming kernel: per-slice A pools, their rank blocks stacked in one shrink
    int32_t b_rank_major;        // B pools laid out [n][r][d_out] (streaming kernel only)
    int32_t ids_after_wait;      // small-batch / streaming kernels: the ids may come from the grid
                                 // before (lora_batch_update): read them only after the wait
    // CTA shares of the tensor-core row space computed by prepare for a grid
    // of tc_share_grid CTAs: boundary b = {first row of CTA b, its segment}
    const int2 *tc_share;
    int32_t tc_share_grid;
    int32_t M_rows;            // rows of x and y
    int32_t n_adapters;
    // tensor-core row space: segment i covers rows [tc_ptr[i], tc_ptr[i+1]),
    // starts at sorted position tc_start[i * tc_rec_stride], adapter tc_adapter[...]
    const int32_t *tc_ptr, *tc_start, *tc_adapter;
    int32_t tc_rec_stride, tc_count_index, tc_rows_index, tc_only;
    // operands
    const void *x;
    int64_t ldx;
    int32_t d_in;
    const void *A;
    int64_t a_stride_adapter, a_stride_r;
    int32_t r_max;
    const int32_t *ranks;
    float scale;
    const float *adapter_scale;
    float *h;            // shrink output / expand input (fp32)
    int64_t ldh;
    void *y;
    int64_t ldy;
    int32_t n_slices;
    int32_t d_out_total;
    SliceDesc slices[LORA_MAX_SLICES];
};

enum Mode { kFused = 0, kShrink = 1, kExpand = 2 };

}  // namespace lora
