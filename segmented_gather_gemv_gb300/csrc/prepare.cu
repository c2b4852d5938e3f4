// prepare.cu -- device-side segment metadata for a batch of per-token
// adapter ids ("III.Punica: Multi-Tenant LoRA Serving", section 代码:
// prepare_lora_batch regroups tokens by adapter and can cut the regrouped
// stream into fixed-size chunks; section SGMV: the segment boundary array).
//
// One CTA builds the whole batch; every working array lives in shared
// memory when it fits (the ids, the per-adapter and per-group tables and
// the per-warp histograms), so the phases below cost shared-memory latency,
// not global-memory round trips.  Nothing is read back by the host.
//   1. per adapter: first row it appears in (atomicMin) and its row count;
//      ids outside [-1, n) are counted as invalid.
//   2. group number of each adapter = number of adapters that appear
//      earlier (block scan of "row i is its adapter's first row").
//   3. per group: row base and segment base (block scans of the row count
//      and of ceil(count / chunk)).
//   4. per segment: start, length and adapter (binary search of the
//      segment's group), written as arrays and 16-byte records, and split
//      by the tensor-core row threshold (block scans).
//   5. stable row positions: every warp owns a contiguous range of rows,
//      counts its rows per group (warp match), the per-group counts are
//      scanned across warps, then each warp re-walks its range and places
//      its rows -- rows inside a group keep ascending order.
//   6. counters.
#include <climits>

#include "common.cuh"

namespace lora {

struct PrepArgs {
    const int32_t *ids;
    int32_t M, n, chunk, tc_min, gcap;
    int32_t *sorted, *indptr, *lens, *widx, *counts;
    SegDesc *desc;
    int32_t max_segs;
    int4 *small, *tc;
    int32_t *tcptr;
    // global fall-backs for tables that do not fit in shared memory
    int32_t *first_pos, *acnt, *agroup;
    int32_t *gadapter, *grow, *gseg;
    int32_t *whist;
    // shared-memory placement (byte offsets into dynamic shared memory, -1 = global)
    int32_t off_ids, off_adapters, off_groups, off_hist;
    int32_t off_bits;   // first-appearance bitmap and its word prefix, or -1
    int32_t off_stage;  // shared-memory copy of the output block (phases 4-5), or -1
    void *out_block;    // the workspace's output block (layout out_layout)
    int2 *shares;       // tensor-core CTA shares: boundary b = {first row, segment}, b <= share_grid
    int32_t ascending;  // 1: groups by increasing adapter id, else by first appearance
    int32_t share_grid;
    // small-batch kernel: hash slots, their table and the group table
    int32_t hs, off_hash, off_gtab;
};

// Shares of the tensor-core row space for a grid of `grid` CTAs: boundary b
// (b <= grid) = {first row of CTA b, the segment holding it}; zeros when the
// batch has no such row.  `tcl` / `tcp` are the tensor-core records and their
// row prefix (nseg of them).  The share end e = rows * b / grid moves to the
// boundary between two adapter groups (runs of records of one adapter: the
// chunks of a chunked group) when one lies within half a share, so that a
// tile holds rows of two adapters only where the groups are short.  The
// boundaries come from a table of the groups' first rows (up to
// kShareGroups groups); with more groups each end looks only at the
// boundaries of its own record, which is exact for unchunked batches.
// plan_shares builds the shares in shared memory (every thread of the block
// calls it; it reads only the block's own records, so it may run before the
// wait on the previous grid); store_shares writes them to the workspace.
constexpr int kShareGroups = 256;
struct ShareTable {
    int2 b[kMaxShareGrid + 1];
    int gstart[kShareGroups + 1];  // first row of group g; [ng] = rows
    int ng;                        // groups in gstart, 0 when they do not fit
};

// largest i < n with v[i] <= r (v ascending, v[0] <= r)
__device__ __forceinline__ int last_le(const int32_t *v, int n, int r) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (v[mid] <= r) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ void plan_shares(const int4 *tcl, const int32_t *tcp, int nseg, int rows, int grid, ShareTable &T) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const bool any = nseg > 0 && rows > 0 && grid > 0;
    __syncthreads();  // the records and tcp[nseg] are complete
    if (tid < 32) {
        // the groups' first rows: a group starts at every record whose
        // adapter differs from the one before
        const int lane = tid;
        int ng = 0;
        for (int base = 0; any && base < nseg && ng <= kShareGroups; base += 32) {
            const int i = base + lane;
            const bool head = i < nseg && (i == 0 || tcl[i - 1].z != tcl[i].z);
            const unsigned bal = __ballot_sync(0xffffffffu, head);
            const int k = ng + __popc(bal & ((1u << lane) - 1u));
            if (head && k < kShareGroups) T.gstart[k] = tcp[i];
            ng += __popc(bal);
        }
        if (lane == 0) {
            T.ng = ng <= kShareGroups ? ng : 0;
            if (ng <= kShareGroups) T.gstart[ng] = rows;
        }
    }
    __syncthreads();
    const int half = grid > 0 ? (int)(rows / (2 * (int64_t)grid)) : 0;
    const int ng = T.ng;
    for (int b = tid; grid > 0 && b <= grid; b += nthr) {
        int e = (int)((int64_t)rows * b / grid), sg = 0;
        if (any) {
            if (nseg >= 2 && e > 0 && e < rows) {
                if (ng > 0) {
                    const int g = last_le(T.gstart, ng, e);
                    const int lo = T.gstart[g], hi = T.gstart[g + 1];
                    if (e - lo <= half && g > 0) e = lo;
                    else if (hi - e <= half && g + 1 < ng) e = hi;
                } else {
                    const int i = last_le(tcp, nseg, e);
                    const int lo = tcp[i], hi = tcp[i + 1], a = tcl[i].z;
                    if (e - lo <= half && i > 0 && tcl[i - 1].z != a) e = lo;
                    else if (hi - e <= half && i + 1 < nseg && tcl[i + 1].z != a) e = hi;
                }
            }
            sg = e < rows ? last_le(tcp, nseg, e) : nseg;
        }
        T.b[b] = make_int2(e, sg);
    }
}

// Each thread writes the boundaries it computed in plan_shares.
__device__ __forceinline__ void store_shares(const ShareTable &T, int grid, int2 *shares) {
    for (int b = threadIdx.x; grid > 0 && b <= grid; b += blockDim.x) shares[b] = T.b[b];
}

// Block-wide exclusive scan of one value per thread.  `ws` is shared scratch
// of 33 ints.  All threads must call it.
__device__ __forceinline__ int block_excl_scan(int v, int *total, int *ws) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
    }
    if (lane == 31) ws[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? ws[lane] : 0;
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += t;
        }
        ws[lane] = s - w;
        if (lane == 31) ws[32] = s;
    }
    __syncthreads();
    int res = ws[warp] + x - v;
    *total = ws[32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(1024, 1) prepare_kernel(const __grid_constant__ PrepArgs p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int scan_ws[33];
    __shared__ int s_invalid;
    __shared__ ShareTable s_shares;

    // Phases 1-3 read only the ids and write only shared memory; when every
    // table of theirs is in shared memory they run before the wait on the
    // previous grid, overlapping it (the previous grid of this library
    // writes y, never ids, and everything before it has completed: see
    // griddep_launch_dependents).  The next kernel may start once this grid
    // has waited; it waits for this grid's completion before it reads what
    // this grid writes.
    // The next grid may start at once: every kernel of this library reads
    // what this grid writes only after its own wait (which returns once this
    // grid has completed), and before that wait reads only data that is
    // fixed before this grid starts (ids, adapter pools).
    griddep_launch_dependents();
    const bool early = p.off_adapters >= 0 && p.off_groups >= 0;
    if (!early) griddep_wait();

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const int M = p.M, n = p.n;
    const int G_cap = p.gcap;

    int32_t *first_pos = p.off_adapters >= 0 ? reinterpret_cast<int32_t *>(smem_raw + p.off_adapters) : p.first_pos;
    int32_t *acnt = p.off_adapters >= 0 ? first_pos + n : p.acnt;
    int32_t *agroup = p.off_adapters >= 0 ? first_pos + 2 * n : p.agroup;
    int32_t *gadapter = p.off_groups >= 0 ? reinterpret_cast<int32_t *>(smem_raw + p.off_groups) : p.gadapter;
    int32_t *grow = p.off_groups >= 0 ? gadapter + G_cap : p.grow;
    int32_t *gseg = p.off_groups >= 0 ? grow + G_cap + 1 : p.gseg;
    int32_t *whist = p.off_hist >= 0 ? reinterpret_cast<int32_t *>(smem_raw + p.off_hist) : p.whist;
    const int32_t *ids = p.ids;
    if (p.off_ids >= 0) {
        int32_t *ids_s = reinterpret_cast<int32_t *>(smem_raw + p.off_ids);
        for (int i = tid; i < M; i += nthr) ids_s[i] = p.ids[i];
        ids = ids_s;
    }

    // Phase 1: first appearance and row count per adapter.
    for (int a = tid; a < n; a += nthr) {
        first_pos[a] = INT_MAX;
        acnt[a] = 0;
    }
    if (tid == 0) s_invalid = 0;
    __syncthreads();
    int bad = 0;
    // Each warp walks its own contiguous rows.  A chunk of 32 equal ids (runs,
    // as in prefill batches) only extends the warp's current run, kept in
    // registers and added once when the run ends; mixed chunks elect one lane
    // per adapter.  So warps do not queue on the same shared-memory counter.
    const int per_warp = (M + nwarps - 1) / nwarps;
    const int w0 = min(M, warp * per_warp), w1 = min(M, w0 + per_warp);
    {
        int run_a = -1, run_cnt = 0, run_first = 0;  // the same in every lane
        for (int b = w0; b < w1; b += 32) {
            const int i = b + lane;
            int a = i < w1 ? ids[i] : -1;
            if (i < w1 && a != -1 && (a < 0 || a >= n)) {
                ++bad;
                a = -1;
            }
            const int a0 = __shfl_sync(0xffffffffu, a, 0);
            if (__all_sync(0xffffffffu, a == a0)) {
                if (a0 != run_a) {
                    if (lane == 0 && run_a >= 0) {
                        atomicMin(&first_pos[run_a], run_first);
                        atomicAdd(&acnt[run_a], run_cnt);
                    }
                    run_a = a0;
                    run_first = b;
                    run_cnt = 0;
                }
                run_cnt += 32;
            } else {
                const unsigned peers = __match_any_sync(0xffffffffu, a);
                if (a >= 0 && lane == __ffs(peers) - 1) {
                    atomicMin(&first_pos[a], i);
                    atomicAdd(&acnt[a], __popc(peers));
                }
            }
        }
        if (lane == 0 && run_a >= 0) {
            atomicMin(&first_pos[run_a], run_first);
            atomicAdd(&acnt[run_a], run_cnt);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);
    __syncthreads();

    // Phase 2: group number by order of first appearance (or, on request,
    // by increasing adapter id: the number of present adapters below it).
    int G = 0;
    if (p.ascending) {
        for (int base = 0; base < n; base += nthr) {
            const int a = base + tid;
            const int flag = a < n && acnt[a] > 0 ? 1 : 0;
            int tot;
            const int ex = block_excl_scan(flag, &tot, scan_ws);
            if (flag) {
                agroup[a] = G + ex;
                gadapter[G + ex] = a;
            }
            G += tot;
        }
        __syncthreads();
    } else if (p.off_bits >= 0 && p.off_adapters >= 0) {
        // The group of a present adapter a is the number of present adapters
        // that first appear before it: set one bit per first appearance, then
        // count the bits below first_pos[a] (word prefix sums + popcount).
        uint32_t *bits = reinterpret_cast<uint32_t *>(smem_raw + p.off_bits);
        const int nw = (M + 31) >> 5;
        int32_t *wpre = reinterpret_cast<int32_t *>(bits + nw);
        for (int w = tid; w < nw; w += nthr) bits[w] = 0u;
        __syncthreads();
        for (int a = tid; a < n; a += nthr)
            if (acnt[a] > 0) atomicOr(&bits[first_pos[a] >> 5], 1u << (first_pos[a] & 31));
        __syncthreads();
        int run = 0;
        for (int base = 0; base < nw; base += nthr) {
            const int w = base + tid;
            int tot;
            const int ex = block_excl_scan(w < nw ? __popc(bits[w]) : 0, &tot, scan_ws);
            if (w < nw) wpre[w] = run + ex;
            run += tot;
        }
        G = run;
        __syncthreads();
        for (int a = tid; a < n; a += nthr)
            if (acnt[a] > 0) {
                const int fp = first_pos[a];
                const int rank = wpre[fp >> 5] + __popc(bits[fp >> 5] & ((1u << (fp & 31)) - 1u));
                agroup[a] = rank;
                gadapter[rank] = a;
            }
        __syncthreads();
    } else if (n <= nthr && n <= 512 && p.off_adapters >= 0) {
        // Small pool: the group of adapter a is the number of present
        // adapters that first appear before it (every thread reads the same
        // entries in step, so the shared-memory reads are broadcasts).
        for (int a0 = 0; a0 < n; a0 += nthr) {
            const int a = a0 + tid;
            const int fa = a < n && acnt[a] > 0 ? first_pos[a] : INT_MAX;
            int rank = 0, present = 0;
            for (int b2 = 0; b2 < n; ++b2) {
                const int fb = first_pos[b2];
                rank += fb < fa ? 1 : 0;
                present += fb != INT_MAX ? 1 : 0;
            }
            if (fa != INT_MAX) {
                agroup[a] = rank;
                gadapter[rank] = a;
            }
            G = present;
        }
        __syncthreads();
    } else
    for (int base = 0; base < M; base += nthr) {
        const int i = base + tid;
        const int a = i < M ? ids[i] : -1;
        const int flag = (i < M && a >= 0 && a < n && first_pos[a] == i) ? 1 : 0;
        int tot;
        const int ex = block_excl_scan(flag, &tot, scan_ws);
        if (flag) {
            agroup[a] = G + ex;
            gadapter[G + ex] = a;
        }
        G += tot;
    }
    __syncthreads();

    // Phase 3: row base and segment base of every group.
    int rows_run = 0, segs_run = 0;
    for (int base = 0; base < G; base += nthr) {
        const int g = base + tid;
        int len = 0, ns = 0;
        if (g < G) {
            len = acnt[gadapter[g]];
            ns = p.chunk > 0 ? (len + p.chunk - 1) / p.chunk : 1;
        }
        int tl, tn;
        const int el = block_excl_scan(len, &tl, scan_ws);
        const int en = block_excl_scan(ns, &tn, scan_ws);
        if (g < G) {
            grow[g] = rows_run + el;
            gseg[g] = segs_run + en;
        }
        rows_run += tl;
        segs_run += tn;
    }
    if (tid == 0) {
        grow[G] = rows_run;
        gseg[G] = segs_run;
    }
    __syncthreads();
    const int S = segs_run, ACT = rows_run;

    // Phases 4-5 write their outputs to shared memory too when they fit
    // (staging), so that only the copy to global memory waits on the
    // previous grid.
    const bool stage = early && p.off_stage >= 0 && p.off_hist >= 0;
    SegDesc *o_desc = p.desc;
    int4 *o_small = p.small, *o_tc = p.tc;
    int32_t *o_indptr = p.indptr, *o_lens = p.lens, *o_widx = p.widx, *o_tcptr = p.tcptr, *o_sorted = p.sorted;
    const OutLayout O = out_layout(p.max_segs, p.M);
    if (stage) {
        // the workspace's output block, byte for byte
        unsigned char *b = smem_raw + p.off_stage;
        o_desc = reinterpret_cast<SegDesc *>(b + O.rec);
        o_small = reinterpret_cast<int4 *>(b + O.small);
        o_tc = reinterpret_cast<int4 *>(b + O.tc);
        o_indptr = reinterpret_cast<int32_t *>(b + O.indptr);
        o_lens = reinterpret_cast<int32_t *>(b + O.lens);
        o_widx = reinterpret_cast<int32_t *>(b + O.widx);
        o_tcptr = reinterpret_cast<int32_t *>(b + O.tcptr);
        o_sorted = reinterpret_cast<int32_t *>(b + O.sorted);
    }
    if (early && !stage) griddep_wait();

    // Phase 4: segments, records and the tensor-core split (by group rows).
    int n_small = 0, n_tc = 0, tc_rows = 0;
    for (int base = 0; base < S; base += nthr) {
        const int s = base + tid;
        int seg_start = 0, seg_len = 0, adapter = 0, grp_len = 0;
        if (s < S) {
            int lo = 0, hi = G - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (gseg[mid] <= s) lo = mid;
                else hi = mid - 1;
            }
            const int g = lo, c = s - gseg[g];
            const int start = grow[g], len = grow[g + 1] - start;
            seg_start = start;
            seg_len = len;
            grp_len = len;
            if (p.chunk > 0) {
                seg_start = start + c * p.chunk;
                seg_len = min(p.chunk, len - c * p.chunk);
            }
            adapter = gadapter[g];
            o_indptr[s] = seg_start;
            o_lens[s] = seg_len;
            o_widx[s] = adapter;
        }
        // The split follows the adapter group's rows: the chunks of a long
        // group stay one dense contraction (and the tensor-core kernel joins
        // consecutive chunks of one group into one tile).
        const int is_tc = (s < S && grp_len >= p.tc_min) ? 1 : 0;
        if (s < S)
            *reinterpret_cast<int4 *>(&o_desc[s]) =
                make_int4(seg_start, seg_len, adapter, s | (is_tc ? LORA_DESC_TC_FLAG : 0));
        const int is_small = (s < S && !is_tc) ? 1 : 0;
        int t1, t2, t3;
        const int es = block_excl_scan(is_small, &t1, scan_ws);
        const int et = block_excl_scan(is_tc, &t2, scan_ws);
        const int er = block_excl_scan(is_tc ? seg_len : 0, &t3, scan_ws);
        const int4 rec = make_int4(seg_start, seg_len, adapter, s);
        if (is_small) o_small[n_small + es] = rec;
        if (is_tc) {
            o_tc[n_tc + et] = rec;
            o_tcptr[n_tc + et] = tc_rows + er;
        }
        n_small += t1;
        n_tc += t2;
        tc_rows += t3;
    }
    if (tid == 0) {
        o_indptr[S] = ACT;
        o_tcptr[n_tc] = tc_rows;
    }
    // Descriptors past the last segment end the list (len 0).
    for (int s = S + tid; s < p.max_segs; s += nthr)
        *reinterpret_cast<int4 *>(&o_desc[s]) = make_int4(0, 0, 0, s);

    // Phase 5: stable row positions.
    for (int k = tid; k < nwarps * G; k += nthr) whist[k] = 0;
    __syncthreads();
    int32_t *wh = whist + warp * G;
    // Rows of this warp per group (the same contiguous rows as phase 1); a
    // run of 32 equal groups is counted in registers.
    {
        int run_g = -1, run_c = 0;
        for (int b = w0; b < w1; b += 32) {
            const int i = b + lane;
            int g = -1;
            if (i < w1) {
                const int a = ids[i];
                if (a >= 0 && a < n) g = agroup[a];
            }
            const int g0 = __shfl_sync(0xffffffffu, g, 0);
            if (__all_sync(0xffffffffu, g == g0)) {
                if (g0 != run_g) {
                    if (lane == 0 && run_g >= 0) wh[run_g] += run_c;
                    __syncwarp();
                    run_g = g0;
                    run_c = 0;
                }
                run_c += 32;
            } else {
                const unsigned peers = __match_any_sync(0xffffffffu, g);
                if (g >= 0 && lane == __ffs(peers) - 1) wh[g] += __popc(peers);
                __syncwarp();
            }
        }
        if (lane == 0 && run_g >= 0) wh[run_g] += run_c;
    }
    __syncthreads();
    for (int g = tid; g < G; g += nthr) {
        int run = grow[g];
        for (int w = 0; w < nwarps; ++w) {
            const int t = whist[w * G + g];
            whist[w * G + g] = run;
            run += t;
        }
    }
    __syncthreads();
    // Positions: the warp's next free slot of each group, in registers for
    // the current run.
    auto place_row = [&](int i, int g, int pos) {
        o_sorted[pos] = i;
        // first rows of every segment, inline in its descriptor
        const int off = pos - grow[g];
        const int s = gseg[g] + (p.chunk > 0 ? off / p.chunk : 0);
        const int k = p.chunk > 0 ? off - (off / p.chunk) * p.chunk : off;
        if (k < kInlineRows) o_desc[s].rows[k] = i;
    };
    {
        int run_g = -1, run_next = 0;
        for (int b = w0; b < w1; b += 32) {
            const int i = b + lane;
            int g = -1;
            if (i < w1) {
                const int a = ids[i];
                if (a >= 0 && a < n) g = agroup[a];
            }
            const int g0 = __shfl_sync(0xffffffffu, g, 0);
            const bool uniform = __all_sync(0xffffffffu, g == g0);
            if (uniform && g0 >= 0) {
                if (g0 != run_g) {
                    if (lane == 0 && run_g >= 0) wh[run_g] = run_next;
                    __syncwarp();
                    run_g = g0;
                    run_next = wh[g0];
                    __syncwarp();
                }
                place_row(i, g0, run_next + lane);
                run_next += 32;
            } else if (!uniform) {
                if (run_g >= 0) {
                    if (lane == 0) wh[run_g] = run_next;
                    run_g = -1;
                }
                __syncwarp();
                const unsigned peers = __match_any_sync(0xffffffffu, g);
                const int base_pos = g >= 0 ? wh[g] : 0;
                __syncwarp();
                if (g >= 0) {
                    place_row(i, g, base_pos + __popc(peers & ((1u << lane) - 1u)));
                    if (lane == __ffs(peers) - 1) wh[g] = base_pos + __popc(peers);
                }
                __syncwarp();
            }
        }
    }

    plan_shares(o_tc, o_tcptr, n_tc, tc_rows, p.share_grid, s_shares);
    if (stage) {
        // copy the staged outputs (descriptors as 16-byte pieces)
        __syncthreads();
        griddep_wait();
        // one contiguous copy of the output block (entries past each
        // array's valid length go along unread)
        const int4 *src = reinterpret_cast<const int4 *>(smem_raw + p.off_stage);
        int4 *dst = reinterpret_cast<int4 *>(p.out_block);
        const int n16 = int(O.total / 16);
        for (int k = tid; k < n16; k += nthr) dst[k] = src[k];
    }

    store_shares(s_shares, p.share_grid, p.shares);

    // Phase 6: counters.
    if (tid == 0) {
        p.counts[LORA_COUNT_SEGS] = S;
        p.counts[LORA_COUNT_ACTIVE] = ACT;
        p.counts[LORA_COUNT_INVALID] = s_invalid;
        p.counts[LORA_COUNT_SMALL_SEGS] = n_small;
        p.counts[LORA_COUNT_TC_SEGS] = n_tc;
        p.counts[LORA_COUNT_TC_ROWS] = tc_rows;
        p.counts[LORA_COUNT_DEVERR] = 0;
        p.counts[LORA_COUNT_GROUPS] = G;
    }
}

// ---------------------------------------------------------------------------
// Small batches (at most kPrepSmallMaxRows rows, groups by first appearance):
// one row per thread and a handful of block-wide steps, every table and the
// whole output block in shared memory, so that the part after the wait on
// the previous grid is one copy.  The outputs are those of prepare_kernel,
// bit for bit.
//   1. a hash slot per adapter with its first row and row count; within each
//      warp, every row's rank among the warp's rows of its adapter;
//   2. one block scan over the rows of (first-row flag | segments << 16 |
//      rows << 32): group number, segment base and row base of every group;
//   3. per segment: start, length, adapter, the tensor-core flag; per warp
//      and group: the warp's row count;
//   4. per group: the warps' row counts turned into their first positions;
//      one block scan over the segments of (tensor-core flag | rows << 32):
//      the small and tensor-core lists and the tensor-core row prefix;
//   5. every row's position (its warp's first position in its group plus its
//      rank in the warp) and the descriptors' inline rows;
//   6. after the wait: the copy, the tensor-core shares and the counters.
constexpr int kPrepSmallThreads = 512;
constexpr int kPrepSmallMaxRows = kPrepSmallThreads;

__global__ void __launch_bounds__(kPrepSmallThreads, 1) prepare_small_kernel(const __grid_constant__ PrepArgs p) {
    constexpr int NW = kPrepSmallThreads / 32;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ unsigned long long wsum[NW];
    __shared__ ShareTable s_shares;
    // The next grid may start at once (see griddep_launch_dependents): this
    // grid writes global memory only after its wait.
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int M = p.M, n = p.n, HS = p.hs, gcap = p.gcap;
    int32_t *key = reinterpret_cast<int32_t *>(smem_raw + p.off_hash), *first = key + HS, *cnt = first + HS;
    int32_t *whist = reinterpret_cast<int32_t *>(smem_raw + p.off_hist);  // [NW][gcap]
    int32_t *gad = reinterpret_cast<int32_t *>(smem_raw + p.off_gtab);
    int32_t *gcnt = gad + gcap, *grb = gcnt + gcap, *gsb = grb + gcap + 1;
    const OutLayout O = out_layout(p.max_segs, M);
    unsigned char *stg = smem_raw + p.off_stage;
    SegDesc *o_desc = reinterpret_cast<SegDesc *>(stg + O.rec);
    int4 *o_small = reinterpret_cast<int4 *>(stg + O.small);
    int4 *o_tc = reinterpret_cast<int4 *>(stg + O.tc);
    int32_t *o_indptr = reinterpret_cast<int32_t *>(stg + O.indptr);
    int32_t *o_lens = reinterpret_cast<int32_t *>(stg + O.lens);
    int32_t *o_widx = reinterpret_cast<int32_t *>(stg + O.widx);
    int32_t *o_tcptr = reinterpret_cast<int32_t *>(stg + O.tcptr);
    int32_t *o_sorted = reinterpret_cast<int32_t *>(stg + O.sorted);

    const int id = tid < M ? __ldcg(p.ids + tid) : -1;
    for (int s = tid; s < HS; s += kPrepSmallThreads) {
        key[s] = -1;
        first[s] = INT_MAX;
        cnt[s] = 0;
    }
    for (int k = tid; k < NW * gcap; k += kPrepSmallThreads) whist[k] = 0;
    const bool valid = tid < M && id >= 0 && id < n;
    const bool invalid = tid < M && id != -1 && !valid;
    __syncthreads();

    // 1. hash slots; ranks inside the warp
    int slot = -1;
    if (valid) {
        slot = (int)(((uint32_t)id * 0x9E3779B1u) >> (32 - (31 - __clz(HS))));
        for (;;) {  // at most M < HS distinct keys: a free slot always exists
            const int k = atomicCAS(&key[slot], -1, id);
            if (k == -1 || k == id) break;
            slot = (slot + 1) & (HS - 1);
        }
        atomicMin(&first[slot], tid);
        atomicAdd(&cnt[slot], 1);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? id : (int)(0x80000000u | (unsigned)lane));
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    const int n_invalid = __syncthreads_count(invalid);

    // 2. groups: number, segment base, row base
    const bool lead = valid && first[slot] == tid;
    const int c = lead ? cnt[slot] : 0;
    const int nseg = lead ? (p.chunk > 0 ? (c + p.chunk - 1) / p.chunk : 1) : 0;
    const unsigned long long v = lead ? (1ull | ((unsigned long long)nseg << 16) | ((unsigned long long)c << 32)) : 0ull;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    unsigned long long base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const unsigned long long s = wsum[w];
        base += w < warp ? s : 0ull;
        total += s;
    }
    const int G = (int)(total & 0xFFFFu), S = (int)((total >> 16) & 0xFFFFu), ACT = (int)(total >> 32);
    if (lead) {
        const unsigned long long ex = base + incl - v;
        const int g = (int)(ex & 0xFFFFu);
        gad[g] = id;
        gcnt[g] = c;
        grb[g] = (int)(ex >> 32);
        gsb[g] = (int)((ex >> 16) & 0xFFFFu);
        first[slot] = g;  // from here on: the slot's group
    }
    if (tid == 0) {
        grb[G] = ACT;
        gsb[G] = S;
    }
    __syncthreads();

    // 3. warps' row counts per group; segments
    const int myg = valid ? first[slot] : -1;
    if (valid && rank_w == 0) whist[warp * gcap + myg] = __popc(peers);
    for (int s = tid; s < S; s += kPrepSmallThreads) {
        int lo = 0, hi = G - 1;  // largest group whose first segment is <= s
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gsb[mid] <= s) lo = mid;
            else hi = mid - 1;
        }
        const int gc = gcnt[lo], cs = s - gsb[lo];
        int st = grb[lo], len = gc;
        if (p.chunk > 0) {
            st += cs * p.chunk;
            len = min(p.chunk, gc - cs * p.chunk);
        }
        o_indptr[s] = st;
        o_lens[s] = len;
        o_widx[s] = gad[lo];
        // the split follows the adapter group's rows (see prepare_kernel)
        *reinterpret_cast<int4 *>(&o_desc[s]) = make_int4(st, len, gad[lo], s | (gc >= p.tc_min ? LORA_DESC_TC_FLAG : 0));
    }
    for (int s = S + tid; s < p.max_segs; s += kPrepSmallThreads)
        *reinterpret_cast<int4 *>(&o_desc[s]) = make_int4(0, 0, 0, s);
    __syncthreads();

    // 4. first position of every warp's rows in each group; the two lists
    if (tid < G) {
        int run = grb[tid];
        for (int w = 0; w < NW; ++w) {
            const int t = whist[w * gcap + tid];
            whist[w * gcap + tid] = run;
            run += t;
        }
    }
    int4 rec = make_int4(0, 0, 0, 0);
    bool is_tc = false;
    if (tid < S) {
        rec = *reinterpret_cast<const int4 *>(&o_desc[tid]);
        is_tc = (rec.w & LORA_DESC_TC_FLAG) != 0;
        rec.w = tid;
    }
    const unsigned long long v2 = is_tc ? (1ull | ((unsigned long long)rec.y << 32)) : 0ull;
    unsigned long long incl2 = v2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o) incl2 += t;
    }
    if (lane == 31) wsum[warp] = incl2;
    __syncthreads();
    unsigned long long base2 = 0, total2 = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const unsigned long long s = wsum[w];
        base2 += w < warp ? s : 0ull;
        total2 += s;
    }
    const int n_tc = (int)(total2 & 0xFFFFFFFFu), tc_rows = (int)(total2 >> 32), n_small = S - n_tc;
    if (tid < S) {
        const unsigned long long ex = base2 + incl2 - v2;
        const int before = (int)(ex & 0xFFFFFFFFu);
        if (is_tc) {
            o_tc[before] = rec;
            o_tcptr[before] = (int)(ex >> 32);
        } else {
            o_small[tid - before] = rec;
        }
    }
    if (tid == 0) {
        o_indptr[S] = ACT;
        o_tcptr[n_tc] = tc_rows;
    }

    // 5. positions and the descriptors' inline rows
    if (valid) {
        const int pos = whist[warp * gcap + myg] + rank_w;
        o_sorted[pos] = tid;
        const int off = pos - grb[myg];
        const int s = gsb[myg] + (p.chunk > 0 ? off / p.chunk : 0);
        const int k = p.chunk > 0 ? off - (off / p.chunk) * p.chunk : off;
        if (k < kInlineRows) o_desc[s].rows[k] = tid;
    }
    __syncthreads();

    // 6. the shares (computed before the wait), then after the previous grid:
    // the copy, the shares, the counters
    plan_shares(o_tc, o_tcptr, n_tc, tc_rows, p.share_grid, s_shares);
    griddep_wait();
    {
        const int4 *src = reinterpret_cast<const int4 *>(stg);
        int4 *dst = reinterpret_cast<int4 *>(p.out_block);
        const int n16 = int(O.total / 16);
        for (int k = tid; k < n16; k += kPrepSmallThreads) dst[k] = src[k];
    }
    store_shares(s_shares, p.share_grid, p.shares);
    if (tid == 0) {
        p.counts[LORA_COUNT_SEGS] = S;
        p.counts[LORA_COUNT_ACTIVE] = ACT;
        p.counts[LORA_COUNT_INVALID] = n_invalid;
        p.counts[LORA_COUNT_SMALL_SEGS] = n_small;
        p.counts[LORA_COUNT_TC_SEGS] = n_tc;
        p.counts[LORA_COUNT_TC_ROWS] = tc_rows;
        p.counts[LORA_COUNT_DEVERR] = 0;
        p.counts[LORA_COUNT_GROUPS] = G;
    }
}

// Shared-memory budget of the prepare kernel.
constexpr size_t kPrepSmemMax = 200 * 1024;

cudaError_t launch_prepare(const int32_t *ids, int32_t M, int32_t n, int32_t chunk,
                           int32_t tc_min, bool ascending, int32_t share_grid, char *ws, const WsLayout &L,
                           lora_batch_t *b, cudaStream_t stream) {
    PrepArgs p{};
    p.ids = ids;
    p.M = M;
    p.n = n;
    p.chunk = chunk;
    p.tc_min = tc_min;
    p.ascending = ascending ? 1 : 0;
    p.gcap = L.g_max;
    auto at = [&](size_t off) { return reinterpret_cast<int32_t *>(ws + off); };
    p.sorted = at(L.sorted);
    p.indptr = at(L.indptr);
    p.lens = at(L.lens);
    p.widx = at(L.widx);
    p.desc = reinterpret_cast<SegDesc *>(ws + L.rec);
    p.out_block = ws;  // the output block starts the workspace
    p.max_segs = L.max_segs;
    p.small = reinterpret_cast<int4 *>(ws + L.small);
    p.tc = reinterpret_cast<int4 *>(ws + L.tc);
    p.tcptr = at(L.tcptr);
    p.counts = at(L.counts);
    p.shares = reinterpret_cast<int2 *>(ws + L.shares);
    p.share_grid = share_grid;
    p.first_pos = at(L.first_pos);
    p.acnt = at(L.adapter_cnt);
    p.agroup = at(L.adapter_group);
    p.gadapter = at(L.group_adapter);
    p.grow = at(L.group_row);
    p.gseg = at(L.group_seg);
    p.whist = at(L.warp_hist);

    const int gcap = L.g_max;
    if (M <= kPrepSmallMaxRows && !ascending) {
        // hash table, warp counts, group table and the output block
        int hs = 64;
        while (hs < 2 * M) hs <<= 1;
        size_t o = 0;
        auto take = [&](size_t bytes) {
            const size_t at = o;
            o += (bytes + 15) & ~size_t(15);
            return (int32_t)at;
        };
        p.hs = hs;
        p.off_hash = take(size_t(3) * hs * 4);
        p.off_hist = take(size_t(kPrepSmallThreads / 32) * gcap * 4);
        p.off_gtab = take((size_t(4) * gcap + 2) * 4);
        p.off_stage = take(out_layout(L.max_segs, M).total);
        if (o <= kPrepSmemMax) {
            static DeviceOnce configured_small;
            cudaError_t e = configured_small.run([] {
                return cudaFuncSetAttribute(prepare_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kPrepSmemMax);
            });
            if (e != cudaSuccess) return e;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1);
            cfg.blockDim = dim3(kPrepSmallThreads);
            cfg.dynamicSmemBytes = o;
            cfg.stream = stream;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, prepare_small_kernel, p);
            if (e != cudaSuccess) return e;
            b->sorted_token_ids = p.sorted;
            b->seg_indptr = p.indptr;
            b->seg_lens = p.lens;
            b->weight_indices = p.widx;
            b->seg_records = reinterpret_cast<int32_t *>(p.desc);
            b->small_segs = reinterpret_cast<int32_t *>(p.small);
            b->tc_segs = reinterpret_cast<int32_t *>(p.tc);
            b->tc_indptr = p.tcptr;
            b->counts = p.counts;
            return cudaSuccess;
        }
    }

    const int threads = M > 8192 ? 1024 : (M > 1024 ? 512 : 256);
    // Place tables in shared memory, most latency-critical first.
    size_t smem = 0;
    auto place = [&](size_t bytes) -> int32_t {
        bytes = (bytes + 15) & ~size_t(15);
        if (smem + bytes > kPrepSmemMax) return -1;
        const int32_t off = (int32_t)smem;
        smem += bytes;
        return off;
    };
    p.off_groups = place(size_t(3 * gcap + 2) * 4);
    p.off_hist = place(size_t(threads / 32) * gcap * 4);
    p.off_adapters = place(size_t(3) * n * 4);
    p.off_bits = M <= 65536 ? place(size_t(2) * ((M + 31) / 32) * 4) : -1;
    p.off_ids = place(size_t(M) * 4);
    p.off_stage = place(out_layout(L.max_segs, M).total);

    static DeviceOnce configured;
    cudaError_t e = configured.run([] {
        return cudaFuncSetAttribute(prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kPrepSmemMax);
    });
    if (e != cudaSuccess) return e;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prepare_kernel, p);
    if (e != cudaSuccess) return e;

    b->sorted_token_ids = p.sorted;
    b->seg_indptr = p.indptr;
    b->seg_lens = p.lens;
    b->weight_indices = p.widx;
    b->seg_records = reinterpret_cast<int32_t *>(p.desc);
    b->small_segs = reinterpret_cast<int32_t *>(p.small);
    b->tc_segs = reinterpret_cast<int32_t *>(p.tc);
    b->tc_indptr = p.tcptr;
    b->counts = p.counts;
    return cudaSuccess;
}

}  // namespace lora
