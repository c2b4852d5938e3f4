// sgmv_small.cu -- fused SGMV kernel for small batches (decode steps): the
// rows are grouped on chip from the ids, the adapter weights are requested
// before the kernel waits on its predecessor, and h is reduced across a
// thread-block cluster by one-way pushes into the peers' shared memory.
//
// What it computes is the fused delta of one batch ("vLLM-Ascend LoRA"
// article, section 3.3: the rows of one adapter are gathered, tmp = rows .
// A^T, delta = (tmp * scale) . B^T is added into the output; the adapter's
// A/B move once and serve every row of the group):
//     y[i] += s_a * (x[i] . A[a]^T) . B[a]^T      for every row i with id a.
//
// Grouping.  Every CTA reads the ids (at most kSmMaxRows) and groups the rows
// itself, in the order in which each adapter first occurs ("III.Punica:
// Multi-Tenant LoRA Serving", section 代码: the regrouping of tokens by
// adapter): a hash table in shared memory gives every adapter its first row
// and its row count, and one block scan over the rows, of "this row is its
// adapter's first" packed with the adapter's tile count, gives every group
// its number and its first tile.  A group of more than kSmRT rows is cut into
// near-equal tiles of at most kSmRT rows; tile t belongs to cluster t mod C.
// The grouping depends only on the ids, so every CTA builds the same tiles,
// and the first row of each group writes the records of its tiles that fall
// to this CTA's cluster.
//
// Work of a tile.  CTA q of a cluster of CL owns
//   - the K slice q of d_in for the shrink (x rows and A rows of that slice),
//   - the N slice q of d_out for the expand (B rows and y rows of that slice),
// so every byte of x, A, B and y of a tile is read once.
//
// Data movement.  A rows and the gathered y rows arrive by 16-byte cp.async
// from every thread (a few per thread: the copy unit takes them faster than
// one bulk copy per 2 KB row piece); the CTA's B rows are one contiguous
// block per output slice and arrive by one bulk copy each.  x never enters
// shared memory: each lane loads its shrink fragments straight into
// registers (8 bytes per row and K step).  The weights (A and B) depend only
// on the adapter, so they are requested before the kernel waits on the
// previous grid in the stream (programmatic dependent launch); x and y are
// requested after that wait.  y + delta leaves by 16-byte stores.  One
// shared-memory region serves three purposes in turn: the hash table of the
// grouping, a tile's A rows, and the warps' partial h.
//
// Compute.  Shrink: warp-level bf16 tensor-core tiles (16 x 8 x 16, fp32
// accumulators in registers; A fragments by 8-byte loads from rows whose
// pitch puts the rows of a half-warp's loads in distinct banks).  The warps
// split the K steps and each takes every 16-column rank block of its steps;
// their partials are summed in warp order.  The CTA's partial h is
// pushed to every CTA of the cluster (st.async, completing on the receiver's
// mbarrier: no cluster barrier per tile), and each CTA sums the CL partials
// in rank order, so every CTA holds the same h.  h is scaled once, masked to
// the adapter's rank and to the tile's rows, and rounded once to bf16.
// Expand: the same tiles with h as the A operand and B rows as the B
// operand, four 8-column tiles per warp in flight, the K slots permuted so
// that B fragments come by conflict-free 64-bit loads; y + delta is formed in
// fp32, rounded once to bf16 and written back into the y rows in shared
// memory, which then leave by 16-byte stores.  The rank mask is exact: h
// columns past the rank are zero and B fragments past the rank are zeroed in
// registers, so padding (even NaN) never enters a result.
#include <algorithm>
#include <climits>

#include "common.cuh"

namespace lora {

constexpr int kSmThreads = 512;
constexpr int kSmWarps = kSmThreads / 32;
constexpr int kSmMaxRows = 1024;  // rows a batch may have for this kernel (two per thread)
constexpr int kSmRT = 16;         // rows per tile: one 16-row MMA tile
constexpr int kSmNtBatch = 4;     // 8-column tiles a warp keeps in flight in the expand
constexpr int kSmXB = 8;          // K steps of x a warp holds in registers at once

// The CTA's columns [n0, n1) by output slice t: columns [cb, ce) (ce <= cb:
// the slice has none of them), y column = column + go, B rows at byte off of
// the B block with a row pitch of str bytes.  Computed on the host for every
// cluster rank and read from the launch parameters.
struct PieceTab {
    int cb[LORA_MAX_SLICES], ce[LORA_MAX_SLICES], str[LORA_MAX_SLICES], go[LORA_MAX_SLICES];
    uint32_t off[LORA_MAX_SLICES];
};

constexpr int kSmMaxCluster = 8;

struct SmGeom {
    int CL;              // CTAs per cluster
    int KC;              // shrink columns per CTA
    int NCmax;           // expand columns per CTA (at most)
    int apitch, ypitch;  // bytes per shared row of A and of y
    int HS;              // hash slots (power of two, >= 2 M)
    int tcap;            // tile records per CTA
    uint32_t ncl_magic;  // ceil(2^32 / clusters): x / clusters = umulhi(x, magic) for x < 2^16
    int ncol0[kSmMaxCluster + 1];  // first expand column of cluster rank q (multiples of 8)
    PieceTab pt[kSmMaxCluster];    // the slices of each cluster rank's columns
    int off_bars, off_scan, off_tl, off_rows, off_recv, off_hbf, off_A, off_y, off_B, total;
};

// One tile of this cluster: adapter, rank, first and last row (exclusive)
// inside its group's rows, scale.
struct TileRec {
    int a, r, lo, hi;
    float sc;
    int pad[3];
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// One test of phase `parity` with cluster-scope acquire (the phase is
// completed by writes from other CTAs of the cluster); the thread may sleep
// in it until the phase completes, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cl(uint64_t *bar, uint32_t parity) {
    const uint32_t b = smem_u32(bar);
    if (mbar_try_wait_cl(b, parity)) return true;
    const long long deadline = clock64() + kWaitLimitCycles;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cl(b, parity)) return true;
        if (clock64() > deadline) return false;
    }
}
// 16 bytes into another CTA's shared memory, completing on its mbarrier.
__device__ __forceinline__ void st_async_f4(uint32_t raddr, const float4 &v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(
                     raddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
                 : "memory");
}
// Shared-memory accesses by 32-bit shared-window address, in program order
// (volatile: they keep their order with the barriers and with each other).
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t hash_slot(int a, int HS) {
    return ((uint32_t)a * 0x9E3779B1u) >> (32 - (31 - __clz(HS)));
}
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ void cp_async16_full(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void add4(float4 &v, const float4 &w) {
    v.x += w.x;
    v.y += w.y;
    v.z += w.z;
    v.w += w.w;
}
template <int R16>
__global__ void __launch_bounds__(kSmThreads, 1)
    sgmv_small_kernel(const __grid_constant__ DeltaArgs p, const __grid_constant__ SmGeom g) {
    constexpr int KS = R16 / 16;  // K steps of the expand (rank blocks of the shrink)
    constexpr int NT = kSmThreads, NW = kSmWarps;
    constexpr int RP = R16 + 4;   // floats per row of a warp's partial h
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar_b = reinterpret_cast<uint64_t *>(smem + g.off_bars);  // B block landed
    uint64_t *recv_bar = bar_b + 1;                                      // [2] partial h received
    // Region A holds the hash table while the rows are grouped, the A rows of
    // a tile during its shrink, and then the warps' partial h.
    int32_t *key = reinterpret_cast<int32_t *>(smem + g.off_A);
    int32_t *first = key + g.HS;
    int32_t *cnt = first + g.HS;
    int32_t *wsum = reinterpret_cast<int32_t *>(smem + g.off_scan);  // [NW]
    int32_t *wsum2 = wsum + 32;                                         // [NW]
    TileRec *tl = reinterpret_cast<TileRec *>(smem + g.off_tl);        // [tcap]
    int32_t *rows_s = reinterpret_cast<int32_t *>(smem + g.off_rows);  // [kSmRT]
    const PieceTab *pt = &g.pt[cluster_ctarank()];  // launch parameters
    float *recv = reinterpret_cast<float *>(smem + g.off_recv);        // [2][CL][16][R16]
    unsigned char *hbf = smem + g.off_hbf;                              // [16][R16 + 8] bf16
    unsigned char *sA = smem + g.off_A, *sY = smem + g.off_y, *sB = smem + g.off_B;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int CL = g.CL;
    const uint32_t q = cluster_ctarank(), cid = cluster_id_x(), ncl = nclusters_x();
    const int M = p.M_rows, n = p.n_adapters;
    const int HS = g.HS;
    const int hpitch = (R16 + 8) * 2;

    // Nothing this grid writes is read by the next one before its own wait,
    // and this grid reads before its wait only what no grid of the stream
    // writes (see griddep_launch_dependents): the next grid may start at once.
    griddep_launch_dependents();
    // ids written by the grid before (an updated batch): read after the wait
    if (p.ids_after_wait) griddep_wait();

    // ---- phase 0: ids (one or two rows per thread), the adapters' ranks and
    // scales, and an empty hash table.  Everything read before the wait (ids,
    // ranks, scales and later the weights) is fixed before the previous grid
    // in the stream started (header contract).
    const int RPT = M > NT ? 2 : 1;
    int idr[2], rkr[2];
    float scr[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = tid * RPT + k;
        idr[k] = (k < RPT && i < M) ? __ldcg(p.ids + i) : -1;
    }
    if (tid == 0) {
        mbar_init(bar_b, 1);
        mbar_init(&recv_bar[0], 1);
        mbar_init(&recv_bar[1], 1);
        fence_mbar_init();
    }
    for (int s = tid; s < HS; s += NT) {
        key[s] = -1;
        first[s] = INT_MAX;
        cnt[s] = 0;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool v = idr[k] >= 0 && idr[k] < n;
        if (!v) idr[k] = -1;
        rkr[k] = v && p.ranks ? __ldcg(p.ranks + idr[k]) : p.r_max;
        scr[k] = v && p.adapter_scale ? __ldcg(p.adapter_scale + idr[k]) : p.scale;
    }
    __syncthreads();
    cluster_arrive_relaxed();  // the barriers exist before any peer pushes into them

    // ---- phase 1: one hash slot per adapter with its first row and count.
    int slot[2] = {-1, -1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (idr[k] >= 0) {
            const int a = idr[k];
            int s = (int)hash_slot(a, HS);
            for (;;) {  // at most M < HS distinct keys: a free slot always exists
                const int kk = atomicCAS(&key[s], -1, a);
                if (kk == -1 || kk == a) break;
                s = (s + 1) & (HS - 1);
            }
            atomicMin(&first[s], tid * RPT + k);
            atomicAdd(&cnt[s], 1);
            slot[k] = s;
        }
    }
    __syncthreads();

    // ---- phase 2: one block scan over the rows of (first-row flag | tiles
    // << 16) gives every group its number and its first tile.
    int ntile[2] = {0, 0}, bad = 0, v = 0;
    bool lead[2] = {false, false};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (slot[k] >= 0 && first[slot[k]] == tid * RPT + k) {
            lead[k] = true;
            const int r = rkr[k];
            if (r < 0 || r > p.r_max) bad = 1;
            else if (r > 0) ntile[k] = (cnt[slot[k]] + kSmRT - 1) / kSmRT;
            v += 1 + (ntile[k] << 16);
        }
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base, total;
    {
        // warp totals, scanned across the warps by shuffles
        const int wv = lane < NW ? wsum[lane] : 0;
        int ws = wv;
#pragma unroll
        for (int o = 1; o < NW; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += t;
        }
        base = __shfl_sync(0xffffffffu, ws - wv, warp);
        total = __shfl_sync(0xffffffffu, ws, NW - 1);
    }
    const int T = total >> 16;  // tiles of the batch
    {
        int run = base + incl - v;  // exclusive prefix of this thread's first row
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (lead[k]) {
                const int tb = run >> 16, nt = ntile[k], c = cnt[slot[k]];
                // tiles tb .. tb + nt - 1 of this group: those of this
                // cluster (tile t is record t / C of cluster t mod C)
                for (int j = 0; j < nt; ++j) {
                    const int t = tb + j;
                    const int e = (int)__umulhi((uint32_t)t, g.ncl_magic);
                    if (t - e * (int)ncl == (int)cid && e < g.tcap) {
                        TileRec rec;
                        rec.a = idr[k];
                        rec.r = rkr[k];
                        rec.lo = nt == 1 ? 0 : c * j / nt;  // c, j, nt <= kSmMaxRows: no overflow
                        rec.hi = nt == 1 ? c : c * (j + 1) / nt;
                        rec.sc = scr[k];
                        rec.pad[0] = rec.pad[1] = rec.pad[2] = 0;
                        tl[e] = rec;
                    }
                }
                run += 1 + (nt << 16);
            }
        }
    }
    // (the barrier also ends every read of the hash table: region A is free)
    const int bad_rank = __syncthreads_or(bad);
    const int my_tiles =
        (int)cid < T ? min((int)__umulhi((uint32_t)(T - 1 - (int)cid), g.ncl_magic) + 1, g.tcap) : 0;

    const int k0 = (int)q * g.KC;
    const int n0 = g.ncol0[q], n1 = g.ncol0[q + 1];
    const int ncols = n1 - n0;
    const int kc8 = g.KC / 8;
    const int nks = g.KC >> 4;  // 16-column K steps of the shrink
    const int g_ = lane >> 2, t4 = lane & 3;

    // The weights of a tile: A rows [0, r) of the K slice (cp.async, one
    // group: warp w takes rows w, w + NW, ..., its lanes the 16-byte pieces),
    // B rows of the N slice (one bulk copy per output slice, on bar_b).
    auto request_weights = [&](const TileRec &ti) {
        const __nv_bfloat16 *Aa = static_cast<const __nv_bfloat16 *>(p.A) + (int64_t)ti.a * p.a_stride_adapter + k0;
        for (int jr = warp; jr < ti.r; jr += NW) {
            const __nv_bfloat16 *src = Aa + (int64_t)jr * p.a_stride_r;
            unsigned char *dst = sA + jr * g.apitch;
            for (int cc = lane; cc < kc8; cc += 32) cp_async16_full(dst + cc * 16, src + cc * 8);
        }
        cp_async_commit();
        if (tid == 0) {
            uint32_t bytes = 0;
            for (int t = 0; t < p.n_slices; ++t)
                if (pt->cb[t] < pt->ce[t]) bytes += (uint32_t)(pt->ce[t] - pt->cb[t]) * (uint32_t)pt->str[t];
            mbar_arrive_expect_tx(bar_b, bytes);
            for (int t = 0; t < p.n_slices; ++t) {
                if (pt->cb[t] < pt->ce[t]) {
                    const SliceDesc &sl = p.slices[t];
                    bulk_g2s(sB + pt->off[t],
                             static_cast<const __nv_bfloat16 *>(sl.B) + (int64_t)ti.a * sl.stride_adapter +
                                 (int64_t)(pt->cb[t] - sl.col_begin) * sl.stride_n,
                             (uint32_t)(pt->ce[t] - pt->cb[t]) * (uint32_t)pt->str[t], bar_b);
                }
            }
        }
    };
    // Rows [lo, hi) of adapter a's group, in ascending row order.
    auto find_rows = [&](int a, int lo, int hi) {
        const unsigned m0 = __ballot_sync(0xffffffffu, idr[0] == a);
        const unsigned m1 = __ballot_sync(0xffffffffu, RPT > 1 && idr[1] == a);
        if (lane == 0) wsum2[warp] = __popc(m0) + __popc(m1);
        __syncthreads();
        int b;
        {
            const int wv = lane < NW ? wsum2[lane] : 0;
            int ws = wv;
#pragma unroll
            for (int o = 1; o < NW; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, ws, o);
                if (lane >= o) ws += t;
            }
            b = __shfl_sync(0xffffffffu, ws - wv, warp);
        }
        const unsigned lt = (1u << lane) - 1u;
        const int p0 = b + __popc(m0 & lt) + __popc(m1 & lt);
        if (idr[0] == a && p0 >= lo && p0 < hi) rows_s[p0 - lo] = tid * RPT;
        const int p1 = p0 + (idr[0] == a ? 1 : 0);
        if (RPT > 1 && idr[1] == a && p1 >= lo && p1 < hi) rows_s[p1 - lo] = tid * RPT + 1;
        __syncthreads();
    };
    // y rows (N slice) of the tile, one cp.async group: warp w takes rows w,
    // w + NW, ..., its lanes the 16-byte pieces.
    auto request_y = [&](int R) {
        for (int row = warp; row < R; row += NW) {
            const __nv_bfloat16 *yrow = static_cast<const __nv_bfloat16 *>(p.y) + (int64_t)rows_s[row] * p.ldy;
            unsigned char *dst = sY + row * g.ypitch;
            for (int t = 0; t < p.n_slices; ++t) {
                const int ce = pt->ce[t], go = pt->go[t];
                for (int col = pt->cb[t] + lane * 8; col < ce; col += 256)
                    cp_async16_full(dst + (col - n0) * 2, yrow + go + col);
            }
        }
        cp_async_commit();
    };
    // x goes straight from global memory into the shrink's B fragments.  The
    // MMA's K slots are permuted inside each 16-column step, the same way for
    // A and x: slots 2t, 2t+1, 2t+8, 2t+9 of lane t take columns 4t .. 4t+3,
    // so a lane's x fragment of one row and step is 8 contiguous bytes (and a
    // warp's load covers 8 rows x 32 bytes).  Lane (g, t) takes rows g and
    // g + 8 of the tile; warp w takes K steps w, w + NW, ...
    const __nv_bfloat16 *xbase = static_cast<const __nv_bfloat16 *>(p.x) + k0 + 4 * t4;
    const __nv_bfloat16 *x0 = nullptr, *x1 = nullptr;
    uint2 xa[kSmXB], xb[kSmXB];
    auto x_rows = [&](int R) {
        x0 = g_ < R ? xbase + (int64_t)rows_s[g_] * p.ldx : nullptr;
        x1 = g_ + 8 < R ? xbase + (int64_t)rows_s[g_ + 8] * p.ldx : nullptr;
    };
    auto load_x = [&](int kb) {
#pragma unroll
        for (int j = 0; j < kSmXB; ++j) {
            const int ks = kb + j * NW;
            xa[j] = (x0 && ks < nks) ? __ldcg(reinterpret_cast<const uint2 *>(x0 + ks * 16)) : make_uint2(0u, 0u);
            xb[j] = (x1 && ks < nks) ? __ldcg(reinterpret_cast<const uint2 *>(x1 + ks * 16)) : make_uint2(0u, 0u);
        }
    };

    TileRec ti{};
    if (my_tiles > 0) {
        ti = tl[0];
        request_weights(ti);
        find_rows(ti.a, ti.lo, ti.hi);
    }
    griddep_wait();
    if (bad_rank && blockIdx.x == 0 && tid == 0) raise_deverr(p.counts, LORA_DEVERR_RANK);
    if (my_tiles > 0) {
        x_rows(ti.hi - ti.lo);
        load_x(warp);
        request_y(ti.hi - ti.lo);
    }
    cluster_wait_acquire();

    bool ok = true;
    for (int e = 0; e < my_tiles; ++e) {
        if (e > 0) {
            // the previous tile is done with every buffer
            ti = tl[e];
            request_weights(ti);
            find_rows(ti.a, ti.lo, ti.hi);
            x_rows(ti.hi - ti.lo);
            load_x(warp);
            request_y(ti.hi - ti.lo);
        }
        const int r = ti.r, R = ti.hi - ti.lo;
        const int r16a = (r + 15) & ~15;
        const int np = r16a / 16;  // 16-column rank blocks
        const int buf = e & 1;
        if (tid == 0) mbar_arrive_expect_tx(&recv_bar[buf], (uint32_t)(CL * 16 * r16a * 4));

        // ---- shrink: h^T = A . x^T on warp-level tensor-core tiles (M = the
        // 16 ranks of a rank block, N = 8 rows, K = 16 columns of d_in): a
        // tile of at most 8 rows takes one product per K step and rank block.
        cp_async_wait<1>();  // A of this thread
        __syncthreads();
        const bool two = R > 8;  // a second 8-row tile
        float acc[KS][2][4];     // [rank block][row tile][fragment]
#pragma unroll
        for (int pb = 0; pb < KS; ++pb)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[pb][u][i] = 0.f;
        // A fragment of rank g (+ 8) of block pb: the 8 bytes of the lane's
        // four permuted columns
        const uint32_t ab = smem_u32(sA) + g_ * g.apitch + 8 * t4;
        for (int kb = warp; kb < nks; kb += NW * kSmXB) {
            if (kb != warp) load_x(kb);
#pragma unroll
            for (int j = 0; j < kSmXB; ++j) {
                const int ks = kb + j * NW;
                if (ks < nks) {
#pragma unroll
                    for (int pb = 0; pb < KS; ++pb) {
                        if (pb < np) {
                            const uint32_t a = ab + pb * 16 * g.apitch + ks * 32;
                            const uint2 lo = lds64(a), hi = lds64(a + 8 * g.apitch);
                            const uint32_t af[4] = {lo.x, hi.x, lo.y, hi.y};
                            mma_bf16_16816(acc[pb][0], af, xa[j].x, xa[j].y);
                            if (two) mma_bf16_16816(acc[pb][1], af, xb[j].x, xb[j].y);
                        }
                    }
                }
            }
        }
        __syncthreads();  // every warp is done with the A rows: the region takes the partials
        // warp partial -> red[warp][row][rank] (row pitch R16 + 4 floats: the
        // fragment's rows 2t and 2t+1 fall in distinct banks).  Rows of a
        // missing second 8-row tile hold leftovers; h masks them.
        {
            const uint32_t rw = smem_u32(sA) + (uint32_t)warp * (16 * RP * 4);
#pragma unroll
            for (int pb = 0; pb < KS; ++pb) {
#pragma unroll
                for (int rt = 0; rt < 2; ++rt) {
                    if (pb < np && (rt == 0 || two)) {
                        const uint32_t a0 = rw + ((rt * 8 + 2 * t4) * RP + pb * 16 + g_) * 4;
                        sts32(a0, __float_as_uint(acc[pb][rt][0]));
                        sts32(a0 + RP * 4, __float_as_uint(acc[pb][rt][1]));
                        sts32(a0 + 8 * 4, __float_as_uint(acc[pb][rt][2]));
                        sts32(a0 + (RP + 8) * 4, __float_as_uint(acc[pb][rt][3]));
                    }
                }
            }
        }
        __syncthreads();
        // CTA partial: the NW warp partials summed in warp order, pushed to
        // every CTA of the cluster: slot q of their receive buffer.
        const int nel4 = 4 * r16a;  // float4 entries of a 16 x r16a block
        const int rq = r16a / 4;    // float4 entries per row
        float *rv = recv + (size_t)buf * CL * 16 * R16;
        if (tid < nel4) {
            const int row = tid / rq, col = (tid - row * rq) * 4;
            const uint32_t a = smem_u32(sA) + (uint32_t)(row * RP + col) * 4;
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const uint4 pv = lds128(a + (uint32_t)w * (16 * RP * 4));
                add4(s4, make_float4(__uint_as_float(pv.x), __uint_as_float(pv.y), __uint_as_float(pv.z),
                                     __uint_as_float(pv.w)));
            }
            const uint32_t la = smem_u32(rv + ((size_t)q * 16 + row) * R16 + col);
            const uint32_t lb = smem_u32(&recv_bar[buf]);
            for (int pr = 0; pr < CL; ++pr) st_async_f4(map_to_rank(la, pr), s4, map_to_rank(lb, pr));
        }
        // h = scale * sum of the CL partials (rank order), masked to the
        // tile's rows and the adapter's rank, rounded once to bf16; only the
        // threads that read the partials wait for them (the others wait at
        // the block barrier below, which also publishes h and the B block)
        if (tid < nel4) {
            if (!mbar_wait_cl(&recv_bar[buf], (uint32_t)(e >> 1) & 1u)) ok = false;
            const int row = tid / rq, col = (tid - row * rq) * 4;
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int pr = 0; pr < 8; ++pr)
                if (pr < CL) add4(s4, *reinterpret_cast<const float4 *>(rv + ((size_t)pr * 16 + row) * R16 + col));
            const bool rok = row < R;
            const float sc = ti.sc;
            const float h0 = rok && col + 0 < r ? s4.x * sc : 0.f;
            const float h1 = rok && col + 1 < r ? s4.y * sc : 0.f;
            const float h2 = rok && col + 2 < r ? s4.z * sc : 0.f;
            const float h3 = rok && col + 3 < r ? s4.w * sc : 0.f;
            *reinterpret_cast<uint2 *>(hbf + row * hpitch + col * 2) =
                make_uint2(bf16x2_bits(h0, h1), bf16x2_bits(h2, h3));
        }
        cp_async_wait<0>();  // y of this thread
        if (tid == NT - 1 && !mbar_wait(bar_b, (uint32_t)e & 1u)) ok = false;
        __syncthreads();

        // ---- expand: warp w takes 8-column tiles w * 4 .. w * 4 + 3, then
        // + 64, ...; the four are in flight together.  Inside each 16-rank
        // K step the MMA's K slots are permuted the same way for h and B:
        // slots 2t, 2t+1 hold ranks 4t, 4t+1 and slots 2t+8, 2t+9 hold ranks
        // 4t+2, 4t+3, so a thread's two B words (and two h words) are eight
        // contiguous bytes: one 64-bit load, and the eight rows of a
        // fragment read 32-byte B rows without bank conflicts.
        uint32_t hf[KS][4];
        const uint32_t hb = smem_u32(hbf) + g_ * hpitch + 8 * t4;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (ks < np) {
                const uint2 lo = lds64(hb + ks * 32);
                const uint2 hi = lds64(hb + 8 * hpitch + ks * 32);
                hf[ks][0] = lo.x;
                hf[ks][1] = hi.x;
                hf[ks][2] = lo.y;
                hf[ks][3] = hi.y;
            }
        }
        uint32_t bm0[KS], bm1[KS];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int kk = ks * 16 + 4 * t4;
            bm0[ks] = (kk + 1 < r ? 0xFFFF0000u : 0u) | (kk < r ? 0x0000FFFFu : 0u);
            bm1[ks] = (kk + 3 < r ? 0xFFFF0000u : 0u) | (kk + 2 < r ? 0x0000FFFFu : 0u);
        }
        const int nnt = ncols >> 3;
        const int bstr0 = (int)p.slices[0].stride_n * 2;  // B row pitch when there is one slice
        const uint32_t sBa = smem_u32(sB) + 8 * t4;
        const uint32_t yr0 = smem_u32(sY) + g_ * g.ypitch + 4 * t4;  // row g_, column 2 t4
        const uint32_t yr1 = yr0 + 8 * g.ypitch;                     // row g_ + 8
        const bool row0 = g_ < R, row1 = g_ + 8 < R;
        for (int nt0 = warp * kSmNtBatch; nt0 < nnt; nt0 += NW * kSmNtBatch) {
            // addresses of the four tiles' B rows (the slice that holds each)
            uint32_t ba[kSmNtBatch];
#pragma unroll
            for (int b = 0; b < kSmNtBatch; ++b) {
                const int col = n0 + (nt0 + b) * 8;
                uint32_t off = 0;
                int beg = n0, str = bstr0;
                if (p.n_slices > 1) {
                    for (int t = 0; t < p.n_slices; ++t)
                        if (col >= pt->cb[t] && col < pt->ce[t]) {
                            beg = pt->cb[t];
                            str = pt->str[t];
                            off = pt->off[t];
                        }
                }
                ba[b] = sBa + off + (col - beg + g_) * str;
            }
            // loads first (B words, then the y words), then the products,
            // then y + delta in fp32, rounded once, back into the y rows
            uint2 bw[kSmNtBatch][KS];
#pragma unroll
            for (int b = 0; b < kSmNtBatch; ++b)
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
                    bw[b][ks] = (nt0 + b < nnt && ks < np) ? lds64(ba[b] + ks * 32) : make_uint2(0u, 0u);
            uint32_t y0[kSmNtBatch], y1[kSmNtBatch];
#pragma unroll
            for (int b = 0; b < kSmNtBatch; ++b) {
                const uint32_t yo = (uint32_t)((nt0 + b) * 16);
                y0[b] = (nt0 + b < nnt && row0) ? lds32(yr0 + yo) : 0u;
                y1[b] = (nt0 + b < nnt && row1) ? lds32(yr1 + yo) : 0u;
            }
            float d[kSmNtBatch][4];
#pragma unroll
            for (int b = 0; b < kSmNtBatch; ++b) {
#pragma unroll
                for (int i = 0; i < 4; ++i) d[b][i] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
                    if (ks < np) mma_bf16_16816(d[b], hf[ks], bw[b][ks].x & bm0[ks], bw[b][ks].y & bm1[ks]);
            }
#pragma unroll
            for (int b = 0; b < kSmNtBatch; ++b) {
                if (nt0 + b < nnt) {
                    const uint32_t yo = (uint32_t)((nt0 + b) * 16);
                    if (row0)
                        sts32(yr0 + yo, bf16x2_bits(__uint_as_float(y0[b] << 16) + d[b][0],
                                                    __uint_as_float(y0[b] & 0xFFFF0000u) + d[b][1]));
                    if (row1)
                        sts32(yr1 + yo, bf16x2_bits(__uint_as_float(y1[b] << 16) + d[b][2],
                                                    __uint_as_float(y1[b] & 0xFFFF0000u) + d[b][3]));
                }
            }
        }
        __syncthreads();
        // the rows leave by 16-byte stores: unit u = (row u / hv, 8-column
        // pieces u % hv, u % hv + hv, ...) goes to warp u % NW (hv = 2 when
        // the rows are at most half the warps)
        {
            const int hv = 2 * R <= NW ? 2 : 1;
            for (int u = warp; u < R * hv; u += NW) {
                const int row = u / hv, part = u - row * hv;
                __nv_bfloat16 *yrow = static_cast<__nv_bfloat16 *>(p.y) + (int64_t)rows_s[row] * p.ldy;
                const uint32_t src = smem_u32(sY) + row * g.ypitch;
                for (int t = 0; t < p.n_slices; ++t) {
                    const int ce = pt->ce[t], go = pt->go[t];
                    for (int col = pt->cb[t] + (part * 32 + lane) * 8; col < ce; col += 256 * hv)
                        *reinterpret_cast<uint4 *>(yrow + go + col) = lds128(src + (col - n0) * 2);
                }
            }
        }
        __syncthreads();  // every buffer may be refilled
    }
    // A wait that gave up may leave the last B block in flight: wait once
    // more (bounded) before the shared memory goes away.
    if (__syncthreads_or(!ok) && tid == 0) {
        raise_deverr(p.counts, LORA_DEVERR_WAIT);
        if (my_tiles > 0) mbar_wait(bar_b, (uint32_t)(my_tiles - 1) & 1u);
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
static int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Shared-memory geometry of one launch with `ncl` clusters of `cl` CTAs;
// false when the shape does not fit.
static bool small_geometry(const DeltaArgs &p, int R16, int cl, int ncl, SmGeom &g) {
    const int M = p.M_rows;
    if (M < 1 || M > kSmMaxRows || cl < 1 || ncl < 1) return false;
    if (p.d_in % (16 * cl)) return false;
    g = SmGeom{};
    g.CL = cl;
    g.KC = p.d_in / cl;
    const int nv = p.d_out_total / 8;
    g.NCmax = ((nv + cl - 1) / cl) * 8;
    int max_stride = 0;
    for (int t = 0; t < p.n_slices; ++t) max_stride = std::max(max_stride, (int)p.slices[t].stride_n);
    g.HS = pow2_at_least(std::max(64, 2 * M));
    g.tcap = (M + ncl - 1) / ncl + 1;
    if (cl > kSmMaxCluster) return false;
    for (int qq = 0; qq <= cl; ++qq) g.ncol0[qq] = (int)((int64_t)nv * qq / cl) * 8;
    for (int qq = 0; qq < cl; ++qq) {
        PieceTab &t = g.pt[qq];
        uint32_t run = 0;
        for (int u = 0; u < LORA_MAX_SLICES; ++u) {
            int cb = 0, ce = 0, str = 0, go = 0;
            if (u < p.n_slices) {
                const SliceDesc &sl = p.slices[u];
                cb = std::max(g.ncol0[qq], sl.col_begin);
                ce = std::min(g.ncol0[qq + 1], sl.col_begin + sl.d_out);
                str = (int)sl.stride_n * 2;
                go = sl.y_col - sl.col_begin;
            }
            t.cb[u] = cb;
            t.ce[u] = ce;
            t.str[u] = str;
            t.go[u] = go;
            t.off[u] = run;
            if (cb < ce) run += (uint32_t)(ce - cb) * (uint32_t)str;
        }
    }
    g.ncl_magic = (uint32_t)((0x100000000ull + (uint64_t)ncl - 1) / (uint64_t)ncl);
    // A row pitch: (pitch / 4) = 8 mod 32 words, so the 8-byte fragment
    // reads of rows g = 0..3 by lanes t = 0..3 (one half-warp) fall in
    // distinct banks; a multiple of 16 bytes for the 16-byte copies
    g.apitch = g.KC * 2 + 4 * (((8 - g.KC / 2) % 32 + 32) % 32);
    g.ypitch = g.NCmax * 2 + 16;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 127) & ~size_t(127);
        return (int)at;
    };
    g.off_bars = take(8 * 4);
    g.off_scan = take(64 * 4);
    g.off_tl = take((size_t)g.tcap * sizeof(TileRec));
    g.off_rows = take(kSmRT * 4);
    g.off_recv = take((size_t)2 * cl * 16 * R16 * 4);
    g.off_hbf = take((size_t)16 * (R16 + 8) * 2);
    // region A: the hash table (key, first, count), the A rows, the warps'
    // partial h, one after the other
    g.off_A = take(std::max({(size_t)R16 * g.apitch, (size_t)3 * g.HS * 4, (size_t)kSmWarps * 16 * (R16 + 4) * 4}));
    g.off_y = take((size_t)kSmRT * g.ypitch);
    // + 32 bytes: the expand's B fragment reads cover 16 rank columns and may
    // reach past a short last B row (those values are masked to zero)
    g.off_B = take((size_t)g.NCmax * max_stride * 2 + 32);
    g.total = (int)o;
    return g.total <= 227 * 1024;
}

static int small_cluster_size(int d_in, int d_out) {
    const int d = d_in > d_out ? d_in : d_out;
    if (d < 1024) return 1;
    if (d < 2048) return 2;
    if (d <= 8192) return 4;
    return 8;
}

// The rank block of a launch: r_max rounded up to 16, 32 or 64.
static int small_r16(int r_max) { return r_max <= 16 ? 16 : (r_max <= 32 ? 32 : 64); }

namespace {
struct SmallResidency {
    const void *fn[16] = {};
    int dev[16] = {}, cl[16] = {}, smem[16] = {}, val[16] = {};
    int n = 0;
};
}  // namespace

template <int R16>
static cudaError_t launch_small_t(const DeltaArgs &p, int cl, int sms, cudaStream_t stream, bool *taken) {
    auto kern = sgmv_small_kernel<R16>;
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (e != cudaSuccess) return e;
    // One SM stays free for the next prepare of the stream, which then runs
    // beside this grid.  The cluster count fixes the tile records per CTA
    // (shared memory); it is checked against residency below.
    int ncl = std::max(1, std::min((sms - 1) / cl, p.M_rows));
    SmGeom g;
    if (!small_geometry(p, R16, cl, ncl, g)) {
        *taken = false;
        return cudaSuccess;
    }
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSmThreads);
    cfg.dynamicSmemBytes = g.total;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    static SmallResidency cache;
    int dev = 0;
    cudaGetDevice(&dev);
    int max_clusters = -1;
    for (int i = 0; i < cache.n; ++i)
        if (cache.fn[i] == (const void *)kern && cache.dev[i] == dev && cache.cl[i] == cl && cache.smem[i] == g.total)
            max_clusters = cache.val[i];
    if (max_clusters < 0) {
        cfg.gridDim = dim3(cl);
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active <= 0) {
            cudaGetLastError();
            active = sms / cl;
        }
        max_clusters = active;
        if (cache.n < 16) {
            cache.fn[cache.n] = (const void *)kern;
            cache.dev[cache.n] = dev;
            cache.cl[cache.n] = cl;
            cache.smem[cache.n] = g.total;
            cache.val[cache.n] = active;
            ++cache.n;
        }
    }
    if (ncl > max_clusters) {
        // fewer clusters fit at once: more tile records per CTA
        ncl = max_clusters;
        if (!small_geometry(p, R16, cl, ncl, g)) {
            *taken = false;
            return cudaSuccess;
        }
        cfg.dynamicSmemBytes = g.total;
    }
    *taken = true;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(ncl * cl);
    return cudaLaunchKernelEx(&cfg, kern, p, g);
}

// Launches the small-batch kernel when the shape is one it takes; returns
// false (launching nothing) otherwise.
bool try_launch_small(const DeltaArgs &p, int sms, cudaStream_t stream, cudaError_t *err) {
    if (p.r_max > 64 || p.ids == nullptr || p.M_rows < 1 || p.M_rows > kSmMaxRows) return false;
    const int R16 = small_r16(p.r_max);
    for (int cl = small_cluster_size(p.d_in, p.d_out_total); cl >= 1; cl >>= 1) {
        if (p.d_in % (16 * cl)) continue;
        bool taken = false;
        if (R16 == 16) *err = launch_small_t<16>(p, cl, sms, stream, &taken);
        else if (R16 == 32) *err = launch_small_t<32>(p, cl, sms, stream, &taken);
        else *err = launch_small_t<64>(p, cl, sms, stream, &taken);
        if (taken || *err != cudaSuccess) return true;
    }
    return false;
}

}  // namespace lora
