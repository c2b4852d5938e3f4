// sgmv_stream.cu -- fused SGMV kernel for batches of up to kSmMaxRows rows:
// the rows are grouped on chip from the ids, the data of each tile streams
// through a ring of shared-memory stages in chunks (the next tile's chunks are
// requested while the current one is computed), and h is reduced across a
// thread-block cluster by one-way pushes into the peers' shared memory.
//
// What it computes is the fused delta of one batch ("vLLM-Ascend LoRA"
// article, section 3.3: the rows of one adapter are gathered, tmp = rows .
// A^T, delta = (tmp * scale) . B^T is added into the output; the adapter's
// A/B move once and serve every row of the group):
//     y[i] += s_a * (x[i] . A[a]^T) . B[a]^T      for every row i with id a.
//
// Grouping.  Every CTA reads the ids and groups the rows itself, in the order
// in which each adapter first occurs ("III.Punica: Multi-Tenant LoRA
// Serving", section 代码: the regrouping of tokens by adapter): a hash table
// in shared memory gives every adapter its first row and its row count, and
// one block scan over the rows, of "this row is its adapter's first" packed
// with the adapter's tile count, gives every group its number and its first
// tile.  A group of more than kSmRT rows is cut into near-equal tiles of at
// most kSmRT rows; tile t belongs to cluster t mod C.  The grouping depends
// only on the ids, so every CTA builds the same tiles, and the first row of
// each group writes the records of its tiles that fall to this CTA's cluster.
// When the call splits by group size, groups of at least the threshold with a
// tensor-core rank get no tiles here (the tensor-core kernel takes them).
//
// Work of a tile.  CTA q of a cluster of CL owns
//   - the K slice q of d_in for the shrink (x rows and A rows of that slice),
//   - the N slice q of d_out for the expand (B rows and y rows of that slice),
// so every byte of x, A, B and y of a tile is read once.  The K slice is
// cut into nK chunks of kc columns (x and A rows), the N slice into nN chunks
// of nc columns (y and B rows); the chunks of all the CTA's tiles form one
// sequence that flows through D shared-memory stages, D - 1 of them in flight
// while one is computed.  A's rows are only the adapter's r ranks, and of
// each B row only the pieces that hold its r ranks are copied, so an adapter
// of a padded pool moves its own rank's bytes (section 3.4 of the same
// article: padding to the largest rank wastes traffic).
//
// Data movement.  Every load is a TMA copy, issued by a producer warp that
// runs ahead of the sixteen consumer warps (a stage is refilled once all of
// them have released it) and completing on the stage's mbarrier: the rank
// rows of A by a 3-D tensor map in 64-column x 16-rank boxes (128-byte
// swizzle), the rank columns of B by a 3-D tensor map in w-rank x 128-column
// boxes, w the adapter's rank rounded up to 16, 32 or 64 (rows of 2w bytes,
// swizzled for w >= 32), and the gathered x and y rows by one bulk copy
// each.  The copy engine's cost grows with the number of rows a box has, not
// with their width, so boxes are a few KB with rows as wide as the adapter's
// rank allows; and the consumers never wait on a copy being issued.  The
// load/store unit stays free for the shared-memory traffic of the compute
// (16-byte cp.async copies in flight slow every shared-memory access behind
// them).  The weights (A and B) depend only on the adapter, so those of the
// first chunks are requested before the kernel waits on the previous grid
// in the stream (programmatic dependent launch), and so are the rows of
// every tile; x and y are requested after that wait.  y + delta leaves by
// 16-byte stores.
//
// Compute.  Shrink: warp-level bf16 tensor-core tiles (16 x 8 x 16, fp32
// accumulators in registers across the K chunks; operands by ldmatrix from
// rows padded by 16 bytes, so the eight rows of a fragment fall in eight bank
// groups).  The warps split the K steps of each chunk (and, for ranks above
// 16, the 16-column rank blocks); their partials are summed in warp order.
// The CTA's partial h is pushed to every CTA of the cluster (st.async,
// completing on the receiver's mbarrier: no cluster barrier per tile), and
// each CTA sums the CL partials in rank order, so every CTA holds the same h.
// h is scaled once, masked to the adapter's rank and to the tile's rows, and
// rounded once to bf16.  Expand: the same tiles with h as the A operand and
// B rows as the B operand, the K slots permuted so that B fragments come by
// 64-bit loads (the 32-byte rank blocks of a B row are XOR-swizzled across
// rows, so the eight rows of a fragment hit distinct bank groups); y + delta
// is formed in fp32, rounded once to bf16 and written back into the y rows
// of the stage, which then leave by 16-byte stores.  The rank mask is exact:
// h columns past the rank are zero and B fragments past the rank are zeroed
// in registers, so padding (even NaN) and stale shared memory never enter a
// result.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cstring>

#include "common.cuh"

namespace lora {
namespace stream {

constexpr int kSmThreads = 512;                       // consumer threads (16 warps): grouping and compute
constexpr int kSmWarps = kSmThreads / 32;
constexpr int kStThreads = kSmThreads + 32;           // + one producer warp that issues every copy
constexpr int kSmMaxRPT = 4;                          // rows per thread at most
constexpr int kSmMaxRows = kSmThreads * kSmMaxRPT;    // rows a batch may have for this kernel
constexpr int kSmRT = 16;                             // rows per tile: one 16-row MMA tile
constexpr int kSmMaxCluster = 8;
constexpr int kSmMaxHashBytes = 48 * 1024;            // hash table (key, first row, count) at most

constexpr int kSmMaxNChunks = 12;                     // N chunks per CTA at most

// One N chunk of a CTA: output slice t, columns [cb, ce) of the
// concatenated output (within slice t).
struct NChunk {
    int t, cb, ce;
};

struct SmGeom {
    int CL;              // CTAs per cluster
    int KC;              // shrink columns per CTA
    int RPT;             // rows per thread (1, 2, 4 or 8)
    int D;               // stages of the chunk ring
    int SB;              // bytes per stage (a multiple of 1024)
    int kc, nK, natoms;  // K chunk columns (a multiple of 64), K chunks per tile, 64-column A atoms per rank block
    int xpitch, offA;    // bytes per x row in a K stage (kc * 2 + 16); A atoms in a K stage
    int ypitch, offB;    // bytes per y row in an N stage; B planes in an N stage
    int ncp;             // rows per B plane (a multiple of 128, >= the widest N chunk)
    int stacked;         // 1: every slice has its own A; their rank blocks are stacked in one shrink
    int rs, nrb_s;       // ranks per slice block when stacked (16, 32 or 64) and its 16-rank blocks
    int HS;              // hash slots (power of two, >= 2 distinct adapters)
    int tcap;            // tile records per CTA
    uint32_t ncl_magic;  // ceil(2^32 / clusters): x / clusters = umulhi(x, magic) for x < 2^16
    int nN[kSmMaxCluster];                  // N chunks of cluster rank q
    NChunk nck[kSmMaxCluster][kSmMaxNChunks];  // the N chunks of cluster rank q
    int off_bars, off_key, off_first, off_cnt, off_scan, off_tl, off_rows, off_ids, off_recv, off_hbf,
        off_stage, total;
};

// Tensor maps: A pool {d_in, r_max, n_adapters} in 64 x 16 boxes (128-byte
// swizzle); B pool of slice t {r_max, d_out, n_adapters} in (16 << wi) x 128
// boxes, wi = 0, 1, 2 (no swizzle, 64-byte and 128-byte swizzle), for the
// widths up to r_max.
struct SmMaps {
    CUtensorMap a[LORA_MAX_SLICES];  // per output slice (all the call's A pool unless stacked)
    CUtensorMap b[LORA_MAX_SLICES][3];
};

// One tile of this cluster: adapter, rank, first and last row (exclusive)
// inside its group's rows, scale.
struct TileRec {
    int a, r, lo, hi;
    float sc;
    int pad[3];
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
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
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
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
__device__ __forceinline__ void add4(float4 &v, const float4 &w) {
    v.x += w.x;
    v.y += w.y;
    v.z += w.z;
    v.w += w.w;
}
__device__ __forceinline__ void tma_3d(uint32_t sdst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(sdst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async_cta() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
// Barrier of the consumer warps only (the producer warp runs its own loop).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kSmThreads) : "memory"); }
__device__ __forceinline__ void mbar_arrive1(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// The expand of the 8-column tiles nt0, nt0 + 16, ... (NB of them) of a
// warp: B words and y words first, then the products, then y + delta in
// fp32, rounded once, back into the y rows of the stage.
__device__ __forceinline__ uint2 ldsm_x2_trans(uint32_t addr) {
    uint2 r;
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n" : "=r"(r.x), "=r"(r.y) : "r"(addr));
    return r;
}
// RM false: B rows of 2w bytes (one output column each), the thread's eight
// bytes of K step ks at boff[ks] (rsh = log2 of the row bytes).  RM true:
// rank-major B in 64-column atoms of w rank rows x 128 bytes (128-byte
// swizzle), read by ldmatrix.trans: lane l < 16 addresses rank row 16 ks + l
// (sBa = the atoms' base + l * 128, boff[ks] = 16 ks * 128, rsh = log2 of an
// atom's bytes), chunk (column tile & 7) ^ (l & 7).
template <int KS, int NB, bool RM>
__device__ __forceinline__ void expand_tiles(int nt0, int np, uint32_t sBa, const uint32_t (&boff)[KS], uint32_t rsh, uint32_t yr0,
                                             uint32_t yr1, bool row0, bool row1, const uint32_t (&hf)[KS][4],
                                             const uint32_t (&bm0)[KS], const uint32_t (&bm1)[KS], uint32_t lsw) {
    uint2 bw[NB][KS];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int nt = nt0 + b * 16;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (RM)
                bw[b][ks] = ks < np ? ldsm_x2_trans(sBa + boff[ks] + ((uint32_t)(nt >> 3) << rsh) +
                                                   ((((uint32_t)nt & 7u) ^ lsw) << 4))
                                    : make_uint2(0u, 0u);
            else
                bw[b][ks] = ks < np ? lds64(sBa + boff[ks] + ((uint32_t)nt << (rsh + 3))) : make_uint2(0u, 0u);
        }
    }
    uint32_t y0[NB], y1[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const uint32_t yo = (uint32_t)((nt0 + b * 16) * 16);
        y0[b] = row0 ? lds32(yr0 + yo) : 0u;
        y1[b] = row1 ? lds32(yr1 + yo) : 0u;
    }
    float d[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int i = 0; i < 4; ++i) d[b][i] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            if (ks < np) mma_bf16_16816(d[b], hf[ks], bw[b][ks].x & bm0[ks], bw[b][ks].y & bm1[ks]);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const uint32_t yo = (uint32_t)((nt0 + b * 16) * 16);
        if (row0)
            sts32(yr0 + yo, bf16x2_bits(__uint_as_float(y0[b] << 16) + d[b][0],
                                        __uint_as_float(y0[b] & 0xFFFF0000u) + d[b][1]));
        if (row1)
            sts32(yr1 + yo, bf16x2_bits(__uint_as_float(y1[b] << 16) + d[b][2],
                                        __uint_as_float(y1[b] & 0xFFFF0000u) + d[b][3]));
    }
}

template <int R16>
__global__ void __launch_bounds__(kStThreads, 1)
    sgmv_stream_kernel(const __grid_constant__ DeltaArgs p, const __grid_constant__ SmGeom g,
                      const __grid_constant__ SmMaps m) {
    constexpr int KS = R16 / 16;  // K steps of the expand (rank blocks of the shrink)
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (the swizzled A atoms need it)
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *recv_bar = reinterpret_cast<uint64_t *>(smem + g.off_bars);  // [2] partial h received
    uint64_t *full = recv_bar + 2;                                         // [D] stage landed
    uint64_t *empty = full + 8;                                            // [D] stage released by the consumers
    int32_t *key = reinterpret_cast<int32_t *>(smem + g.off_key);
    int32_t *first = reinterpret_cast<int32_t *>(smem + g.off_first);
    int32_t *cnt = reinterpret_cast<int32_t *>(smem + g.off_cnt);
    int32_t *wsum = reinterpret_cast<int32_t *>(smem + g.off_scan);  // [kSmWarps]
    int32_t *wsum2 = wsum + 32;                                         // [kSmWarps]
    TileRec *tl = reinterpret_cast<TileRec *>(smem + g.off_tl);        // [tcap]
    int32_t *rows_all = reinterpret_cast<int32_t *>(smem + g.off_rows);  // [tcap][kSmRT]: rows of tile e
    int32_t *ids_s = reinterpret_cast<int32_t *>(smem + g.off_ids);    // [512 RPT]: valid id or -1 per row
    float *recv = reinterpret_cast<float *>(smem + g.off_recv);        // [2][CL][16][R16]
    unsigned char *hbf = smem + g.off_hbf;                              // [16][R16 + 8] bf16
    unsigned char *stages = smem + g.off_stage;                         // [D][SB]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int CL = g.CL, D = g.D, RPT = g.RPT;
    const uint32_t q = cluster_ctarank(), cid = cluster_id_x(), ncl = nclusters_x();
    const int M = p.M_rows, n = p.n_adapters;
    const int HS = g.HS;
    const int hpitch = (R16 + 8) * 2;

    // Nothing this grid writes is read by the next one before its own wait,
    // and this grid reads before its wait only what no grid of the stream
    // writes (see griddep_launch_dependents): the next grid may start at once.
    // A tensor-core grid launched after this one for the same call reads the
    // batch metadata at its start: then this grid triggers only after its
    // wait on prepare.
    if (!p.trigger_after_wait) griddep_launch_dependents();
    if (warp == kSmWarps) {
        // the producer's tensor maps, one per lane: A per stacked slice, B
        // per slice and box width
        const CUtensorMap *mp = nullptr;
        if (lane < (g.stacked ? p.n_slices : 1)) mp = &m.a[lane];
        else if (lane >= 4 && lane < 4 + 3 * p.n_slices) {
            const int t = (lane - 4) / 3, wi = (lane - 4) - 3 * t;
            if ((16 << wi) <= p.r_max) mp = &m.b[t][wi];
        }
        if (mp) prefetch_tensormap(mp);
    }
    // ids written by the grid before (an updated batch): read after the wait
    if (p.ids_after_wait) griddep_wait();

    // ---- phase 0: ids (rows tid * RPT .. tid * RPT + RPT - 1), the adapters'
    // ranks and scales, and an empty hash table.  Everything read before the
    // wait (ids, ranks, scales and later the weights) is fixed before the
    // previous grid in the stream started (header contract).
    int idr[kSmMaxRPT], rkr[kSmMaxRPT];
    float scr[kSmMaxRPT];
#pragma unroll
    for (int k = 0; k < kSmMaxRPT; ++k) {
        const int i = tid * RPT + k;
        idr[k] = (k < RPT && i < M) ? __ldcg(p.ids + i) : -1;
    }
    if (tid == 0) {
        mbar_init(&recv_bar[0], 1);
        mbar_init(&recv_bar[1], 1);
        for (int s2 = 0; s2 < g.D; ++s2) {
            mbar_init(&full[s2], 1);
            mbar_init(&empty[s2], kSmWarps);
        }
        fence_mbar_init();
    }
    for (int s = tid; s < HS && tid < kSmThreads; s += kSmThreads) {
        key[s] = -1;
        first[s] = INT_MAX;
        cnt[s] = 0;
    }
#pragma unroll
    for (int k = 0; k < kSmMaxRPT; ++k) {
        const bool v = idr[k] >= 0 && idr[k] < n;
        if (!v) idr[k] = -1;
        rkr[k] = v && p.ranks ? __ldcg(p.ranks + idr[k]) : p.r_max;
        scr[k] = v && p.adapter_scale ? __ldcg(p.adapter_scale + idr[k]) : p.scale;
        if (k < RPT && tid < kSmThreads) ids_s[tid * RPT + k] = idr[k];
    }
    __syncthreads();
    cluster_arrive_relaxed();  // the barriers exist before any peer pushes into them

    // ---- phase 1: one hash slot per adapter with its first row and count.
    int slot[kSmMaxRPT];
#pragma unroll
    for (int k = 0; k < kSmMaxRPT; ++k) {
        slot[k] = -1;
        if (idr[k] >= 0) {
            const int a = idr[k];
            int s = (int)hash_slot(a, HS);
            for (;;) {  // fewer distinct keys than slots: a free slot always exists
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
    int ntile[kSmMaxRPT], bad = 0, v = 0;
    bool lead[kSmMaxRPT];
#pragma unroll
    for (int k = 0; k < kSmMaxRPT; ++k) {
        ntile[k] = 0;
        lead[k] = false;
        if (slot[k] >= 0 && first[slot[k]] == tid * RPT + k) {
            lead[k] = true;
            const int r = rkr[k];
            // groups of at least max_len rows with a tensor-core rank belong to
            // the tensor-core kernel when the call splits (prepare's rule)
            const bool to_tc = p.split_tc && cnt[slot[k]] >= p.max_len && tc_rank_ok(r);
            if (r < 0 || r > p.r_max) bad = 1;
            else if (r > 0 && !to_tc) ntile[k] = (cnt[slot[k]] + kSmRT - 1) / kSmRT;
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
        const int wv = lane < kSmWarps ? wsum[lane] : 0;
        int ws = wv;
#pragma unroll
        for (int o = 1; o < kSmWarps; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += t;
        }
        base = __shfl_sync(0xffffffffu, ws - wv, warp);
        total = __shfl_sync(0xffffffffu, ws, kSmWarps - 1);
    }
    const int T = total >> 16;  // tiles of the batch
    {
        int run = base + incl - v;  // exclusive prefix of this thread's first row
#pragma unroll
        for (int k = 0; k < kSmMaxRPT; ++k) {
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
    const int bad_rank = __syncthreads_or(bad);
    const int my_tiles =
        (int)cid < T ? min((int)__umulhi((uint32_t)(T - 1 - (int)cid), g.ncl_magic) + 1, g.tcap) : 0;

    const int k0 = (int)q * g.KC;
    const NChunk *nck = g.nck[q];  // launch parameters
    const int nch = g.nK + g.nN[q];  // chunks per tile (>= D - 1)
    const int J = my_tiles * nch;

    // Rows [lo, hi) of adapter a's group, in ascending row order, into dst
    // (consumer warps only).
    auto find_rows = [&](int a, int lo, int hi, int32_t *dst) {
        int idv[kSmMaxRPT];
        const int rb = tid * RPT;
        if (RPT == 4) {
            const int4 u0 = *reinterpret_cast<const int4 *>(ids_s + rb);
            idv[0] = u0.x; idv[1] = u0.y; idv[2] = u0.z; idv[3] = u0.w;
        } else if (RPT == 2) {
            const int2 u0 = *reinterpret_cast<const int2 *>(ids_s + rb);
            idv[0] = u0.x; idv[1] = u0.y;
        } else {
            idv[0] = ids_s[rb];
        }
        int mine = 0;
#pragma unroll
        for (int k = 0; k < kSmMaxRPT; ++k)
            if (k < RPT && idv[k] == a) ++mine;
        int inc = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        if (lane == 31) wsum2[warp] = inc;
        consumers_sync();
        int b;
        {
            const int wv = lane < kSmWarps ? wsum2[lane] : 0;
            int ws = wv;
#pragma unroll
            for (int o = 1; o < kSmWarps; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, ws, o);
                if (lane >= o) ws += t;
            }
            b = __shfl_sync(0xffffffffu, ws - wv, warp);
        }
        if (mine) {
            int pos = b + inc - mine;
#pragma unroll
            for (int k = 0; k < kSmMaxRPT; ++k) {
                if (k < RPT && idv[k] == a) {
                    if (pos >= lo && pos < hi) dst[pos - lo] = rb + k;
                    ++pos;
                }
            }
        }
        consumers_sync();
    };

    // The copies of chunk (e, c) into stage st: the weights (A or B boxes)
    // and / or the activations (x or y rows), spread over the lanes of the
    // producer warp, all completing on full[st].  The call with the weights
    // sets the stage's expected bytes (weights and activations).
    auto issue = [&](int e, int c, int st, bool w, bool act) {
        if (e >= my_tiles) return;
        const TileRec ti = tl[e];
        const uint32_t sb = smem_u32(stages) + (uint32_t)(st * g.SB);
        uint64_t *fb = &full[st];
        const int R = ti.hi - ti.lo;
        const int32_t *rws = rows_all + e * kSmRT;
        const int wi = ti.r <= 16 ? 0 : (ti.r <= 32 ? 1 : 2);  // B box of 16 << wi ranks
        if (c < g.nK) {
            const int kb = k0 + c * g.kc;
            const int nbl = ((ti.r + 15) >> 4) * g.natoms;         // 16-rank blocks x atoms of one slice
            const int nA = (g.stacked ? p.n_slices : 1) * nbl;
            if (w && lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(nA * 2048 + R * g.kc * 2));
            {
                // A: box (columns 64 at .., ranks 16 pb ..) of slice t's pool
                // -> atom (t nrb_s + pb) natoms + at (stacked), pb natoms + at
                if (w)
                    for (int i = lane; i < nA; i += 32) {
                        const int t = i / nbl, rem = i - t * nbl;
                        const int pb = rem / g.natoms, at = rem - pb * g.natoms;
                        tma_3d(sb + g.offA + (uint32_t)(((t * g.nrb_s + pb) * g.natoms + at) * 2048), &m.a[t],
                               kb + at * 64, pb * 16, ti.a, fb);
                    }
                // x rows
                if (act)
                    for (int i = lane; i < R; i += 32)
                        bulk_g2s(stages + st * g.SB + i * g.xpitch,
                                 static_cast<const __nv_bfloat16 *>(p.x) + (int64_t)rws[i] * p.ldx + kb,
                                 (uint32_t)(g.kc * 2), fb);
            }
        } else {
            const NChunk ck = nck[c - g.nK];
            const SliceDesc &sl = p.slices[ck.t];
            const int ncols = ck.ce - ck.cb;
            // B boxes of 128 columns x (16 << wi) ranks (rank-contiguous
            // rows), or 64 columns x (16 << wi) rank rows (rank-major)
            const int cw = p.b_rank_major ? 64 : 128;
            const int nbx = (ncols + cw - 1) / cw;
            const uint32_t bb = (uint32_t)cw * (32u << wi);  // bytes per box
            if (w && lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(nbx * bb + R * ncols * 2));
            {
                if (w)
                    for (int bx = lane; bx < nbx; bx += 32) {
                        if (p.b_rank_major)
                            tma_3d(sb + g.offB + (uint32_t)bx * bb, &m.b[ck.t][wi], ck.cb - sl.col_begin + bx * cw, 0,
                                   ti.a, fb);
                        else
                            tma_3d(sb + g.offB + (uint32_t)bx * bb, &m.b[ck.t][wi], 0, ck.cb - sl.col_begin + bx * cw,
                                   ti.a, fb);
                    }
                // y rows
                if (act)
                    for (int i = lane; i < R; i += 32)
                        bulk_g2s(stages + st * g.SB + i * g.ypitch,
                                 static_cast<const __nv_bfloat16 *>(p.y) + (int64_t)rws[i] * p.ldy + sl.y_col +
                                     (ck.cb - sl.col_begin),
                                 (uint32_t)(ncols * 2), fb);
            }
        }
    };

    // ---- every tile's rows, found before the wait on the previous grid (the
    // ids are fixed before it started); then the producer warp streams the
    // chunks and the consumer warps compute them.
    if (warp < kSmWarps)
        for (int e = 0; e < my_tiles; ++e) {
            const TileRec t0 = tl[e];
            find_rows(t0.a, t0.lo, t0.hi, rows_all + e * kSmRT);
        }
    __syncthreads();
    bool ok = true;
    if (warp == kSmWarps) {
        // ---- producer: the weights of the first D chunks (every stage is
        // free) before the wait, then their activations, then each further
        // chunk once the consumers have released its stage
        const int npre = min(D, J);
        int pe = 0, pc = 0;
        for (int j = 0; j < npre; ++j) {
            issue(pe, pc, j, true, false);
            if (++pc == nch) {
                pc = 0;
                ++pe;
            }
        }
        griddep_wait();
        pe = 0;
        pc = 0;
        for (int j = 0; j < npre; ++j) {
            issue(pe, pc, j, false, true);
            if (++pc == nch) {
                pc = 0;
                ++pe;
            }
        }
        int pst = npre % D, pu = npre / D;  // stage of chunk j and its use
        for (int j = npre; j < J; ++j) {
            if (lane == 0 && !mbar_wait(&empty[pst], (uint32_t)(pu - 1) & 1u)) ok = false;
            __syncwarp();
            issue(pe, pc, pst, true, true);
            if (++pc == nch) {
                pc = 0;
                ++pe;
            }
            if (++pst == D) {
                pst = 0;
                ++pu;
            }
        }
        cluster_wait_acquire();
    } else {
    griddep_wait();
    if (p.trigger_after_wait) griddep_launch_dependents();
    if (bad_rank && blockIdx.x == 0 && tid == 0) raise_deverr(p.counts, LORA_DEVERR_RANK);
    cluster_wait_acquire();

    const int g_ = lane >> 2, t4 = lane & 3;
    // tile state
    TileRec ti{};
    int r = 0, R = 0, r16a = 16, np = 1, npe = 1;
    float acc[2][2][4];
    uint32_t hf[KS][4], bm0[KS], bm1[KS];
    int st = 0;                        // stage of chunk j
    uint32_t ph = 0;                   // phase parity of its barrier
    int e = 0, c = 0;                  // chunk j = (e, c)
    for (int j = 0; j < J; ++j) {
        // chunk j has landed (one thread waits; the consumer barrier passes
        // its view of the copies on)
        if (tid == 0 && !mbar_wait(&full[st], ph)) ok = false;
        consumers_sync();
        if (c == 0) {
            ti = tl[e];
            r = ti.r;
            R = ti.hi - ti.lo;
            // rank blocks of the shrink (all slices' when stacked) and K
            // steps of the expand
            np = g.stacked ? p.n_slices * g.nrb_s : (r + 15) >> 4;
            r16a = np * 16;
            npe = (r + 15) >> 4;
            if (tid == 0) mbar_arrive_expect_tx(&recv_bar[e & 1], (uint32_t)(CL * 16 * r16a * 4));
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[u][t][i] = 0.f;
        }
        unsigned char *sb = stages + st * g.SB;
        const int buf = e & 1;
        if (c < g.nK) {
            // ---- shrink over this K chunk: h^T += A . x^T on warp-level
            // tensor-core tiles (M = the 16 ranks of a rank block, N = 8
            // rows, K = 16 columns): warp w takes rank block w % np and the
            // K steps w / np, w / np + kw, ...
            const int kw = kSmWarps / np;
            const int my_pb = warp % np, my_kq = warp / np;
            const bool two = R > 8;  // a second 8-row tile
            if (my_kq < kw) {
                const int nks = g.kc >> 4;
                // A operand: rank (lane & 15) of block my_pb, K half lane >> 4:
                // atom (my_pb, ks / 4), row lane & 15, 16-byte chunk
                // (2 (ks % 4) + half) ^ (lane & 7) (128-byte swizzle);
                // B operand: x rows (lane & 7) (+ 8 for lanes 16-31), K half (lane >> 3) & 1
                const int ra = lane & 7, hs = lane >> 4;
                const uint32_t ab =
                    smem_u32(sb) + g.offA + (uint32_t)(my_pb * g.natoms * 2048 + (lane & 15) * 128);
                const uint32_t xb = smem_u32(sb) + ((lane & 7) + ((lane >> 4) << 3)) * g.xpitch + ((lane >> 3) & 1) * 16;
                int u = 0;
#pragma unroll 4
                for (int ks = my_kq; ks < nks; ks += kw) {
                    uint32_t af[4], xf[4];
                    ldsm_x4(af, ab + (ks >> 2) * 2048 + (((((ks & 3) << 1) | hs) ^ ra) << 4));
                    if (two) ldsm_x4(xf, xb + ks * 32);
                    else ldsm_x2(xf, xb + ks * 32);
                    if (u == 0) {
                        mma_bf16_16816(acc[0][0], af, xf[0], xf[1]);
                        if (two) mma_bf16_16816(acc[1][0], af, xf[2], xf[3]);
                    } else {
                        mma_bf16_16816(acc[0][1], af, xf[0], xf[1]);
                        if (two) mma_bf16_16816(acc[1][1], af, xf[2], xf[3]);
                    }
                    u ^= 1;
                }
            }
            if (c == g.nK - 1) {
                // warp partial -> red[warp][row][rank in block] (row pitch 20
                // floats: the fragment's rows 2t and 2t+1 fall in distinct
                // banks), in this K stage, whose x and A every warp has read
                float *red = reinterpret_cast<float *>(sb);
                consumers_sync();
                if (my_kq < kw) {
                    const uint32_t rw = smem_u32(red) + (uint32_t)warp * (16 * 20 * 4);
#pragma unroll
                    for (int rt = 0; rt < 2; ++rt) {
                        if (rt == 0 || two) {
                            const uint32_t a0 = rw + ((rt * 8 + 2 * t4) * 20 + g_) * 4;
                            sts32(a0, __float_as_uint(acc[rt][0][0] + acc[rt][1][0]));
                            sts32(a0 + 20 * 4, __float_as_uint(acc[rt][0][1] + acc[rt][1][1]));
                            sts32(a0 + 8 * 4, __float_as_uint(acc[rt][0][2] + acc[rt][1][2]));
                            sts32(a0 + 28 * 4, __float_as_uint(acc[rt][0][3] + acc[rt][1][3]));
                        }
                    }
                }
                fence_proxy_async_cta();  // writes into the stage come before the producer's next copies
                consumers_sync();
                // CTA partial: the kw partials of each rank block summed in
                // two levels (pairs kq, kq + 8 by all threads in place, then
                // the eight sums in order), pushed to every CTA of the
                // cluster: slot q of their receive buffer.  Rows of a missing
                // second 8-row tile hold leftovers; h masks them.
                const int nel4 = 4 * r16a;  // float4 entries of a 16 x r16a block
                const int rq = r16a / 4;    // float4 entries per row
                float *rv = recv + (size_t)buf * CL * 16 * R16;
                const uint32_t redb = smem_u32(red);
                if (kw > 8) {
                    // kw == 16 (np == 1): warp partials kq and kq + 8
                    const int e4 = tid & 63, part = tid >> 6;  // 64 float4 x 8 parts
                    const uint32_t a = redb + ((uint32_t)part * 320 + (e4 >> 2) * 20 + (e4 & 3) * 4) * 4;
                    const uint4 x4 = lds128(a), y4 = lds128(a + 8 * 320 * 4);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(a),
                                 "f"(__uint_as_float(x4.x) + __uint_as_float(y4.x)),
                                 "f"(__uint_as_float(x4.y) + __uint_as_float(y4.y)),
                                 "f"(__uint_as_float(x4.z) + __uint_as_float(y4.z)),
                                 "f"(__uint_as_float(x4.w) + __uint_as_float(y4.w))
                                 : "memory");
                    fence_proxy_async_cta();
                    consumers_sync();
                }
                if (tid < nel4) {
                    const int row = tid / rq, col = (tid - row * rq) * 4;
                    const int pb = col >> 4, cl = col & 15;
                    const int kn = kw > 8 ? 8 : kw;
                    uint4 pv[8];
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq)
                        pv[kq] = kq < kn ? lds128(redb + ((uint32_t)(kq * np + pb) * 320 + row * 20 + cl) * 4)
                                         : make_uint4(0u, 0u, 0u, 0u);
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq)
                        add4(s4, make_float4(__uint_as_float(pv[kq].x), __uint_as_float(pv[kq].y),
                                             __uint_as_float(pv[kq].z), __uint_as_float(pv[kq].w)));
                    const uint32_t la = smem_u32(rv + ((size_t)q * 16 + row) * R16 + col);
                    const uint32_t lb = smem_u32(&recv_bar[buf]);
                    for (int pr = 0; pr < CL; ++pr) st_async_f4(map_to_rank(la, pr), s4, map_to_rank(lb, pr));
                }
                // h = scale * sum of the CL partials (rank order), masked to
                // the tile's rows and the adapter's rank, rounded once to
                // bf16 (one thread waits for the partials; the next chunk's
                // block barrier publishes h)
                if (tid == 0 && !mbar_wait_cl(&recv_bar[buf], (uint32_t)(e >> 1) & 1u)) ok = false;
                consumers_sync();
                if (tid < nel4) {
                    const int row = tid / rq, col = (tid - row * rq) * 4;
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int pr = 0; pr < 8; ++pr)
                        if (pr < CL)
                            add4(s4, *reinterpret_cast<const float4 *>(rv + ((size_t)pr * 16 + row) * R16 + col));
                    const bool rok = row < R;
                    const float sc = ti.sc;
                    const int cin = g.stacked ? (col & (g.rs - 1)) : col;  // rank within its slice
                    const float h0 = rok && cin + 0 < r ? s4.x * sc : 0.f;
                    const float h1 = rok && cin + 1 < r ? s4.y * sc : 0.f;
                    const float h2 = rok && cin + 2 < r ? s4.z * sc : 0.f;
                    const float h3 = rok && cin + 3 < r ? s4.w * sc : 0.f;
                    *reinterpret_cast<uint2 *>(hbf + row * hpitch + col * 2) =
                        make_uint2(bf16x2_bits(h0, h1), bf16x2_bits(h2, h3));
                }
            }
        } else {
            // ---- expand over this N chunk: columns [lo, hi).  Inside each
            // 16-rank K step the MMA's K slots are permuted the same way for
            // h and B: slots 2t, 2t+1 hold ranks 4t, 4t+1 and slots 2t+8,
            // 2t+9 hold ranks 4t+2, 4t+3, so a thread's two B words (and two
            // h words) are eight contiguous bytes: one 64-bit load.
            const NChunk ck = nck[c - g.nK];
            if (c == g.nK || g.stacked) {
                // h of this chunk's slice: its block of columns when stacked
                const uint32_t hb = smem_u32(hbf) + g_ * hpitch + 8 * t4 + (g.stacked ? ck.t * g.rs * 2 : 0);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    if (p.b_rank_major) {
                        // natural K order (ldmatrix.trans gives B in it):
                        // slots 2t, 2t + 1 and 2t + 8, 2t + 9
                        const uint32_t hn = hb - 8 * t4 + 4 * t4 + ks * 32;
                        if (ks < npe) {
                            hf[ks][0] = lds32(hn);
                            hf[ks][1] = lds32(hn + 8 * hpitch);
                            hf[ks][2] = lds32(hn + 16);
                            hf[ks][3] = lds32(hn + 8 * hpitch + 16);
                        }
                        const int kk = ks * 16 + 2 * t4;
                        bm0[ks] = (kk + 1 < r ? 0xFFFF0000u : 0u) | (kk < r ? 0x0000FFFFu : 0u);
                        bm1[ks] = (kk + 9 < r ? 0xFFFF0000u : 0u) | (kk + 8 < r ? 0x0000FFFFu : 0u);
                    } else {
                        if (ks < npe) {
                            const uint2 lo2 = lds64(hb + ks * 32);
                            const uint2 hi2 = lds64(hb + 8 * hpitch + ks * 32);
                            hf[ks][0] = lo2.x;
                            hf[ks][1] = hi2.x;
                            hf[ks][2] = lo2.y;
                            hf[ks][3] = hi2.y;
                        }
                        const int kk = ks * 16 + 4 * t4;
                        bm0[ks] = (kk + 1 < r ? 0xFFFF0000u : 0u) | (kk < r ? 0x0000FFFFu : 0u);
                        bm1[ks] = (kk + 3 < r ? 0xFFFF0000u : 0u) | (kk + 2 < r ? 0x0000FFFFu : 0u);
                    }
                }
            }
            const int nnt = (ck.ce - ck.cb) >> 3;
            // B fragment of K step ks, 8-column tile nt: row n = 8 nt + g_
            // (2w bytes, w = 16 << wi ranks), 16-byte chunk 2 ks + t4 / 2
            // (swizzled: ^ g_ for w = 64, ^ (g_ / 2) % 4 for w = 32), bytes
            // 8 (t4 % 2) .. + 8: ranks 16 ks + 4 t4 ..; the eight rows of a
            // fragment fall in distinct bank groups
            const int wi = r <= 16 ? 0 : (r <= 32 ? 1 : 2);
            uint32_t rsh, sBa, lsw = 0;
            uint32_t boff[KS];
            if (p.b_rank_major) {
                // atoms of 64 columns x (16 << wi) rank rows of 128 bytes
                const uint32_t l = (uint32_t)(lane & 15);
                rsh = 11u + (uint32_t)wi;  // log2 bytes per atom
                sBa = smem_u32(sb) + g.offB + l * 128u;
                lsw = l & 7u;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) boff[ks] = (uint32_t)ks * 16u * 128u;
            } else {
                rsh = 5u + (uint32_t)wi;  // log2 bytes per B row
                const int swz = wi == 2 ? g_ : (wi == 1 ? (g_ >> 1) & 3 : 0);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) boff[ks] = ((((2 * ks + (t4 >> 1)) ^ swz) << 4) + (t4 & 1) * 8);
                sBa = smem_u32(sb) + g.offB + ((uint32_t)g_ << rsh);
            }
            const uint32_t yr0 = smem_u32(sb) + g_ * g.ypitch + 4 * t4;  // row g_, column 2 t4
            const uint32_t yr1 = yr0 + 8 * g.ypitch;                     // row g_ + 8
            const bool row0 = g_ < R, row1 = g_ + 8 < R;
            // warp w takes the 8-column tiles w, w + 16, ...: two at a time
            // (in flight together) while two remain, then one
            int nt = warp;
            if (p.b_rank_major) {
                for (; nt + kSmWarps < nnt; nt += 2 * kSmWarps)
                    expand_tiles<KS, 2, true>(nt, npe, sBa, boff, rsh, yr0, yr1, row0, row1, hf, bm0, bm1, lsw);
                for (; nt < nnt; nt += kSmWarps)
                    expand_tiles<KS, 1, true>(nt, npe, sBa, boff, rsh, yr0, yr1, row0, row1, hf, bm0, bm1, lsw);
            } else {
                for (; nt + kSmWarps < nnt; nt += 2 * kSmWarps)
                    expand_tiles<KS, 2, false>(nt, npe, sBa, boff, rsh, yr0, yr1, row0, row1, hf, bm0, bm1, lsw);
                for (; nt < nnt; nt += kSmWarps)
                    expand_tiles<KS, 1, false>(nt, npe, sBa, boff, rsh, yr0, yr1, row0, row1, hf, bm0, bm1, lsw);
            }
            fence_proxy_async_cta();  // the y + delta writes come before the producer's next copies
            consumers_sync();
            // the rows leave by 16-byte stores: warp w takes row w / hv and
            // the 8-column pieces w % hv, w % hv + hv, ... (hv = 2 when R <= 8)
            {
                const int hv = R > 8 ? 1 : 2;
                const int row = warp / hv, part = warp - row * hv;
                if (row < R) {
                    __nv_bfloat16 *yrow =
                        static_cast<__nv_bfloat16 *>(p.y) + (int64_t)rows_all[e * kSmRT + row] * p.ldy;
                    const uint32_t src = smem_u32(sb) + row * g.ypitch;
                    const SliceDesc &sl = p.slices[ck.t];
                    const int go = sl.y_col - sl.col_begin;
                    for (int col = ck.cb + (part * 32 + lane) * 8; col < ck.ce; col += 256 * hv)
                        *reinterpret_cast<uint4 *>(yrow + go + col) = lds128(src + (col - ck.cb) * 2);
                }
            }
        }
        // release the stage (its writes were fenced where they happened;
        // the reads are ordered by the barrier)
        __syncwarp();
        if (lane == 0) mbar_arrive1(&empty[st]);
        if (++st == D) {
            st = 0;
            ph ^= 1u;
        }
        if (++c == nch) {
            c = 0;
            ++e;
        }
    }
    }
    // A wait that gave up may leave copies in flight: wait once more
    // (bounded) for the last use of every stage before the shared memory
    // goes away.
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            raise_deverr(p.counts, LORA_DEVERR_WAIT);
            for (int s2 = 0; s2 < D && s2 < J; ++s2) mbar_wait(&full[s2], (uint32_t)((J - 1 - s2) / D) & 1u);
        }
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
    if (M < 1 || M > kSmMaxRows || cl < 1 || cl > kSmMaxCluster || ncl < 1) return false;
    if (p.d_in % (64 * cl)) return false;
    g = SmGeom{};
    g.CL = cl;
    g.KC = p.d_in / cl;
    g.stacked = p.stacked ? 1 : 0;
    g.rs = p.r_max <= 16 ? 16 : (p.r_max <= 32 ? 32 : 64);
    g.nrb_s = g.rs / 16;
    if (g.stacked && p.n_slices * g.rs > R16) return false;
    g.RPT = M <= kSmThreads ? 1 : (M <= 2 * kSmThreads ? 2 : 4);
    const int nv = p.d_out_total / 8;
    int ncol0[kSmMaxCluster + 1];
    for (int qq = 0; qq <= cl; ++qq) ncol0[qq] = (int)((int64_t)nv * qq / cl) * 8;
    // distinct adapters G <= min(M, n); tiles T <= sum over groups of
    // ceil(c / 16) <= (M + 15 G) / 16
    const int G = std::min(M, p.n_adapters);
    g.HS = pow2_at_least(std::max(64, 2 * G));
    if ((size_t)g.HS * 12 > (size_t)kSmMaxHashBytes) return false;
    const int Tmax = (M + 15 * G + 15) / 16;
    g.tcap = (Tmax + ncl - 1) / ncl;
    g.ncl_magic = (uint32_t)((0x100000000ull + (uint64_t)ncl - 1) / (uint64_t)ncl);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 127) & ~size_t(127);
        return (int)at;
    };
    g.off_bars = take(8 * (2 + 8 + 8));
    g.off_key = take((size_t)g.HS * 4);
    g.off_first = take((size_t)g.HS * 4);
    g.off_cnt = take((size_t)g.HS * 4);
    g.off_scan = take(64 * 4);
    g.off_tl = take((size_t)g.tcap * sizeof(TileRec));
    g.off_rows = take((size_t)g.tcap * kSmRT * 4);
    g.off_ids = take((size_t)kSmThreads * g.RPT * 4);
    g.off_recv = take((size_t)2 * cl * 16 * R16 * 4);
    g.off_hbf = take((size_t)16 * (R16 + 8) * 2);
    g.off_stage = (int)((o + 1023) & ~size_t(1023));
    // the kernel aligns its base to 1024 bytes: up to 1023 bytes of slack
    const int limit = 227 * 1024 - 1024;
    if (g.off_stage >= limit) return false;
    const int avail = limit - g.off_stage;
    const int ng = R16 / 8;  // 8-rank B planes
    auto r1k = [](int v) { return (v + 1023) & ~1023; };
    // a K stage: x rows, then (R16 / 16) x (kc / 64) A atoms of 2 KB; an N
    // stage: y rows, then R16 / 8 B planes of nc (rounded up to 128) rows;
    // either holds the 20 KB of warp partials of the h reduction
    constexpr int kRedBytes = kSmWarps * 16 * 20 * 4;
    auto kbytes = [&](int kc) { return std::max(kRedBytes, r1k(kSmRT * (2 * kc + 16)) + (R16 / 16) * (kc / 64) * 2048); };
    auto nbytes = [&](int nc) { return std::max(kRedBytes, r1k(kSmRT * (2 * nc + 16)) + ng * ((nc + 127) & ~127) * 16); };
    // The N chunks of cluster rank q: its columns cut at the output slices,
    // each piece into near-equal chunks of at most nc columns (multiples of 8).
    auto make_chunks = [&](int nc, int *max_cols) {
        *max_cols = 0;
        for (int qq = 0; qq < cl; ++qq) {
            int k = 0;
            for (int t = 0; t < p.n_slices; ++t) {
                const SliceDesc &sl = p.slices[t];
                const int cb = std::max(ncol0[qq], sl.col_begin), ce = std::min(ncol0[qq + 1], sl.col_begin + sl.d_out);
                if (cb >= ce) continue;
                const int parts = (ce - cb + nc - 1) / nc;
                const int step = (((ce - cb + parts - 1) / parts) + 7) & ~7;
                for (int c0 = cb; c0 < ce; c0 += step) {
                    if (k == kSmMaxNChunks) return false;
                    g.nck[qq][k].t = t;
                    g.nck[qq][k].cb = c0;
                    g.nck[qq][k].ce = std::min(c0 + step, ce);
                    *max_cols = std::max(*max_cols, g.nck[qq][k].ce - c0);
                    ++k;
                }
            }
            g.nN[qq] = k;
        }
        return true;
    };
    // Whole slices as one chunk where three stages hold them, else chunks of
    // at least `want` columns with as many stages (up to five) as hold them.
    const int NCq = ncol0[1] - ncol0[0] + 8;  // columns of a cluster rank, at most
    for (int want : {1 << 30, 512, 256, 128, 64}) {
        for (int D = 5; D >= 3; --D) {
            const int lim = (avail / D) & ~1023;
            int kc = 0;
            for (int k = 64; k <= g.KC; k <<= 1)
                if (g.KC % k == 0 && kbytes(k) <= lim) kc = k;
            int nc = 0;
            for (int c = 64; nbytes(c) <= lim && c <= 4096; c += 64) nc = c;
            if (kc < std::min(want, g.KC) || nc < std::min(want, NCq)) continue;
            int maxc = 0;
            if (!make_chunks(nc, &maxc)) continue;
            int minN = kSmMaxNChunks;
            for (int qq = 0; qq < cl; ++qq) minN = std::min(minN, g.nN[qq]);
            g.kc = kc;
            g.nK = g.KC / kc;
            g.natoms = kc / 64;
            g.ncp = (maxc + 127) & ~127;
            g.xpitch = 2 * kc + 16;
            g.offA = r1k(kSmRT * g.xpitch);
            g.ypitch = 2 * maxc + 16;
            g.offB = r1k(kSmRT * g.ypitch);
            g.SB = std::max(kbytes(kc), std::max(kRedBytes, g.offB + ng * g.ncp * 16));
            // the rows of tile e + 1 are found when tile e starts: at most one
            // tile's chunks ahead
            g.D = std::min(D, g.nK + minN + 1);
            g.total = g.off_stage + g.D * g.SB + 1024;
            if (g.total > 227 * 1024) continue;
            return true;
        }
    }
    return false;
}

// Cluster size by the larger of d_in and d_out: a CTA's K and N slices stay
// at most about 4096 columns, in clusters of at least two above 1024.  Fewer,
// wider CTAs per tile measured faster than the 2048-column slices of the
// single-pass kernel: mixed serving (4096 -> 6144) 54.4 -> 50.9 us per launch
// in clusters of 2 instead of 4 (59.5 in clusters of 1), mixed rank (4096 ->
// 14336) 49.7 -> 41.8 us in clusters of 4 instead of 8.
static int small_cluster_size(int d_in, int d_out) {
    const int d = d_in > d_out ? d_in : d_out;
    if (d < 1024) return 1;
    if (d <= 8192) return 2;
    if (d <= 16384) return 4;
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

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn small_encode_fn() {
    static EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// A 3-D bf16 tensor map {d0, d1, d2} with byte strides {s1, s2} and box
// {b0, b1, 1}; the last few encodings are kept per thread, so a call with the
// pools of an earlier call encodes nothing.
struct MapKey {
    const void *base;
    uint64_t d0, d1, d2, s1, s2;
    uint32_t b0, b1, swz;
};
struct MapCache {
    MapKey key[16];
    CUtensorMap map[16];
    int n = 0, next = 0;
};
// swz: 0 none, 1 64-byte, 2 128-byte swizzle
bool encode_3d(CUtensorMap *out, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b0, uint32_t b1, int swz) {
    static thread_local MapCache cache;
    MapKey k;
    memset(&k, 0, sizeof(k));
    k.base = base;
    k.d0 = d0;
    k.d1 = d1;
    k.d2 = d2;
    k.s1 = s1;
    k.s2 = s2;
    k.b0 = b0;
    k.b1 = b1;
    k.swz = (uint32_t)swz;
    for (int i = 0; i < cache.n; ++i)
        if (memcmp(&cache.key[i], &k, sizeof(k)) == 0) {
            *out = cache.map[i];
            return true;
        }
    EncodeTiledFn fn = small_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, 1}, elem[3] = {1, 1, 1};
    // No L2 promotion for boxes of narrow rows (a few ranks of a padded B
    // row): promotion would fetch the padding around every row.
    const CUtensorMapL2promotion promo = b0 * 2 >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_NONE;
    if (fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE,
           swz == 2 ? CU_TENSOR_MAP_SWIZZLE_128B : (swz == 1 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
           promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const int i = cache.n < 16 ? cache.n++ : (cache.next++ & 15);
    cache.key[i] = k;
    cache.map[i] = *out;
    return true;
}

// The tensor maps of a call: A in 64-column x 16-rank boxes (128-byte
// swizzle), every slice's B in 16-, 32- and 64-rank x 128-column boxes.
bool small_maps(const DeltaArgs &p, SmMaps &m) {
    memset(&m, 0, sizeof(m));
    // B boxes of 16, 32 or 64 ranks, none wider than the pool: pools padded
    // to one of those widths
    if (p.r_max != 16 && p.r_max != 32 && p.r_max != 64) return false;
    for (int t = 0; t < (p.stacked ? p.n_slices : 1); ++t) {
        const void *A = p.stacked && p.slices[t].A ? p.slices[t].A : p.A;
        if (!encode_3d(&m.a[t], A, (uint64_t)p.d_in, (uint64_t)p.r_max, (uint64_t)p.n_adapters,
                       (uint64_t)p.a_stride_r * 2, (uint64_t)p.a_stride_adapter * 2, 64, 16, 2))
            return false;
    }
    for (int t = 0; t < p.n_slices; ++t) {
        const SliceDesc &sl = p.slices[t];
        for (int wi = 0; wi < 3 && (16 << wi) <= p.r_max; ++wi) {
            const bool ok =
                p.b_rank_major
                    ? encode_3d(&m.b[t][wi], sl.B, (uint64_t)sl.d_out, (uint64_t)p.r_max, (uint64_t)p.n_adapters,
                                (uint64_t)sl.stride_r * 2, (uint64_t)sl.stride_adapter * 2, 64, 16u << wi, 2)
                    : encode_3d(&m.b[t][wi], sl.B, (uint64_t)p.r_max, (uint64_t)sl.d_out, (uint64_t)p.n_adapters,
                                (uint64_t)sl.stride_n * 2, (uint64_t)sl.stride_adapter * 2, 16u << wi, 128, wi);
            if (!ok) return false;
        }
    }
    return true;
}
}  // namespace

static_assert(sizeof(DeltaArgs) + sizeof(SmGeom) + sizeof(SmMaps) <= 4096, "kernel parameters above 4 KB");

template <int R16>
static cudaError_t launch_small_t(const DeltaArgs &p, const SmMaps &maps, int cl, int sms, cudaStream_t stream,
                                  bool *taken) {
    auto kern = sgmv_stream_kernel<R16>;
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
    cfg.blockDim = dim3(kStThreads);
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
    return cudaLaunchKernelEx(&cfg, kern, p, g, maps);
}

}  // namespace stream

// Launches the streaming kernel when the shape is one it takes; returns
// false (launching nothing) otherwise.
bool try_launch_stream(const DeltaArgs &p, int sms, cudaStream_t stream, cudaError_t *err) {
    using namespace stream;
    if (p.r_max > 64 || p.ids == nullptr || p.M_rows < 1 || p.M_rows > kSmMaxRows) return false;
    SmMaps maps;
    if (!small_maps(p, maps)) return false;
    const int rs = p.r_max <= 16 ? 16 : (p.r_max <= 32 ? 32 : 64);
    if (p.stacked && p.n_slices * rs > 64) return false;
    const int R16 = p.stacked ? small_r16(p.n_slices * rs) : small_r16(p.r_max);
    const int cl0 = small_cluster_size(p.d_in, p.d_out_total);
    // the preferred cluster size first, then larger ones, then smaller ones
    int order[8], no = 0;
    order[no++] = cl0;
    for (int cl = cl0 * 2; cl <= kSmMaxCluster; cl *= 2) order[no++] = cl;
    for (int cl = cl0 / 2; cl >= 1; cl /= 2) order[no++] = cl;
    for (int i = 0; i < no; ++i) {
        const int cl = order[i];
        if (p.d_in % (64 * cl) || cl > sms - 1) continue;
        bool taken = false;
        if (R16 == 16) *err = launch_small_t<16>(p, maps, cl, sms, stream, &taken);
        else if (R16 == 32) *err = launch_small_t<32>(p, maps, cl, sms, stream, &taken);
        else *err = launch_small_t<64>(p, maps, cl, sms, stream, &taken);
        if (taken || *err != cudaSuccess) return true;
    }
    return false;
}

}  // namespace lora
