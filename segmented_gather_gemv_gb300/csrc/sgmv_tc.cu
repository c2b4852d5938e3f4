// sgmv_tc.cu -- tensor-core (tcgen05 / TMEM) SGMV for segments with many rows
// (prefill).  "vLLM-Ascend LoRA" article, section 3.4: the rows of one
// adapter form a (tokens_i x d) matrix; (x A^T) gives (tokens_i x r) and
// (. B^T) returns to (tokens_i x d) -- a grouped GEMM over segments of
// different lengths; section 4.1: segments with enough rows go to the matrix
// unit.
//
// Work split: the rows of all segments routed here form one row space; CTA b
// of a persistent grid takes rows [M b / G, M (b+1) / G), so every CTA moves
// the same amount of x and y whatever the segment lengths.  Its rows are cut
// into tiles of up to 128 rows that share one adapter (consecutive chunks of
// the same adapter group merge into one tile).
//
// Per tile:
//   shrink  D1[128 x r] (TMEM, fp32) = x_tile[128 x d_in] . A_a^T, K in
//           64-element blocks, operands staged in the 128-byte swizzle;
//   scale   the epilogue warps read D1, multiply by s_a, round to bf16 and
//           write H[128 x r] to shared memory (never to global memory);
//   expand  per 128-column n-tile: D2[128 x 128] (TMEM, triple buffered)
//           = H . B_a[cols]^T;
//   store   y_tile += D2 in fp32, rounded once to bf16, stored from registers.
// Ranks are masked exactly: A rows / B columns at or past the adapter's rank
// are zero-filled in shared memory (never read), so padding never reaches y.
//
// Warp roles (448 threads): warps 0-1 x/A loaders, warp 2 MMA issuer (one
// thread) and TMEM owner, warp 3 B loader, warps 4-5 y loaders, warps 6..13
// epilogue (warp w
// owns TMEM lanes 32 (w % 4) .. +31, i.e. tile rows, and one half of the
// columns of every n-tile; four of them also build H).
//
// Loads are 16-byte cp.async issued by the loader warps (they write the
// swizzled operand layouts themselves and signal the stage barrier with
// cp.async.mbarrier.arrive.noinc): rows gathered through sorted_token_ids
// are 128- or 256-byte pieces of rows far apart, and bulk / tensor async
// copies of such pieces run several times slower than 16-byte copies.
#include "common.cuh"

namespace lora {

constexpr int kTcThreads = 448;
constexpr int kBM = 128;        // tile rows (MMA M)
constexpr int kBK = 128;        // shrink K block: two 64-element (128-byte) swizzle atoms
constexpr int kBN = 128;        // expand n-tile (MMA N)
constexpr int kSX = 2;          // x/A stages
constexpr int kSB = 4;          // B stages
constexpr int kSY = 3;          // y stages
constexpr int kST = 3;          // TMEM D2 buffers
constexpr int kTcMaxRank = 32;  // ranks above this use the CUDA-core kernel
constexpr int kSnapRows = 16;   // CTA row ranges end on a segment boundary this close
constexpr int kYPitch = kBN * 2 + 16;  // bytes per y row in a y stage (padded)

// Shared-memory layout (bytes, from a 1024-aligned base).
constexpr int kXAtom = kBM * 128;                    // 16 KB: 128 rows x 64 columns
constexpr int kAAtom = kTcMaxRank * 128;             // 4 KB: 32 rank rows x 64 columns
constexpr int kXBytes = 2 * kXAtom;                  // 32 KB
constexpr int kABytes = 2 * kAAtom;                  // 8 KB
constexpr int kXStage = kXBytes + kABytes;           // 24 KB
constexpr int kBChunk = kBN * 16;                    // 2 KB: 8 rank columns x 128 rows
constexpr int kBStage = (kTcMaxRank / 8) * kBChunk;  // 16 KB
constexpr int kHChunk = kBM * 16;                    // 2 KB
constexpr int kHBytes = (kTcMaxRank / 8) * kHChunk;  // 16 KB
constexpr int kYStage = kBM * kYPitch;               // 34 KB
constexpr int kOffX = 0;
constexpr int kOffB = kOffX + kSX * kXStage;
constexpr int kOffH = kOffB + kSB * kBStage;
constexpr int kOffY = kOffH + kHBytes;
constexpr int kOffRows = kOffY + kSY * kYStage;      // 3 x 128 ints (per loader role)
constexpr int kOffBars = kOffRows + 3 * kBM * 4;
constexpr int kNumBars = 2 * kSX + 2 * kSB + 2 * kSY + 3 + 2 * kST + 1;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kTcSmem = kOffMisc + 64 + 1024;        // + alignment slack


// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst), "r"(smem_u32(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4, leading and stride
// byte offsets >> 4, descriptor version 1, layout type.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(layout & 7) << 61;
    return d;
}
constexpr uint32_t kLayoutNone = 0, kLayoutSw128 = 2;

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both
// K-major, shape M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// Bounded waits: false (and `ok` cleared) when the wait timed out or another
// role aborted; the caller then leaves its loop.  wait1 is for a single
// thread; wait_warp is called by all 32 lanes and returns the same answer on
// every lane (so warp-collective instructions that follow stay converged).
__device__ __forceinline__ bool wait1(uint64_t *bar, uint32_t parity, bool &ok, volatile int *abort) {
    if (mbar_wait_abort(bar, parity, abort)) return true;
    ok = false;
    return false;
}
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, bool &ok, volatile int *abort) {
    const bool mine = mbar_wait_abort(bar, parity, abort);
    const bool all = __all_sync(0xffffffffu, mine);
    if (!all) ok = false;
    return all;
}

// One tile of the row space: `n` rows starting at sorted position `pos`,
// all on adapter `a`.
struct Tile {
    int pos, n, a;
};

// Walks the tiles of one CTA's row range.  Every role runs its own copy and
// sees the same sequence.
struct TileWalker {
    const DeltaArgs *p;
    int r, r1, nseg;
    __device__ __forceinline__ int seg_of(int row) const {
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p->tc_ptr[mid] <= row) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    }
    __device__ __forceinline__ bool next(Tile &t) {
        if (r >= r1) return false;
        int i = seg_of(r);
        const int a = p->tc_adapter[(int64_t)i * p->tc_rec_stride];
        const int start = p->tc_start[(int64_t)i * p->tc_rec_stride];
        t.pos = start + (r - p->tc_ptr[i]);
        t.a = a;
        int end = p->tc_ptr[i + 1];  // row-space end of the current run
        int run_end_pos = start + (end - p->tc_ptr[i]);
        // Consecutive segments of the same adapter that continue the run
        // (chunks of one adapter group) join the tile.
        while (end < r1 && end - r < kBM && i + 1 < nseg) {
            const int a2 = p->tc_adapter[(int64_t)(i + 1) * p->tc_rec_stride];
            const int s2 = p->tc_start[(int64_t)(i + 1) * p->tc_rec_stride];
            if (a2 != a || s2 != run_end_pos) break;
            ++i;
            run_end_pos += p->tc_ptr[i + 1] - p->tc_ptr[i];
            end = p->tc_ptr[i + 1];
        }
        t.n = min(min(kBM, r1 - r), end - r);
        r += t.n;
        return true;
    }
};

// Column range of expand n-tile `nt`: slice t, first column c within it.
__device__ __forceinline__ void ntile_cols(const DeltaArgs &p, int nt, int &slice, int &c0, int &ncols) {
    int t = 0;
    for (;;) {
        const int nts = (p.slices[t].d_out + kBN - 1) / kBN;
        if (nt < nts || t + 1 >= p.n_slices) break;
        nt -= nts;
        ++t;
    }
    slice = t;
    c0 = nt * kBN;
    ncols = min(kBN, p.slices[t].d_out - c0);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    sgmv_tc_kernel(const __grid_constant__ DeltaArgs p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint64_t *xf = bars, *xe = xf + kSX, *bf = xe + kSX, *be = bf + kSB, *yf = be + kSB, *ye = yf + kSY;
    uint64_t *d1f = ye + kSY, *hr = d1f + 1, *he = hr + 1, *tf = he + 1, *te = tf + kST, *fin = te + kST;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kSX; ++s) { mbar_init(&xf[s], 64); mbar_init(&xe[s], 1); }
        for (int s = 0; s < kSB; ++s) { mbar_init(&bf[s], 32); mbar_init(&be[s], 1); }
        for (int s = 0; s < kSY; ++s) { mbar_init(&yf[s], 64); mbar_init(&ye[s], 256); }
        mbar_init(d1f, 1);
        mbar_init(hr, 128);
        mbar_init(he, 1);
        for (int s = 0; s < kST; ++s) { mbar_init(&tf[s], 1); mbar_init(&te[s], 256); }
        mbar_init(fin, 1);
        fence_mbar_init();
        *abort = 0;
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    griddep_launch_dependents();
    griddep_wait();

    const int nseg = min(p.counts[p.tc_count_index], p.max_list);
    const int Mrows = p.counts[p.tc_rows_index];
    const int G = gridDim.x, b = blockIdx.x;
    TileWalker walker{&p, 0, 0, nseg};
    if (nseg > 0) {
        // Equal row shares, each end moved to a segment boundary that lies
        // within kSnapRows: a tile costs a full pass over the K blocks and
        // n-tiles however few rows it holds, so a CTA should not end a few
        // rows into the next segment.  Both neighbours compute the same end.
        auto snap = [&](int r) {
            if (r <= 0 || r >= Mrows) return r <= 0 ? 0 : Mrows;
            const int i = walker.seg_of(r);
            const int lo = p.tc_ptr[i], hi = p.tc_ptr[i + 1];
            if (r - lo <= kSnapRows) return lo;
            if (hi - r <= kSnapRows) return hi;
            return r;
        };
        walker.r = snap((int)((int64_t)Mrows * b / G));
        walker.r1 = snap((int)((int64_t)Mrows * (b + 1) / G));
        if (walker.r1 < walker.r) walker.r1 = walker.r;
    }

    int n_nt = 0;
    for (int t = 0; t < p.n_slices; ++t) n_nt += (p.slices[t].d_out + kBN - 1) / kBN;
    const int nkb = (p.d_in + kBK - 1) / kBK;
    // Every CTA walks the K blocks and the n-tiles from its own starting
    // point.  Rows of x and y are a power-of-two stride apart; if all CTAs
    // read the same column block at the same time, their requests fall on the
    // same memory channels.
    const int kb_rot = (int)(((uint32_t)b * 2654435761u) >> 7) % nkb;
    const int nt_rot = (int)(((uint32_t)b * 2246822519u) >> 7) % (n_nt > 0 ? n_nt : 1);
    bool ok = true;

    if (warp < 2) {
        // ------------------------------------------------------------ x/A loaders
        const int lt = tid;  // 0..63
        int32_t *rows = reinterpret_cast<int32_t *>(smem + kOffRows);
        const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(p.x);
        const __nv_bfloat16 *Ag = static_cast<const __nv_bfloat16 *>(p.A);
        uint32_t xs = 0;
        Tile t;
        while (walker.next(t)) {
            const int r = p.ranks ? p.ranks[t.a] : p.r_max;
            const bool live = r <= p.r_max && tc_rank_ok(r);
            if (!live) continue;
            asm volatile("bar.sync 1, 64;\n" ::: "memory");  // previous tile done with rows
            for (int i = lt; i < t.n; i += 64) rows[i] = p.sorted[t.pos + i];
            asm volatile("bar.sync 1, 64;\n" ::: "memory");
            const int n16 = (r + 15) / 16;
            const __nv_bfloat16 *Aa = Ag + (int64_t)t.a * p.a_stride_adapter;
            for (int kbi = 0; kbi < nkb; ++kbi, ++xs) {
                const int kb = kbi + kb_rot < nkb ? kbi + kb_rot : kbi + kb_rot - nkb;
                const int s = xs % kSX;
                if (!wait_warp(&xe[s], ((xs / kSX) & 1) ^ 1, ok, abort)) goto role_done;
                unsigned char *xst = smem + kOffX + s * kXStage;
                // x rows: 16 chunks of 16 bytes per row (256 contiguous bytes),
                // two 64-column atoms in the 128-byte swizzle
                for (int e = lt; e < t.n * 16; e += 64) {
                    const int i = e >> 4, c = e & 15, k = kb * kBK + c * 8;
                    const __nv_bfloat16 *row = xg + (int64_t)rows[i] * p.ldx;
                    cp_async16(xst + (c >> 3) * kXAtom + i * 128 + (((c & 7) ^ (i & 7)) << 4), k < p.d_in ? row + k : row,
                               k < p.d_in ? 16 : 0);
                }
                // A rows of the adapter (rows >= rank zero-filled)
                for (int e = lt; e < 16 * n16 * 16; e += 64) {
                    const int j = e >> 4, c = e & 15, k = kb * kBK + c * 8;
                    const bool in = j < r && k < p.d_in;
                    cp_async16(xst + kXBytes + (c >> 3) * kAAtom + j * 128 + (((c & 7) ^ (j & 7)) << 4),
                               in ? Aa + (int64_t)j * p.a_stride_r + k : Aa, in ? 16 : 0);
                }
                cp_async_arrive_noinc(&xf[s]);
            }
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ B loader
        uint32_t bs = 0;
        Tile t;
        while (walker.next(t)) {
            const int r = p.ranks ? p.ranks[t.a] : p.r_max;
            const bool live = r <= p.r_max && tc_rank_ok(r);
            if (!live) continue;
            const int n16 = (r + 15) / 16, n8mma = 2 * n16, sh8 = n16 == 1 ? 1 : 2;
            for (int nti = 0; nti < n_nt; ++nti, ++bs) {
                const int nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                int sl, c0, nc;
                ntile_cols(p, nt, sl, c0, nc);
                const SliceDesc &S = p.slices[sl];
                // B rows c0 .. c0+127 of this slice, 8 rank columns per 2 KB chunk
                const int sb = bs % kSB;
                if (!wait_warp(&be[sb], ((bs / kSB) & 1) ^ 1, ok, abort)) goto role_done;
                unsigned char *bst = smem + kOffB + sb * kBStage;
                const __nv_bfloat16 *Ba = static_cast<const __nv_bfloat16 *>(S.B) + (int64_t)t.a * S.stride_adapter;
                for (int e = lane; e < kBN * n8mma; e += 32) {
                    const int n = e >> sh8, c = e & (n8mma - 1);
                    const bool in = c0 + n < S.d_out && c * 8 < r;
                    cp_async16(bst + c * kBChunk + n * 16, in ? Ba + (int64_t)(c0 + n) * S.stride_n + c * 8 : Ba,
                               in ? 16 : 0);
                }
                cp_async_arrive_noinc(&bf[sb]);
            }
        }
    } else if (warp == 4 || warp == 5) {
        // ------------------------------------------------------------ y loaders
        const int lt = tid - 128;  // 0..63
        int32_t *rows = reinterpret_cast<int32_t *>(smem + kOffRows + kBM * 4);
        uint32_t ys = 0;
        Tile t;
        while (walker.next(t)) {
            const int r = p.ranks ? p.ranks[t.a] : p.r_max;
            const bool live = r <= p.r_max && tc_rank_ok(r);
            if (!live) continue;
            asm volatile("bar.sync 2, 64;\n" ::: "memory");  // previous tile done with rows
            for (int i = lt; i < t.n; i += 64) rows[i] = p.sorted[t.pos + i];
            asm volatile("bar.sync 2, 64;\n" ::: "memory");
            for (int nti = 0; nti < n_nt; ++nti, ++ys) {
                const int nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                int sl, c0, nc;
                ntile_cols(p, nt, sl, c0, nc);
                const SliceDesc &S = p.slices[sl];
                const int sy = ys % kSY;
                if (!wait_warp(&ye[sy], ((ys / kSY) & 1) ^ 1, ok, abort)) goto role_done;
                unsigned char *yst = smem + kOffY + sy * kYStage;
                const int nch = nc >> 3;
                const __nv_bfloat16 *yc = static_cast<const __nv_bfloat16 *>(p.y) + S.y_col + c0;
                if (nch == kBN / 8) {
                    for (int e = lt; e < t.n * (kBN / 8); e += 64) {
                        const int i = e >> 4, c = e & 15;
                        cp_async16(yst + i * kYPitch + c * 16, yc + (int64_t)rows[i] * p.ldy + c * 8, 16);
                    }
                } else {
                    for (int e = lt; e < t.n * nch; e += 64) {
                        const int i = e / nch, c = e - i * nch;
                        cp_async16(yst + i * kYPitch + c * 16, yc + (int64_t)rows[i] * p.ldy + c * 8, 16);
                    }
                }
                cp_async_arrive_noinc(&yf[sy]);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t xs = 0, bs = 0, ts = 0, tiles = 0;
            const uint32_t id2 = idesc_bf16(kBM, kBN);
            const uint32_t x_base = smem_u32(smem + kOffX), b_base = smem_u32(smem + kOffB);
            const uint32_t h_base = smem_u32(smem + kOffH);
            Tile t;
            while (walker.next(t)) {
                const int r = p.ranks ? p.ranks[t.a] : p.r_max;
                const bool live = r <= p.r_max && tc_rank_ok(r);
                if (!live) continue;
                const int n16 = (r + 15) / 16;
                const uint32_t id1 = idesc_bf16(kBM, 16 * n16);
                // D1 is free again: the previous tile's expand was issued only
                // after the epilogue had read D1 (hr).
                for (int kbi = 0; kbi < nkb; ++kbi, ++xs) {
                    const int s = xs % kSX;
                    if (!wait1(&xf[s], (xs / kSX) & 1, ok, abort)) goto role_done;
                    tc_fence_after();
                    const uint32_t xa = x_base + s * kXStage, aa = xa + kXBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kXAtom + (kk & 3) * 32, aoff = (kk >> 2) * kAAtom + (kk & 3) * 32;
                        umma(tmem, smem_desc(xa + off, 16, 1024, kLayoutSw128),
                             smem_desc(aa + aoff, 16, 1024, kLayoutSw128), id1, (kbi | kk) != 0);
                    }
                    umma_commit(&xe[s]);
                }
                umma_commit(d1f);
                // H of this tile is ready once the epilogue has written it.
                if (!wait1(hr, tiles & 1, ok, abort)) goto role_done;
                tc_fence_after();
                for (int nt = 0; nt < n_nt; ++nt, ++bs, ++ts) {
                    const int sb = bs % kSB, st = ts % kST;
                    if (!wait1(&bf[sb], (bs / kSB) & 1, ok, abort)) goto role_done;
                    if (!wait1(&te[st], ((ts / kST) & 1) ^ 1, ok, abort)) goto role_done;
                    tc_fence_after();
                    const uint32_t bb = b_base + sb * kBStage;
                    const uint32_t d2 = tmem + 128 + 128 * st;
                    for (int kc = 0; kc < n16; ++kc)
                        umma(d2, smem_desc(h_base + kc * 2 * kHChunk, kHChunk, 128, kLayoutNone),
                             smem_desc(bb + kc * 2 * kBChunk, kBChunk, 128, kLayoutNone), id2, kc != 0);
                    umma_commit(&be[sb]);
                    umma_commit(&tf[st]);
                }
                umma_commit(he);
                ++tiles;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;              // TMEM lane quadrant
        const int chalf = (warp - 6) >> 2;    // which 64 columns of an n-tile
        const int row = q4 * 32 + lane;       // tile row owned by this thread
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        unsigned char *H = smem + kOffH;
        uint32_t ys = 0, ts = 0, tiles = 0;
        Tile t;
        while (walker.next(t)) {
            const int r = p.ranks ? p.ranks[t.a] : p.r_max;
            const bool live = r <= p.r_max && tc_rank_ok(r);
            if (!live) {
                // Tiles the tensor cores cannot take are the CUDA-core
                // kernel's; with the tensor-core path forced they are an error.
                if (p.tc_only && row == 0 && chalf == 0 && r != 0) raise_deverr(p.counts, LORA_DEVERR_RANK);
                continue;
            }
            const float sc = p.adapter_scale ? p.adapter_scale[t.a] : p.scale;
            const int n16 = (r + 15) / 16;
            const int my_row = row < t.n ? p.sorted[t.pos + row] : 0;  // this thread's token row
            if (chalf == 0) {
                // ---- D1 -> scale -> bf16 H (cols >= r are zero)
                if (!wait_warp(d1f, tiles & 1, ok, abort)) goto role_done;
                tc_fence_after();
                if (tiles > 0)
                    if (!wait_warp(he, (tiles - 1) & 1, ok, abort)) goto role_done;  // previous expand done with H
                for (int c16 = 0; c16 < kTcMaxRank / 16; ++c16) {
                    if (c16 >= n16) break;
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_off + 16 * c16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int c8 = 2 * c16 + half;
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 8 * c8 + 2 * e;
                            const float f0 = j < r ? __uint_as_float(v[8 * half + 2 * e]) * sc : 0.f;
                            const float f1 = j + 1 < r ? __uint_as_float(v[8 * half + 2 * e + 1]) * sc : 0.f;
                            const __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
                            w[e] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        *reinterpret_cast<uint4 *>(H + c8 * kHChunk + row * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(hr);
            }
            // ---- expand n-tiles: y += D2 (this thread: its row, 64 columns)
            for (int nti = 0; nti < n_nt; ++nti, ++ys, ++ts) {
                const int nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                const int sy = ys % kSY, st = ts % kST;
                int sl, c0, nc;
                ntile_cols(p, nt, sl, c0, nc);
                const SliceDesc &S = p.slices[sl];
                if (!wait_warp(&tf[st], (ts / kST) & 1, ok, abort)) goto role_done;
                if (!wait_warp(&yf[sy], (ys / kSY) & 1, ok, abort)) goto role_done;
                tc_fence_after();
                const unsigned char *yrow = smem + kOffY + sy * kYStage + row * kYPitch;
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.y) + (int64_t)my_row * p.ldy + S.y_col + c0;
                uint4 outv[8];
                const int cbase = 64 * chalf;
#pragma unroll
                for (int c32 = 0; c32 < 2; ++c32) {
                    uint32_t v0[16], v1[16];
                    const uint32_t ta = tmem + 128 + 128 * st + lane_off + cbase + 32 * c32;
                    tmem_ld16(ta, v0);
                    tmem_ld16(ta + 16, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 yv = *reinterpret_cast<const uint4 *>(yrow + (cbase + 32 * c32) * 2 + q * 16);
                        uint32_t *yw = reinterpret_cast<uint32_t *>(&yv);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = q * 8 + 2 * e;
                            const uint32_t a0 = j < 16 ? v0[j] : v1[j - 16];
                            const uint32_t a1 = j + 1 < 16 ? v0[j + 1] : v1[j + 1 - 16];
                            const float y0 = __uint_as_float(yw[e] << 16) + __uint_as_float(a0);
                            const float y1 = __uint_as_float(yw[e] & 0xFFFF0000u) + __uint_as_float(a1);
                            const __nv_bfloat162 o = __floats2bfloat162_rn(y0, y1);
                            yw[e] = *reinterpret_cast<const uint32_t *>(&o);
                        }
                        outv[c32 * 4 + q] = yv;
                    }
                }
                // TMEM buffer and y stage are free as soon as they are read
                tc_fence_before();
                mbar_arrive(&te[st]);
                mbar_arrive(&ye[sy]);
                if (row < t.n) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (cbase + 8 * k < nc) *reinterpret_cast<uint4 *>(dst + cbase + 8 * k) = outv[k];
                }
            }
            ++tiles;
        }
    }
role_done:
    bulk_wait0();
    if (warp == 2 && lane == 0) {
        // every MMA this CTA issued has completed before TMEM is released
        umma_commit(fin);
        if (!mbar_wait(fin, 0)) ok = false;
    }
    if (!ok) raise_deverr(p.counts, LORA_DEVERR_WAIT);
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
bool tc_available() { return true; }

cudaError_t launch_tc(const DeltaArgs &p, int mode, int sms, cudaStream_t stream) {
    if (mode != kFused) return cudaErrorNotSupported;
    static DeviceOnce once;
    cudaError_t e = once.run([] {
        return cudaFuncSetAttribute(sgmv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sgmv_tc_kernel, p);
}

}  // namespace lora
