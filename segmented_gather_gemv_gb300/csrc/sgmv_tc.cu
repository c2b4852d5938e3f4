// sgmv_tc.cu -- tensor-core (tcgen05 / TMEM) SGMV for segments with many rows
// (prefill).  "vLLM-Ascend LoRA" article, section 3.4: the rows of one
// adapter form a (tokens_i x d) matrix; (x A^T) gives (tokens_i x r) and
// (. B^T) returns to (tokens_i x d) -- a grouped GEMM over segments of
// different lengths; section 4.1: segments with enough rows go to the matrix
// unit.
//
// Work split: the rows of all segments routed here form one row space; CTA b
// of a persistent grid takes the equal share [M b / G, M (b+1) / G), its end
// moved to a nearby boundary between adapters (prepare computes the shares
// for this grid), so every CTA moves about the same amount of x and y
// whatever the segment lengths.  The grid has one CTA per 64 batch rows, at
// most one per SM, and leaves one SM free.  A share is cut into tiles of up to 128 rows; a tile may
// span several segments (pieces, see Tile below), so a share never costs two
// passes.
//
// Per tile:
//   shrink  D1[128 x K] (TMEM, fp32) = x_tile[128 x d_in] . A^T, where A
//           stacks the rank rows of the tile's adapters (K <= 32), K in
//           128-element blocks, operands in the 128-byte swizzle;
//   scale   the epilogue warps read D1, keep for each row only its own
//           adapter's columns, multiply by s_a, round to bf16 and write
//           H[128 x K] to shared memory (never to global memory);
//   expand  per 128-column n-tile: D2[128 x 128] (TMEM, triple buffered)
//           = y_tile . I + H . B^T: the y stage times a 16 x 16 identity puts
//           y into the fp32 accumulator exactly, then B stacks the adapters'
//           rows of that n-tile;
//   store   D2 rounded once to bf16 and written back as y.  An output that
//           comes out non-finite (a non-finite y reaches its whole 16-column
//           group through the identity: 0 * inf is NaN) is formed again as y
//           + sum_j h_j B_j in fp32, so every element is y + delta exactly.
// Ranks are masked exactly: A rows / B columns past an adapter's rank are
// never read, H columns past it are zero, so padding never reaches y.
//
// Split calls (one instantiation per mode): a shrink runs the x jobs only and
// the epilogue writes each row's D1 columns to h in global memory (fp32,
// unscaled, zero past the rank); an expand runs the y jobs only, with H
// built from h in global memory (scaled, rounded to bf16) instead of D1.
//
// Data movement.  The kernel streams x once and y twice (read, write); the
// adapter weights are small and stay in L2.  All staging goes through ONE
// ring of stages, filled in program order: a tile's nkb "x jobs" (x rows of
// one K block + the A block), then its n_nt "y jobs" (y rows of one n-tile +
// the B block).  So the y of a tile is already on its way while its last K
// blocks are multiplied, and the next tile's x while its last n-tiles are
// stored.  An x stage is released by the MMA (tcgen05.commit); a y stage by
// the epilogue warps once they have stored it.  A stage holds `cap` rows,
// cap = the CTA's share rounded up to 8 (at most 128), so a short share gets
// more, smaller stages: the bytes in flight per SM set the DRAM throughput,
// and a job's round trip (load, MMA, epilogue, release) takes microseconds.
// Rows of a tile past its end may hold anything: row i of D1 and D2 depends
// only on row i of the operands, so the MMA may also read whatever lies in
// shared memory past a stage's `cap` rows (up to 120 rows of 128 bytes, kept
// inside the allocation by kOverrun).
//
// Copies.  Rows of a tile that sit on consecutive token rows within one
// piece (a prefill sequence keeps its tokens adjacent and in order in
// sorted_token_ids) move by TMA: tiled copies of 64 columns x 64, 32 or 8
// rows in the 128-byte swizzle, for x and y; the A block comes by TMA from a
// 3-D map of the pool.  Rows that no box covers (a group of 8 split by a
// piece boundary or by a break in the token rows, and in tiles of 32 rows or
// more a partial last group) and the B block (16-byte pieces of L2-resident
// rows) move by 16-byte cp.async.  A loader that
// issues one cp.async per 16 bytes for everything spends its time issuing
// and waiting on its own instruction stream, which is why the boxes matter.
// y is stored with st.global, eight 64-byte row pieces per warp
// instruction: TMA stores mixed with such stores in one CTA stalled the
// CTA's loads.
//
// Warp roles (672 threads): warps 0, 1, 2 and 4 loaders (lane 0 of warps 0
// and 1 issue the boxes of atoms 0 and 1; warps 2 and 4 the cp.async
// copies), warp 3 MMA issuer (one thread) and TMEM owner, warps 5..20
// epilogue.  The MMA thread shares a scheduler with neither TMA issuer: next
// to one, its MMAs slowed that issuer's boxes.  Epilogue warp w owns TMEM
// lanes 32 (w % 4) .. +31 (tile rows) and one quarter of the columns of every
// n-tile; four of them also build H.  Without tensor maps every loader thread
// copies by cp.async.
#include <cuda.h>
#include <cstring>

#include "common.cuh"

namespace lora {

constexpr int kLoaderWarps = 4;                      // warps 0, 1, 2 and 4
constexpr int kLoaderThreads = kLoaderWarps * 32;
constexpr int kMmaWarp = 3;
constexpr int kLoaderWarp3 = 4;                      // the fourth loader warp
constexpr int kEpiWarp0 = 5;                         // warps 5..20
constexpr int kEpiWarps = 16;                        // 4 per TMEM lane quadrant
constexpr int kEpiCols = 128 * 4 / kEpiWarps;        // columns of an n-tile per epilogue warp
constexpr int kEpiChunks = kEpiCols / 8;             // 16-byte chunks of a row per epilogue warp
constexpr int kTcThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kBM = 128;        // tile rows (MMA M)
constexpr int kBK = 128;        // shrink K block: two 64-element (128-byte) swizzle atoms
constexpr int kBN = 128;        // expand n-tile (MMA N)
constexpr int kMaxNS = 16;      // ring stages at most
constexpr int kST = 3;          // TMEM D2 buffers
constexpr int kTcMaxRank = 32;  // ranks above this use the CUDA-core kernel
// Tensor maps of x and of the y column block of every slice (bf16, 128-byte
// swizzle), with boxes of 64 columns x 64, 32 and 8 rows; use = 0 when they
// could not be made.
// Also 3-D maps of the pools: A [adapter][rank row][d_in] in boxes of 64
// columns x 8 rank rows (128-byte swizzle), and for every slice B
// [adapter][d_out row][rank] in boxes of 8 rank columns x 128 rows (no
// swizzle: one 2 KB chunk of the MMA's core-matrix layout).  A box placed
// past the last rank row / column reads zeros.  use_ab = 0 when those maps
// could not be made.
struct TcMaps {
    CUtensorMap x64, x32, x8;
    CUtensorMap y64[LORA_MAX_SLICES], y32[LORA_MAX_SLICES], y8[LORA_MAX_SLICES];
    CUtensorMap a8, a16, a32, b[LORA_MAX_SLICES];
    int32_t use, use_ab, r_pad;  // r_pad: first rank index past every adapter's rank, a multiple of 8
    int32_t a_box_max;           // largest rank box encoded: 8, 16 or 32
};


// Shared-memory layout (bytes, from a 1024-aligned base).  A stage of a
// CTA whose tiles have at most `cap` rows (a multiple of 8) and whose ranks
// need n16 16-column MMA steps:
//   x job: x   two 64-column atoms of cap rows x 128 bytes (128-byte swizzle),
//          then A  two atoms of 16 n16 rank rows x 128 bytes;
//   y job: y   two 64-column atoms of cap rows x 128 bytes (same swizzle),
//          then B  2 n16 chunks of 128 rows x 16 bytes (8 rank columns each).
// Both take cap * 256 + 4096 * n16 bytes: at most 40 KB.
constexpr int kBChunk = kBN * 16;                    // 2 KB: 8 rank columns x 128 rows
constexpr int kRingBytes = 200 * 1024;
constexpr int kHChunk = kBM * 16;                    // 2 KB
constexpr int kHBytes = (kTcMaxRank / 8) * kHChunk;  // 8 KB
constexpr int kOffH = kRingBytes;
constexpr int kOffBars = kOffH + kHBytes;
constexpr int kNumBars = 2 * kMaxNS + 3 + 2 * kST + 1;
constexpr int kOffMisc = kOffBars + kNumBars * 8;    // TMEM address, abort flag, CTA row range
constexpr int kOffLdr = kOffMisc + 64;               // loader tables: row tokens, group tokens, TMA boxes
// loader tables, at kOffLdr: row tokens [4 warps][32] ints, group tokens
// [2][16] ints, TMA boxes [2][16] uint2, then the helpers' row lists [2][128] int2
constexpr int kLdrGtok = 4 * 32 * 4, kLdrBox = kLdrGtok + 2 * 16 * 4, kLdrRows = kLdrBox + 2 * 16 * 8;
// each TMA issuer's resolved copies of the tile: {smem offset, map code, row or rank, adapter}
constexpr int kCmdMax = 24;  // <= 16 row boxes + <= 4 rank boxes + 1 zero box
constexpr int kLdrCmd = kLdrRows + 2 * kBM * 8;
constexpr int kLdrBytes = kLdrCmd + 2 * kCmdMax * 16;
// 16 x 16 bf16 identity, the B operand that adds a y stage into D2
constexpr int kOffIdent = (kOffLdr + kLdrBytes + 127) & ~127;
constexpr int kIdentBytes = 16 * 16 * 2;
constexpr int kOverrun = (kBM - 8) * 128;            // MMA reads past the last stage
constexpr int kTcSmemUsed =
    kOffIdent + kIdentBytes > kRingBytes + kOverrun ? kOffIdent + kIdentBytes : kRingBytes + kOverrun;
constexpr int kTcSmem = kTcSmemUsed + 1024;          // + alignment slack

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
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

__device__ __forceinline__ void tma_load_2d(void *sdst, const CUtensorMap *map, int c, int r, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_u32(sdst)),
        "l"(map), "r"(c), "r"(r), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *sdst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(
            smem_u32(sdst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

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

// Largest i in [0, nseg) with ptr[i] <= r (ptr[0] = 0 <= r).  Called by all
// 32 lanes of a warp; each round probes 32 entries at once.
__device__ __forceinline__ int warp_seg_of(const int32_t *ptr, int nseg, int r, int lane) {
    int lo = 0, hi = nseg - 1;
    while (hi > lo) {
        const int step = (hi - lo + 32) >> 5;
        const int q = lo + lane * step;
        const bool le = q <= hi && ptr[q] <= r;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        lo += (31 - __clz(m)) * step;
        hi = min(hi, lo + step - 1);
    }
    return lo;
}

// One tile: `n` consecutive rows of the row space (at most 128), made of up
// to kMaxPieces pieces.  Piece q covers tile rows [off[q], off[q+1]); they
// are the rows at sorted positions pos[q] .., all on adapter a[q], whose rank
// is rank[q]; rk[q] = rank[q] if the tensor cores take it, else 0.  Piece q
// owns rank columns [kofs[q], kofs[q] + rk[q]) of the tile's stacked A and B
// blocks (K of them in all, at most 32): its rows see only its own adapter,
// because H is zero outside those columns.  So a CTA's row range never has to
// end at a segment boundary, and a tile costs one pass over the K blocks and
// n-tiles however many adapters share it.
constexpr int kMaxPieces = 4;
struct Tile {
    int n, np, K;
    int off[kMaxPieces + 1], pos[kMaxPieces], a[kMaxPieces], rank[kMaxPieces], rk[kMaxPieces], kofs[kMaxPieces];
    __device__ __forceinline__ int piece_of(int i) const {
        int q = 0;
#pragma unroll
        for (int u = 1; u < kMaxPieces; ++u) q += (u < np && i >= off[u]) ? 1 : 0;
        return q;
    }
};
// arr[q] for a run-time q, with compile-time indices only (keeps tiles in registers)
__device__ __forceinline__ int sel(const int (&arr)[kMaxPieces], int q) {
    int v = arr[0];
#pragma unroll
    for (int u = 1; u < kMaxPieces; ++u) v = q == u ? arr[u] : v;
    return v;
}

// Walks the tiles of one CTA's row range [r, r1); i is the segment holding
// row r.  Every role runs its own copy and sees the same sequence.
struct TileWalker {
    const DeltaArgs *p;
    int r, r1, i;
    __device__ __forceinline__ bool next(Tile &t) {
        if (r >= r1) return false;
        t.n = 0;
        t.np = 0;
        t.K = 0;
#pragma unroll
        for (int u = 0; u <= kMaxPieces; ++u) t.off[u] = 0;
        int last_a = -1, last_end = -1;  // adapter and sorted end position of the last piece
        while (r < r1 && t.n < kBM) {
            while (p->tc_ptr[i + 1] <= r) ++i;
            const int a = p->tc_adapter[(int64_t)i * p->tc_rec_stride];
            const int pos = p->tc_start[(int64_t)i * p->tc_rec_stride] + (r - p->tc_ptr[i]);
            const int cnt = min(min(p->tc_ptr[i + 1] - r, r1 - r), kBM - t.n);
            // a new piece, unless this segment continues the last one (the
            // next chunk of the same adapter group)
            const bool fresh = !(a == last_a && pos == last_end);
            const int rank = p->ranks ? p->ranks[a] : p->r_max;
            const int rk = rank <= p->r_max && tc_rank_ok(rank) ? rank : 0;
            if (fresh && (t.np == kMaxPieces || t.K + rk > kTcMaxRank)) break;
#pragma unroll
            for (int u = 0; u < kMaxPieces; ++u)
                if (fresh && u == t.np) {
                    t.pos[u] = pos;
                    t.a[u] = a;
                    t.rank[u] = rank;
                    t.rk[u] = rk;
                    t.kofs[u] = t.K;
                    t.off[u] = t.n;
                }
            if (fresh) {
                t.K += rk;
                ++t.np;
            }
            last_a = a;
            last_end = pos + cnt;
            t.n += cnt;
            r += cnt;
        }
#pragma unroll
        for (int u = 1; u <= kMaxPieces; ++u)
            if (u == t.np) t.off[u] = t.n;
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

// Byte offset of 16-byte chunk c (of 16) of row i in an x or y stage: atom
// c / 8, 128-byte rows, chunk index XORed with the row's low bits (the
// 128-byte swizzle of TMA and of the MMA operands; a warp reading one chunk
// of 32 rows, or 8 chunks of 4 rows, spreads over all banks).
__device__ __forceinline__ int schunk(int xatom, int i, int c) { return (c >> 3) * xatom + i * 128 + (((c & 7) ^ (i & 7)) << 4); }

// Token row (row of x and y) of tile row i.
__device__ __forceinline__ int tile_token(const DeltaArgs &p, const Tile &t, int i) {
    const int q = t.piece_of(i);
    int pos = t.pos[0], off = t.off[0];
#pragma unroll
    for (int u = 1; u < kMaxPieces; ++u)
        if (q == u) {
            pos = t.pos[u];
            off = t.off[u];
        }
    return p.sorted[pos + (i - off)];
}

// Which 8-row groups (bit g: tile rows 8g .. 8g+7, the last group possibly
// partial), 32-row groups (bit j: rows 32j .. 32j+31, full) and 64-row
// groups (bit h) lie in one piece on consecutive token rows, so that one TMA
// box moves them.  Called by all 32 lanes of a warp; every lane gets the
// same masks.
__device__ __forceinline__ void tile_box_masks(const DeltaArgs &p, const TcMaps &m, const Tile &t, int lane,
                                               uint32_t &mask8, uint32_t &mask32, uint32_t &mask64, int &tok8) {
    bool ok = false;
    tok8 = 0;  // lanes 0-15: token row of tile row 8 lane (0 past the tile or without maps)
    if (m.use) {
        int i0 = -1, i1 = 0;
        if (lane < 16 && 8 * lane < t.n && (8 * lane + 8 <= t.n || t.n < 32)) {
            // In a tile of 32 rows or more, full groups only: a partial last
            // group costs a whole TMA issue for a few rows, which the cp.async
            // helpers copy for much less (in small tiles they are busy enough).
            i0 = 8 * lane;
            i1 = min(i0 + 7, t.n - 1);
        } else if (lane >= 16 && lane < 20 && 32 * (lane - 16) + 32 <= t.n) {
            i0 = 32 * (lane - 16);
            i1 = i0 + 31;
        } else if (lane >= 20 && lane < 22 && 64 * (lane - 20) + 64 <= t.n) {
            i0 = 64 * (lane - 20);
            i1 = i0 + 63;
        }
        if (i0 >= 0) {
            const int k0 = tile_token(p, t, i0);
            ok = t.piece_of(i0) == t.piece_of(i1) && tile_token(p, t, i1) - k0 == i1 - i0;
            if (lane < 16) tok8 = k0;
        }
    }
    const uint32_t b = __ballot_sync(0xffffffffu, ok);
    mask8 = b & 0xFFFFu;
    mask32 = (b >> 16) & 0xFu;
    mask64 = (b >> 20) & 0x3u;
}

// y + delta in fp32 for element e of a stage chunk of tile row `row` (yword:
// the chunk's 32-bit word holding it): delta = sum over the adapter's rank
// columns j of H[row][k_lo + j]
// (bf16, scaled) times B[a][col][j] (the rare path of outputs the identity
// product made non-finite).
__device__ __forceinline__ float exact_output(uint32_t yword, int e, const unsigned char *H, int row, int k_lo, int rk,
                                              const SliceDesc &S, int a, int col) {
    const float yv = __uint_as_float((e & 1) ? (yword & 0xFFFF0000u) : (yword << 16));
    const __nv_bfloat16 *Bp = static_cast<const __nv_bfloat16 *>(S.B) + (int64_t)a * S.stride_adapter +
                              (int64_t)col * S.stride_n;
    float dsum = 0.f;
#pragma unroll 1
    for (int j = 0; j < rk; ++j) {
        const int kc = k_lo + j;
        const float hj =
            __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(H + (kc >> 3) * kHChunk + row * 16 + (kc & 7) * 2));
        dsum = fmaf(hj, __bfloat162float(Bp[j]), dsum);
    }
    return yv + dsum;
}

// MODE: kFused, kShrink (x jobs only; h out, unscaled) or kExpand (h in;
// y jobs only).
template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    sgmv_tc_kernel(const __grid_constant__ DeltaArgs p, const __grid_constant__ TcMaps m) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint64_t *full = bars, *empty = full + kMaxNS;
    uint64_t *d1f = empty + kMaxNS, *hr = d1f + 1, *he = hr + 1, *tf = he + 1, *te = tf + kST, *fin = te + kST;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 16);
    int *range = reinterpret_cast<int *>(smem + kOffMisc + 32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        // the tensor maps of the TMA copies, one per lane: x, y per slice, A
        const CUtensorMap *mp = nullptr;
        if (m.use && MODE != kExpand && lane < 3) mp = lane == 0 ? &m.x64 : lane == 1 ? &m.x32 : &m.x8;
        else if (m.use && MODE != kShrink && lane >= 3 && lane < 3 + 3 * p.n_slices) {
            const int t = (lane - 3) / 3, k = (lane - 3) - 3 * t;
            mp = k == 0 ? &m.y64[t] : k == 1 ? &m.y32[t] : &m.y8[t];
        } else if (m.use_ab && lane >= 16 && lane < 19 && (8 << (lane - 16)) <= m.a_box_max)
            mp = lane == 16 ? &m.a8 : lane == 17 ? &m.a16 : &m.a32;
        if (mp) prefetch_tensormap(mp);
    }
    if (tid == 0) {
        for (int s = 0; s < kMaxNS; ++s) {
            // TMA path: the two issuers' expect_tx and the 64 helper threads;
            // cp.async path: every loader thread and the two issuers
            mbar_init(&full[s], m.use_ab ? 2 + 64 : kLoaderThreads + 2);
            mbar_init(&empty[s], kEpiWarps);  // the epilogue warps, or the MMA thread (kEpiWarps - 1 arrivals + commit)
        }
        mbar_init(d1f, 1);
        mbar_init(hr, 4);
        mbar_init(he, 1);
        for (int s = 0; s < kST; ++s) { mbar_init(&tf[s], 1); mbar_init(&te[s], kEpiWarps); }
        mbar_init(fin, 1);
        fence_mbar_init();
        *abort = 0;
    }
    // Launched right after the CUDA-core kernel (which triggers only after
    // its own wait on prepare), this grid starts at once and waits for its
    // predecessor only before it exits, so that its completion implies the
    // predecessor's.  Otherwise it waits first.
    if (!p.after_cc) griddep_wait();
    griddep_launch_dependents();

    if (tid < 256) {
        // identity I[n][k] = (n == k), K-major without swizzle: 8-column
        // halves 256 bytes apart, 16 bytes per row
        const int n = tid >> 4, k = tid & 15;
        *reinterpret_cast<uint16_t *>(smem + kOffIdent + (k >> 3) * 256 + n * 16 + (k & 7) * 2) =
            n == k ? (uint16_t)0x3F80 : (uint16_t)0;
        fence_proxy_async_smem();
    }
    bool planned = false;
    if (warp == kMmaWarp && p.tc_share != nullptr && p.tc_share_grid == (int)gridDim.x) {
        // the shares prepare computed for this grid over its tensor-core
        // list; a call that routes every segment here (tc_only) takes them
        // when that list holds every segment (the two row spaces are then
        // the same)
        const int2 s0 = p.tc_share[blockIdx.x], s1 = p.tc_share[blockIdx.x + 1];
        planned = !p.tc_only || p.counts[LORA_COUNT_TC_SEGS] == p.counts[LORA_COUNT_SEGS];
        if (planned && lane == 0) {
            range[0] = s0.x;
            range[1] = max(s0.x, s1.x);
            range[2] = s0.x < s1.x ? s0.y : 0;
        }
    }
    if (warp == kMmaWarp && !planned) {
        // This CTA's row range: an equal share of the row space.
        const int nseg = min(p.counts[p.tc_count_index], p.max_list);
        const int Mrows = nseg > 0 ? p.counts[p.tc_rows_index] : 0;
        const int G = gridDim.x, b = blockIdx.x;
        // A share end moves to a boundary between two adapters when one lies
        // within half a share: a tile of one adapter needs no row split by a
        // piece boundary (its rows move by TMA boxes alone) and no second
        // pass when two ranks do not fit one tile.  Chunks of one adapter do
        // not count as boundaries, but only the boundaries of the record
        // holding the end are seen (prepare's table looks at whole adapter
        // groups).  Both neighbours compute the same end.
        const int half = (int)(Mrows / (2 * (int64_t)G));
        auto adapter_of = [&](int i) { return p.tc_adapter[(int64_t)i * p.tc_rec_stride]; };
        auto share_end = [&](int e) {
            if (nseg < 2 || e <= 0 || e >= Mrows) return e;
            const int i = warp_seg_of(p.tc_ptr, nseg, e, lane);
            const int lo = p.tc_ptr[i], hi = p.tc_ptr[i + 1];
            const int a = adapter_of(i);
            if (e - lo <= half && i > 0 && adapter_of(i - 1) != a) return lo;
            if (hi - e <= half && i + 1 < nseg && adapter_of(i + 1) != a) return hi;
            return e;
        };
        const int r0 = share_end((int)((int64_t)Mrows * b / G));
        const int r1 = max(r0, share_end((int)((int64_t)Mrows * (b + 1) / G)));
        const int i0 = r0 < r1 ? warp_seg_of(p.tc_ptr, nseg, r0, lane) : 0;
        if (lane == 0) {
            range[0] = r0;
            range[1] = r1;
            range[2] = i0;
        }
    }
    __syncthreads();
    // A CTA without rows (no tensor-core segments in this batch, or fewer
    // rows than CTAs) leaves before it takes TMEM.
    if (range[0] >= range[1]) {
        if (p.after_cc) griddep_wait();
        return;
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    TileWalker walker{&p, range[0], range[1], range[2]};
    // Stage geometry of this CTA (same in every role).
    const int cap = min(kBM, (range[1] - range[0] + 7) & ~7);
    const int xatom = cap * 128, xbytes = cap * 256, aatom = 4096;
    const int stage_bytes = xbytes + 2 * aatom;
    const int NS = cap > 0 ? min(kMaxNS, kRingBytes / stage_bytes) : 1;

    int n_nt = 0;
    for (int t = 0; t < p.n_slices; ++t) n_nt += (p.slices[t].d_out + kBN - 1) / kBN;
    const int nkb = (p.d_in + kBK - 1) / kBK;
    // Every CTA walks the K blocks and the n-tiles from its own starting
    // point, so that the CTAs do not all hit the same column block at once.
    const int kb_rot = nkb > 0 ? (int)(((uint32_t)blockIdx.x * 2654435761u) >> 7) % nkb : 0;
    const int nt_rot = (int)(((uint32_t)blockIdx.x * 2246822519u) >> 7) % (n_nt > 0 ? n_nt : 1);
    const __nv_bfloat16 *yg = static_cast<const __nv_bfloat16 *>(p.y);
    bool ok = true;

    if (warp < kMmaWarp || warp == kLoaderWarp3) {
        // loader warps 0, 1, 2 and 4 (warp 3 issues the MMAs, so that the
        // MMA thread shares a scheduler with neither TMA issuer); lw numbers
        // them 0-3
        const int lw = warp == kLoaderWarp3 ? 3 : warp;
        // ------------------------------------------------------------ loaders
        // Thread lt copies chunk (lt & 15) of tile rows (lt >> 4) + 8q (row
        // group q) by cp.async where no TMA box covers them; lane 0 of warps
        // 0 and 1 issues the TMA boxes of atoms 0 and 1.  Per tile, each warp
        // writes its tables (row tokens; box list) to shared memory once, so
        // the per-stage loop only reads them.
        const int lt = lw * 32 + lane, c = lt & 15, i0 = lt >> 4;
        const int hq = lw;  // the atom of an issuing warp (0 or 1)
        int32_t *lrow = reinterpret_cast<int32_t *>(smem + kOffLdr) + 32 * lw;      // [slot]: token row
        int32_t *lgt = reinterpret_cast<int32_t *>(smem + kOffLdr + kLdrGtok) + 16 * (lw & 1);  // [g]: token of row 8g
        uint2 *lbox = reinterpret_cast<uint2 *>(smem + kOffLdr + kLdrBox) + 16 * (lw & 1);     // {row | height code << 8, token}
        const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(p.x);
        const __nv_bfloat16 *Ag = static_cast<const __nv_bfloat16 *>(p.A);
        int s = 0;
        uint32_t ph = 0;
        Tile t;
        while (walker.next(t)) {
            if (t.K == 0) continue;
            uint32_t mask8, mask32, mask64;
            int tok8;
            tile_box_masks(p, m, t, lane, mask8, mask32, mask64, tok8);
            // token rows of the 8-row groups (the boxes' first rows), from the masks' reads
            {
                __syncwarp();  // the previous tile's readers are done
                if (lw < 2 && lane < 16) lgt[lane] = 8 * lane < t.n ? (m.use ? tok8 : tile_token(p, t, 8 * lane)) : 0;
                __syncwarp();
            }
            int nbox = 0;
            if (lw < 2 && lane == 0) {
                for (int h = 0; h < 2; ++h) {
                    if ((mask64 >> h) & 1) {
                        lbox[nbox++] = make_uint2(64 * h | 2u << 8, lgt[8 * h]);
                        continue;
                    }
                    for (int j = 2 * h; j < 2 * h + 2; ++j) {
                        if ((mask32 >> j) & 1) {
                            lbox[nbox++] = make_uint2(32 * j | 1u << 8, lgt[4 * j]);
                            continue;
                        }
                        for (int g = 4 * j; g < 4 * j + 4; ++g)
                            if ((mask8 >> g) & 1) lbox[nbox++] = make_uint2(8 * g, lgt[g]);
                    }
                }
            }
            const uint32_t box_bytes = (uint32_t)__popc(mask8) * 8 * 128;  // per atom
            const int K16 = (t.K + 15) & ~15;
            const int n8 = K16 / 8, sh8 = n8 == 2 ? 1 : 2;
            if (m.use_ab) {
                // TMA path.  Lane 0 of warp 0 issues the boxes of atom 0, lane 0 of
                // warp 1 those of atom 1, A block included.  The 64 threads of the
                // other two loader warps copy the B block (small and in L2; a TMA
                // box of it would move 16-byte pieces) and the rows that no box
                // covers (a group split by a piece boundary or by a break in the
                // token rows), from a list built once per tile.  The other lanes
                // of warps 0 and 1 sit these stages out (the full barriers do not
                // count them).
                const int njobs = nkb + n_nt;
                int covered = 0;
                for (int g = 0; g < 16; ++g)
                    if ((mask8 >> g) & 1) covered += min(8, t.n - 8 * g);
                const int nu = t.n - covered;  // rows moved by cp.async
                if (lw < 2 && lane == 0) {
                    // This atom's copies of the tile, resolved once into shared
                    // memory: row boxes first, then the stacked A block in rank
                    // boxes of 32/16/8 (and zero boxes up to K16); the job loop
                    // only adds the column.
                    uint4 *cmd = reinterpret_cast<uint4 *>(smem + kOffLdr + kLdrCmd) + kCmdMax * lw;
                    int ncmd = 0;
                    for (int q = 0; q < nbox; ++q) {
                        const uint2 bx = lbox[q];
                        cmd[ncmd++] = make_uint4((uint32_t)(hq * xatom + (int)(bx.x & 255) * 128), 2u - (bx.x >> 8), bx.y, 0u);
                    }
                    const int nrow = ncmd;
                    const uint32_t abase_off = (uint32_t)(xbytes + hq * aatom);
                    for (int u = 0; u < t.np; ++u) {
                        const int rk = sel(t.rk, u), ko = sel(t.kofs, u), au = sel(t.a, u);
                        for (int j = 0; j < rk;) {
                            const int w = (rk - j >= 32 && m.a_box_max >= 32) ? 32 : (rk - j >= 16 && m.a_box_max >= 16) ? 16 : 8;
                            cmd[ncmd++] = make_uint4(abase_off + (uint32_t)(ko + j) * 128, w == 32 ? 5u : w == 16 ? 4u : 3u,
                                                     (uint32_t)j, (uint32_t)au);
                            j += w;
                        }
                    }
                    for (int j = t.K; j < K16; j += 8)
                        cmd[ncmd++] = make_uint4(abase_off + (uint32_t)j * 128, 3u, (uint32_t)m.r_pad, 0u);
                    const uint32_t x_tx = box_bytes + (uint32_t)(K16 / 8) * 1024;
                    for (int jb = 0; jb < njobs; ++jb) {
                        if (!wait1(&empty[s], ph ^ 1, ok, abort)) goto role_done;
                        unsigned char *st = smem + s * stage_bytes;
                        if (jb < nkb) {
                            const int kb = jb + kb_rot < nkb ? jb + kb_rot : jb + kb_rot - nkb;
                            const int col = kb * kBK + 64 * hq;
                            mbar_arrive_expect_tx(&full[s], x_tx);
                            for (int q = 0; q < ncmd; ++q) {
                                const uint4 c = cmd[q];
                                const int cd = (int)c.y;
                                if (cd < 3)
                                    tma_load_2d(st + c.x, cd == 0 ? &m.x64 : cd == 1 ? &m.x32 : &m.x8, col, (int)c.z, &full[s]);
                                else
                                    tma_load_3d(st + c.x, cd == 5 ? &m.a32 : cd == 4 ? &m.a16 : &m.a8, col, (int)c.z, (int)c.w,
                                                &full[s]);
                            }
                        } else {
                            const int nti = jb - nkb, nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                            int sl, c0, nc;
                            ntile_cols(p, nt, sl, c0, nc);
                            const int col = c0 + 64 * hq;
                            mbar_arrive_expect_tx(&full[s], box_bytes);
                            for (int q = 0; q < nrow; ++q) {
                                const uint4 c = cmd[q];
                                const int cd = (int)c.y;
                                tma_load_2d(st + c.x, cd == 0 ? &m.y64[sl] : cd == 1 ? &m.y32[sl] : &m.y8[sl], col, (int)c.z,
                                            &full[s]);
                            }
                        }
                        if (++s == NS) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                } else if (lw >= 2) {
                    // the uncovered rows: tile row and token row, in this warp's list
                    int2 *ul = reinterpret_cast<int2 *>(smem + kOffLdr + kLdrRows) + kBM * (lw - 2);
                    {
                        int cnt = 0;
                        __syncwarp();
                        for (int i0r = 0; i0r < t.n; i0r += 32) {
                            const int i = i0r + lane;
                            const bool need = i < t.n && !((mask8 >> (i >> 3)) & 1);
                            const unsigned bal = __ballot_sync(0xffffffffu, need);
                            if (need) ul[cnt + __popc(bal & ((1u << lane) - 1))] = make_int2(i, tile_token(p, t, i));
                            cnt += __popc(bal);
                        }
                        __syncwarp();
                    }
                    const int hl = lt - 64, hc = hl & 15, hr0 = hl >> 4;  // chunk; first list entry (then every 4th)
                    // B: chunk hb (8 rank columns) of rows hn0 + (64 / n8) k
                    const int hb = hl & (n8 - 1), hn0 = hl >> (sh8), hstep = 64 >> sh8;
                    int hb_a = 0, hb_j = -1;
#pragma unroll
                    for (int u = 0; u < kMaxPieces; ++u)
                        if (u < t.np && 8 * hb >= t.kofs[u] && 8 * hb < t.kofs[u] + t.rk[u]) {
                            hb_a = t.a[u];
                            hb_j = 8 * hb - t.kofs[u];
                        }
                    for (int jb = 0; jb < njobs; ++jb) {
                        if (!wait_warp(&empty[s], ph ^ 1, ok, abort)) goto role_done;
                        unsigned char *st = smem + s * stage_bytes;
                        if (jb < nkb) {
                            const int kb = jb + kb_rot < nkb ? jb + kb_rot : jb + kb_rot - nkb;
                            const int k = kb * kBK + hc * 8;
                            const bool kin = k < p.d_in;
                            for (int e = hr0; e < nu; e += 4) {
                                const int2 ri = ul[e];
                                const __nv_bfloat16 *row = xg + (int64_t)ri.y * p.ldx;
                                cp_async16(st + schunk(xatom, ri.x, hc), kin ? row + k : row, kin ? 16 : 0);
                            }
                        } else {
                            const int nti = jb - nkb, nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                            int sl, c0, nc;
                            ntile_cols(p, nt, sl, c0, nc);
                            const SliceDesc &S = p.slices[sl];
                            const __nv_bfloat16 *yc = yg + S.y_col + c0;
                            // chunks past the n-tile's last column are zero-filled: the
                            // MMA adds the whole stage (times the identity) into D2
                            for (int e = hr0; e < nu; e += 4) {
                                const int2 ri = ul[e];
                                const __nv_bfloat16 *yr = yc + (int64_t)ri.y * p.ldy;
                                cp_async16(st + schunk(xatom, ri.x, hc), hc * 8 < nc ? yr + hc * 8 : yr, hc * 8 < nc ? 16 : 0);
                            }
                            // the stacked B block: rows c0 .. c0+nc-1 of the slice (columns of no piece zero-filled)
                            const __nv_bfloat16 *Bb =
                                static_cast<const __nv_bfloat16 *>(S.B) + (int64_t)hb_a * S.stride_adapter + hb_j;
                            for (int n = hn0; n < nc; n += hstep)
                                cp_async16(st + xbytes + hb * kBChunk + n * 16,
                                           hb_j >= 0 ? Bb + (int64_t)(c0 + n) * S.stride_n : S.B, hb_j >= 0 ? 16 : 0);
                        }
                        cp_async_arrive_noinc(&full[s]);
                        if (++s == NS) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                } else {
                    for (int jb = 0; jb < njobs; ++jb)
                        if (++s == NS) {
                            s = 0;
                            ph ^= 1;
                        }
                }
                continue;
            }
            // cp.async path: this lane's slot, tile row (2 warp + (lane & 1)) + 8 (lane >> 1)
            {
                const int i = 2 * lw + (lane & 1) + 8 * (lane >> 1);
                __syncwarp();  // the previous tile's readers are done
                lrow[lane] = i < t.n ? tile_token(p, t, i) : 0;
                __syncwarp();
            }
            // cp.async rows of this thread: bit q = row i0 + 8q
            uint32_t mine = 0;
#pragma unroll
            for (int q = 0; q < kBM / 8; ++q) mine |= (i0 + 8 * q < t.n && !((mask8 >> q) & 1)) ? 1u << q : 0u;
            // per-thread tables of the A rows and the B chunk
            // A rows j = i0 + 8q of the stacked block: adapter row, or -1 (zero)
            int arow[kTcMaxRank / 8];
            const __nv_bfloat16 *abase[kTcMaxRank / 8];
#pragma unroll
            for (int q = 0; q < kTcMaxRank / 8; ++q) {
                const int j = i0 + 8 * q;
                arow[q] = -1;
                abase[q] = Ag;
#pragma unroll
                for (int u = 0; u < kMaxPieces; ++u)
                    if (u < t.np && j >= t.kofs[u] && j < t.kofs[u] + t.rk[u]) {
                        arow[q] = j - t.kofs[u];
                        abase[q] = Ag + (int64_t)t.a[u] * p.a_stride_adapter;
                    }
            }
            // this thread's B chunk (8 rank columns; the same in every y job):
            // adapter and first column, or -1 (zero)
            const int bcb = lt & (n8 - 1);
            int b_a = 0, b_j = -1;
#pragma unroll
            for (int u = 0; u < kMaxPieces; ++u)
                if (u < t.np && 8 * bcb >= t.kofs[u] && 8 * bcb < t.kofs[u] + t.rk[u]) {
                    b_a = t.a[u];
                    b_j = 8 * bcb - t.kofs[u];
                }
            const int slot_hi = (lt >> 4) & 1;  // lrow index of row i0 + 8q is 2q + slot_hi
            for (int kbi = 0; kbi < nkb; ++kbi) {
                const int kb = kbi + kb_rot < nkb ? kbi + kb_rot : kbi + kb_rot - nkb;
                if (!wait_warp(&empty[s], ph ^ 1, ok, abort)) goto role_done;
                unsigned char *st = smem + s * stage_bytes;
                const int k = kb * kBK + c * 8;
                const bool kin = k < p.d_in;
                if (lw < 2 && lane == 0) {
                    // the expected bytes are announced before the boxes are issued
                    mbar_arrive_expect_tx(&full[s], box_bytes);
                    unsigned char *dst = st + hq * xatom;
                    const int col = kb * kBK + 64 * hq;
                    for (int e = 0; e < nbox; ++e) {
                        const uint2 bx = lbox[e];
                        const int code = bx.x >> 8, i = bx.x & 255;
                        tma_load_2d(dst + i * 128, code == 2 ? &m.x64 : code == 1 ? &m.x32 : &m.x8, col, (int)bx.y,
                                    &full[s]);
                    }
                }
                // x rows not moved by TMA: two 64-column atoms in the 128-byte swizzle
                unsigned char *xd = st + (c >> 3) * xatom + (((c & 7) ^ (i0 & 7)) << 4);
#pragma unroll
                for (int q = 0; q < kBM / 8; ++q) {
                    if (!((mine >> q) & 1)) continue;
                    const __nv_bfloat16 *row = xg + (int64_t)lrow[2 * q + slot_hi] * p.ldx;
                    cp_async16(xd + (i0 + 8 * q) * 128, kin ? row + k : row, kin ? 16 : 0);
                }
                // the stacked A block (rows of no piece, or past a rank, zero-filled)
                unsigned char *ad = st + xbytes + (c >> 3) * aatom + (((c & 7) ^ (i0 & 7)) << 4);
#pragma unroll
                for (int q = 0; q < kTcMaxRank / 8; ++q) {
                    if (i0 + 8 * q >= K16) break;
                    const bool in = arow[q] >= 0 && kin;
                    cp_async16(ad + (i0 + 8 * q) * 128, in ? abase[q] + (int64_t)arow[q] * p.a_stride_r + k : Ag,
                               in ? 16 : 0);
                }
                cp_async_arrive_noinc(&full[s]);
                if (++s == NS) {
                    s = 0;
                    ph ^= 1;
                }
            }
            for (int nti = 0; nti < n_nt; ++nti) {
                const int nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                int sl, c0, nc;
                ntile_cols(p, nt, sl, c0, nc);
                const SliceDesc &S = p.slices[sl];
                if (!wait_warp(&empty[s], ph ^ 1, ok, abort)) goto role_done;
                unsigned char *st = smem + s * stage_bytes;
                if (lw < 2 && lane == 0) {
                    mbar_arrive_expect_tx(&full[s], box_bytes);
                    unsigned char *dst = st + hq * xatom;
                    const int col = c0 + 64 * hq;
                    for (int e = 0; e < nbox; ++e) {
                        const uint2 bx = lbox[e];
                        const int code = bx.x >> 8, i = bx.x & 255;
                        tma_load_2d(dst + i * 128, code == 2 ? &m.y64[sl] : code == 1 ? &m.y32[sl] : &m.y8[sl], col,
                                    (int)bx.y, &full[s]);
                    }
                }
                const __nv_bfloat16 *yc = yg + S.y_col + c0;
                if (nc == kBN) {
#pragma unroll
                    for (int q = 0; q < kBM / 8; ++q) {
                        if (!((mine >> q) & 1)) continue;
                        cp_async16(st + schunk(xatom, i0 + 8 * q, c), yc + (int64_t)lrow[2 * q + slot_hi] * p.ldy + c * 8, 16);
                    }
                } else {
                    // chunks past the n-tile's last column are zero-filled
                    const int nch = nc >> 3;
                    for (int e = lt; e < t.n * 16; e += kLoaderThreads) {
                        const int i = e >> 4, cc = e & 15;
                        if ((mask8 >> (i >> 3)) & 1) continue;
                        const __nv_bfloat16 *yr = yc + (int64_t)tile_token(p, t, i) * p.ldy;
                        cp_async16(st + schunk(xatom, i, cc), cc < nch ? yr + cc * 8 : yr, cc < nch ? 16 : 0);
                    }
                }
                // the stacked B block: rows c0 .. c0+nc-1 of the slice, 8 rank
                // columns per 2 KB chunk (columns of no piece zero-filled)
                const __nv_bfloat16 *Bb = static_cast<const __nv_bfloat16 *>(S.B) + (int64_t)b_a * S.stride_adapter + b_j;
                for (int e = lt; e < nc * n8; e += kLoaderThreads) {
                    const int n = e >> sh8;
                    cp_async16(st + xbytes + bcb * kBChunk + n * 16, b_j >= 0 ? Bb + (int64_t)(c0 + n) * S.stride_n : S.B,
                               b_j >= 0 ? 16 : 0);
                }
                cp_async_arrive_noinc(&full[s]);
                if (++s == NS) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t job = 0, ts = 0, tiles = 0;
            const uint32_t id2 = idesc_bf16(kBM, kBN), idi = idesc_bf16(kBM, 16);
            const uint32_t ring = smem_u32(smem), h_base = smem_u32(smem + kOffH);
            const uint64_t ident = smem_desc(smem_u32(smem + kOffIdent), 256, 128, kLayoutNone);
            Tile t;
            while (walker.next(t)) {
                if (t.K == 0) continue;
                const int n16 = (t.K + 15) / 16;
                const uint32_t id1 = idesc_bf16(kBM, 16 * n16);
                // D1 is free again: the previous tile's expand was issued only
                // after the epilogue had read D1 (hr).
                for (int kbi = 0; kbi < nkb; ++kbi, ++job) {
                    const int s = job % NS;
                    if (!wait1(&full[s], (job / NS) & 1, ok, abort)) goto role_done;
                    tc_fence_after();
                    fence_proxy_async_smem();  // rows the helpers wrote by cp.async
                    const uint32_t xa = ring + s * stage_bytes, aa = xa + xbytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * xatom + (kk & 3) * 32, aoff = (kk >> 2) * aatom + (kk & 3) * 32;
                        // four accumulators (TMEM columns 32 q) take the K steps in
                        // turn, so consecutive MMAs do not wait on one another
                        umma(tmem + 32 * (kk & 3), smem_desc(xa + off, 16, 1024, kLayoutSw128),
                             smem_desc(aa + aoff, 16, 1024, kLayoutSw128), id1, (kbi | (kk >> 2)) != 0);
                    }
                    // the stage is free once these MMAs have read it
                    mbar_arrive_n(&empty[s], kEpiWarps - 1);
                    umma_commit(&empty[s]);
                }
                if (MODE != kExpand) umma_commit(d1f);
                // H of this tile is ready once the epilogue has written it
                // (shrink only: the epilogue has read D1)
                if (!wait1(hr, tiles & 1, ok, abort)) goto role_done;
                tc_fence_after();
                for (int nt = 0; nt < n_nt; ++nt, ++job, ++ts) {
                    const int s = job % NS, sd = ts % kST;
                    if (!wait1(&full[s], (job / NS) & 1, ok, abort)) goto role_done;
                    if (!wait1(&te[sd], ((ts / kST) & 1) ^ 1, ok, abort)) goto role_done;
                    tc_fence_after();
                    fence_proxy_async_smem();  // rows the helpers wrote by cp.async
                    const uint32_t ya = ring + s * stage_bytes, bb = ya + xbytes;
                    const uint32_t d2 = tmem + 128 + 128 * sd;
                    // D2 = y: columns 16 kk .. +15 take the y stage's K block kk
                    // times the identity (exact: one product per column is y, the
                    // others are zero), so the epilogue needs no y of its own
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        umma(d2 + 16 * kk, smem_desc(ya + (kk >> 2) * xatom + (kk & 3) * 32, 16, 1024, kLayoutSw128),
                             ident, idi, 0);
                    // D2 += H . B^T
                    for (int kc = 0; kc < n16; ++kc)
                        umma(d2, smem_desc(h_base + kc * 2 * kHChunk, kHChunk, 128, kLayoutNone),
                             smem_desc(bb + kc * 2 * kBChunk, kBChunk, 128, kLayoutNone), id2, 1);
                    umma_commit(&tf[sd]);
                }
                if (MODE != kShrink) umma_commit(he);
                ++tiles;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kEpiWarp0;     // 0..7
        const int q4 = warp & 3;             // TMEM lane quadrant
        const int chalf = ew >> 2;           // which kEpiCols columns of an n-tile
        const int row = q4 * 32 + lane;      // tile row owned by this thread
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        unsigned char *H = smem + kOffH;
        __nv_bfloat16 *yw = static_cast<__nv_bfloat16 *>(p.y);
        uint32_t job = 0, ts = 0, tiles = 0;
        Tile t;
        while (walker.next(t)) {
            // Pieces the tensor cores cannot take are the CUDA-core kernel's;
            // with the tensor-core path forced they are an error.
            if (p.tc_only && ew == 0 && lane < t.np && sel(t.rk, lane) == 0 && sel(t.rank, lane) != 0)
                raise_deverr(p.counts, LORA_DEVERR_RANK);
            if (MODE == kShrink && p.tc_only && chalf == 0 && row < t.n && sel(t.rank, t.piece_of(row)) == 0) {
                // every segment is this kernel's: h rows of rank-0 adapters are zero
                float *hrow = p.h + (int64_t)tile_token(p, t, row) * p.ldh;
                for (int j = 0; j < p.r_max; ++j) hrow[j] = 0.f;
            }
            if (t.K == 0) continue;
            job += nkb;  // the x stages of this tile are the MMA's
            const int K16 = (t.K + 15) & ~15;
            // this thread's row: token row, piece, rank columns and scale
            const int pq = row < t.n ? t.piece_of(row) : 0;
            const bool live = row < t.n && sel(t.rk, pq) > 0;
            const int my_tok = row < t.n ? tile_token(p, t, row) : 0;
            const int k_lo = live ? sel(t.kofs, pq) : 0, k_hi = live ? sel(t.kofs, pq) + sel(t.rk, pq) : 0;
            const float sc = live ? (p.adapter_scale ? p.adapter_scale[sel(t.a, pq)] : p.scale) : 0.f;
            if (chalf == 0 && MODE == kExpand) {
                // ---- h (global, fp32) -> scale -> bf16 H (columns of other pieces are zero)
                if (tiles > 0)
                    if (!wait_warp(he, (tiles - 1) & 1, ok, abort)) goto role_done;  // previous expand done with H
                const float *hrow = p.h + (int64_t)my_tok * p.ldh;
                for (int c8 = 0; c8 < kTcMaxRank / 8; ++c8) {
                    if (8 * c8 >= K16) break;
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 8 * c8 + 2 * e;
                        const float f0 = j >= k_lo && j < k_hi ? hrow[j - k_lo] * sc : 0.f;
                        const float f1 = j + 1 >= k_lo && j + 1 < k_hi ? hrow[j + 1 - k_lo] * sc : 0.f;
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
                        w[e] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    *reinterpret_cast<uint4 *>(H + c8 * kHChunk + row * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(hr);
            } else if (chalf == 0) {
                // ---- D1 -> scale -> bf16 H (columns of other pieces are
                // zero), or (shrink) D1 -> h in global memory, unscaled, zero
                // past the rank
                if (!wait_warp(d1f, tiles & 1, ok, abort)) goto role_done;
                tc_fence_after();
                if (tiles > 0 && MODE != kShrink)
                    if (!wait_warp(he, (tiles - 1) & 1, ok, abort)) goto role_done;  // previous expand done with H
                float *hout = MODE == kShrink && live ? p.h + (int64_t)my_tok * p.ldh : nullptr;
                for (int c16 = 0; c16 < kTcMaxRank / 16; ++c16) {
                    if (16 * c16 >= K16) break;
                    uint32_t v[16], u[3][16];
                    tmem_ld16(tmem + lane_off + 16 * c16, v);
#pragma unroll
                    for (int q = 0; q < 3; ++q) tmem_ld16(tmem + lane_off + 32 * (q + 1) + 16 * c16, u[q]);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        v[e] = __float_as_uint((__uint_as_float(v[e]) + __uint_as_float(u[0][e])) +
                                               (__uint_as_float(u[1][e]) + __uint_as_float(u[2][e])));
                    if (MODE == kShrink) {
                        if (hout) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int j = 16 * c16 + e - k_lo;
                                if (j >= 0 && j < k_hi - k_lo) hout[j] = __uint_as_float(v[e]);
                            }
                        }
                        continue;
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int c8 = 2 * c16 + half;
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 8 * c8 + 2 * e;
                            const float f0 = j >= k_lo && j < k_hi ? __uint_as_float(v[8 * half + 2 * e]) * sc : 0.f;
                            const float f1 = j + 1 >= k_lo && j + 1 < k_hi ? __uint_as_float(v[8 * half + 2 * e + 1]) * sc : 0.f;
                            const __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
                            w[e] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        *reinterpret_cast<uint4 *>(H + c8 * kHChunk + row * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                if (hout)
                    for (int j = k_hi - k_lo; j < p.r_max; ++j) hout[j] = 0.f;
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(hr);
            }
            // ---- expand n-tiles: y = D2 (this warp: 32 rows x kEpiCols columns)
            // Per tile, once: the rows this lane stores (8 k + lane / kEpiChunks
            // of the warp's quadrant) as offsets into y (-1: no row or rank 0),
            // the stage offsets it reads them from (rows 8 apart: + 1024 k)
            // and the offsets of its own row's chunks.
            static_assert(kEpiChunks == 4, "store map: 4 chunks per row piece, 8 rows per instruction");
            int64_t srow[kEpiChunks];
#pragma unroll
            for (int k = 0; k < kEpiChunks; ++k) {
                const int rl = 8 * k + lane / kEpiChunks;
                const int tok = __shfl_sync(0xffffffffu, my_tok, rl);
                const bool lv = __shfl_sync(0xffffffffu, live, rl);
                srow[k] = lv ? (int64_t)tok * p.ldy : -1;
            }
            const int ccol = kEpiChunks * chalf + lane % kEpiChunks;  // this lane's 16-byte chunk of a row
            const int ld_off = schunk(xatom, q4 * 32 + lane / kEpiChunks, ccol);
            int st_off[kEpiChunks];
#pragma unroll
            for (int q = 0; q < kEpiChunks; ++q) st_off[q] = schunk(xatom, row, kEpiChunks * chalf + q);
            // this row's first H column and rank (for the rare exact path)
            const int rinfo = k_lo | ((k_hi - k_lo) << 8), radapter = live ? sel(t.a, pq) : 0;
            for (int nti = 0; nti < n_nt; ++nti, ++job, ++ts) {
                const int nt = nti + nt_rot < n_nt ? nti + nt_rot : nti + nt_rot - n_nt;
                const int s = job % NS, sd = ts % kST;
                int sl, c0, nc;
                ntile_cols(p, nt, sl, c0, nc);
                const SliceDesc &S = p.slices[sl];
                // D2 holds y + delta (the MMA read this job's y stage before it
                // committed tf)
                if (!wait_warp(&tf[sd], (ts / kST) & 1, ok, abort)) goto role_done;
                tc_fence_after();
                uint32_t v[kEpiCols / 16][16];
                const uint32_t ta = tmem + 128 + 128 * sd + lane_off + kEpiCols * chalf;
#pragma unroll
                for (int q = 0; q < kEpiCols / 16; ++q) tmem_ld16(ta + 16 * q, v[q]);
                tmem_wait_ld();
                // the TMEM buffer is free as soon as it is read
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&te[sd]);
                // round once to bf16, into the stage in place of y (rows of the
                // tile only: the stage holds cap rows per atom)
                unsigned char *ys = smem + s * stage_bytes;
#pragma unroll
                for (int q = 0; q < kEpiChunks; ++q) {
                    if (!live) break;
                    // Any output not finite?  (x * 0 is 0 for finite x and NaN
                    // for an infinity or NaN; the sum of eight such products is
                    // NaN exactly when one of the eight is.)
                    float z = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) z = fmaf(__uint_as_float(v[q >> 1][(q & 1) * 8 + e]), 0.f, z);
                    if (z == z) {
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[q >> 1][(q & 1) * 8 + 2 * e]),
                                                                            __uint_as_float(v[q >> 1][(q & 1) * 8 + 2 * e + 1]));
                            o[e] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        *reinterpret_cast<uint4 *>(ys + st_off[q]) = make_uint4(o[0], o[1], o[2], o[3]);
                    } else {
                        // A y value that is not finite reaches every output of its
                        // row's 16-column group through the identity product
                        // (0 * inf is NaN).  This chunk's outputs are formed again,
                        // y + delta in fp32 from the chunk's y (still in the
                        // stage), the row's H and the adapter's B rows (see
                        // exact_output): exact for every element.
                        unsigned char *yc = ys + st_off[q];
#pragma unroll 1
                        for (int e = 0; e < 8; ++e) {
                            const uint32_t w = reinterpret_cast<const uint32_t *>(yc)[e >> 1];
                            const float out = exact_output(w, e, H, row, rinfo & 0xFF, rinfo >> 8, S, radapter,
                                                           c0 + kEpiCols * chalf + 8 * q + e);
                            *reinterpret_cast<__nv_bfloat16 *>(yc + 2 * e) = __float2bfloat16_rn(out);
                        }
                    }
                }
                __syncwarp();
                // store the warp's live rows: 8 row pieces of kEpiCols columns
                // per instruction (st.global: TMA stores mixed with these in
                // one CTA stalled its loads)
                if (ccol * 8 < nc) {
                    __nv_bfloat16 *ydst = yw + S.y_col + c0 + ccol * 8;
#pragma unroll
                    for (int k = 0; k < kEpiChunks; ++k)
                        if (srow[k] >= 0)
                            *reinterpret_cast<uint4 *>(ydst + srow[k]) = *reinterpret_cast<const uint4 *>(ys + ld_off + 1024 * k);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            ++tiles;
        }
    }
role_done:
    if (warp < kMmaWarp || warp == kLoaderWarp3) asm volatile("cp.async.wait_all;\n" ::: "memory");
    if (warp == kMmaWarp && lane == 0) {
        // every MMA this CTA issued has completed before TMEM is released
        umma_commit(fin);
        if (!mbar_wait(fin, 0)) ok = false;
    }
    if (!ok) raise_deverr(p.counts, LORA_DEVERR_WAIT);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
    }
    if (p.after_cc) griddep_wait();
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
bool tc_available() { return true; }

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (no link-time dependency on it).
EncodeTiledFn encode_fn() {
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

// Row-major bf16 matrix of `rows` x `cols` with row pitch `ld` elements;
// boxes of 64 columns x box_rows rows, 128-byte swizzle, zero fill.
bool encode_rows(EncodeTiledFn fn, CUtensorMap *map, const void *base, int64_t cols, int64_t rows, int64_t ld,
                 int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc(const DeltaArgs &p, int mode, int sms, cudaStream_t stream) {
    if (mode != kFused && mode != kShrink && mode != kExpand) return cudaErrorNotSupported;
    static DeviceOnce once[3];
    auto kern = mode == kShrink ? sgmv_tc_kernel<kShrink> : mode == kExpand ? sgmv_tc_kernel<kExpand> : sgmv_tc_kernel<kFused>;
    cudaError_t e = once[mode].run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    });
    if (e != cudaSuccess) return e;
    // Tensor maps for the TMA copies of contiguous row groups; without them
    // (no driver entry point, a shape the encoder refuses) every row moves
    // by cp.async.
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    EncodeTiledFn fn = encode_fn();
    // (shrink: x and A only; expand: y and B only)
    bool use = fn != nullptr;
    if (use && mode != kExpand)
        use = encode_rows(fn, &maps.x64, p.x, p.d_in, p.M_rows, p.ldx, 64) &&
              encode_rows(fn, &maps.x32, p.x, p.d_in, p.M_rows, p.ldx, 32) &&
              encode_rows(fn, &maps.x8, p.x, p.d_in, p.M_rows, p.ldx, 8);
    for (int t = 0; use && mode != kShrink && t < p.n_slices; ++t) {
        const void *yb = static_cast<const __nv_bfloat16 *>(p.y) + p.slices[t].y_col;
        use = encode_rows(fn, &maps.y64[t], yb, p.slices[t].d_out, p.M_rows, p.ldy, 64) &&
              encode_rows(fn, &maps.y32[t], yb, p.slices[t].d_out, p.M_rows, p.ldy, 32) &&
              encode_rows(fn, &maps.y8[t], yb, p.slices[t].d_out, p.M_rows, p.ldy, 8);
    }
    maps.use = use ? 1 : 0;
    // A and B pools as 3-D maps (rank rows / columns past r_pad read zeros)
    bool use_ab = use;
    maps.r_pad = (p.r_max + 7) & ~7;
    if (use_ab && mode != kExpand) {
        const cuuint64_t dims[3] = {(cuuint64_t)p.d_in, (cuuint64_t)p.r_max, (cuuint64_t)p.n_adapters};
        const cuuint64_t strides[2] = {(cuuint64_t)(p.a_stride_r * 2), (cuuint64_t)(p.a_stride_adapter * 2)};
        const cuuint32_t box[3] = {64, 8, 1}, elem[3] = {1, 1, 1};
        use_ab = fn(&maps.a8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.A), dims, strides, box, elem,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        // wider rank boxes, one TMA copy per 16 or 32 rank rows of a piece
        maps.a_box_max = 8;
        CUtensorMap *wide[2] = {&maps.a16, &maps.a32};
        for (int w = 0; use_ab && w < 2 && p.r_max >= 16 << w; ++w) {
            const cuuint32_t boxw[3] = {64, (cuuint32_t)(16 << w), 1};
            if (fn(wide[w], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.A), dims, strides, boxw, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                break;
            maps.a_box_max = 16 << w;
        }
    }
    for (int t = 0; use_ab && mode != kShrink && t < p.n_slices; ++t) {
        const SliceDesc &S = p.slices[t];
        const cuuint64_t dims[3] = {(cuuint64_t)p.r_max, (cuuint64_t)S.d_out, (cuuint64_t)p.n_adapters};
        const cuuint64_t strides[2] = {(cuuint64_t)(S.stride_n * 2), (cuuint64_t)(S.stride_adapter * 2)};
        const cuuint32_t box[3] = {8, (cuuint32_t)kBN, 1}, elem[3] = {1, 1, 1};
        use_ab = fn(&maps.b[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(S.B), dims, strides, box, elem,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    maps.use_ab = use_ab ? 1 : 0;
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
    return cudaLaunchKernelEx(&cfg, kern, p, maps);
}

}  // namespace lora
