// sgmv_cc.cu -- SGMV kernel for small segments (decode): clusters of CTAs,
// warp-level tensor-core tiles for bf16 (the "CUDA-core" path of the API,
// where fp32 inputs run on CUDA-core FMAs).
//
// Each segment (rows that share one adapter) is handled by one thread-block
// cluster of CL CTAs ("vLLM-Ascend LoRA" article, section 3.3: the rows of
// one adapter are gathered, tmp = rows . A^T, delta = (tmp * scale) . B^T,
// scatter-added; the adapter's A/B are moved once and reused by all rows of
// the segment).  CTA q of the cluster owns
//   - the K slice q of d_in for the shrink (A rows r x K/CL, x rows R x K/CL),
//   - the N slice q of d_out for the expand (B rows N/CL x r, y rows R x N/CL),
// so every byte of x, A, B and y is read once per segment tile.  The partial
// h of the K slices is pushed to every CTA of the cluster through
// distributed shared memory and summed in a fixed order, so every CTA holds
// the same h; h never leaves the chip.
//
// Order: cluster c takes segments c, c + C, ... (C clusters); with
// per-adapter ranks and more segments than clusters, the CTAs first deal the
// tiles to the clusters by an estimate of their time (the work plan below).
//
// Latency: a segment is reached through one 128-byte descriptor that holds
// its first rows inline, so every load address of the tile is known after a
// single dependent read.  All x/A (shrink) and y/B (expand) bytes of a tile
// are then requested at once with 16-byte cp.async (gathered rows cost the
// same as contiguous ones; bulk async copies of row pieces are far slower on
// row-gathered data); B rows land in an XOR-swizzled layout and are read only
// up to the adapter's rank.
//
// Compute, bf16 inputs: warp-level tensor-core products (16 x 8 x 16 bf16
// tiles, fp32 accumulators in registers).  Shrink -- the R x r output is cut
// into 16 x 8 tiles; each warp takes one tile and every (16 / tiles)-th K
// step, with four accumulators so that four products are in flight; the
// warps' partial tiles are summed in warp order.  Expand -- h (scaled fp32)
// is rounded once to bf16 in fragment order; each warp takes eight 8-column
// tiles at a time (four when the tile has more than 16 rows), adds y in the
// stage and the stage leaves in 16-byte row pieces.  A tile of a few rows costs a handful of instructions per warp,
// with no tensor-memory allocation or commit round trip on the path.
// fp32 inputs (packed FFMA2, exact fp32 products): shrink -- every thread
// owns a 4-row x 4-rank block of h and strides over K with its accumulators
// live across all K chunks; lanes sharing a block are reduced once, at the
// end.  Expand -- every thread owns two adjacent output columns and all rows
// of the tile.
#include <type_traits>

#include "common.cuh"

namespace lora {

constexpr int kCcThreads = 512;
constexpr int kCcStages = 3;
constexpr int kCcMaxCluster = 8;
// Work plan limits: segment lists and tile counts above these are walked
// round-robin instead.
constexpr int kPlanMaxSegs = 256;
constexpr int kPlanMaxTiles = 512;

// Shared-memory layout of one launch (computed on the host).
struct CcGeom {
    int RT;           // rows per tile (multiple of 4, <= kInlineRows)
    int HP;           // r_max rounded up to 8
    int stage_bytes;  // bytes per ring stage (multiple of 128)
    int off_bars, off_desc, off_rows, off_slots, off_recv, off_hfull, off_plan, off_ring;
    int total;
};

__host__ __device__ __forceinline__ int cc_rows_per_tile(int r_max) {
    int rt = 1024 / (r_max > 0 ? r_max : 1);
    rt = rt > kInlineRows ? kInlineRows : rt;
    rt = rt < 8 ? 8 : rt;
    return rt & ~3;
}

__device__ __forceinline__ int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}
__device__ __forceinline__ int ilog2(int v) { return 31 - __clz(v); }

// Position of 16-byte chunk c of B row n in a stage whose rows hold rvp
// chunks: an XOR swizzle that spreads rows read together over the banks.
__device__ __forceinline__ int b_swizzle(int n, int c, int rvp) {
    if (rvp >= 8) return c ^ (n & 7);
    const int sh = rvp == 1 ? 3 : rvp == 2 ? 2 : 1;
    return c ^ ((n >> sh) & (rvp - 1));
}

// Maps a column of the concatenated output range to its slice.
__device__ __forceinline__ int slice_of(const DeltaArgs &p, int col) {
    int t = 0;
#pragma unroll
    for (int u = 1; u < LORA_MAX_SLICES; ++u)
        if (u < p.n_slices && col >= p.slices[u].col_begin) t = u;
    return t;
}

// Reduces 16 values over groups of KS adjacent lanes (KS a power of two,
// 1..32).  Afterwards v[i] (i < 16 >> min(log2 KS, 4)) holds the group total
// of entry idx(i, lane) = i + sum_s bit_{S-1-s}(lane) * (16 >> (s+1)).
__device__ __forceinline__ void group_reduce16(float (&v)[16], int lane, int S) {
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        if (st >= S) break;
        const int off = 1 << (S - 1 - st);
        if (st < 4) {
            const int half = 8 >> st;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
}

// bf16 products of a tile: D[16 x 8] += A[16 x 16] . B[16 x 8] on the warp's
// tensor cores, fp32 accumulators in registers.  With g = lane / 4 and
// t = lane % 4: a[0] holds A row g, k = 2t, 2t+1 (lower k in the low half),
// a[1] row g + 8, a[2] row g with k + 8, a[3] row g + 8 with k + 8; b0 holds
// B column g at k = 2t, 2t+1 and b1 the same column at k + 8; d[0], d[1] are
// D row g, columns 2t, 2t+1 and d[2], d[3] row g + 8.  No shared-memory
// staging of operands or accumulators is needed, so a tile of a few rows
// costs a handful of instructions per warp.
__device__ __forceinline__ void mma_16x8x16_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds_u32(const unsigned char *p) { return *reinterpret_cast<const uint32_t *>(p); }

template <typename T, int MODE>
__global__ void __launch_bounds__(kCcThreads, 1)
    sgmv_cc_kernel(const __grid_constant__ DeltaArgs p, const __grid_constant__ CcGeom g) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int PV = V / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    int32_t *desc_s = reinterpret_cast<int32_t *>(smem + g.off_desc);  // [32]
    int32_t *rows_s = reinterpret_cast<int32_t *>(smem + g.off_rows);  // [RT]
    float *slots = reinterpret_cast<float *>(smem + g.off_slots);      // 16 KB: fp32 block totals, bf16 partial tiles + h fragments
    float *recv = reinterpret_cast<float *>(smem + g.off_recv);        // [CL][RT][HP]
    float *h_full = reinterpret_cast<float *>(smem + g.off_hfull);     // [RT][HP]
    unsigned char *ring = smem + g.off_ring;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t CL = cluster_nctarank(), q = cluster_ctarank();
    const uint32_t cid = cluster_id_x(), ncl = nclusters_x();
    const int RT = g.RT, HP = g.HP, SB = g.stage_bytes;

    griddep_wait();
    griddep_launch_dependents();

    const int kv_total = p.d_in / V;
    const int kv0 = (int)((int64_t)kv_total * q / CL), kv1 = (int)((int64_t)kv_total * (q + 1) / CL);
    const int nv_total = p.d_out_total / V;
    const int nv0 = (int)((int64_t)nv_total * q / CL), nv1 = (int)((int64_t)nv_total * (q + 1) / CL);
    const T *xg = static_cast<const T *>(p.x);
    const T *Ag = static_cast<const T *>(p.A);
    uint32_t gjob = 0;  // jobs issued so far by this CTA (ring position and barrier phase)
    bool pushed = false;  // this CTA has pushed a tile's partial h before

    // Segments this kernel takes (the others belong to the tensor-core
    // kernel, or add nothing).
    auto seg_taken = [&](int len, int flags, int r) {
        if (len == 0 || len < p.min_len) return false;
        // segments of long adapter groups (flagged by prepare) belong to the
        // tensor-core kernel when it can take their rank
        if (p.split_tc && (flags & LORA_DESC_TC_FLAG) && tc_rank_ok(r)) return false;
        if (r == 0 && MODE != kShrink) return false;  // rank 0: nothing to add
        return true;
    };

    // ---- work plan.  By default cluster c walks segments c, c + C, ...
    // (C clusters).  With per-adapter ranks the tiles differ in cost several
    // fold, and that order can leave one cluster with several heavy tiles;
    // then, with more segments than clusters, every CTA builds the same
    // plan: each tile of a taken segment gets an estimate of its time (a
    // fixed part plus the bytes a CTA moves), the tiles are ranked by it
    // (ties by position) and dealt to the clusters in snake order -- 0..C-1,
    // then C-1..0, ... -- largest first.  The descriptors, ranks and the
    // segment count are read in one round trip.
    int32_t *plan = reinterpret_cast<int32_t *>(smem + g.off_plan);  // [0] = tiles of this cluster, then the tiles
    int n_plan = -1;  // -1: round-robin over segments
    const bool may_plan = p.ranks != nullptr && p.counts != nullptr && p.n_adapters <= kCcThreads;
    int4 pd = make_int4(0, 0, 0, 0);  // this thread's descriptor head {start, len, adapter, flags}
    int32_t *p_rank = reinterpret_cast<int32_t *>(ring);  // scratch in the (still unused) ring
    // With a small-segment list (every adapter at the pool's rank, one the
    // tensor cores take) the segments of this kernel are exactly that list:
    // the round robin walks it instead of every descriptor.
    const bool by_list = p.split_tc && p.small_list != nullptr;
    const int n_list = by_list ? min(__ldcg(p.counts + LORA_COUNT_SMALL_SEGS), p.max_list) : 0;
    if (tid < 32 && !by_list) desc_s[tid] = reinterpret_cast<const int32_t *>(p.desc + cid)[tid];  // round-robin's first
    if (may_plan) {
        if (tid < min(p.max_list, kPlanMaxSegs)) pd = *reinterpret_cast<const int4 *>(p.desc + tid);
        if (tid < p.n_adapters) p_rank[tid] = p.ranks[tid];
        if (tid == 32) plan[0] = min(p.counts[LORA_COUNT_SEGS], p.max_list);
    }
    __syncthreads();
    const int S_all = may_plan ? plan[0] : -1;
    if (S_all > (int)ncl && S_all <= kPlanMaxSegs) {
        // per segment its tile count, then per tile its cost and code
        // (segment << 16 | tile)
        int32_t *s_tiles = p_rank + kCcThreads;                                 // [kPlanMaxSegs + 1]
        float *t_cost = reinterpret_cast<float *>(s_tiles + kPlanMaxSegs + 1);  // [kPlanMaxTiles]
        int32_t *t_code = reinterpret_cast<int32_t *>(t_cost + kPlanMaxTiles);  // [kPlanMaxTiles]
        int my_r = 0, my_nt = 0;
        if (tid < S_all) {
            my_r = pd.z >= 0 && pd.z < p.n_adapters ? p_rank[pd.z] : -1;
            if (seg_taken(pd.y, pd.w, my_r)) {
                if (my_r < 0 || my_r > p.r_max) {
                    if (cid == 0 && q == 0) raise_deverr(p.counts, LORA_DEVERR_RANK);
                } else {
                    my_nt = (pd.y + RT - 1) / RT;
                }
            }
        }
        // exclusive prefix sum of the tile counts over the first S_all
        // threads (warp scans, then the warp totals)
        int x = my_nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        int *wsum = reinterpret_cast<int *>(t_code + kPlanMaxTiles);  // [16]
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += wsum[w];
        if (tid < S_all) s_tiles[tid] = base + x - my_nt;
        if (tid == kCcThreads - 1) s_tiles[S_all] = base + x;  // total (threads past S_all add 0)
        __syncthreads();
        const int NT = s_tiles[S_all];
        if (NT > (int)ncl && NT <= kPlanMaxTiles) {
            const float es = (float)sizeof(T);
            const float per_rank = (float)(p.d_in + p.d_out_total) * es / (float)CL;
            const float per_row = (float)(p.d_in + 2 * p.d_out_total) * es / (float)CL;
            const float fixed = 120000.f;  // about 3 us of one CTA's streaming, in bytes
            if (tid < S_all) {
                const int b0 = s_tiles[tid];
                for (int t = 0; t < my_nt; ++t) {
                    const int R = min(RT, pd.y - t * RT);
                    t_cost[b0 + t] = fixed + per_rank * (float)my_r + per_row * (float)R;
                    t_code[b0 + t] = (tid << 16) | t;
                }
            }
            __syncthreads();
            const int C = (int)ncl;
            for (int j = tid; j < NT; j += kCcThreads) {
                const float cj = t_cost[j];
                int pos = 0;
                for (int k = 0; k < NT; ++k) {
                    const float ck = t_cost[k];
                    pos += (ck > cj || (ck == cj && k < j)) ? 1 : 0;
                }
                const int round = pos / C, m = pos - round * C;
                const int cl = (round & 1) ? C - 1 - m : m;
                if (cl == (int)cid) plan[1 + round] = t_code[j];
            }
            if (tid == 0) {
                // rounds 0 .. full - 1 give every cluster a tile; the last
                // round gives one to the clusters whose place is below its size
                const int full = NT / C, rest = NT - full * C;
                const int m = (full & 1) ? C - 1 - (int)cid : (int)cid;
                plan[0] = full + (m < rest ? 1 : 0);
            }
            __syncthreads();
            n_plan = plan[0];
        }
    }
    __syncthreads();  // the scratch is dead before the ring is used

    for (int e = 0;; ++e) {
        int li, tb, te;  // segment and tiles [tb, te) of this entry
        if (n_plan >= 0) {
            if (e >= n_plan) break;
            const int code = plan[1 + e];
            li = code >> 16;
            tb = code & 0xFFFF;
            te = tb + 1;
        } else {
            li = (int)cid + e * (int)ncl;
            if (by_list) {
                if (li >= n_list) break;
                li = __ldcg(&p.small_list[li].w);
            } else if (li >= p.max_list) {
                break;
            }
            tb = 0;
            te = 0x7fffffff;
        }
        if (n_plan >= 0 || e > 0 || by_list) {
            __syncthreads();  // the previous segment is done with desc_s / rows_s
            if (tid < 32) desc_s[tid] = reinterpret_cast<const int32_t *>(p.desc + li)[tid];
            __syncthreads();
        }
        const int start = desc_s[0], len = desc_s[1], a = desc_s[2];
        if (len == 0) break;  // descriptors are compacted: the list ends here
        const int r = p.ranks ? p.ranks[a] : p.r_max;
        if (!seg_taken(len, desc_s[3], r)) continue;
        if (r < 0 || r > p.r_max) {
            if (q == 0 && tid == 0) raise_deverr(p.counts, LORA_DEVERR_RANK);
            continue;
        }
        const float sc = p.adapter_scale ? p.adapter_scale[a] : p.scale;
        const int rv = (r + V - 1) / V;
        const int rvp = next_pow2(rv > 0 ? rv : 1);
        const int njg = (r + 3) / 4;

        for (int tt = tb; tt < te && tt * RT < len; ++tt) {
            const int t0 = tt * RT;
            const int R = min(RT, len - t0);
            const int nrb = (R + 3) / 4, Rp = nrb * 4;
            if (t0 > 0) __syncthreads();  // the previous tile is done with rows_s
            if (tid < R) rows_s[tid] = t0 + tid < kInlineRows ? desc_s[4 + t0 + tid] : p.sorted[start + t0 + tid];
            __syncthreads();

            // Shrink thread map: block ob = (row block, rank group) of 4x4
            // outputs, KS lanes per block striding over K.
            const int n_ob = nrb * (njg > 0 ? njg : 1);
            const int KS = kCcThreads / next_pow2(n_ob);
            const int ob = tid / KS, ks = tid - ob * KS;
            const int my_rb = ob / (njg > 0 ? njg : 1), my_jg = ob - my_rb * (njg > 0 ? njg : 1);
            const bool has_block = ob < n_ob && njg > 0;

            // bf16 tensor-core map: the shrink output (R rows x r ranks) in
            // mt x ntr tiles of 16 x 8; warp w takes tile w % ntt and the K
            // steps w / ntt, w / ntt + kp_n, ... (ntt <= 16: a tile of 17 or
            // more rows only exists for r_max <= 60, so ntr <= 8 then).
            const int mt = (R + 15) >> 4, ntr = max(1, (r + 7) >> 3), ntt = mt * ntr;
            const int kp_n = kCcThreads / 32 / ntt;
            const int my_t = warp % ntt, my_kp = warp / ntt;
            const bool mma_on = my_kp < kp_n;
            const int kr = (r + 15) >> 4;  // K steps of the expand (K = rank)

            // Jobs: shrink stages hold R + r rows of kc 16-byte chunks (kc
            // even, so that K steps of 16 elements stay within a job), expand
            // stages R rows of nc chunks of y and nc * V rows of B.  Rows are
            // kcs = kc + 1 and ncs = nc | 1 chunks apart: an odd stride puts
            // the eight rows a fragment load touches in eight different bank
            // groups.
            int nK = 0, kc = 2, nN = 0, nc = 1;
            if (MODE != kExpand && kv1 > kv0) {
                const int kcmax = max(2, (SB / ((Rp + r) * 16) - 1) & ~1);
                nK = (kv1 - kv0 + kcmax - 1) / kcmax;
                kc = (((kv1 - kv0 + nK - 1) / nK) + 1) & ~1;
            }
            if (MODE != kShrink && nv1 > nv0) {
                const int ncmax = max(1, (SB / 16 - R) / (R + V * rvp));
                nN = (nv1 - nv0 + ncmax - 1) / ncmax;
                nc = (nv1 - nv0 + nN - 1) / nN;
            }
            const int kcs = kc + 1, ncs = nc | 1;
            const int total = nK + nN;

            // ---- issue one job into its stage (called by every thread): all
            // loads are 16-byte cp.async, so rows gathered from anywhere cost
            // no more than contiguous ones.
            auto issue = [&](int j) {
                const uint32_t G = gjob + j;
                unsigned char *sb = ring + (size_t)(G % kCcStages) * SB;
                if (j < nK) {
                    const int kb = kv0 + j * kc, kn = min(kc, kv1 - kb);
                    // bf16: an odd last chunk gets a zero partner, so that
                    // its K step reads no stale bytes
                    const int knf = sizeof(T) == 2 ? (kn + 1) & ~1 : kn;
                    for (int row = warp; row < R + r; row += kCcThreads / 32) {
                        const T *src = row < R ? xg + (int64_t)rows_s[row] * p.ldx + (int64_t)kb * V
                                               : Ag + (int64_t)a * p.a_stride_adapter +
                                                     (int64_t)(row - R) * p.a_stride_r + (int64_t)kb * V;
                        unsigned char *dst = sb + (size_t)(row < R ? row : Rp + (row - R)) * kcs * 16;
                        for (int c = lane; c < knf; c += 32)
                            cp_async16(dst + c * 16, c < kn ? src + c * V : src, c < kn ? 16 : 0);
                    }
                } else {
                    const int nb = nv0 + (j - nK) * nc, nn = min(nc, nv1 - nb);
                    const int c0 = nb * V;
                    for (int row = warp; row < R; row += kCcThreads / 32) {
                        const int64_t yrow = (int64_t)rows_s[row] * p.ldy;
                        unsigned char *dst = sb + (size_t)row * ncs * 16;
                        for (int c = lane; c < nn; c += 32) {
                            const int col = c0 + c * V;
                            const SliceDesc &S = p.slices[slice_of(p, col)];
                            cp_async16(dst + c * 16, static_cast<const T *>(p.y) + yrow + S.y_col + (col - S.col_begin), 16);
                        }
                    }
                    unsigned char *bst = sb + (size_t)R * ncs * 16;
                    const int nrows = nn * V;
                    const int rv_shift = (rv & (rv - 1)) == 0 ? ilog2(rv) : -1;
                    for (int e = tid; e < nrows * rv; e += kCcThreads) {
                        const int br = rv_shift >= 0 ? e >> rv_shift : e / rv;
                        const int c = e - br * rv;
                        const int col = c0 + br;
                        const SliceDesc &S = p.slices[slice_of(p, col)];
                        const T *src = static_cast<const T *>(S.B) + (int64_t)a * S.stride_adapter +
                                       (int64_t)(col - S.col_begin) * S.stride_n + c * V;
                        const int bytes = min(16, (r - c * V) * (int)sizeof(T));
                        cp_async16(bst + (size_t)(br * rvp + b_swizzle(br, c, rvp)) * 16, src, bytes);
                    }
                }
                cp_async_commit();
            };

            float2 acc[4][4];  // fp32: 4 rows x 4 ranks (pairs of K)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[i][jj] = make_float2(0.f, 0.f);
            // bf16: this warp's 16 x 8 tile in four accumulators (K steps
            // round-robin), so that four products are in flight at once
            float macc[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) macc[u][0] = macc[u][1] = macc[u][2] = macc[u][3] = 0.f;
            // bf16 partial tiles [warp][lane][4] and the expand's h fragments
            // [m tile][K step][lane][4] share the slot area (8 KB + 4 KB).
            float *red = slots;
            uint32_t *hfrag = reinterpret_cast<uint32_t *>(slots) + 2048;

            // ---- partial h of this CTA -> every CTA of the cluster -> h_full.
            auto finish_shrink = [&]() {
                const int S = ilog2(KS < 32 ? KS : 32);
                const int wpb = KS > 32 ? KS / 32 : 1;  // warps per block
                if constexpr (sizeof(T) == 2) {
                    if (mma_on)
                        *reinterpret_cast<float4 *>(red + (warp * 32 + lane) * 4) =
                            make_float4((macc[0][0] + macc[1][0]) + (macc[2][0] + macc[3][0]),
                                        (macc[0][1] + macc[1][1]) + (macc[2][1] + macc[3][1]),
                                        (macc[0][2] + macc[1][2]) + (macc[2][2] + macc[3][2]),
                                        (macc[0][3] + macc[1][3]) + (macc[2][3] + macc[3][3]));
                } else {
                float v[16];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) v[i * 4 + jj] = acc[i][jj].x + acc[i][jj].y;
                group_reduce16(v, lane, S);
                const int nvals = 16 >> (S < 4 ? S : 4);
                if (has_block) {
                    // this lane's share of the block's 16 totals
                    int base = 0;
#pragma unroll
                    for (int st = 0; st < 4; ++st)
                        if (st < S) base += ((lane >> (S - 1 - st)) & 1) * (16 >> (st + 1));
                    const bool writer = S <= 4 || (lane & 1) == 0;
                    if (writer) {
                        const int wslot = ob * wpb + (KS > 32 ? (ks >> 5) : 0);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < nvals) slots[wslot * 16 + base + i] = v[i];
                    }
                }
                }
                __syncthreads();
                // Before a second push: every CTA of the cluster is done reading
                // its receive buffer for the previous tile (all CTAs of a cluster
                // walk the same tiles).  A CTA's last tile needs no barrier after
                // it, so the CTA leaves right after its expand.
                if (pushed) {
                    cluster_arrive_release();
                    cluster_wait_acquire();
                }
                pushed = true;
                for (int e = tid; e < R * r; e += kCcThreads) {
                    const int row = e / r, j = e - row * r;
                    const int b = (row >> 2) * njg + (j >> 2), idx = (row & 3) * 4 + (j & 3);
                    float s = 0.f;
                    if constexpr (sizeof(T) == 2) {
                        // tile of (row, j), then its K-split partials in warp order
                        const int t = (row >> 4) * ntr + (j >> 3);
                        const int at = (((row & 7) << 2) + ((j & 7) >> 1)) * 4 + ((row >> 3) & 1) * 2 + (j & 1);
                        for (int kp = 0; kp < kp_n; ++kp) s += red[(kp * ntt + t) * 128 + at];
                    } else {
                        for (int w = 0; w < wpb; ++w) s += slots[(b * wpb + w) * 16 + idx];
                    }
                    const uint32_t local = smem_u32(recv + ((int)q * RT + row) * HP + j);
                    for (uint32_t pr = 0; pr < CL; ++pr) st_dsmem_f32(map_to_rank(local, pr), s);
                }
                cluster_arrive_release();
                cluster_wait_acquire();
                for (int e = tid; e < RT * HP; e += kCcThreads) {
                    const int row = e / HP, j = e - row * HP;
                    float s = 0.f;
                    if (row < R && j < r)
                        for (uint32_t pq = 0; pq < CL; ++pq) s += recv[((int)pq * RT + row) * HP + j];
                    h_full[e] = (MODE == kFused) ? s * sc : s;
                }
                __syncthreads();
                if (MODE == kShrink && q == 0) {
                    for (int e = tid; e < R * p.r_max; e += kCcThreads) {
                        const int row = e / p.r_max, j = e - row * p.r_max;
                        p.h[(int64_t)rows_s[row] * p.ldh + j] = j < r ? h_full[row * HP + j] : 0.f;
                    }
                }
            };

            if (MODE == kExpand) {
                for (int e = tid; e < RT * HP; e += kCcThreads) {
                    const int row = e / HP, j = e - row * HP;
                    h_full[e] = (row < R && j < r) ? p.h[(int64_t)rows_s[row] * p.ldh + j] * sc : 0.f;
                }
            }

#pragma unroll 1
            for (int j = 0; j < kCcStages; ++j) {
                if (j < total) issue(j);
                else cp_async_commit();
            }
            if (MODE != kExpand && nK == 0) finish_shrink();

#pragma unroll 1
            for (int j = 0; j < total; ++j) {
                const uint32_t G = gjob + j;
                cp_async_wait<kCcStages - 1>();
                __syncthreads();
                const unsigned char *sb = ring + (size_t)(G % kCcStages) * SB;
                if (j < nK) {
                    // ---- shrink job: acc += x[rows of my block, K] . A[ranks of my block, K]
                    const int kn = min(kc, kv1 - (kv0 + j * kc));
                    if constexpr (sizeof(T) == 2) {
                        // tensor-core tile (rows 16 mi.., ranks 8 ni..) over this
                        // warp's K steps; rows past R and ranks past r are zero
                        if (mma_on) {
                            const int mi = my_t / ntr, ni = my_t - mi * ntr;
                            const int gq = lane >> 2, tq = lane & 3;
                            const int xr = mi * 16 + gq, an = ni * 8 + gq;
                            const bool v0 = xr < R, v1 = xr + 8 < R, va = an < r;
                            const unsigned char *x0 = sb + (size_t)xr * kcs * 16 + tq * 4;
                            const unsigned char *x1 = x0 + (size_t)8 * kcs * 16;
                            const unsigned char *ap = sb + (size_t)(Rp + an) * kcs * 16 + tq * 4;
                            const int nks = (kn + 1) >> 1;
                            for (int st0 = my_kp; st0 < nks; st0 += 4 * kp_n) {
                                uint32_t af[4][4], b0[4], b1[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const int st = st0 + u * kp_n;
                                    const bool in = st < nks;
                                    af[u][0] = in && v0 ? lds_u32(x0 + st * 32) : 0u;
                                    af[u][1] = in && v1 ? lds_u32(x1 + st * 32) : 0u;
                                    af[u][2] = in && v0 ? lds_u32(x0 + st * 32 + 16) : 0u;
                                    af[u][3] = in && v1 ? lds_u32(x1 + st * 32 + 16) : 0u;
                                    b0[u] = in && va ? lds_u32(ap + st * 32) : 0u;
                                    b1[u] = in && va ? lds_u32(ap + st * 32 + 16) : 0u;
                                }
#pragma unroll
                                for (int u = 0; u < 4; ++u) mma_16x8x16_bf16(macc[u], af[u], b0[u], b1[u]);
                            }
                        }
                    } else if (has_block) {
                        const uint4 *xs = reinterpret_cast<const uint4 *>(sb) + (my_rb * 4) * kcs;
                        const uint4 *As = reinterpret_cast<const uint4 *>(sb + (size_t)Rp * kcs * 16) + (my_jg * 4) * kcs;
                        const int jvalid = r - my_jg * 4;  // ranks of this block that exist
                        for (int kv = ks; kv < kn; kv += KS) {
                            uint4 av[4], xv[4];
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) av[jj] = jj < jvalid ? As[jj * kcs + kv] : make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int i = 0; i < 4; ++i) xv[i] = xs[i * kcs + kv];
#pragma unroll
                            for (int qq = 0; qq < PV; ++qq) {
                                float2 ap[4], xp[4];
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj) ap[jj] = pair_of<T>(av[jj], qq);
#pragma unroll
                                for (int i = 0; i < 4; ++i) xp[i] = pair_of<T>(xv[i], qq);
#pragma unroll
                                for (int i = 0; i < 4; ++i)
#pragma unroll
                                    for (int jj = 0; jj < 4; ++jj) acc[i][jj] = __ffma2_rn(xp[i], ap[jj], acc[i][jj]);
                            }
                        }
                    }
                    if (j == nK - 1) finish_shrink();
                } else {
                    // ---- expand job: y[rows, c..c+1] += h . B[c..c+1]^T
                    const int nb = nv0 + (j - nK) * nc, nn = min(nc, nv1 - nb);
                    const int npairs = nn * V / 2;
                    const uint4 *Bs = reinterpret_cast<const uint4 *>(sb + (size_t)R * ncs * 16);
                    const typename E::PairT *ys = reinterpret_cast<const typename E::PairT *>(sb);
                    const int ystride = ncs * V / 2;
                    if constexpr (sizeof(T) == 2) {
                        if (j == nK) {
                            // h (scaled, fp32) rounded once to bf16, in fragment
                            // order: [m tile][K step][lane][a0..a3]
                            for (int e = tid; e < mt * kr * 128; e += kCcThreads) {
                                const int rg = e & 3, ln = (e >> 2) & 31, blk = e >> 7;
                                const int mi = blk / kr, st = blk - mi * kr;
                                const int row = mi * 16 + (ln >> 2) + ((rg & 1) ? 8 : 0);
                                const int col = st * 16 + 2 * (ln & 3) + ((rg & 2) ? 8 : 0);
                                const float lo = row < R && col < r ? h_full[row * HP + col] : 0.f;
                                const float hi = row < R && col + 1 < r ? h_full[row * HP + col + 1] : 0.f;
                                const __nv_bfloat162 hv = __floats2bfloat162_rn(lo, hi);
                                hfrag[e] = *reinterpret_cast<const uint32_t *>(&hv);
                            }
                            __syncthreads();
                        }
                        // warp per 8-column tile: y[rows, 8 cols] += h . B[8 cols]^T,
                        // B fragments from the swizzled rows (chunks past the
                        // rank are zero); the sums replace y in the stage, which
                        // then goes out in 16-byte row pieces
                        const int gq = lane >> 2, tq = lane & 3;
                        uint32_t *yst = reinterpret_cast<uint32_t *>(const_cast<unsigned char *>(sb));
                        const unsigned char *Bb = reinterpret_cast<const unsigned char *>(Bs);
                        constexpr int kW = kCcThreads / 32;
                        // swizzle of B row n: chunk c sits at c ^ ((n >> bsh) & bmask)
                        const int bsh = rvp >= 8 ? 0 : (rvp == 1 ? 3 : rvp == 2 ? 2 : 1);
                        const int bmask = rvp >= 8 ? 7 : rvp - 1;
                        // NB column tiles per warp at a time (eight when the
                        // tile has at most 16 rows), MT row tiles of 16
                        auto expand_tiles = [&](auto nb_c, auto mt_c) {
                            constexpr int NB = decltype(nb_c)::value, MT = decltype(mt_c)::value;
                            for (int jt0 = warp; jt0 < nn; jt0 += NB * kW) {
                                float d[MT][NB][4];
#pragma unroll
                                for (int mi = 0; mi < MT; ++mi)
#pragma unroll
                                    for (int u = 0; u < NB; ++u) d[mi][u][0] = d[mi][u][1] = d[mi][u][2] = d[mi][u][3] = 0.f;
                                uint32_t boff[NB];
                                int bsw[NB];
#pragma unroll
                                for (int u = 0; u < NB; ++u) {
                                    const int n = (jt0 + u * kW) * 8 + gq;
                                    boff[u] = (uint32_t)(n * rvp) * 16u + (uint32_t)tq * 4u;
                                    bsw[u] = (n >> bsh) & bmask;
                                }
                                for (int st = 0; st < kr; ++st) {
                                    const int c0 = 2 * st, c1 = c0 + 1;
                                    uint32_t bq0[NB], bq1[NB];
#pragma unroll
                                    for (int u = 0; u < NB; ++u) {
                                        const bool in = jt0 + u * kW < nn;
                                        bq0[u] = in && c0 < rv ? lds_u32(Bb + boff[u] + ((uint32_t)(c0 ^ bsw[u]) << 4)) : 0u;
                                        bq1[u] = in && c1 < rv ? lds_u32(Bb + boff[u] + ((uint32_t)(c1 ^ bsw[u]) << 4)) : 0u;
                                    }
#pragma unroll
                                    for (int mi = 0; mi < MT; ++mi) {
                                        const uint4 av = *reinterpret_cast<const uint4 *>(hfrag + ((mi * kr + st) * 32 + lane) * 4);
                                        const uint32_t af[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                                        for (int u = 0; u < NB; ++u) mma_16x8x16_bf16(d[mi][u], af, bq0[u], bq1[u]);
                                    }
                                }
#pragma unroll
                                for (int u = 0; u < NB; ++u) {
                                    const int jt = jt0 + u * kW;
                                    if (jt < nn) {
#pragma unroll
                                        for (int mi = 0; mi < MT; ++mi) {
                                            const int row0 = mi * 16 + gq, row1 = row0 + 8;
                                            if (row0 < R) {
                                                const int at = row0 * ystride + jt * 4 + tq;
                                                const float2 yv = E::pair_to_f32(yst[at]);
                                                const __nv_bfloat162 o = __floats2bfloat162_rn(yv.x + d[mi][u][0], yv.y + d[mi][u][1]);
                                                yst[at] = *reinterpret_cast<const uint32_t *>(&o);
                                            }
                                            if (row1 < R) {
                                                const int at = row1 * ystride + jt * 4 + tq;
                                                const float2 yv = E::pair_to_f32(yst[at]);
                                                const __nv_bfloat162 o = __floats2bfloat162_rn(yv.x + d[mi][u][2], yv.y + d[mi][u][3]);
                                                yst[at] = *reinterpret_cast<const uint32_t *>(&o);
                                            }
                                        }
                                    }
                                }
                            }
                        };
                        if (mt == 1) expand_tiles(std::integral_constant<int, 8>{}, std::integral_constant<int, 1>{});
                        else expand_tiles(std::integral_constant<int, 4>{}, std::integral_constant<int, 2>{});
                        __syncthreads();
                        for (int row = warp; row < R; row += kCcThreads / 32) {
                            T *yrow = static_cast<T *>(p.y) + (int64_t)rows_s[row] * p.ldy;
                            for (int c = lane; c < nn; c += 32) {
                                const int col = nb * V + c * V;
                                const SliceDesc &S = p.slices[slice_of(p, col)];
                                *reinterpret_cast<uint4 *>(yrow + S.y_col + (col - S.col_begin)) =
                                    *reinterpret_cast<const uint4 *>(sb + ((size_t)row * ncs + c) * 16);
                            }
                        }
                    } else
                    for (int cp = tid; cp < npairs; cp += kCcThreads) {
                        const int c0 = 2 * cp, c1 = c0 + 1;
                        const int col = nb * V + c0;
                        const SliceDesc &S = p.slices[slice_of(p, col)];
                        T *yg = static_cast<T *>(p.y) + S.y_col + (col - S.col_begin);
                        for (int rb = 0; rb < nrb; ++rb) {
                            float2 o0[4], o1[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) o0[i] = o1[i] = make_float2(0.f, 0.f);
                            for (int jc = 0; jc < rv; ++jc) {
                                const uint4 b0 = Bs[c0 * rvp + b_swizzle(c0, jc, rvp)];
                                const uint4 b1 = Bs[c1 * rvp + b_swizzle(c1, jc, rvp)];
#pragma unroll
                                for (int qq = 0; qq < PV; qq += 2) {
                                    const float2 p00 = pair_of<T>(b0, qq), p01 = pair_of<T>(b0, qq + 1);
                                    const float2 p10 = pair_of<T>(b1, qq), p11 = pair_of<T>(b1, qq + 1);
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const float4 hh = *reinterpret_cast<const float4 *>(
                                            h_full + (rb * 4 + i) * HP + jc * V + 2 * qq);
                                        const float2 h0 = make_float2(hh.x, hh.y), h1 = make_float2(hh.z, hh.w);
                                        o0[i] = __ffma2_rn(p00, h0, o0[i]);
                                        o0[i] = __ffma2_rn(p01, h1, o0[i]);
                                        o1[i] = __ffma2_rn(p10, h0, o1[i]);
                                        o1[i] = __ffma2_rn(p11, h1, o1[i]);
                                    }
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int row = rb * 4 + i;
                                if (row < R) {
                                    float2 yv = E::pair_to_f32(ys[row * ystride + cp]);
                                    yv.x += o0[i].x + o0[i].y;
                                    yv.y += o1[i].x + o1[i].y;
                                    E::store_pair(yg + (int64_t)rows_s[row] * p.ldy, yv);
                                }
                            }
                        }
                    }
                }
                __syncthreads();
                if (j + kCcStages < total) issue(j + kCcStages);
                else cp_async_commit();
            }
            gjob += (uint32_t)total;
        }
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
static CcGeom cc_geometry(int r_max, int cluster) {
    CcGeom g{};
    g.RT = cc_rows_per_tile(r_max);
    g.HP = (r_max + 7) & ~7;
    int o = 0;
    auto take = [&](int bytes) {
        const int at = o;
        o = (o + bytes + 127) & ~127;
        return at;
    };
    g.off_bars = take(kCcStages * 8);
    g.off_desc = take(32 * 4);
    g.off_rows = take(g.RT * 4);
    g.off_slots = take(256 * 16 * 4);
    g.off_recv = take(cluster * g.RT * g.HP * 4);
    g.off_hfull = take(g.RT * g.HP * 4);
    g.off_plan = take((kPlanMaxTiles + 4) * 4);
    g.off_ring = o;
    const int budget = 225 * 1024;
    g.stage_bytes = ((budget - o) / kCcStages) & ~127;
    g.total = o + kCcStages * g.stage_bytes;
    return g;
}

// Co-resident clusters for a kernel / cluster size / shared-memory size,
// queried once and cached.
struct ResidencyCache {
    struct Entry {
        const void *fn;
        int dev, cluster, smem, value;
    };
    Entry e[64] = {};
    int n = 0;
    int get(const void *fn, int dev, int cluster, int smem) const {
        for (int i = 0; i < n; ++i)
            if (e[i].fn == fn && e[i].dev == dev && e[i].cluster == cluster && e[i].smem == smem) return e[i].value;
        return -1;
    }
    void put(const void *fn, int dev, int cluster, int smem, int v) {
        if (n < 64) e[n++] = {fn, dev, cluster, smem, v};
    }
};

template <typename T, int MODE>
static cudaError_t launch_cc_t(const DeltaArgs &p, int cluster, int sms, cudaStream_t stream) {
    auto kern = sgmv_cc_kernel<T, MODE>;
    const CcGeom g = cc_geometry(p.r_max, cluster);
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        // the block's 227 KB less the kernel's static shared memory
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, kern);
        if (r != cudaSuccess) return r;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    227 * 1024 - (int)fa.sharedSizeBytes);
    });
    if (e != cudaSuccess) return e;

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kCcThreads);
    cfg.dynamicSmemBytes = g.total;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;

    static ResidencyCache cache;
    int dev = 0;
    cudaGetDevice(&dev);
    int max_clusters = cache.get((const void *)kern, dev, cluster, g.total);
    if (max_clusters < 0) {
        cfg.gridDim = dim3(cluster);
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active <= 0) {
            cudaGetLastError();
            active = sms / cluster;
        }
        cfg.numAttrs = 2;
        max_clusters = active;
        cache.put((const void *)kern, dev, cluster, g.total, active);
    }
    // No more clusters than the SMs left to this kernel hold (a tensor-core
    // grid may hold the others: clusters that cannot start with the rest
    // finish their segments last, and the next kernel in the stream starts
    // only once every CTA has), but at least kCcMinClusters, so that a large
    // batch whose tensor-core grid fills the GPU still spreads many small
    // segments widely once that grid's CTAs leave.
    constexpr int kCcMinClusters = 8;
    int nclusters = p.max_list < max_clusters ? p.max_list : max_clusters;
    const int cap = sms / cluster > kCcMinClusters ? sms / cluster : kCcMinClusters;
    if (nclusters > cap) nclusters = cap;
    if (nclusters < 1) nclusters = 1;
    cfg.gridDim = dim3(nclusters * cluster);
    return cudaLaunchKernelEx(&cfg, kern, p, g);
}

// Cluster size: enough CTAs per segment to spread one adapter's weights over
// several SMs, not so many that the slices become too thin to stream well.
int cc_cluster_size(int d_in, int d_out) {
    const int d = d_in > d_out ? d_in : d_out;
    if (d < 1024) return 1;
    if (d < 2048) return 2;
    if (d <= 8192) return 4;
    return 8;
}

cudaError_t launch_cc(const DeltaArgs &p, int dtype, int mode, int cluster, int sms, cudaStream_t stream) {
    if (cluster > kCcMaxCluster) cluster = kCcMaxCluster;
    if (dtype == LORA_F32) {
        if (mode == kFused) return launch_cc_t<float, kFused>(p, cluster, sms, stream);
        if (mode == kShrink) return launch_cc_t<float, kShrink>(p, cluster, sms, stream);
        return launch_cc_t<float, kExpand>(p, cluster, sms, stream);
    }
    if (mode == kFused) return launch_cc_t<__nv_bfloat16, kFused>(p, cluster, sms, stream);
    if (mode == kShrink) return launch_cc_t<__nv_bfloat16, kShrink>(p, cluster, sms, stream);
    return launch_cc_t<__nv_bfloat16, kExpand>(p, cluster, sms, stream);
}

}  // namespace lora
