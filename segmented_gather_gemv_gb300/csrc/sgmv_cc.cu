// sgmv_cc.cu -- CUDA-core SGMV kernel for small segments (decode).
//
// Each segment (rows that share one adapter) is handled by one thread-block
// cluster of CL CTAs ("vLLM-Ascend LoRA" article, section 3.3: the rows of
// one adapter are gathered, tmp = rows . A^T, delta = (tmp * scale) . B^T,
// scatter-added; the adapter's A/B are moved once and reused by all rows of
// the segment).  CTA q of the cluster owns
//   - the K slice q of d_in for the shrink (A rows r x K/CL, x rows R x K/CL),
//   - the N slice q of d_out for the expand (B rows N/CL x r, y rows R x N/CL),
// so every byte of x, A, B and y is read exactly once per segment.  The
// partial h of the K slices is summed across the cluster through distributed
// shared memory (fixed order, so every CTA holds the same h); h never leaves
// the chip.
//
// Loads: 16-byte cp.async into a ring of kCcStages stages.  All x/A (shrink)
// and y/B (expand) tiles of a segment are "jobs"; the first kCcStages-1 jobs
// are issued before any compute, so the expand's B and y tiles are in flight
// while the shrink runs.  Gathered rows (sorted_token_ids) cost nothing
// extra: every 16-byte copy carries its own address.  B rows are read only up
// to the adapter's rank (the rest of the last vector is zero-filled).
//
// Compute (fp32 FMA): shrink -- warp w owns rank rows j = w + 8*jj, lanes
// stride over the K vectors, a transposing butterfly reduces the lanes;
// expand -- every thread owns CPT output columns and all rows of the tile.
#include "common.cuh"

namespace lora {

constexpr int kCcThreads = 256;
constexpr int kCcWarps = kCcThreads / 32;
constexpr int kCcStages = 8;
constexpr int kCcCpt = 4;  // output columns per thread per expand pass

__host__ __device__ __forceinline__ int cc_hp(int r_max) { return (r_max + 7) & ~7; }

template <int RT>
static inline size_t cc_smem_bytes(int stage_bytes, int r_max) {
    return (size_t)kCcStages * stage_bytes + (size_t)3 * RT * cc_hp(r_max) * 4 + RT * 4;
}

// After this, lane l holds in v[0 .. NV/32) the sums over the 32 lanes of the
// original entries i + (NV/32) * l.
template <int NV>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[NV], int lane) {
    static_assert(NV >= 32 && (NV & (NV - 1)) == 0, "NV must be a power of two >= 32");
#pragma unroll
    for (int stage = 0; stage < 5; ++stage) {
        const int off = 16 >> stage;
        const int half = NV >> (stage + 1);
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
}

// Maps a column of the concatenated output range to its slice.
__device__ __forceinline__ int slice_of(const DeltaArgs &p, int col) {
    int t = 0;
#pragma unroll
    for (int u = 1; u < LORA_MAX_SLICES; ++u)
        if (u < p.n_slices && col >= p.slices[u].col_begin) t = u;
    return t;
}

template <typename T, int MODE, int JW, int RT>
__global__ void __launch_bounds__(kCcThreads, 1)
    sgmv_cc_kernel(const __grid_constant__ DeltaArgs p, const int stage_bytes) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int NA = RT * JW;
    constexpr int NV = NA < 32 ? 32 : NA;
    extern __shared__ __align__(16) unsigned char smem[];

    const int HP = cc_hp(p.r_max);
    unsigned char *ring = smem;
    float *h_part = reinterpret_cast<float *>(smem + (size_t)kCcStages * stage_bytes);
    float *h_full = h_part + 2 * RT * HP;
    int32_t *rows_s = reinterpret_cast<int32_t *>(h_full + RT * HP);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t CL = cluster_nctarank(), q = cluster_ctarank();
    const uint32_t cid = cluster_id_x(), ncl = nclusters_x();

    int nlist = p.counts[p.count_index];
    if (nlist > p.max_list) nlist = p.max_list;

    const int kv_total = p.d_in / V;
    const int kv0 = (int)((int64_t)kv_total * q / CL), kv1 = (int)((int64_t)kv_total * (q + 1) / CL);
    const int nv_total = p.d_out_total / V;
    const int nv0 = (int)((int64_t)nv_total * q / CL), nv1 = (int)((int64_t)nv_total * (q + 1) / CL);

    int hbuf = 0;
    for (int li = (int)cid; li < nlist; li += (int)ncl) {
        const int s = p.seg_list ? p.seg_list[li] : li;
        const int a = p.widx[s], len = p.lens[s], start = p.indptr[s];
        const int r = p.ranks ? p.ranks[a] : p.r_max;
        if (r < 0 || r > p.r_max) {
            if (q == 0 && tid == 0) raise_deverr(p.counts, LORA_DEVERR_RANK);
            continue;
        }
        const float sc = p.adapter_scale ? p.adapter_scale[a] : p.scale;
        const int rv = (r + V - 1) / V;  // 16-byte vectors per B row

        for (int t0 = 0; t0 < len; t0 += RT) {
            const int R = min(RT, len - t0);
            __syncthreads();  // the previous tile is done with rows_s and h_full
            if (tid < R) rows_s[tid] = p.sorted[start + t0 + tid];
            __syncthreads();

            int kc = stage_bytes / ((R + r) * 16);
            int nc = stage_bytes / ((R + V * rv) * 16);
            kc = kc < 1 ? 1 : kc;
            nc = nc < 1 ? 1 : nc;
            const int nK = (MODE == kExpand) ? 0 : (kv1 - kv0 + kc - 1) / kc;
            const int nN = (MODE == kShrink) ? 0 : (nv1 - nv0 + nc - 1) / nc;
            const int total = nK + nN;

            float acc[RT][JW];
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int jj = 0; jj < JW; ++jj) acc[i][jj] = 0.f;

            // ---- job issue: all 16-byte copies of one job into its stage.
            auto issue = [&](int j) {
                unsigned char *st = ring + (size_t)(j % kCcStages) * stage_bytes;
                if (j < nK) {
                    const int kb = kv0 + j * kc, kn = min(kc, kv1 - kb);
                    for (int row = warp; row < R + r; row += kCcWarps) {
                        const T *src;
                        if (row < R)
                            src = static_cast<const T *>(p.x) + (int64_t)rows_s[row] * p.ldx + (int64_t)kb * V;
                        else
                            src = static_cast<const T *>(p.A) + (int64_t)a * p.a_stride_adapter +
                                  (int64_t)(row - R) * p.a_stride_r + (int64_t)kb * V;
                        unsigned char *dst = st + (size_t)row * kc * 16;
                        for (int c = lane; c < kn; c += 32) cp_async16(dst + c * 16, src + c * V, 16);
                    }
                } else {
                    const int nb = nv0 + (j - nK) * nc, nn = min(nc, nv1 - nb);
                    for (int row = warp; row < R; row += kCcWarps) {
                        const int64_t yrow = (int64_t)rows_s[row] * p.ldy;
                        unsigned char *dst = st + (size_t)row * nc * 16;
                        for (int c = lane; c < nn; c += 32) {
                            const int col = (nb + c) * V;
                            const SliceDesc &S = p.slices[slice_of(p, col)];
                            const T *src = static_cast<const T *>(p.y) + yrow + S.y_col + (col - S.col_begin);
                            cp_async16(dst + c * 16, src, 16);
                        }
                    }
                    unsigned char *bst = st + (size_t)R * nc * 16;
                    const int nrows = nn * V;
                    for (int e = tid; e < nrows * rv; e += kCcThreads) {
                        const int br = e / rv, c = e - br * rv;
                        const int col = nb * V + br;
                        const SliceDesc &S = p.slices[slice_of(p, col)];
                        const T *src = static_cast<const T *>(S.B) + (int64_t)a * S.stride_adapter +
                                       (int64_t)(col - S.col_begin) * S.stride_n + c * V;
                        const int bytes = min(16, (r - c * V) * (int)sizeof(T));
                        cp_async16(bst + (size_t)e * 16, src, bytes);
                    }
                }
            };

            // ---- h reduction across the cluster (shrink/fused only).
            auto reduce_h = [&]() {
                float v[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i) v[i] = i < NA ? acc[i / JW][i % JW] : 0.f;
                warp_transpose_reduce<NV>(v, lane);
                float *hp = h_part + hbuf * RT * HP;
#pragma unroll
                for (int i = 0; i < NV / 32; ++i) {
                    const int idx = i + (NV / 32) * lane;
                    if (idx < NA) {
                        const int row = idx / JW, j = warp + kCcWarps * (idx % JW);
                        if (row < R && j < r) hp[row * HP + j] = v[i];
                    }
                }
                __syncthreads();
                cluster_sync();
                for (int e = tid; e < R * HP; e += kCcThreads) {
                    const int row = e / HP, j = e - row * HP;
                    float sum = 0.f;
                    if (j < r) {
                        const uint32_t addr = smem_u32(hp + row * HP + j);
                        for (uint32_t pr = 0; pr < CL; ++pr) sum += ld_dsmem_f32(map_to_rank(addr, pr));
                    }
                    h_full[e] = (MODE == kFused) ? sum * sc : sum;
                }
                __syncthreads();
                if (MODE == kShrink && q == 0) {
                    for (int e = tid; e < R * p.r_max; e += kCcThreads) {
                        const int row = e / p.r_max, j = e - row * p.r_max;
                        p.h[(int64_t)rows_s[row] * p.ldh + j] = j < r ? h_full[row * HP + j] : 0.f;
                    }
                }
                hbuf ^= 1;
            };

            if (MODE == kExpand) {
                for (int e = tid; e < R * HP; e += kCcThreads) {
                    const int row = e / HP, j = e - row * HP;
                    h_full[e] = j < r ? p.h[(int64_t)rows_s[row] * p.ldh + j] * sc : 0.f;
                }
                __syncthreads();
            }

#pragma unroll 1
            for (int j = 0; j < kCcStages - 1; ++j) {
                if (j < total) issue(j);
                cp_async_commit();
            }
            if (MODE != kExpand && nK == 0) reduce_h();

#pragma unroll 1
            for (int j = 0; j < total; ++j) {
                const int jn = j + kCcStages - 1;
                if (jn < total) issue(jn);
                cp_async_commit();
                cp_async_wait<kCcStages - 1>();
                __syncthreads();
                const unsigned char *st = ring + (size_t)(j % kCcStages) * stage_bytes;
                if (j < nK) {
                    // ---- shrink job: acc[row][jj] += x[row, K] . A[j, K]
                    const int kb = kv0 + j * kc, kn = min(kc, kv1 - kb);
                    const unsigned char *xs = st;
                    const unsigned char *As = st + (size_t)R * kc * 16;
                    if (warp < r) {
                        for (int c = lane; c < kn; c += 32) {
                            float af[JW][V];
#pragma unroll
                            for (int jj = 0; jj < JW; ++jj) {
                                const int jr = warp + kCcWarps * jj;
                                if (jr < r) {
                                    const uint4 u = *reinterpret_cast<const uint4 *>(As + ((size_t)jr * kc + c) * 16);
                                    E::to_f32(u, af[jj]);
                                } else {
#pragma unroll
                                    for (int e = 0; e < V; ++e) af[jj][e] = 0.f;
                                }
                            }
#pragma unroll
                            for (int row = 0; row < RT; ++row) {
                                if (row < R) {
                                    const uint4 u = *reinterpret_cast<const uint4 *>(xs + ((size_t)row * kc + c) * 16);
                                    float xf[V];
                                    E::to_f32(u, xf);
#pragma unroll
                                    for (int jj = 0; jj < JW; ++jj)
#pragma unroll
                                        for (int e = 0; e < V; ++e) acc[row][jj] = fmaf(xf[e], af[jj][e], acc[row][jj]);
                                }
                            }
                        }
                    }
                    if (j == nK - 1) reduce_h();
                } else {
                    // ---- expand job: y[row, col] += h[row, :] . B[col, :]
                    const int nb = nv0 + (j - nK) * nc, nn = min(nc, nv1 - nb);
                    T *ys = reinterpret_cast<T *>(const_cast<unsigned char *>(st));
                    const unsigned char *bs = st + (size_t)R * nc * 16;
                    const int ncols = nn * V, ystride = nc * V;
                    for (int c0 = tid; c0 < ncols; c0 += kCcThreads * kCcCpt) {
                        float out[kCcCpt][RT];
#pragma unroll
                        for (int u = 0; u < kCcCpt; ++u)
#pragma unroll
                            for (int row = 0; row < RT; ++row) out[u][row] = 0.f;
                        for (int cv = 0; cv < rv; ++cv) {
                            float bf[kCcCpt][V];
#pragma unroll
                            for (int u = 0; u < kCcCpt; ++u) {
                                const int col = c0 + u * kCcThreads;
                                if (col < ncols) {
                                    const uint4 w = *reinterpret_cast<const uint4 *>(bs + ((size_t)col * rv + cv) * 16);
                                    E::to_f32(w, bf[u]);
                                } else {
#pragma unroll
                                    for (int e = 0; e < V; ++e) bf[u][e] = 0.f;
                                }
                            }
#pragma unroll
                            for (int e = 0; e < V; e += 4) {
                                const int jb = cv * V + e;
#pragma unroll
                                for (int row = 0; row < RT; ++row) {
                                    if (row < R) {
                                        const float4 h4 = *reinterpret_cast<const float4 *>(h_full + row * HP + jb);
#pragma unroll
                                        for (int u = 0; u < kCcCpt; ++u) {
                                            float t = out[u][row];
                                            t = fmaf(h4.x, bf[u][e + 0], t);
                                            t = fmaf(h4.y, bf[u][e + 1], t);
                                            t = fmaf(h4.z, bf[u][e + 2], t);
                                            t = fmaf(h4.w, bf[u][e + 3], t);
                                            out[u][row] = t;
                                        }
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kCcCpt; ++u) {
                            const int col = c0 + u * kCcThreads;
                            if (col < ncols) {
#pragma unroll
                                for (int row = 0; row < RT; ++row) {
                                    if (row < R) {
                                        T *yp = ys + row * ystride + col;
                                        E::store1(yp, E::load1(yp) + out[u][row]);
                                    }
                                }
                            }
                        }
                    }
                    __syncthreads();
                    for (int row = warp; row < R; row += kCcWarps) {
                        const int64_t yrow = (int64_t)rows_s[row] * p.ldy;
                        const unsigned char *src = st + (size_t)row * nc * 16;
                        for (int c = lane; c < nn; c += 32) {
                            const int col = (nb + c) * V;
                            const SliceDesc &S = p.slices[slice_of(p, col)];
                            T *dst = static_cast<T *>(p.y) + yrow + S.y_col + (col - S.col_begin);
                            *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src + c * 16);
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
    // Keep this CTA's shared memory alive until every peer has finished its
    // distributed-shared-memory reads.
    if (MODE != kExpand) cluster_sync();
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <typename T, int MODE, int JW, int RT>
static cudaError_t launch_cc_t(const DeltaArgs &p, int cluster, int sms, cudaStream_t stream) {
    auto kern = sgmv_cc_kernel<T, MODE, JW, RT>;
    constexpr int kSmemBudget = 200 * 1024;
    const int fixed = 3 * RT * cc_hp(p.r_max) * 4 + RT * 4;
    int stage_bytes = ((kSmemBudget - fixed) / kCcStages) & ~127;
    const size_t smem = cc_smem_bytes<RT>(stage_bytes, p.r_max);
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (e != cudaSuccess) return e;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kCcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    // Co-resident clusters for this shape (queried once per device and
    // cluster size; the answer does not depend on the batch).
    static int resident[64][9] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int max_clusters = sms / cluster;
    if (dev >= 0 && dev < 64 && cluster <= 8) {
        if (!resident[dev][cluster]) {
            cfg.gridDim = dim3(cluster);
            int active = 0;
            if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active <= 0) {
                cudaGetLastError();
                active = sms / cluster;
            }
            resident[dev][cluster] = active;
        }
        max_clusters = resident[dev][cluster];
    }
    int nclusters = p.max_list < max_clusters ? p.max_list : max_clusters;
    if (nclusters < 1) nclusters = 1;
    cfg.gridDim = dim3(nclusters * cluster);
    e = cudaLaunchKernelEx(&cfg, kern, p, stage_bytes);
    return e;
}

template <typename T, int MODE>
static cudaError_t launch_cc_mode(const DeltaArgs &p, int cluster, int sms, cudaStream_t stream) {
    const int jw = (p.r_max + kCcWarps - 1) / kCcWarps;
    if (jw <= 1) return launch_cc_t<T, MODE, 1, 16>(p, cluster, sms, stream);
    if (jw <= 2) return launch_cc_t<T, MODE, 2, 16>(p, cluster, sms, stream);
    if (jw <= 4) return launch_cc_t<T, MODE, 4, 16>(p, cluster, sms, stream);
    if (jw <= 8) return launch_cc_t<T, MODE, 8, 8>(p, cluster, sms, stream);
    return launch_cc_t<T, MODE, 16, 4>(p, cluster, sms, stream);
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
    if (dtype == LORA_F32) {
        if (mode == kFused) return launch_cc_mode<float, kFused>(p, cluster, sms, stream);
        if (mode == kShrink) return launch_cc_mode<float, kShrink>(p, cluster, sms, stream);
        return launch_cc_mode<float, kExpand>(p, cluster, sms, stream);
    }
    if (mode == kFused) return launch_cc_mode<__nv_bfloat16, kFused>(p, cluster, sms, stream);
    if (mode == kShrink) return launch_cc_mode<__nv_bfloat16, kShrink>(p, cluster, sms, stream);
    return launch_cc_mode<__nv_bfloat16, kExpand>(p, cluster, sms, stream);
}

}  // namespace lora
