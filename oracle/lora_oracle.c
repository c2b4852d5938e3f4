/*
 * lora_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of the multi-LoRA delta
 * path, in double precision.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code; the product library
 * never calls it and shares no source with it.
 *
 * What it computes, and where that is stated:
 *
 *   - Unmerged LoRA delta with its scaling factor: for every token row i
 *     that carries an adapter id a = ids[i],
 *         y[i, :] += s_a * (x[i, :] . A[a]^T) . B[a]^T
 *     ("vLLM-Ascend LoRA" article, section 1.1, the unmerged forward
 *     y = Wx + (alpha/r)(x A^T) B^T; section 2.3, "out += delta").
 *   - The same per-token loop as the reference test of the "09. Triton
 *     Fused LoRA" tutorial (Step 4, test_multi_lora): h_r = x_i A^T, then
 *     y_i = h_r B^T, one token at a time.
 *   - Pool layout: A pool (num_loras, r, in_features), B pool
 *     (num_loras, out_features, r) ("09. Triton Fused LoRA", Step 1 and
 *     the test's pool shapes).
 *   - Tokens whose id is -1 carry no adapter and are skipped ("vLLM-Ascend
 *     LoRA" article, section 5.3: empty-adapter sequences must be skipped).
 *   - Mixed ranks: each adapter uses only its own rank r_a <= r_max; the
 *     padded rows of A and padded columns of B are never read
 *     ("vLLM-Ascend LoRA" article, section 3.4, padding to the maximum
 *     rank with the excess masked out).
 *   - Segmentation: tokens are grouped by adapter (segment boundary array
 *     s, "III.Punica: Multi-Tenant LoRA Serving", section SGMV: ids
 *     2 2 2 5 5 1 1 give s = [0, 3, 5, 7]); groups appear in the order in
 *     which their adapter first occurs in the batch, rows inside a group
 *     keep ascending token order, and each group may be cut into fixed-size
 *     chunks, each chunk a segment of its own (same page, section 代码:
 *     prepare_lora_batch regroups tokens by adapter, then cuts the
 *     regrouped stream into chunks).  Optionally the groups come by
 *     increasing adapter id instead (the same "regroup by adapter" read as
 *     a sort by id).
 *
 * Numerics: every input element is read as stored (fp32 storage; bf16
 * inputs are exactly representable in fp32) and widened to double; every
 * product and sum is carried in double.  No blocking, no reordering beyond
 * the plain loops below.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR (-1)

/* Is `id` a usable pool slot?  -1 means "no adapter"; anything else
 * outside [0, n_adapters) is an invalid id, skipped and counted. */
static int id_valid(int32_t id, int32_t n_adapters)
{
    return id >= 0 && id < n_adapters;
}

/*
 * Segmentation oracle.
 *
 * Inputs : ids[M], n_adapters, chunk_size (0 = no chunking).
 * Outputs: sorted_token_ids[num_active]   token rows, grouped;
 *          seg_indptr[num_segs + 1]       exclusive prefix of seg_lens;
 *          seg_lens[num_segs];
 *          weight_indices[num_segs]       adapter of each segment;
 *          counts[0..2] = num_segs, num_active, num_invalid.
 * Buffers must hold M entries (seg_indptr M + 1); with chunking a group of
 * L rows yields ceil(L / chunk_size) segments, never more than L.
 */
int oracle_prepare_batch_ordered(const int32_t *ids, int32_t M, int32_t n_adapters,
                                 int32_t chunk_size, int32_t ascending,
                                 int32_t *sorted_token_ids, int32_t *seg_indptr,
                                 int32_t *seg_lens, int32_t *weight_indices,
                                 int32_t *counts)
{
    if (M < 0 || n_adapters < 0 || chunk_size < 0 || (ascending != 0 && ascending != 1))
        return ORACLE_ERR;
    char *seen = (char *)calloc((size_t)(n_adapters > 0 ? n_adapters : 1), 1);
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(M > 0 ? M : 1));
    if (!seen || !order) {
        free(seen);
        free(order);
        return ORACLE_ERR;
    }
    /* Distinct valid adapters in order of first appearance. */
    int32_t n_groups = 0, n_invalid = 0;
    for (int32_t i = 0; i < M; ++i) {
        int32_t a = ids[i];
        if (a == -1)
            continue;
        if (!id_valid(a, n_adapters)) {
            ++n_invalid;
            continue;
        }
        if (!seen[a]) {
            seen[a] = 1;
            order[n_groups++] = a;
        }
    }
    /* Ascending order (the page's "regroup tokens by adapter" read as a sort
     * by adapter id): the present adapters by increasing id instead. */
    if (ascending) {
        n_groups = 0;
        for (int32_t a = 0; a < n_adapters; ++a)
            if (seen[a])
                order[n_groups++] = a;
    }
    /* Each group lists its token rows in ascending order, then is cut into
     * chunks of chunk_size rows (the last one may be shorter). */
    int32_t pos = 0, s = 0;
    for (int32_t g = 0; g < n_groups; ++g) {
        int32_t a = order[g];
        int32_t start = pos;
        for (int32_t i = 0; i < M; ++i)
            if (ids[i] == a)
                sorted_token_ids[pos++] = i;
        if (chunk_size > 0) {
            for (int32_t c = start; c < pos; c += chunk_size) {
                int32_t len = pos - c < chunk_size ? pos - c : chunk_size;
                seg_indptr[s] = c;
                seg_lens[s] = len;
                weight_indices[s] = a;
                ++s;
            }
        } else {
            seg_indptr[s] = start;
            seg_lens[s] = pos - start;
            weight_indices[s] = a;
            ++s;
        }
    }
    seg_indptr[s] = pos;
    counts[0] = s;
    counts[1] = pos;
    counts[2] = n_invalid;
    free(seen);
    free(order);
    return ORACLE_OK;
}

int oracle_prepare_batch(const int32_t *ids, int32_t M, int32_t n_adapters,
                         int32_t chunk_size, int32_t *sorted_token_ids,
                         int32_t *seg_indptr, int32_t *seg_lens,
                         int32_t *weight_indices, int32_t *counts)
{
    return oracle_prepare_batch_ordered(ids, M, n_adapters, chunk_size, 0, sorted_token_ids,
                                        seg_indptr, seg_lens, weight_indices, counts);
}

/* Rank used by adapter a: its own rank when a rank table is given, else the
 * pool's (uniform) rank. */
static int32_t rank_of(const int32_t *ranks, int32_t a, int32_t r_max)
{
    return ranks ? ranks[a] : r_max;
}

/*
 * Shrink: h[i, j] = sum_k x[i, k] * A[a, j, k] for j < r_a, a = ids[i]
 * ("09. Triton Fused LoRA", Step 4 test: h_r = x[i] @ A.T).
 * Rows with no valid adapter are left untouched; columns j >= r_a of an
 * active row are set to 0.
 */
int oracle_shrink(int32_t M, int32_t d_in, int32_t r_max, const float *x,
                  int64_t ldx, const int32_t *ids, int32_t n_adapters,
                  const float *A, int64_t sA_adapter, int64_t sA_r,
                  const int32_t *ranks, double *h, int64_t ldh)
{
    for (int32_t i = 0; i < M; ++i) {
        int32_t a = ids[i];
        if (!id_valid(a, n_adapters))
            continue;
        int32_t r = rank_of(ranks, a, r_max);
        if (r < 0 || r > r_max)
            return ORACLE_ERR;
        for (int32_t j = 0; j < r_max; ++j) {
            double acc = 0.0;
            if (j < r) {
                const float *arow = A + (int64_t)a * sA_adapter + (int64_t)j * sA_r;
                const float *xrow = x + (int64_t)i * ldx;
                for (int32_t k = 0; k < d_in; ++k)
                    acc += (double)xrow[k] * (double)arow[k];
            }
            h[(int64_t)i * ldh + j] = acc;
        }
    }
    return ORACLE_OK;
}

/*
 * Expand: y[i, off_t + n] += s_a * sum_{j < r_a} h[i, j] * B_t[a, n, j]
 * for every output slice t ("09. Triton Fused LoRA", Step 4 test:
 * y_i = h_r @ B.T; "vLLM-Ascend LoRA" article, section 3.3: the delta is
 * (tmp * scale) @ B^T and is added into the output).
 *
 * s_a = adapter_scale[a] when adapter_scale is given, else `scale`.
 * The scale multiplies the finished dot product once.
 * Slices: B_t points at slice t's pool, d_out[t] rows, written to y
 * columns [col_off[t], col_off[t] + d_out[t]).
 */
int oracle_expand(int32_t M, int32_t r_max, const double *h, int64_t ldh,
                  const int32_t *ids, int32_t n_adapters, const int32_t *ranks,
                  double scale, const double *adapter_scale, int32_t n_slices,
                  const float *const *B, const int64_t *sB_adapter,
                  const int64_t *sB_n, const int32_t *d_out,
                  const int32_t *col_off, double *y, int64_t ldy)
{
    for (int32_t i = 0; i < M; ++i) {
        int32_t a = ids[i];
        if (!id_valid(a, n_adapters))
            continue;
        int32_t r = rank_of(ranks, a, r_max);
        if (r < 0 || r > r_max)
            return ORACLE_ERR;
        double s = adapter_scale ? adapter_scale[a] : scale;
        const double *hrow = h + (int64_t)i * ldh;
        for (int32_t t = 0; t < n_slices; ++t) {
            for (int32_t n = 0; n < d_out[t]; ++n) {
                const float *brow = B[t] + (int64_t)a * sB_adapter[t] + (int64_t)n * sB_n[t];
                double acc = 0.0;
                for (int32_t j = 0; j < r; ++j)
                    acc += hrow[j] * (double)brow[j];
                y[(int64_t)i * ldy + col_off[t] + n] += s * acc;
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Fused delta: the two steps above for each token row in turn, with the
 * r-wide intermediate held in a local row buffer
 * ("vLLM-Ascend LoRA" article, sections 3.2 and 4.3: shrink to r, then
 * expand back, the M x r intermediate never leaving the computation).
 * `h_out` may be NULL; when given, it receives the unscaled intermediate.
 */
int oracle_delta(int32_t M, int32_t d_in, int32_t r_max, const float *x,
                 int64_t ldx, const int32_t *ids, int32_t n_adapters,
                 const float *A, int64_t sA_adapter, int64_t sA_r,
                 const int32_t *ranks, double scale,
                 const double *adapter_scale, int32_t n_slices,
                 const float *const *B, const int64_t *sB_adapter,
                 const int64_t *sB_n, const int32_t *d_out,
                 const int32_t *col_off, double *y, int64_t ldy,
                 double *h_out, int64_t ldh)
{
    double *hrow = (double *)malloc(sizeof(double) * (size_t)(r_max > 0 ? r_max : 1));
    if (!hrow)
        return ORACLE_ERR;
    int rc = ORACLE_OK;
    for (int32_t i = 0; i < M && rc == ORACLE_OK; ++i) {
        int32_t one_id = ids[i];
        if (!id_valid(one_id, n_adapters))
            continue;
        rc = oracle_shrink(1, d_in, r_max, x + (int64_t)i * ldx, ldx, &one_id,
                           n_adapters, A, sA_adapter, sA_r, ranks, hrow, r_max);
        if (rc != ORACLE_OK)
            break;
        if (h_out)
            memcpy(h_out + (int64_t)i * ldh, hrow, sizeof(double) * (size_t)r_max);
        rc = oracle_expand(1, r_max, hrow, r_max, &one_id, n_adapters, ranks,
                           scale, adapter_scale, n_slices, B, sB_adapter, sB_n,
                           d_out, col_off, y + (int64_t)i * ldy, ldy);
    }
    free(hrow);
    return rc;
}

/*
 * The same fused delta with the token rows shared out over `threads` host
 * threads (OpenMP when the oracle is built with it; otherwise one thread).
 * Every row runs exactly the arithmetic of oracle_delta -- rows are
 * independent and each writes only its own y row -- so the result is
 * bit-identical; only the time differs.  Returns the threads used.
 */
int oracle_delta_parallel(int32_t M, int32_t d_in, int32_t r_max, const float *x,
                          int64_t ldx, const int32_t *ids, int32_t n_adapters,
                          const float *A, int64_t sA_adapter, int64_t sA_r,
                          const int32_t *ranks, double scale,
                          const double *adapter_scale, int32_t n_slices,
                          const float *const *B, const int64_t *sB_adapter,
                          const int64_t *sB_n, const int32_t *d_out,
                          const int32_t *col_off, double *y, int64_t ldy,
                          int32_t threads, int32_t *threads_used)
{
    int rc_all = ORACLE_OK, used = 1;
    if (threads < 1)
        threads = 1;
#ifdef _OPENMP
#pragma omp parallel num_threads(threads)
#endif
    {
        int rc = ORACLE_OK;
#ifdef _OPENMP
#pragma omp single
        used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 4)
#endif
        for (int32_t i = 0; i < M; ++i) {
            if (rc != ORACLE_OK)
                continue;
            rc = oracle_delta(1, d_in, r_max, x + (int64_t)i * ldx, ldx, ids + i, n_adapters, A,
                              sA_adapter, sA_r, ranks, scale, adapter_scale, n_slices, B,
                              sB_adapter, sB_n, d_out, col_off, y + (int64_t)i * ldy, ldy,
                              NULL, 0);
        }
        if (rc != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            rc_all = rc;
        }
    }
    if (threads_used)
        *threads_used = used;
    return rc_all;
}

