/*
 * Plain fp64 CPU oracle for the paged-KV chunk attention with a shared
 * Transformer-XL relative-position term (OASR documentation pages).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (each function below restates its passage):
 *
 *   Streaming chunk attention (Scheduler page, section 4.3 "Heterogeneous-offset
 *   batching": a block mask from each stream's cache_seqlens plus a score
 *   modification that adds the rel-pos bias matrix_bd / sqrt(d_k); Model Layer
 *   page, table "Three optional encoder declarations", row fixed_attention_window:
 *   a Transformer-XL table whose distances are cache + i - j, shared by a cohort
 *   with uniform cache_seqlens; Model Layer page, Nemotron ASR section:
 *   Transformer-XL relative position with rel_shift).  For stream b, head h,
 *   query i in [0,T) and key j in [0, C+T):
 *
 *       Kc_j = cache_k[b][j]      (j <  C)      Vc_j likewise
 *            = k_new [b][j-C]     (j >= C)
 *       s_ij = scale * ( sum_d (q_i[d] + u[d]) * Kc_j[d]
 *                      + sum_d (q_i[d] + v[d]) * rel[rho][d] )
 *       rho  = z - (C + i - j),   z = R - T           (rel_shift order: row 0 holds
 *                                                      the largest distance)
 *       p_ij = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)
 *       out_i = sum_j p_ij * Vc_j
 *
 *   Every cached key and the whole chunk are visible (no causal mask inside the
 *   chunk).  The scale multiplies the sum of the content and position terms.
 *
 *   Packed varlen attention (ASR Engine page, section 4.1: with sequence packing each
 *   micro-batch is one gapless varlen-attention row; Model Layer page, engine-facing
 *   surface table, forward_offline_packed).  Segment s owns rows
 *   [cu[s], cu[s+1]); query i and key j (both local to the segment) see each other
 *   in both directions, with distance i - j and rho = z - (i - j), z = (R-1)/2.
 *
 *   Chunked-limited packed attention (Model Layer page, Nemotron ASR section: the
 *   chunked_limited mask applies offline too; a query sees its own chunk of
 *   num_lookahead_tokens + 1 frames plus (sliding_window - 1) // chunk earlier chunks,
 *   and the offline pass runs in query blocks scored against their frames plus that
 *   history).  As the packed attention, but query i of a segment sees key j only if
 *   i/cs - left <= j/cs <= i/cs, cs = chunk frames, left = earlier chunks (integer
 *   division of positions local to the segment).  The query blocks are how the pass is
 *   organised, not what it computes, so the definition below is the masked attention.
 *
 *   Paged append (ASR Engine page, section 4.3 "Batched paged forward": the chunk's
 *   rows are written through each stream's block_table, and the cache length is
 *   committed afterwards by the caller).  Row t of stream b goes to logical
 *   position p = cache_seqlens[b] + t, physical block block_table[b][p / bs],
 *   slot p % bs.
 *
 * Inputs arrive as float32 arrays holding exactly the stored values (bf16 values
 * widen to float32 without rounding); all arithmetic is in double.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

/* Index of element (b, t, h, d) of a [B, T, H, D] row-major array. */
static size_t idx4(int b, int t, int h, int d, int T, int H, int D)
{
    return (((size_t)b * T + t) * H + h) * (size_t)D + d;
}

/*
 * Paged append.  Byte copy of each (b, t, h) row of D elements of elem_size
 * bytes from k_new/v_new [B,T,H,D] into k_pool/v_pool [num_blocks, bs, H, D].
 * Rows whose logical block lies past max_blocks_per_seq, or whose physical
 * block id is outside [0, num_blocks), are not written; their count is
 * returned.
 */
long oracle_paged_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                         int num_blocks, int block_size, const int32_t *block_table,
                         int max_blocks_per_seq, const int32_t *cache_seqlens,
                         int B, int T, int H, int D, int elem_size)
{
    long skipped = 0;
    size_t row_bytes = (size_t)D * elem_size;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            long p = (long)cache_seqlens[b] + t;          /* logical position */
            long logical_block = p / block_size;
            long slot = p % block_size;
            if (p < 0 || logical_block >= max_blocks_per_seq) { skipped += H; continue; }
            int32_t blk = block_table[(size_t)b * max_blocks_per_seq + logical_block];
            if (blk < 0 || blk >= num_blocks) { skipped += H; continue; }
            for (int h = 0; h < H; ++h) {
                size_t src = idx4(b, t, h, 0, T, H, D) * elem_size;
                size_t dst = ((((size_t)blk * block_size + slot) * H + h) * D) * elem_size;
                memcpy((char *)k_pool + dst, (const char *)k_new + src, row_bytes);
                memcpy((char *)v_pool + dst, (const char *)v_new + src, row_bytes);
            }
        }
    }
    return skipped;
}

/*
 * Softmax-weighted sum for one query row: given the n scores s[0..n) and the
 * n value rows (val(j) returns a pointer to D floats), writes out[0..D).
 */
static void softmax_pv(const double *s, int n, const float *const *vrows, int D, double *out)
{
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) if (s[j] > m) m = s[j];
    double denom = 0.0;
    for (int j = 0; j < n; ++j) denom += exp(s[j] - m);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(s[j] - m) / denom;
        for (int d = 0; d < D; ++d) out[d] += p * (double)vrows[j][d];
    }
}

/*
 * Streaming chunk attention for one (b, i, h) output row; see the header.
 * cache_k/cache_v: [B, C, H, D]; q, k_new, v_new, out: [B, T, H, D];
 * u, vb: [H, D]; rel: [R, H, D].  Returns 0, or -1 if a needed rel row is
 * outside [0, R).
 */
static int chunk_row(const float *q, const float *cache_k, const float *cache_v,
                     const float *k_new, const float *v_new, const float *u,
                     const float *vb, const float *rel, int R, int T, int C, int H, int D,
                     double scale, int b, int i, int h, double *s, const float **vrows,
                     double *out_row)
{
    int K = C + T;
    int z = R - T;
    const float *qi = q + idx4(b, i, h, 0, T, H, D);
    const float *uh = u + (size_t)h * D;
    const float *vh = vb + (size_t)h * D;
    for (int j = 0; j < K; ++j) {
        const float *kj = (j < C) ? cache_k + idx4(b, j, h, 0, C, H, D)
                                  : k_new + idx4(b, j - C, h, 0, T, H, D);
        vrows[j] = (j < C) ? cache_v + idx4(b, j, h, 0, C, H, D)
                           : v_new + idx4(b, j - C, h, 0, T, H, D);
        int rho = z - (C + i - j);
        if (rho < 0 || rho >= R) return -1;
        const float *rr = rel + ((size_t)rho * H + h) * D;
        double ac = 0.0, bd = 0.0;
        for (int d = 0; d < D; ++d) {
            ac += ((double)qi[d] + (double)uh[d]) * (double)kj[d];
            bd += ((double)qi[d] + (double)vh[d]) * (double)rr[d];
        }
        s[j] = (ac + bd) * scale;
    }
    softmax_pv(s, K, vrows, D, out_row);
    return 0;
}

/*
 * Streaming chunk attention over an un-paged copy of the cache.
 * rows: n_rows triples (b, i, h) to compute, or NULL for every row.
 * out: [B, T, H, D] doubles; rows not requested are left untouched.
 * Returns the number of rows that needed a rel row outside the table (those
 * rows are written as NaN).
 */
long oracle_chunk_relattn(const float *q, const float *cache_k, const float *cache_v,
                          const float *k_new, const float *v_new, const float *u,
                          const float *vb, const float *rel, int R, int B, int T, int C,
                          int H, int D, double scale, const int32_t *rows, long n_rows,
                          double *out)
{
    long total = rows ? n_rows : (long)B * T * H;
    long bad = 0;
    int K = C + T;
#pragma omp parallel reduction(+ : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)K);
        const float **vrows = (const float **)malloc(sizeof(float *) * (size_t)K);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < total; ++r) {
            int b, i, h;
            if (rows) { b = rows[3 * r]; i = rows[3 * r + 1]; h = rows[3 * r + 2]; }
            else { h = (int)(r % H); i = (int)((r / H) % T); b = (int)(r / ((long)H * T)); }
            double *o = out + idx4(b, i, h, 0, T, H, D);
            if (chunk_row(q, cache_k, cache_v, k_new, v_new, u, vb, rel, R, T, C, H, D,
                          scale, b, i, h, s, vrows, o) != 0) {
                for (int d = 0; d < D; ++d) o[d] = NAN;
                ++bad;
            }
        }
        free(s);
        free((void *)vrows);
    }
    return bad;
}

/*
 * Packed varlen attention over one gapless row of segments.
 * q, k, v, out: [total, H, D]; cu_seqlens: [num_seqs + 1], cu[0] = 0,
 * non-decreasing; rel: [R, H, D] with z = (R - 1) / 2.
 * rows: n_rows pairs (token, h) to compute, or NULL for every row.
 * Returns the number of rows that needed a rel row outside the table, or
 * whose token lies in no segment (those rows are written as NaN).
 */
long oracle_packed_relattn(const float *q, const float *k, const float *v,
                           const int32_t *cu_seqlens, int num_seqs, int total,
                           const float *u, const float *vb, const float *rel, int R,
                           int H, int D, double scale, const int32_t *rows, long n_rows,
                           double *out)
{
    long nrow = rows ? n_rows : (long)total * H;
    int z = (R - 1) / 2;
    int lmax = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int L = cu_seqlens[s + 1] - cu_seqlens[s];
        if (L > lmax) lmax = L;
    }
    long bad = 0;
#pragma omp parallel reduction(+ : bad)
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(lmax > 0 ? lmax : 1));
        const float **vrows = (const float **)malloc(sizeof(float *) * (size_t)(lmax > 0 ? lmax : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < nrow; ++r) {
            int t, h;
            if (rows) { t = rows[2 * r]; h = rows[2 * r + 1]; }
            else { h = (int)(r % H); t = (int)(r / H); }
            double *o = out + ((size_t)t * H + h) * D;
            /* the segment holding token t */
            int seg = -1;
            for (int s = 0; s < num_seqs; ++s)
                if (t >= cu_seqlens[s] && t < cu_seqlens[s + 1]) { seg = s; break; }
            int ok = seg >= 0;
            if (ok) {
                int start = cu_seqlens[seg];
                int L = cu_seqlens[seg + 1] - start;
                int i = t - start;
                const float *qi = q + ((size_t)t * H + h) * D;
                const float *uh = u + (size_t)h * D;
                const float *vh = vb + (size_t)h * D;
                for (int j = 0; j < L && ok; ++j) {
                    const float *kj = k + ((size_t)(start + j) * H + h) * D;
                    vrows[j] = v + ((size_t)(start + j) * H + h) * D;
                    int rho = z - (i - j);
                    if (rho < 0 || rho >= R) { ok = 0; break; }
                    const float *rr = rel + ((size_t)rho * H + h) * D;
                    double ac = 0.0, bd = 0.0;
                    for (int d = 0; d < D; ++d) {
                        ac += ((double)qi[d] + (double)uh[d]) * (double)kj[d];
                        bd += ((double)qi[d] + (double)vh[d]) * (double)rr[d];
                    }
                    sc[j] = (ac + bd) * scale;
                }
                if (ok) softmax_pv(sc, L, vrows, D, o);
            }
            if (!ok) {
                for (int d = 0; d < D; ++d) o[d] = NAN;
                ++bad;
            }
        }
        free(sc);
        free((void *)vrows);
    }
    return bad;
}

/* Number of OpenMP threads the oracle runs with (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the oracle's later parallel regions (timing only; results do not depend on
 * it: every output element is computed by one thread in a fixed order). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Chunked-limited packed attention: the packed attention restricted, per query, to the
 * keys of its own chunk and the `left` chunks before it (chunk = cs frames of the
 * segment).  Every key of the segment is tested against that condition. */
long oracle_packed_relattn_chunked(const float *q, const float *k, const float *v,
                                   const int32_t *cu_seqlens, int num_seqs, int total,
                                   const float *u, const float *vb, const float *rel, int R,
                                   int H, int D, double scale, int cs, int left,
                                   const int32_t *rows, long n_rows, double *out)
{
    long nrow = rows ? n_rows : (long)total * H;
    int z = (R - 1) / 2;
    int lmax = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int L = cu_seqlens[s + 1] - cu_seqlens[s];
        if (L > lmax) lmax = L;
    }
    long bad = 0;
#pragma omp parallel reduction(+ : bad)
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(lmax > 0 ? lmax : 1));
        const float **vrows = (const float **)malloc(sizeof(float *) * (size_t)(lmax > 0 ? lmax : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < nrow; ++r) {
            int t, h;
            if (rows) { t = rows[2 * r]; h = rows[2 * r + 1]; }
            else { h = (int)(r % H); t = (int)(r / H); }
            double *o = out + ((size_t)t * H + h) * D;
            int seg = -1;
            for (int s = 0; s < num_seqs; ++s)
                if (t >= cu_seqlens[s] && t < cu_seqlens[s + 1]) { seg = s; break; }
            int ok = seg >= 0;
            if (ok) {
                int start = cu_seqlens[seg];
                int L = cu_seqlens[seg + 1] - start;
                int i = t - start;
                const float *qi = q + ((size_t)t * H + h) * D;
                const float *uh = u + (size_t)h * D;
                const float *vh = vb + (size_t)h * D;
                int n = 0;   /* visible keys, in order */
                for (int j = 0; j < L && ok; ++j) {
                    if (j / cs < i / cs - left || j / cs > i / cs) continue;
                    const float *kj = k + ((size_t)(start + j) * H + h) * D;
                    vrows[n] = v + ((size_t)(start + j) * H + h) * D;
                    int rho = z - (i - j);
                    if (rho < 0 || rho >= R) { ok = 0; break; }
                    const float *rr = rel + ((size_t)rho * H + h) * D;
                    double ac = 0.0, bd = 0.0;
                    for (int d = 0; d < D; ++d) {
                        ac += ((double)qi[d] + (double)uh[d]) * (double)kj[d];
                        bd += ((double)qi[d] + (double)vh[d]) * (double)rr[d];
                    }
                    sc[n++] = (ac + bd) * scale;
                }
                if (ok) softmax_pv(sc, n, vrows, D, o);
            }
            if (!ok) {
                for (int d = 0; d < D; ++d) o[d] = NAN;
                ++bad;
            }
        }
        free(sc);
        free((void *)vrows);
    }
    return bad;
}
