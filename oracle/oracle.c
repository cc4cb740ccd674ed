/*
 * oracle.c -- plain, slow, obviously correct CPU model of the tovl hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this file's library.  The CUDA
 * product path never includes, links or calls it, and it includes nothing
 * from the CUDA path: the two share no code, table or helper.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] Astro Bear, "Fused compute/communication operators (4): cross-GPU
 *        sync protocols on PCIe -- single writer, election and watermarks"
 *        section 2 (slot + monotonic sequence), section 3 (local election and
 *        single-writer publish), section 4 (64-row chunk watermarks),
 *        section 5 (row-block counters pre-seeded with the padding count),
 *        section 7 (expected table recomputed on the host by naive loops).
 *   [P3] "DeepEP FIFO/Streaming Pipeline analysis", notify stage (per-expert
 *        token counting before dispatch).
 *
 * Every function is the plain definition of what the path computes:
 *   gather        G[s*R + i, :] = X_s[i, :]
 *   dispatch      D[dst(t,j), :] = x[t, :], every other row zero
 *   copy_perm     dst[perm[i], :] = src[i, :]
 *   reduce        O[m, :] = bf16( sum_{s=0..S-1} f32(P_s[m, :]) ), fp32 sums in
 *                 ascending s (the reduce-scatter that follows a K-split GEMM)
 *   combine       S[t*k + j, :] = Y[dst(t,j), :]  (token-ordered staging) and
 *                 C[t, :] = bf16( sum_{j=0..k-1} w[t,j] * f32(S[t*k + j, :]) ),
 *                 each product and each sum rounded to fp32 in ascending j
 *   matmul_f32    O[m,n] = sum_{k=0..K-1} f32(A[m,k]) * f32(W[k,n]),
 *                 accumulated in fp32 in ascending k (the accumulate precision
 *                 the method fixes: bf16 inputs, fp32 accumulation)
 *   plans/tables  by naive loops over rows and routing entries
 *   ctrl state    closed forms of the monotonic protocol after R rounds
 *
 * Readings where the pages are silent (stable (t,j) row order inside an
 * expert segment, per-round padding seeds for every counter, bf16 output by
 * round-to-nearest-even) are stated beside the function that takes them.
 *
 * Parity pins: every function here is checked by tests against numpy /
 * torch library routines, closed forms, brute force on tiny inputs and
 * special cases (identity weights, all-padding blocks).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 <-> f32                                                        */
/* ------------------------------------------------------------------ */

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round binary32 to bf16, nearest-even (the IEEE default rounding).  NaN is
 * kept a quiet NaN with its sign.  Method: add half an ulp of the target
 * format minus one, plus the parity of the kept lsb, then truncate. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

void oracle_bf16_to_f32(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f32(in[i]);
}

void oracle_f32_to_bf16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* ------------------------------------------------------------------ */
/* data plane                                                          */
/* ------------------------------------------------------------------ */

/* All-gather of logical shards into one buffer: shard s, row i lands at
 * row s*R + i (the tensor-parallel all-gather whose volume the platform page
 * [P4 section 3] shows hiding under the GEMM).  Shards are given as a table of
 * base pointers, each [R][K] row-major bf16. */
void oracle_gather(const uint16_t *const *shards, int S, int R, int K, uint16_t *G)
{
    for (int s = 0; s < S; ++s)
        for (int i = 0; i < R; ++i)
            for (int k = 0; k < K; ++k)
                G[((int64_t)s * R + i) * K + k] = shards[s][(int64_t)i * K + k];
}

/* Dispatch scatter: every routed pair (t, j) copies token row t to its
 * destination row dst[t*k + j]; rows that no pair targets are padding and
 * hold zero ([P1 section 5]: padding rows are never written by producers). */
void oracle_dispatch(const uint16_t *x, int T, int H, const int32_t *dst, int k,
                     int64_t m_pad, uint16_t *D)
{
    memset(D, 0, (size_t)m_pad * (size_t)H * sizeof(uint16_t));
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t r = dst[(int64_t)t * k + j];
            for (int h = 0; h < H; ++h)
                D[r * H + h] = x[(int64_t)t * H + h];
        }
}

/* Combine, the reverse of dispatch ([P1 section 3]: the "layer1 combine"
 * pushes every expert-output row back to its token's staging row, counted
 * and published per chunk by the elected last writer).  Pair (t, j) was
 * dispatched to row dst[t*k + j] of the expert layout; its output row comes
 * back to staging row t*k + j.  The combined token row is the gate-weighted
 * sum of its k staged rows.  Reading where the pages are silent: weights are
 * fp32, the sum runs over j in ascending order with every product and every
 * partial sum rounded to fp32 (no fused multiply-add), and the result is
 * rounded to bf16, nearest even. */
void oracle_combine(const uint16_t *Y, int N, const int32_t *dst, const float *w, int T, int k,
                    uint16_t *S, uint16_t *C)
{
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t s = (int64_t)t * k + j;
            memcpy(S + s * N, Y + (int64_t)dst[s] * N, (size_t)N * sizeof(uint16_t));
        }
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int64_t s = (int64_t)t * k + j;
                float prod = w[s] * bf16_to_f32(S[s * N + n]);
                acc = acc + prod;
            }
            C[(int64_t)t * N + n] = f32_to_bf16_rne(acc);
        }
}

/* Reduction of S partial products, the reduce half of a row-parallel
 * layer's reduce-scatter (ReduceScatter is the collective the platform page
 * [P4 section 3] benchmarks beside AllGather).  Shard s holds the partial
 * P_s = bf16(X_s W_s) of its K-slice; the output row m is the sum over
 * shards.  Readings where the pages are silent: partials travel as bf16 (the
 * rounded output of each shard's GEMM), the sum runs over s in ascending
 * order with every partial sum rounded to fp32, and the result is rounded
 * to bf16, nearest even.  P is [S][M][N], O is [M][N]. */
void oracle_reduce_partials(const uint16_t *P, int S, int64_t M, int N, uint16_t *O)
{
    for (int64_t m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int s = 0; s < S; ++s)
                acc = acc + bf16_to_f32(P[((int64_t)s * M + m) * N + n]);
            O[m * N + n] = f32_to_bf16_rne(acc);
        }
}

/* Permuted row copy: source row i goes to destination row perm[i]. */
void oracle_copy_perm(const uint8_t *src, int64_t n_rows, int row_bytes,
                      const int32_t *perm, uint8_t *dst)
{
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t r = perm[i];
        for (int b = 0; b < row_bytes; ++b)
            dst[r * row_bytes + b] = src[i * (int64_t)row_bytes + b];
    }
}

/* ------------------------------------------------------------------ */
/* dense contraction                                                   */
/* ------------------------------------------------------------------ */

/* O[m,n] = sum_k f32(A[m,k]) * f32(W[k,n]), fp32 accumulation, k ascending.
 * A is [M][K] row-major, W is [K][N] row-major, O is [M][N] fp32.
 * Output rows are independent, so they are shared among threads; the sum for
 * one element is always taken in the same k order. */
void oracle_matmul_f32(const uint16_t *A, const uint16_t *W, int M, int N, int K, float *O)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; ++m) {
        float *o = O + (int64_t)m * N;
        for (int n = 0; n < N; ++n) o[n] = 0.0f;
        for (int k = 0; k < K; ++k) {
            float a = bf16_to_f32(A[(int64_t)m * K + k]);
            const uint16_t *w = W + (int64_t)k * N;
            for (int n = 0; n < N; ++n) {
                float p = a * bf16_to_f32(w[n]);
                o[n] = o[n] + p;
            }
        }
    }
}

/* Same definition on a chosen subset of rows of A (row indices rows[0..nr)),
 * for sampled checks of outputs too large to compute whole. */
void oracle_matmul_rows_f32(const uint16_t *A, const uint16_t *W, int N, int K,
                            const int64_t *rows, int nr, float *O)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nr; ++i) {
        int64_t m = rows[i];
        float *o = O + (int64_t)i * N;
        for (int n = 0; n < N; ++n) o[n] = 0.0f;
        for (int k = 0; k < K; ++k) {
            float a = bf16_to_f32(A[m * K + k]);
            const uint16_t *w = W + (int64_t)k * N;
            for (int n = 0; n < N; ++n) {
                float p = a * bf16_to_f32(w[n]);
                o[n] = o[n] + p;
            }
        }
    }
}

/* Grouped contraction over padded expert segments: rows [off[e], off[e+1])
 * of D are multiplied by expert e's weight W[e] ([K][N] row-major). */
void oracle_grouped_matmul_f32(const uint16_t *D, const uint16_t *W, int E, const int32_t *off,
                               int N, int K, float *O)
{
    for (int e = 0; e < E; ++e) {
        int64_t r0 = off[e], r1 = off[e + 1];
        if (r1 > r0)
            oracle_matmul_f32(D + r0 * K, W + (int64_t)e * K * N, (int)(r1 - r0), N, K,
                              O + r0 * N);
    }
}

/* ------------------------------------------------------------------ */
/* expected tables and routing plan (naive loops, [P1 section 7])      */
/* ------------------------------------------------------------------ */

/* Gather: the number of real rows that land in each chunk of chunk_rows
 * destination rows, by a loop over every destination row.  A chunk's
 * remaining chunk_rows - expected[c] arrivals are the padding seed. */
void oracle_gather_expected(int64_t n_rows, int chunk_rows, int n_chunks, int32_t *expected)
{
    for (int c = 0; c < n_chunks; ++c) expected[c] = 0;
    for (int64_t r = 0; r < n_rows; ++r) expected[r / chunk_rows] += 1;
}

/* Permuted copy: the number of source rows whose destination falls in each
 * destination chunk. */
void oracle_perm_expected(const int32_t *perm, int64_t n_rows, int chunk_rows, int n_chunks,
                          int32_t *expected)
{
    for (int c = 0; c < n_chunks; ++c) expected[c] = 0;
    for (int64_t i = 0; i < n_rows; ++i) expected[perm[i] / chunk_rows] += 1;
}

/* Dispatch plan for top-k routing topk[T][k] over E experts.
 *   counts[e]   number of pairs (t,j) routed to e (the notify-stage count)
 *   off[e]      start row of expert e's segment; segments are padded up to a
 *               multiple of block_rows, off[E] = total padded rows
 *   dst[t*k+j]  destination row: off[e] plus the number of earlier pairs
 *               (row-major (t,j) order) routed to the same e.  (Reading: the
 *               pages leave the in-segment order open; a stable order makes
 *               the dispatched buffer a function of the routing alone.)
 *   src[r]      token that fills row r, or -1 for a padding row
 *   pad[b]      rows of block b that no pair fills (the counter seed)
 *   blk_e[b]    expert that owns block b
 * Returns the number of padded blocks, or -1 if an expert id is outside
 * [0, E) or the outputs would exceed max_rows. */
int oracle_dispatch_plan(const int32_t *topk, int T, int k, int E, int block_rows,
                         int64_t max_rows, int32_t *counts, int32_t *off, int32_t *dst,
                         int32_t *src, int32_t *pad, int32_t *blk_e)
{
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < (int64_t)T * k; ++i) {
        int e = topk[i];
        if (e < 0 || e >= E) return -1;
        counts[e] += 1;
    }
    off[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t padded = ((int64_t)counts[e] + block_rows - 1) / block_rows * block_rows;
        if ((int64_t)off[e] + padded > max_rows) return -1;
        off[e + 1] = off[e] + (int32_t)padded;
    }
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = topk[(int64_t)t * k + j];
            dst[(int64_t)t * k + j] = off[e] + fill[e];
            fill[e] += 1;
        }
    free(fill);
    int64_t m_pad = off[E];
    for (int64_t r = 0; r < m_pad; ++r) src[r] = -1;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) src[dst[(int64_t)t * k + j]] = t;
    int n_blocks = (int)(m_pad / block_rows);
    for (int b = 0; b < n_blocks; ++b) {
        int real = 0;
        for (int r = 0; r < block_rows; ++r)
            if (src[(int64_t)b * block_rows + r] >= 0) real += 1;
        pad[b] = block_rows - real;
        int owner = -1;
        for (int e = 0; e < E; ++e)
            if ((int64_t)b * block_rows >= off[e] && (int64_t)b * block_rows < off[e + 1]) owner = e;
        blk_e[b] = owner;
    }
    return n_blocks;
}

/* ------------------------------------------------------------------ */
/* control-plane end state ([P1 sections 2, 4, 5])                     */
/* ------------------------------------------------------------------ */

/* After the R-th call on one handle, with sequence numbers 1, 2, ..., R and
 * never reset:
 *   every chunk watermark slot holds R (the last published sequence; round k
 *   waits for >= k, so older values are harmless),
 *   every chunk arrival counter holds R * chunk_rows (each round adds the
 *   chunk's real arrivals plus its padding seed, i.e. exactly chunk_rows),
 *   every row-block counter holds R * block_rows (real arrivals plus the
 *   padding seed reach ROW_BLOCK exactly, once per round). */
void oracle_ctrl_state(int64_t R, int n_chunks, int n_blocks, int chunk_rows, int block_rows,
                       int32_t *slots, int32_t *cnts, int32_t *rbcnts)
{
    for (int c = 0; c < n_chunks; ++c) {
        slots[c] = (int32_t)R;
        cnts[c] = (int32_t)(R * chunk_rows);
    }
    for (int b = 0; b < n_blocks; ++b) rbcnts[b] = (int32_t)(R * block_rows);
}
