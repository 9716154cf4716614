/*
 * swa_oracle.c -- the CPU oracle for causal sliding-window attention with
 * attention sinks.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * It is deliberately plain and slow: fp64 throughout, an explicit mask built
 * set by set, and a naive loop over every key position of every query row.
 * There is no tiling, no online softmax and no slot arithmetic beyond the
 * definition of the rolling buffer.
 *
 * Sources (web pages on the subject; section / figure named on each routine):
 *   [SW]  "Sliding Window and Sparse Attention, from Longformer to CSA2"
 *   [LS]  "Local and Sparse Attention: Reading Fewer Token Positions"
 *   [QA]  "How does sliding window attention (SWA) reduce memory usage in
 *          long-context models?"
 *
 * Readings taken where the pages are silent (each is a choice, listed with
 * the rest of the design notes):
 *   - the window holds w cells including the current one ([LS] Fig. 1);
 *   - sinks are the token positions 0..g-1, united with the window, a key in
 *     both sets counted once, and never a future key ([LS] Fig. 2);
 *   - GQA maps query head h to key/value head h / (H / Hkv);
 *   - `scale` multiplies q.k before masking;
 *   - the rolling cache keeps ring slots 0..w-1 (position p in slot p mod w)
 *     followed by g sink slots (position p < g also in slot w + p).
 *
 * Pins: every public routine here is checked by tests that do not call back
 * into it for the expected value (worked examples printed on the pages,
 * closed forms, textbook special cases and torch routines).  None is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* The mask.                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * One row i of the explicit n x n mask (1 = the query at position i reads the
 * key at position j, 0 = blocked), built the way the pages build it:
 *   1. the causal lower triangle: j <= i            ([SW] §1, causal models)
 *   2. cut to the band of the last w cells:
 *      keep i-w+1 <= j <= i                         ([SW] §2 definition;
 *                                                    [QA] Example: the
 *                                                    triu(tril(.), -w+1) mask;
 *                                                    [LS] Fig. 1)
 *   3. add the sink columns j < g, still only where j <= i
 *                                                   ([SW] §2 attention sinks;
 *                                                    [LS] Fig. 2: a key in the
 *                                                    window and the designated
 *                                                    set is read once, and no
 *                                                    future key is read)
 */
void oracle_mask_row(int64_t i, int64_t n, int64_t w, int64_t g, uint8_t *row)
{
    int64_t j;
    /* step 1: causal triangle */
    for (j = 0; j < n; ++j)
        row[j] = (uint8_t)(j <= i);
    /* step 2: keep only the band i-w+1 .. i */
    for (j = 0; j < n; ++j)
        if (j < i - w + 1)
            row[j] = 0;
    /* step 3: the sink columns, where causal */
    for (j = 0; j < n && j < g; ++j)
        if (j <= i)
            row[j] = 1;
}

/* The whole n x n mask, row-major (n*n bytes, caller-owned). */
void oracle_mask(int64_t n, int64_t w, int64_t g, uint8_t *mask)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i)
        oracle_mask_row(i, n, w, g, mask + (size_t)i * (size_t)n);
}

/*
 * The number of connections: the count of ones in the mask.  [LS] Fig. 1
 * counts 21 connections for eight tokens and a window of three, against 36
 * for full causal attention.
 */
int64_t oracle_count_pairs(int64_t n, int64_t w, int64_t g)
{
    int64_t total = 0;
#pragma omp parallel reduction(+ : total)
    {
        uint8_t *row = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        int64_t ii;
#pragma omp for schedule(static)
        for (ii = 0; ii < n; ++ii) {
            int64_t j, c = 0;
            oracle_mask_row(ii, n, w, g, row);
            for (j = 0; j < n; ++j)
                c += row[j];
            total += c;
        }
        free(row);
    }
    return total;
}

/*
 * Block sparsity ([SW] §1 last paragraph and §4 "Block-sparse attention"):
 * the n x n mask seen as a grid of BM x BN tiles.  For tile (qt, kt), rows
 * qt*BM .. qt*BM+BM-1 that exist (< n) and columns kt*BN .. kt*BN+BN-1:
 *   0 = no allowed pair (skipped), 1 = some but not all pairs allowed
 *   (partial: needs the element mask), 2 = every pair allowed (full).
 * Columns at or past n count as blocked cells.  Output is
 * cls[qt * n_kt + kt], n_qt = ceil(n/BM), n_kt = ceil(n/BN).  Brute force over
 * the explicit mask.
 */
void oracle_tiles(int64_t n, int64_t w, int64_t g, int64_t BM, int64_t BN, int32_t *cls)
{
    int64_t n_qt = (n + BM - 1) / BM, n_kt = (n + BN - 1) / BN, qt;
#pragma omp parallel
    {
        uint8_t *row = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        int64_t *cnt = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_kt > 0 ? n_kt : 1));
#pragma omp for schedule(dynamic, 1)
        for (qt = 0; qt < n_qt; ++qt) {
            int64_t kt, i, rows = 0;
            for (kt = 0; kt < n_kt; ++kt)
                cnt[kt] = 0;
            for (i = qt * BM; i < qt * BM + BM && i < n; ++i) {
                int64_t j;
                ++rows;
                oracle_mask_row(i, n, w, g, row);
                for (j = 0; j < n; ++j)
                    cnt[j / BN] += row[j];
            }
            for (kt = 0; kt < n_kt; ++kt) {
                int64_t cells = rows * BN; /* includes columns past n */
                int32_t c = 0;
                if (cnt[kt] == cells)
                    c = 2;
                else if (cnt[kt] > 0)
                    c = 1;
                cls[qt * n_kt + kt] = c;
            }
        }
        free(row);
        free(cnt);
    }
}

/* ------------------------------------------------------------------------ */
/* Other fixed patterns.                                                     */
/* ------------------------------------------------------------------------ */

/*
 * Pattern codes (the same numbers as the library's public enum, which this
 * file does not include):
 *   0  window     the band of the last w cells plus the sinks (above);
 *   1  dilated    every r-th key in a band r times wider: the keys i, i-r,
 *                 ..., i-(w-1)r ([SW] §2 "Dilated windows": the cost of a
 *                 window of w, a reach r times longer; [SW] §10 glossary:
 *                 a window that attends to every r-th key);
 *   2  strided    the Sparse Transformer's strided head: every j with
 *                 (i - j) mod r = 0 ([SW] §4, Sparse Transformer);
 *   3  landmark   the band of the last w cells plus positions designated at
 *                 regular intervals, j mod r = 0 ([LS] Fig. 2, right: with
 *                 w = 3 and r = 4, position 7 reads 0, 4, 5, 6, 7).
 * In every pattern the sink columns j < g are added where causal, and no key
 * is read twice (a mask is a set).
 */
void oracle_pattern_mask_row(int64_t i, int64_t n, int64_t w, int64_t g, int64_t r,
                             int pattern, uint8_t *row)
{
    int64_t j;
    if (pattern == 0) {
        oracle_mask_row(i, n, w, g, row);
        return;
    }
    /* causal triangle */
    for (j = 0; j < n; ++j)
        row[j] = (uint8_t)(j <= i);
    if (pattern == 1 || pattern == 2) {
        /* only keys a whole number of strides back */
        for (j = 0; j < n; ++j)
            if ((i - j) % r != 0)
                row[j] = 0;
        /* dilated: only the w nearest of them */
        if (pattern == 1)
            for (j = 0; j < n; ++j)
                if (i - j > (w - 1) * r)
                    row[j] = 0;
    } else if (pattern == 3) {
        /* the band of the last w cells ... */
        for (j = 0; j < n; ++j)
            if (j < i - w + 1)
                row[j] = 0;
        /* ... plus the landmark positions, where causal */
        for (j = 0; j < n; j += r)
            if (j <= i)
                row[j] = 1;
    }
    /* the sink columns, where causal */
    for (j = 0; j < n && j < g; ++j)
        if (j <= i)
            row[j] = 1;
}

/* The whole n x n mask of a pattern, row-major (n*n bytes, caller-owned). */
void oracle_pattern_mask(int64_t n, int64_t w, int64_t g, int64_t r, int pattern, uint8_t *mask)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i)
        oracle_pattern_mask_row(i, n, w, g, r, pattern, mask + (size_t)i * (size_t)n);
}

/* The number of connections of a pattern: the count of ones in its mask. */
int64_t oracle_pattern_count_pairs(int64_t n, int64_t w, int64_t g, int64_t r, int pattern)
{
    int64_t total = 0;
#pragma omp parallel reduction(+ : total)
    {
        uint8_t *row = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        int64_t ii;
#pragma omp for schedule(static)
        for (ii = 0; ii < n; ++ii) {
            int64_t j, c = 0;
            oracle_pattern_mask_row(ii, n, w, g, r, pattern, row);
            for (j = 0; j < n; ++j)
                c += row[j];
            total += c;
        }
        free(row);
    }
    return total;
}

/* ------------------------------------------------------------------------ */
/* Attention.                                                                */
/* ------------------------------------------------------------------------ */

/*
 * One query row: Attention = softmax(q K^T * scale) V over the keys the mask
 * row allows ([SW] §1 first formula), masked keys given -inf before the
 * softmax ([LS] Fig. 1 text; [QA] Example).  With zero_score != 0 the masked
 * keys get a score of 0 instead -- the computation [LS] Fig. 1 warns is a
 * different one; it exists only so that a test can show the two differ.
 *
 * Softmax in fp64 with the maximum subtracted.  lse = log(sum_j exp(s_j)),
 * natural log ([SW] §6 stage 3 and §10: the log-sum-exp lets results over
 * disjoint key sets be normalised jointly).
 *
 * sink_logit: the learned per-head attention sink of [SW] §6 stage 3 (a
 * logit that absorbs probability mass when nothing is relevant), taken as
 * one more entry of the softmax with score sink_logit and a value vector of
 * zeros: it enters the maximum and the normalising sum, not the output.
 * -INFINITY means no such sink (the plain softmax above).
 */
static void attend_row(const double *q, const double *K, const double *V,
                       const uint8_t *row, int64_t nkeys, int64_t d, double scale,
                       int zero_score, double sink_logit, double *s, double *o, double *lse)
{
    int64_t j, k;
    double mx = sink_logit, sum = 0.0;
    for (j = 0; j < nkeys; ++j) {
        if (row[j]) {
            double dot = 0.0;
            for (k = 0; k < d; ++k)
                dot += q[k] * K[j * d + k];
            s[j] = scale * dot;
        } else {
            s[j] = zero_score ? 0.0 : -INFINITY;
        }
        if (s[j] > mx)
            mx = s[j];
    }
    for (k = 0; k < d; ++k)
        o[k] = 0.0;
    for (j = 0; j < nkeys; ++j) {
        double p = exp(s[j] - mx); /* exp(-inf) = 0 for masked keys */
        if (p == 0.0)
            continue;
        sum += p;
        for (k = 0; k < d; ++k)
            o[k] += p * V[j * d + k];
    }
    sum += exp(sink_logit - mx); /* the sink: in the sum, value zero */
    for (k = 0; k < d; ++k)
        o[k] /= sum;
    if (lse)
        *lse = mx + log(sum);
}

/* sink_logits [H] or NULL: the per-head sink logit of query head h. */
static double sink_of(const double *sink_logits, int64_t h)
{
    return sink_logits ? sink_logits[h] : -INFINITY;
}

/*
 * Prefill over full sequences.  Layouts (row-major, contiguous):
 *   Q, O [B][H][n][d],  K, V [B][Hkv][n][d],  LSE [B][H][n] (may be NULL).
 * Query head h reads key/value head h / (H / Hkv) (grouped-query attention,
 * [SW] §10 glossary).  Every (b, h, i) row is independent.
 */
void oracle_prefill(const double *Q, const double *K, const double *V, double *O, double *LSE,
                    int64_t B, int64_t H, int64_t Hkv, int64_t n, int64_t d,
                    int64_t w, int64_t g, double scale, int zero_score,
                    const double *sink_logits)
{
    int64_t r, rows = B * H * n, G = H / Hkv;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for schedule(dynamic, 16)
        for (r = 0; r < rows; ++r) {
            int64_t i = r % n, h = (r / n) % H, b = r / (n * H);
            int64_t kvh = h / G;
            const double *Kbh = K + ((b * Hkv + kvh) * n) * d;
            const double *Vbh = V + ((b * Hkv + kvh) * n) * d;
            oracle_mask_row(i, n, w, g, mrow);
            attend_row(Q + r * d, Kbh, Vbh, mrow, n, d, scale, zero_score,
                       sink_of(sink_logits, h), s, O + r * d, LSE ? LSE + r : NULL);
        }
        free(mrow);
        free(s);
    }
}

/*
 * Prefill on a sample of rows only (for sequences too long to run whole).
 * rows[3*t .. 3*t+2] = (b, h, i); q_rows [nrows][d] holds Q[b][h][i][:] for
 * each sampled row; O_rows [nrows][d], LSE_rows [nrows] or NULL.
 * Same arithmetic as oracle_prefill, row by row.
 */
void oracle_prefill_rows(const double *q_rows, const double *K, const double *V,
                         int64_t B, int64_t H, int64_t Hkv, int64_t n, int64_t d,
                         int64_t w, int64_t g, double scale,
                         const int64_t *rows, int64_t nrows, double *O_rows, double *LSE_rows,
                         const double *sink_logits)
{
    int64_t t, G = H / Hkv;
    (void)B;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for schedule(dynamic, 1)
        for (t = 0; t < nrows; ++t) {
            int64_t b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
            int64_t kvh = h / G;
            const double *q = q_rows + t * d;
            const double *Kbh = K + ((b * Hkv + kvh) * n) * d;
            const double *Vbh = V + ((b * Hkv + kvh) * n) * d;
            oracle_mask_row(i, n, w, g, mrow);
            attend_row(q, Kbh, Vbh, mrow, n, d, scale, 0, sink_of(sink_logits, h), s,
                       O_rows + t * d, LSE_rows ? LSE_rows + t : NULL);
        }
        free(mrow);
        free(s);
    }
}

/*
 * Prefill under one of the fixed patterns above (pattern 0 is oracle_prefill
 * itself).  Same layouts and arithmetic as oracle_prefill; only the mask row
 * differs.
 */
void oracle_prefill_pattern(const double *Q, const double *K, const double *V, double *O,
                            double *LSE, int64_t B, int64_t H, int64_t Hkv, int64_t n,
                            int64_t d, int64_t w, int64_t g, int64_t r, int pattern,
                            double scale, const double *sink_logits)
{
    int64_t t, rows = B * H * n, G = H / Hkv;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for schedule(dynamic, 16)
        for (t = 0; t < rows; ++t) {
            int64_t i = t % n, h = (t / n) % H, b = t / (n * H);
            int64_t kvh = h / G;
            const double *Kbh = K + ((b * Hkv + kvh) * n) * d;
            const double *Vbh = V + ((b * Hkv + kvh) * n) * d;
            oracle_pattern_mask_row(i, n, w, g, r, pattern, mrow);
            attend_row(Q + t * d, Kbh, Vbh, mrow, n, d, scale, 0, sink_of(sink_logits, h), s,
                       O + t * d, LSE ? LSE + t : NULL);
        }
        free(mrow);
        free(s);
    }
}

/* oracle_prefill_rows under a fixed pattern: sampled (b, h, i) rows only. */
void oracle_prefill_pattern_rows(const double *q_rows, const double *K, const double *V,
                                 int64_t B, int64_t H, int64_t Hkv, int64_t n, int64_t d,
                                 int64_t w, int64_t g, int64_t r, int pattern, double scale,
                                 const int64_t *rows, int64_t nrows, double *O_rows,
                                 double *LSE_rows, const double *sink_logits)
{
    int64_t t, G = H / Hkv;
    (void)B;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for schedule(dynamic, 1)
        for (t = 0; t < nrows; ++t) {
            int64_t b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
            int64_t kvh = h / G;
            const double *Kbh = K + ((b * Hkv + kvh) * n) * d;
            const double *Vbh = V + ((b * Hkv + kvh) * n) * d;
            oracle_pattern_mask_row(i, n, w, g, r, pattern, mrow);
            attend_row(q_rows + t * d, Kbh, Vbh, mrow, n, d, scale, 0, sink_of(sink_logits, h),
                       s, O_rows + t * d, LSE_rows ? LSE_rows + t : NULL);
        }
        free(mrow);
        free(s);
    }
}

/* ------------------------------------------------------------------------ */
/* Decode.                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * One-token decode against the unbounded history of every position seen so
 * far ([SW] §1: decode is one query against the cached keys).  The query of
 * sequence b sits at position pos[b] and reads, among positions 0..pos[b],
 * the ones row pos[b] of the mask allows.  No slot arithmetic: the history
 * is indexed by position.
 *   q, O [B][H][d];  Khist, Vhist [B][Hkv][P][d] with P > max(pos);
 *   LSE [B][H] or NULL.
 */
void oracle_decode_history(const double *q, const double *Khist, const double *Vhist,
                           const int64_t *pos, int64_t P,
                           int64_t B, int64_t H, int64_t Hkv, int64_t d,
                           int64_t w, int64_t g, double scale, double *O, double *LSE,
                           const double *sink_logits)
{
    int64_t r, G = H / Hkv;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)(P > 0 ? P : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1));
#pragma omp for schedule(dynamic, 1)
        for (r = 0; r < B * H; ++r) {
            int64_t b = r / H, h = r % H, kvh = h / G, p = pos[b];
            const double *Kbh = Khist + ((b * Hkv + kvh) * P) * d;
            const double *Vbh = Vhist + ((b * Hkv + kvh) * P) * d;
            oracle_mask_row(p, p + 1, w, g, mrow);
            attend_row(q + r * d, Kbh, Vbh, mrow, p + 1, d, scale, 0, sink_of(sink_logits, h), s,
                       O + r * d, LSE ? LSE + r : NULL);
        }
        free(mrow);
        free(s);
    }
}

/*
 * Where the rolling cache keeps position p ([SW] §2: position i overwrites
 * slot i mod w; [SW] §2 attention sinks and [LS] Fig. 4 text: the first
 * positions must stay stored after they leave the window).
 *   ring slot = p mod w;  sink slot = w + p if p < g, else -1.
 */
void oracle_cache_slots(int64_t p, int64_t w, int64_t g, int64_t *ring, int64_t *sink)
{
    *ring = p % w;
    *sink = (p < g) ? w + p : -1;
}

/*
 * One-token decode from a rolling cache Kc, Vc [B][Hkv][w+g][d] that holds
 * the most recent positions in their ring slots and positions 0..g-1 in their
 * sink slots.  For each key position j that row pos[b] of the mask allows,
 * the key is fetched from where the cache keeps it: its ring slot while it is
 * still inside the window (j > pos-w), its sink slot once it has left it.
 * Then the same attention as above over those keys.
 */
void oracle_decode_cache(const double *q, const double *Kc, const double *Vc,
                         const int64_t *pos, int64_t B, int64_t H, int64_t Hkv, int64_t d,
                         int64_t w, int64_t g, double scale, double *O, double *LSE,
                         const double *sink_logits)
{
    int64_t r, G = H / Hkv, S = w + g;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < B * H; ++r) {
        int64_t b = r / H, h = r % H, kvh = h / G, p = pos[b], j, k, cnt = 0;
        const double *Kb = Kc + ((b * Hkv + kvh) * S) * d;
        const double *Vb = Vc + ((b * Hkv + kvh) * S) * d;
        uint8_t *mrow = (uint8_t *)malloc((size_t)(p + 1));
        double *Kg, *Vg, *s;
        uint8_t *ones;
        oracle_mask_row(p, p + 1, w, g, mrow);
        for (j = 0; j <= p; ++j)
            cnt += mrow[j];
        Kg = (double *)malloc(sizeof(double) * (size_t)(cnt * d));
        Vg = (double *)malloc(sizeof(double) * (size_t)(cnt * d));
        s = (double *)malloc(sizeof(double) * (size_t)cnt);
        ones = (uint8_t *)malloc((size_t)cnt);
        cnt = 0;
        for (j = 0; j <= p; ++j) {
            int64_t ring, sink, slot;
            if (!mrow[j])
                continue;
            oracle_cache_slots(j, w, g, &ring, &sink);
            slot = (j <= p - w) ? sink : ring; /* left the window: only the sink copy remains */
            for (k = 0; k < d; ++k) {
                Kg[cnt * d + k] = Kb[slot * d + k];
                Vg[cnt * d + k] = Vb[slot * d + k];
            }
            ones[cnt] = 1;
            ++cnt;
        }
        attend_row(q + r * d, Kg, Vg, ones, cnt, d, scale, 0, sink_of(sink_logits, h), s, O + r * d,
                   LSE ? LSE + r : NULL);
        free(mrow);
        free(Kg);
        free(Vg);
        free(s);
        free(ones);
    }
}

/* Threads the OpenMP runtime will use (for reporting the CPU baseline). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int t)
{
#ifdef _OPENMP
    if (t > 0)
        omp_set_num_threads(t);
#else
    (void)t;
#endif
}
