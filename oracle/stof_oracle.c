/*
 * CPU oracle for the STOF masked-attention hot path.  TEST INFRASTRUCTURE
 * ONLY: it is called by the tests, by the package's smoke check and by the
 * benchmark's CPU-baseline leg, never by the library it checks.  It shares
 * no code with the CUDA path.
 *
 * Everything here is the plain definition, written for a reader to check by
 * eye: direct loops, fp64 arithmetic, no blocking or fusion.
 *
 * Citations (all to "Accelerating Sparse Transformer Inference on GPU"):
 *   [ABS]  arXiv abstract (catalogue record page): STOF maps MHA to row-wise
 *          or block-wise kernels with their own storage formats.
 *   [FMT]  gist.science technical summary, Methodology 1 "Unified MHA
 *          module", two-level storage format: a BSR of outer tiles (OT);
 *          empty OTs are skipped; "full" OTs (every element valid) and
 *          "partial" OTs (valid and invalid mixed) are tracked by pointer
 *          arrays; inside a partial OT each 8x8 inner tile (IT) is one
 *          64-bit bitmap, giving exact masking without materialising the
 *          sparse matrix.
 *   [PROB] same page, Problem statement: masks (causal, sliding window,
 *          random, BigBird) make attention skip work; resetting the score
 *          matrix after the fact is the inefficient alternative.
 *
 * Readings where the pages are silent (each is a convention of this
 * library, not of the pages):
 *   - a mask byte is valid iff it is non-zero;
 *   - the pointer arrays are two CSRs (full, partial) over OT rows, rows
 *     numbered mask-major then OT row, offsets global across masks, column
 *     indices ascending;
 *   - inside an IT, bit (8*r + c) is element (r, c) (row-major, bit 0 =
 *     top-left); the ITs of a partial OT are stored row-major; bitmaps are
 *     stored only for partial OTs, in the order of the partial list;
 *   - a query row with no valid key has output 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Masked softmax attention, fp64 ([ABS], [FMT] "exact masking", [PROB]).    */
/*                                                                          */
/* For query row i with valid key set V_i = { j : mask[i][j] != 0 }:        */
/*   s_ij = scale * sum_t q[i][t] * k[j][t]                                 */
/*   M_i  = max_{j in V_i} s_ij                                             */
/*   o[i] = sum_{j in V_i} exp(s_ij - M_i) v[j] / sum_{j in V_i} exp(s_ij - M_i) */
/*   o[i] = 0 when V_i is empty.                                            */
/* Masked keys are skipped, exactly as if their weight were zero.           */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t row_begin, row_end, lk;
    int d;
    double scale;
    const double *q, *k, *v;
    const uint8_t *mask;
    double *o;
} attn_job;

static void attention_rows(const attn_job *jb)
{
    const int d = jb->d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->lk > 0 ? jb->lk : 1));
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i) {
        const double *qi = jb->q + i * d;
        const uint8_t *mi = jb->mask + i * jb->lk;
        double *oi = jb->o + i * d;
        int any = 0;
        double mx = -INFINITY;
        /* pass 1: scores of the valid keys and their maximum */
        for (int64_t j = 0; j < jb->lk; ++j) {
            if (!mi[j]) continue;
            const double *kj = jb->k + j * d;
            double dot = 0.0;
            for (int t = 0; t < d; ++t) dot += qi[t] * kj[t];
            s[j] = jb->scale * dot;
            if (!any || s[j] > mx) mx = s[j];
            any = 1;
        }
        for (int t = 0; t < d; ++t) oi[t] = 0.0;
        if (!any) continue; /* fully masked row: output 0 */
        /* pass 2: weights exp(s - max), their sum, and the weighted sum of v */
        double den = 0.0;
        for (int64_t j = 0; j < jb->lk; ++j) {
            if (!mi[j]) continue;
            const double w = exp(s[j] - mx);
            const double *vj = jb->v + j * d;
            den += w;
            for (int t = 0; t < d; ++t) oi[t] += w * vj[t];
        }
        for (int t = 0; t < d; ++t) oi[t] /= den;
    }
    free(s);
}

static void *attention_thread(void *arg)
{
    attention_rows((const attn_job *)arg);
    return NULL;
}

/* q: [n_q][d] query rows; k, v: [lk][d] keys and values of the same head;
 * mask: [n_q][lk] the mask rows of those queries; o: [n_q][d] output.
 * Rows are split over n_threads threads (<= 0: one thread). */
int stof_oracle_attention(int64_t n_q, int64_t lk, int d, double scale,
                          const double *q, const double *k, const double *v,
                          const uint8_t *mask, double *o, int n_threads)
{
    if (n_q < 0 || lk < 0 || d <= 0) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > n_q) n_threads = (int)(n_q > 0 ? n_q : 1);
    attn_job jobs[256];
    pthread_t tid[256];
    int64_t per = (n_q + n_threads - 1) / n_threads;
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].row_begin = t * per < n_q ? t * per : n_q;
        jobs[t].row_end = (t + 1) * per < n_q ? (t + 1) * per : n_q;
        jobs[t].lk = lk;
        jobs[t].d = d;
        jobs[t].scale = scale;
        jobs[t].q = q;
        jobs[t].k = k;
        jobs[t].v = v;
        jobs[t].mask = mask;
        jobs[t].o = o;
    }
    if (n_threads == 1) {
        attention_rows(&jobs[0]);
        return 0;
    }
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&tid[t], NULL, attention_thread, &jobs[t]) != 0) break;
        ++started;
    }
    for (int t = started; t < n_threads; ++t) attention_rows(&jobs[t]);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Brute-force encoder into the two-level format ([FMT]).                   */
/* ------------------------------------------------------------------------ */

static int64_t ot_ones(const uint8_t *m, int64_t lk, int64_t r0, int64_t c0, int bm, int bn)
{
    int64_t ones = 0;
    for (int r = 0; r < bm; ++r)
        for (int c = 0; c < bn; ++c)
            ones += m[(r0 + r) * lk + (c0 + c)] != 0;
    return ones;
}

static int bad_shape(int n_masks, int lq, int lk, int bm, int bn)
{
    return n_masks < 1 || lq < 1 || lk < 1 || bm < 8 || bn < 8 || bm % 8 || bn % 8 ||
           lq % bm || lk % bn;
}

/* counts[0] = number of full OTs, counts[1] = number of partial OTs,
 * counts[2] = number of valid mask elements. */
int stof_oracle_encode_count(const uint8_t *mask, int n_masks, int lq, int lk, int bm, int bn,
                             int64_t *counts)
{
    if (bad_shape(n_masks, lq, lk, bm, bn)) return -1;
    int64_t n_full = 0, n_part = 0, nnz = 0;
    for (int m = 0; m < n_masks; ++m) {
        const uint8_t *mm = mask + (int64_t)m * lq * lk;
        for (int I = 0; I < lq / bm; ++I)
            for (int J = 0; J < lk / bn; ++J) {
                int64_t ones = ot_ones(mm, lk, (int64_t)I * bm, (int64_t)J * bn, bm, bn);
                nnz += ones;
                if (ones == (int64_t)bm * bn) ++n_full;
                else if (ones > 0) ++n_part;
            }
    }
    counts[0] = n_full;
    counts[1] = n_part;
    counts[2] = nnz;
    return 0;
}

/* Fills the format.  Array sizes: row pointers n_masks*(lq/bm)+1 each;
 * full_col_idx n_full; part_col_idx n_part; bitmaps n_part*(bm/8)*(bn/8). */
int stof_oracle_encode(const uint8_t *mask, int n_masks, int lq, int lk, int bm, int bn,
                       int32_t *full_row_ptr, int32_t *full_col_idx,
                       int32_t *part_row_ptr, int32_t *part_col_idx, uint64_t *bitmaps)
{
    if (bad_shape(n_masks, lq, lk, bm, bn)) return -1;
    const int n_tr = lq / bm, n_tc = lk / bn, itr = bm / 8, itc = bn / 8;
    int64_t nf = 0, np = 0;
    for (int m = 0; m < n_masks; ++m) {
        const uint8_t *mm = mask + (int64_t)m * lq * lk;
        for (int I = 0; I < n_tr; ++I) {
            const int64_t row = (int64_t)m * n_tr + I;
            full_row_ptr[row] = (int32_t)nf;
            part_row_ptr[row] = (int32_t)np;
            for (int J = 0; J < n_tc; ++J) { /* ascending column order */
                const int64_t r0 = (int64_t)I * bm, c0 = (int64_t)J * bn;
                int64_t ones = ot_ones(mm, lk, r0, c0, bm, bn);
                if (ones == 0) continue;                      /* empty: skipped */
                if (ones == (int64_t)bm * bn) {               /* full */
                    full_col_idx[nf++] = J;
                    continue;
                }
                part_col_idx[np] = J;                         /* partial */
                uint64_t *words = bitmaps + np * (int64_t)itr * itc;
                for (int p = 0; p < itr; ++p)
                    for (int qq = 0; qq < itc; ++qq) {
                        uint64_t w = 0;
                        for (int r = 0; r < 8; ++r)
                            for (int c = 0; c < 8; ++c)
                                if (mm[(r0 + 8 * p + r) * lk + (c0 + 8 * qq + c)])
                                    w |= (uint64_t)1 << (8 * r + c);
                        words[p * itc + qq] = w;
                    }
                ++np;
            }
        }
    }
    full_row_ptr[(int64_t)n_masks * n_tr] = (int32_t)nf;
    part_row_ptr[(int64_t)n_masks * n_tr] = (int32_t)np;
    return 0;
}

/* Rebuilds the dense 0/1 mask [n_masks][lq][lk] from the format: unlisted
 * OTs are 0, full OTs are 1, partial OTs take their IT bits. */
int stof_oracle_decode(int n_masks, int lq, int lk, int bm, int bn,
                       const int32_t *full_row_ptr, const int32_t *full_col_idx,
                       const int32_t *part_row_ptr, const int32_t *part_col_idx,
                       const uint64_t *bitmaps, uint8_t *mask_out)
{
    if (bad_shape(n_masks, lq, lk, bm, bn)) return -1;
    const int n_tr = lq / bm, itr = bm / 8, itc = bn / 8;
    memset(mask_out, 0, (size_t)n_masks * lq * lk);
    for (int m = 0; m < n_masks; ++m) {
        uint8_t *mm = mask_out + (int64_t)m * lq * lk;
        for (int I = 0; I < n_tr; ++I) {
            const int64_t row = (int64_t)m * n_tr + I;
            for (int32_t e = full_row_ptr[row]; e < full_row_ptr[row + 1]; ++e) {
                const int64_t c0 = (int64_t)full_col_idx[e] * bn;
                for (int r = 0; r < bm; ++r)
                    for (int c = 0; c < bn; ++c)
                        mm[((int64_t)I * bm + r) * lk + c0 + c] = 1;
            }
            for (int32_t e = part_row_ptr[row]; e < part_row_ptr[row + 1]; ++e) {
                const int64_t c0 = (int64_t)part_col_idx[e] * bn;
                const uint64_t *words = bitmaps + (int64_t)e * itr * itc;
                for (int p = 0; p < itr; ++p)
                    for (int qq = 0; qq < itc; ++qq)
                        for (int r = 0; r < 8; ++r)
                            for (int c = 0; c < 8; ++c)
                                if ((words[p * itc + qq] >> (8 * r + c)) & 1)
                                    mm[((int64_t)I * bm + 8 * p + r) * lk + c0 + 8 * qq + c] = 1;
            }
        }
    }
    return 0;
}
