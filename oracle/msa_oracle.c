/*
 * msa_oracle.c -- plain fp64 CPU oracle of the MiniMax Sparse Attention (MSA)
 * layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares no
 * code, header, table or helper with the CUDA path, and the CUDA path never
 * calls it.
 *
 * Every bf16 input is widened exactly to double; all arithmetic is double with
 * no blocking, fusion or reordering beyond the definitions below.  OpenMP only
 * splits independent rows across threads.
 *
 * What it computes (MSA, two stages).  Sources, by page title and passage:
 *   [serving]  "MiniMax M3 preparado para inferencia en produccion" (community
 *              post on the M3 serving report): paragraphs "KV-Block-Major",
 *              "MSA con paged attention" and "MSA opera en dos etapas".
 *   [M2]       article on the MiniMax M2 report, section "MiniMax Sparse
 *              Attention (MSA) y escalado subcuadratico entrante".
 *   [agents]   "MiniMax M3: Como la atencion dispersa hace practicos a los
 *              agentes de largo alcance": the MSA paragraph, the figure caption
 *              under it and the bullet "Costo predecible a cualquier longitud".
 *
 *   1. index score.  A light Index Branch scores the context in blocks
 *      ([agents], MSA paragraph and caption).  The pages never print the
 *      formula; the library and this oracle both take:
 *          s_t = sum_h w_h * ReLU(q_idx_h . k_idx_t)
 *          c_j = max over the tokens t of block j of s_t
 *      Only blocks strictly before the query's own block are scored; the own
 *      block and later blocks get -inf (the own block is forced in step 2).
 *   2. selection.  Per query and KV group keep the own block plus the k-1 best
 *      earlier blocks ordered by (score desc, block index asc); with at most
 *      k-1 earlier blocks keep them all.  Bk = 128 and k = 16 give 2048 tokens
 *      per query and GQA group ([agents], "Costo predecible").
 *   3. attention.  Exact softmax attention of each query head against the
 *      tokens of the selected blocks of its GQA group, causally clipped
 *      (t <= i in prefill, t < L in decode), on uncompressed keys and values
 *      ([M2]; [serving], "MSA opera en dos etapas").
 *   4. log-sum-exp merge of partial results over blocks ([serving],
 *      "KV-Block-Major").
 *   5. decode page table built from the selected blocks, with the KV-group
 *      dimension flattened into the batch ([serving], "MSA con paged
 *      attention").
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* exact bf16 -> double widening */
static double bf16(uint16_t h)
{
    union { uint32_t u; float f; } c;
    c.u = ((uint32_t)h) << 16;
    return (double)c.f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* s_t for one token: sum_h w[h] * max(0, sum_e q[h][e] * k[e]) */
static double token_score(int HI, int dI, const double *q, const float *w, const uint16_t *k)
{
    double s = 0.0;
    for (int h = 0; h < HI; ++h) {
        double dot = 0.0;
        for (int e = 0; e < dI; ++e) dot += q[h * dI + e] * bf16(k[e]);
        double r = dot > 0.0 ? dot : 0.0;
        s += (double)w[h] * r;
    }
    return s;
}

/*
 * Prefill block scores for a list of query rows.
 *   qidx [B,S,Hkv,HI,dI] bf16, kidx [B,S,Hkv,dI] bf16, w [B,S,Hkv,HI] fp32.
 *   rows[r] = b*S + i.   C [nrows, Hkv, nb_stride]: c_j for j < b_i, else -inf.
 */
void orc_prefill_scores(int B, int S, int Hkv, int HI, int dI, int Bk,
                        const uint16_t *qidx, const uint16_t *kidx, const float *w,
                        int64_t nrows, const int64_t *rows, int nb_stride, double *C)
{
    (void)B;
    int64_t total = nrows * (int64_t)Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rg = 0; rg < total; ++rg) {
        int64_t r = rg / Hkv;
        int g = (int)(rg % Hkv);
        int64_t bi = rows[r];
        int64_t b = bi / S, i = bi % S;
        int own = (int)(i / Bk);
        double *c = C + rg * nb_stride;
        double *q = (double *)malloc(sizeof(double) * HI * dI);
        const uint16_t *qr = qidx + ((bi * Hkv + g) * HI) * (int64_t)dI;
        for (int e = 0; e < HI * dI; ++e) q[e] = bf16(qr[e]);
        const float *wr = w + (bi * Hkv + g) * (int64_t)HI;
        for (int j = 0; j < nb_stride; ++j) c[j] = -INFINITY;
        for (int j = 0; j < own; ++j) {
            double m = -INFINITY;
            for (int t = j * Bk; t < (j + 1) * Bk; ++t) {
                const uint16_t *kr = kidx + (((b * S) + t) * Hkv + g) * (int64_t)dI;
                double s = token_score(HI, dI, q, wr, kr);
                if (s > m) m = s;
            }
            c[j] = m;
        }
        free(q);
    }
}

/*
 * Decode block scores over paged index keys.
 *   qidx [B,Hkv,HI,dI] bf16, w [B,Hkv,HI] fp32,
 *   kidx_pool [P,Hkv,Bk,dI] bf16, seq_pt [B,max_pages] int32, seq_len [B] int32.
 *   The query sits at position L-1; its own block is (L-1)/Bk.
 *   C [B,Hkv,nb_stride]: c_j for j < own, else -inf.
 */
void orc_decode_scores(int B, int Hkv, int HI, int dI, int Bk,
                       const uint16_t *qidx, const float *w, const uint16_t *kidx_pool,
                       const int32_t *seq_pt, int max_pages, const int32_t *seq_len,
                       int nb_stride, double *C)
{
    int64_t total = (int64_t)B * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bg = 0; bg < total; ++bg) {
        int b = (int)(bg / Hkv), g = (int)(bg % Hkv);
        int own = (seq_len[b] - 1) / Bk;
        double *c = C + bg * nb_stride;
        double *q = (double *)malloc(sizeof(double) * HI * dI);
        const uint16_t *qr = qidx + bg * (int64_t)HI * dI;
        for (int e = 0; e < HI * dI; ++e) q[e] = bf16(qr[e]);
        const float *wr = w + bg * (int64_t)HI;
        for (int j = 0; j < nb_stride; ++j) c[j] = -INFINITY;
        for (int j = 0; j < own && j < max_pages; ++j) {
            int64_t p = seq_pt[(int64_t)b * max_pages + j];
            double m = -INFINITY;
            for (int t = 0; t < Bk; ++t) {
                const uint16_t *kr = kidx_pool + ((p * Hkv + g) * Bk + t) * (int64_t)dI;
                double s = token_score(HI, dI, q, wr, kr);
                if (s > m) m = s;
            }
            c[j] = m;
        }
        free(q);
    }
}

/* ordering of candidate blocks: score descending, then block index ascending */
typedef struct { double c; int32_t j; } cand_t;

static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->c > b->c) return -1;
    if (a->c < b->c) return 1;
    return (a->j < b->j) ? -1 : (a->j > b->j);
}

static int int_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * Block selection for rows of block scores.
 *   C [nrows, nb_stride]; own[r] is the row's own block (candidates j < own[r]).
 *   sel [nrows, k] ascending, padded with -1; count [nrows].
 *   c_last[r] / c_next[r]: scores of the (k-1)-th kept and the first dropped
 *   earlier block in (score desc, index asc) order; NaN when nothing is dropped.
 */
void orc_select(int64_t nrows, int nb_stride, const double *C, const int32_t *own, int k,
                int32_t *sel, int32_t *count, double *c_last, double *c_next)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t r = 0; r < nrows; ++r) {
        int n = own[r];
        int32_t *s = sel + r * k;
        for (int x = 0; x < k; ++x) s[x] = -1;
        c_last[r] = NAN;
        c_next[r] = NAN;
        if (n <= k - 1) {
            for (int j = 0; j < n; ++j) s[j] = j;
            s[n] = n;
            count[r] = n + 1;
            continue;
        }
        cand_t *cs = (cand_t *)malloc(sizeof(cand_t) * n);
        for (int j = 0; j < n; ++j) { cs[j].c = C[r * nb_stride + j]; cs[j].j = j; }
        qsort(cs, n, sizeof(cand_t), cand_cmp);
        for (int x = 0; x < k - 1; ++x) s[x] = cs[x].j;
        qsort(s, k - 1, sizeof(int32_t), int_cmp);
        s[k - 1] = n;
        count[r] = k;
        c_last[r] = (k >= 2) ? cs[k - 2].c : NAN;
        c_next[r] = cs[k - 1].c;
        free(cs);
    }
}

/*
 * Softmax attention of one query vector over an explicit key list.
 *   z_t = scale * q . K_t,   O = sum_t softmax(z)_t V_t,   LSE = ln sum_t e^{z_t}.
 */
static void attend_keys(int D, double scale, const double *q, int nk,
                        const uint16_t **kr, const uint16_t **vr, double *z,
                        double *O, double *LSE)
{
    for (int d = 0; d < D; ++d) O[d] = 0.0;
    if (nk == 0) { *LSE = -INFINITY; return; }
    double m = -INFINITY;
    for (int t = 0; t < nk; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * bf16(kr[t][d]);
        z[t] = scale * dot;
        if (z[t] > m) m = z[t];
    }
    double l = 0.0;
    for (int t = 0; t < nk; ++t) {
        double p = exp(z[t] - m);
        l += p;
        for (int d = 0; d < D; ++d) O[d] += p * bf16(vr[t][d]);
    }
    for (int d = 0; d < D; ++d) O[d] /= l;
    *LSE = m + log(l);
}

/*
 * Prefill sparse attention for a list of query rows with a given selection.
 *   Q [B,S,Hq,D], K, V [B,S,Hkv,D] bf16.  rows[r] = b*S + i.
 *   sel [nrows,Hkv,k] (ascending, -1 padded), count [nrows,Hkv].
 *   Keys of head hq (group g = hq / (Hq/Hkv)): tokens t of the selected blocks
 *   of (row, g) with t <= i and t < S.
 *   O [nrows,Hq,D], LSE [nrows,Hq].
 */
void orc_prefill_attend(int B, int S, int Hq, int Hkv, int D, int Bk, double scale,
                        const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                        int64_t nrows, const int64_t *rows, int k,
                        const int32_t *sel, const int32_t *count, double *O, double *LSE)
{
    (void)B;
    int G = Hq / Hkv;
    int64_t total = nrows * (int64_t)Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < total; ++rh) {
        int64_t r = rh / Hq;
        int hq = (int)(rh % Hq), g = hq / G;
        int64_t bi = rows[r], b = bi / S, i = bi % S;
        int cnt = count[r * Hkv + g];
        const int32_t *s = sel + (r * Hkv + g) * (int64_t)k;
        int maxk = cnt * Bk;
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (maxk + 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (maxk + 1));
        double *z = (double *)malloc(sizeof(double) * (maxk + 1));
        double *q = (double *)malloc(sizeof(double) * D);
        int nk = 0;
        for (int x = 0; x < cnt; ++x) {
            int j = s[x];
            for (int t = j * Bk; t < (j + 1) * Bk; ++t) {
                if (t > i || t >= S) break;
                kr[nk] = K + ((b * S + t) * Hkv + g) * (int64_t)D;
                vr[nk] = V + ((b * S + t) * Hkv + g) * (int64_t)D;
                ++nk;
            }
        }
        const uint16_t *qr = Q + (bi * Hq + hq) * (int64_t)D;
        for (int d = 0; d < D; ++d) q[d] = bf16(qr[d]);
        attend_keys(D, scale, q, nk, kr, vr, z, O + rh * D, LSE + rh);
        free(kr); free(vr); free(z); free(q);
    }
}

/*
 * Decode sparse attention over paged K/V with a given per-(b, g) selection.
 *   Q [B,Hq,D]; K_pool, V_pool [P,Hkv,Bk,D] bf16; seq_pt [B,max_pages];
 *   seq_len [B]; sel [B,Hkv,k], count [B,Hkv].  Keys: tokens t < L_b of the
 *   selected blocks.  O [B,Hq,D], LSE [B,Hq].
 */
void orc_decode_attend(int B, int Hq, int Hkv, int D, int Bk, double scale,
                       const uint16_t *Q, const uint16_t *K_pool, const uint16_t *V_pool,
                       const int32_t *seq_pt, int max_pages, const int32_t *seq_len,
                       int k, const int32_t *sel, const int32_t *count,
                       double *O, double *LSE)
{
    int G = Hq / Hkv;
    int64_t total = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < total; ++bh) {
        int b = (int)(bh / Hq), hq = (int)(bh % Hq), g = hq / G;
        int L = seq_len[b];
        int cnt = count[b * Hkv + g];
        const int32_t *s = sel + ((int64_t)b * Hkv + g) * k;
        int maxk = cnt * Bk;
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (maxk + 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (maxk + 1));
        double *z = (double *)malloc(sizeof(double) * (maxk + 1));
        double *q = (double *)malloc(sizeof(double) * D);
        int nk = 0;
        for (int x = 0; x < cnt; ++x) {
            int j = s[x];
            int64_t p = seq_pt[(int64_t)b * max_pages + j];
            for (int t = 0; t < Bk; ++t) {
                if (j * Bk + t >= L) break;
                kr[nk] = K_pool + ((p * Hkv + g) * Bk + t) * (int64_t)D;
                vr[nk] = V_pool + ((p * Hkv + g) * Bk + t) * (int64_t)D;
                ++nk;
            }
        }
        const uint16_t *qr = Q + bh * (int64_t)D;
        for (int d = 0; d < D; ++d) q[d] = bf16(qr[d]);
        attend_keys(D, scale, q, nk, kr, vr, z, O + bh * D, LSE + bh);
        free(kr); free(vr); free(z); free(q);
    }
}

/*
 * Log-sum-exp merge of partial softmax results.
 *   Op [rows,parts,D], LSEp [rows,parts] (-inf marks an empty part).
 *   LSE = ln sum_p e^{LSEp},  O = sum_p e^{LSEp - LSE} Op.
 *   A row with no non-empty part gets O = 0, LSE = -inf.
 */
void orc_lse_merge(int64_t rows, int parts, int D, const double *Op, const double *LSEp,
                   double *O, double *LSE)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double *l = LSEp + r * parts;
        double m = -INFINITY;
        for (int p = 0; p < parts; ++p) if (l[p] > m) m = l[p];
        double *o = O + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (m == -INFINITY) { LSE[r] = -INFINITY; continue; }
        double sum = 0.0;
        for (int p = 0; p < parts; ++p) if (l[p] != -INFINITY) sum += exp(l[p] - m);
        double lse = m + log(sum);
        for (int p = 0; p < parts; ++p) {
            if (l[p] == -INFINITY) continue;
            double a = exp(l[p] - lse);
            const double *op = Op + (r * parts + p) * (int64_t)D;
            for (int d = 0; d < D; ++d) o[d] += a * op[d];
        }
        LSE[r] = lse;
    }
}

/*
 * Decode page table from the selected blocks, KV group flattened into batch.
 *   Row r = b*Hkv + g.  pt[r][s] = seq_pt[b][sel[b,g,s]] for s < count, else -1;
 *   n[r] = count[b,g]; last_len[r] = number of valid tokens in the row's last
 *   selected page (the own block, the largest selected index): L_b - Bk*own.
 */
void orc_page_table(int B, int Hkv, int k, int Bk, const int32_t *sel, const int32_t *count,
                    const int32_t *seq_pt, int max_pages, const int32_t *seq_len,
                    int32_t *pt, int32_t *n, int32_t *last_len)
{
    for (int64_t r = 0; r < (int64_t)B * Hkv; ++r) {
        int b = (int)(r / Hkv);
        int cnt = count[r];
        for (int s = 0; s < k; ++s)
            pt[r * k + s] = (s < cnt) ? seq_pt[(int64_t)b * max_pages + sel[r * k + s]] : -1;
        n[r] = cnt;
        int own = (seq_len[b] - 1) / Bk;
        last_len[r] = seq_len[b] - Bk * own;
    }
}
