/*
 * gca_oracle.c -- plain fp64 CPU oracle for Grouped Cross Attention (GCA).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the GCA hot path computes.  It exists so that the CUDA
 * library can be checked against it.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark may load it; the product path
 * (the CUDA library and its Python binding) never does, and the two share no
 * code, headers or constants.
 *
 * Source: "Efficient Length-Generalizable Attention via Causal Retrieval for
 * Long-Context Language Modeling" (Hu, Teng, Zhao, Wu, Tu; ICML 2025,
 * arXiv 2410.01651), as available in these web pages:
 *   [P1] paperlayer.ai summary, sections 1, 3, 3.1, 3.2, 4.3 and App. B;
 *   [P2] PaperHub/OpenReview rebuttal to reviewer 1, comment "Cmt 1"
 *        (the G=1 special case of Eq. 1: r_t^k = l_t^T l_k / sqrt(d)),
 *        answer to W2 (Eq. 2 is the batch form of Figure 2) and to Q4
 *        (Eq. 3 is the "softmax off by one");
 *   [P5] the official repository README, "Model Architecture" (two-stage
 *        attention: per-retrieved-chunk attention, then a weighted sum with
 *        the softmax-normalised retrieval scores) and the
 *        `enable_softmax_one` switch.
 *
 * Readings taken where the pages are silent (each is a parameter or is
 * stated here):
 *   - query chunk c is served by the landmark of chunk c-1; its candidates
 *     are chunks kappa < c-1 (strict) or kappa <= c-1 (include_self);
 *   - one score per (batch, query chunk, slot), shared by all heads;
 *   - top-k order: score descending, then chunk index ascending; fewer
 *     than k candidates leaves idx = -1, weight 0 in the remaining slots;
 *   - off-by-one softmax: w_j = e^{r_j} / (1 + sum_i e^{r_i});
 *   - inside a retrieved chunk there is no mask; attention scale is a
 *     parameter (1/sqrt(head dim) by default);
 *   - the log-sum-exp of an empty slot is -infinity.
 *
 * Everything is computed in double precision with straightforward loops.
 * The scores of integer landmarks are exact in fp64, so the top-k indices
 * are exact.  OpenMP, if enabled, only splits independent outer loops.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Softmax over the selected relevance scores (Figure 2 / Eq. 2 weights,   */
/* Eq. 3 "softmax off by one" per the rebuttal answer to Q4).             */
/* r[0..m-1] are the valid scores; writes w[0..m-1].                       */
/* ---------------------------------------------------------------------- */
void oracle_weights_from_scores(int m, const double* r, int off_by_one, double* w)
{
    if (m <= 0) return;
    double mx = r[0];
    for (int i = 1; i < m; ++i) if (r[i] > mx) mx = r[i];
    /* off-by-one: an implicit extra logit 0 joins the denominator. */
    if (off_by_one && mx < 0.0) mx = 0.0;
    double den = off_by_one ? exp(0.0 - mx) : 0.0;
    for (int i = 0; i < m; ++i) den += exp(r[i] - mx);
    for (int i = 0; i < m; ++i) w[i] = exp(r[i] - mx) / den;
}

typedef struct { double s; int kappa; } cand_t;

/* order: score descending, chunk index ascending */
static int cand_cmp(const void* a, const void* b)
{
    const cand_t* x = (const cand_t*)a;
    const cand_t* y = (const cand_t*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->kappa > y->kappa) - (x->kappa < y->kappa);
}

/* Select the top-k of n scored candidates and fill one (idx, score, weight) row. */
static void select_row(cand_t* cand, int n, int topk, int off_by_one, double score_scale,
                       int32_t* idx, double* score, double* weight)
{
    qsort(cand, (size_t)n, sizeof(cand_t), cand_cmp);
    int m = n < topk ? n : topk;
    double r[64];
    for (int j = 0; j < m; ++j) r[j] = cand[j].s * score_scale;
    for (int j = 0; j < topk; ++j) { idx[j] = -1; score[j] = 0.0; weight[j] = 0.0; }
    for (int j = 0; j < m; ++j) { idx[j] = cand[j].kappa; score[j] = r[j]; }
    oracle_weights_from_scores(m, r, off_by_one, weight);
}

/* ---------------------------------------------------------------------- */
/* Causal relevance scoring + top-k + softmax ([P2] Cmt 1, [P1] 3.1/3.2,  */
/* [P5] Model Architecture).                                              */
/*   lm     [B, nC, D]  landmark representations                          */
/*   idx    [B, nC, topk]  retrieved chunk per slot, -1 = empty            */
/*   score  [B, nC, topk]  r = score_scale * l_{c-1}^T l_kappa             */
/*   weight [B, nC, topk]  softmax (or off-by-one) of the valid r          */
/* Returns 0, or -1 if topk is outside [1, 64].                           */
/* ---------------------------------------------------------------------- */
int oracle_score_topk(int B, int nC, int D, int topk, int include_self, int off_by_one,
                      double score_scale, const double* lm, int32_t* idx, double* score,
                      double* weight)
{
    if (topk < 1 || topk > 64) return -1;
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < nC; ++c) {
            int32_t* ir = idx + ((size_t)b * nC + c) * topk;
            double* sr = score + ((size_t)b * nC + c) * topk;
            double* wr = weight + ((size_t)b * nC + c) * topk;
            int t = c - 1;                         /* landmark chunk */
            int n = (t < 0) ? 0 : (include_self ? t + 1 : t);
            cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
            const double* lt = lm + ((size_t)b * nC + (t < 0 ? 0 : t)) * D;
            for (int kappa = 0; kappa < n; ++kappa) {
                const double* lk = lm + ((size_t)b * nC + kappa) * D;
                double s = 0.0;
                for (int e = 0; e < D; ++e) s += lt[e] * lk[e];
                cand[kappa].s = s;
                cand[kappa].kappa = kappa;
            }
            select_row(cand, n, topk, off_by_one, score_scale, ir, sr, wr);
            free(cand);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Decode-time retrieval ([P1] 3.2 and 4.3: retrieval runs once per chunk  */
/* of generated tokens, against every stored landmark).                   */
/*   lm [N, D], ql [D]  ->  idx/score/weight [topk]                        */
/* ---------------------------------------------------------------------- */
int oracle_decode_retrieve(int N, int D, int topk, int off_by_one, double score_scale,
                           const double* lm, const double* ql, int32_t* idx, double* score,
                           double* weight)
{
    if (topk < 1 || topk > 64) return -1;
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(N > 0 ? N : 1));
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        double s = 0.0;
        for (int e = 0; e < D; ++e) s += ql[e] * lm[(size_t)n * D + e];
        cand[n].s = s;
        cand[n].kappa = n;
    }
    select_row(cand, N, topk, off_by_one, score_scale, idx, score, weight);
    free(cand);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Per-slot attention of one query token against one retrieved chunk     */
/* (stage 1, [P5] "first stage"; Figure 1/2 chunk-wise cross attention).  */
/* Writes o_j[d] = sum_s p_s v_s and returns lse = ln sum_s exp(a_s).      */
/* ---------------------------------------------------------------------- */
static double attend_one(int S, int H, int d, double attn_scale, const double* qt,
                         const double* kchunk, const double* vchunk, int h, double* a,
                         double* o_j)
{
    double mx = -INFINITY;
    for (int s = 0; s < S; ++s) {
        const double* ks = kchunk + ((size_t)s * H + h) * d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += qt[e] * ks[e];
        a[s] = attn_scale * dot;
        if (a[s] > mx) mx = a[s];
    }
    double l = 0.0;
    for (int s = 0; s < S; ++s) l += exp(a[s] - mx);
    for (int e = 0; e < d; ++e) o_j[e] = 0.0;
    for (int s = 0; s < S; ++s) {
        double p = exp(a[s] - mx) / l;
        const double* vs = vchunk + ((size_t)s * H + h) * d;
        for (int e = 0; e < d; ++e) o_j[e] += p * vs[e];
    }
    return mx + log(l);
}

/* ---------------------------------------------------------------------- */
/* GCA forward: stage 1 + stage 2 ([P5] Model Architecture; [P2] W2: Eq. 2 */
/* is the batch form of Figure 2; [P1] App. B: returns O and the LSE).     */
/*   q    [B, Lq, H, d]            (Lq = nQ * S query tokens)              */
/*   k, v [B, nP * S, H, d]        (pool of nP chunks)                     */
/*   idx, w [B, nQ, topk]          query chunk c uses row c                */
/*   o    [B, Lq, H, d]            O_t = sum_j w_j O_t^j (0 if no slot)    */
/*   lse  [B, Lq, H, topk] or NULL (-inf for an empty slot)               */
/*   qmask [B, nQ] or NULL: only chunks with qmask != 0 are computed.      */
/* ---------------------------------------------------------------------- */
void oracle_fwd(int B, int nQ, int nP, int S, int H, int d, int topk, double attn_scale,
                const double* q, const double* k, const double* v, const int32_t* idx,
                const double* w, double* o, double* lse, const uint8_t* qmask)
{
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < nQ; ++c) {
            if (qmask && !qmask[(size_t)b * nQ + c]) continue;
            double* a = (double*)malloc(sizeof(double) * (size_t)S);
            double* oj = (double*)malloc(sizeof(double) * (size_t)d);
            const int32_t* ir = idx + ((size_t)b * nQ + c) * topk;
            const double* wr = w + ((size_t)b * nQ + c) * topk;
            for (int t = 0; t < S; ++t) {
                size_t tok = (size_t)b * nQ * S + (size_t)c * S + t;
                for (int h = 0; h < H; ++h) {
                    const double* qt = q + (tok * H + h) * d;
                    double* ot = o + (tok * H + h) * d;
                    for (int e = 0; e < d; ++e) ot[e] = 0.0;
                    for (int j = 0; j < topk; ++j) {
                        double* lsep = lse ? lse + (tok * H + h) * topk + j : NULL;
                        int kappa = ir[j];
                        if (kappa < 0) { if (lsep) *lsep = -INFINITY; continue; }
                        size_t row0 = (size_t)b * nP * S + (size_t)kappa * S;
                        double l = attend_one(S, H, d, attn_scale, qt, k + row0 * H * d,
                                              v + row0 * H * d, h, a, oj);
                        if (lsep) *lsep = l;
                        for (int e = 0; e < d; ++e) ot[e] += wr[j] * oj[e];
                    }
                }
            }
            free(a);
            free(oj);
        }
    }
}

/* ---------------------------------------------------------------------- */
/* GCA backward ([P1] App. B backward: gradients for Q, K, V and the       */
/* weights; [P1] section 3 and [P5]: the relevance scores receive          */
/* gradients through the weights).  Direct chain rule with every per-slot  */
/* output O_t^j materialised, no recomputation tricks:                     */
/*   dO_t^j = w_j dO_t,   dw_j = sum_{t in c, h} dO_t . O_t^j              */
/*   dV_s  += p_ts w_j dO_t                                                */
/*   dp_ts  = w_j dO_t . v_s,  da_ts = p_ts (dp_ts - w_j dO_t . O_t^j)     */
/*   dq_t  += attn_scale sum_s da_ts k_s,  dk_s += attn_scale da_ts q_t     */
/*   dr_j   = sum_i dw_i (dw_i/dr_j) = w_j (dw_j - sum_i w_i dw_i)          */
/*            (identical for the vanilla and the off-by-one softmax).      */
/* Inputs as oracle_fwd plus dout [B, Lq, H, d].  Outputs dq [B,Lq,H,d],    */
/* dk, dv [B, nP*S, H, d] (fully overwritten), dscore [B, nQ, topk].        */
/* qmask [B,nQ] limits dq/dscore to selected query chunks; kmask [B,nP]     */
/* limits dk/dv to selected key chunks (unselected entries are left 0).    */
/* ---------------------------------------------------------------------- */
void oracle_bwd(int B, int nQ, int nP, int S, int H, int d, int topk, double attn_scale,
                const double* q, const double* k, const double* v, const int32_t* idx,
                const double* w, const double* dout, double* dq, double* dk, double* dv,
                double* dscore, const uint8_t* qmask, const uint8_t* kmask)
{
    size_t Lq = (size_t)nQ * S, Lp = (size_t)nP * S;
    memset(dq, 0, sizeof(double) * (size_t)B * Lq * H * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Lp * H * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Lp * H * d);
    memset(dscore, 0, sizeof(double) * (size_t)B * nQ * topk);

    /* Query side: dq and dscore for each selected query chunk. */
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < nQ; ++c) {
            if (qmask && !qmask[(size_t)b * nQ + c]) continue;
            const int32_t* ir = idx + ((size_t)b * nQ + c) * topk;
            const double* wr = w + ((size_t)b * nQ + c) * topk;
            double* a = (double*)malloc(sizeof(double) * (size_t)S);
            double* p = (double*)malloc(sizeof(double) * (size_t)S);
            double* dp = (double*)malloc(sizeof(double) * (size_t)S);
            double* oj = (double*)malloc(sizeof(double) * (size_t)d);
            double dwj[64];
            for (int j = 0; j < topk; ++j) dwj[j] = 0.0;
            for (int j = 0; j < topk; ++j) {
                int kappa = ir[j];
                if (kappa < 0) continue;
                size_t row0 = (size_t)b * Lp + (size_t)kappa * S;
                const double* kc = k + row0 * H * d;
                const double* vc = v + row0 * H * d;
                for (int t = 0; t < S; ++t) {
                    size_t tok = (size_t)b * Lq + (size_t)c * S + t;
                    for (int h = 0; h < H; ++h) {
                        const double* qt = q + (tok * H + h) * d;
                        const double* gt = dout + (tok * H + h) * d;
                        double lse = attend_one(S, H, d, attn_scale, qt, kc, vc, h, a, oj);
                        double delta = 0.0;             /* dO_t . O_t^j */
                        for (int e = 0; e < d; ++e) delta += gt[e] * oj[e];
                        dwj[j] += delta;
                        for (int s = 0; s < S; ++s) {
                            const double* vs = vc + ((size_t)s * H + h) * d;
                            double g = 0.0;
                            for (int e = 0; e < d; ++e) g += gt[e] * vs[e];
                            p[s] = exp(a[s] - lse);
                            dp[s] = wr[j] * g;
                        }
                        double* dqt = dq + (tok * H + h) * d;
                        for (int s = 0; s < S; ++s) {
                            double da = p[s] * (dp[s] - wr[j] * delta);
                            const double* ks = kc + ((size_t)s * H + h) * d;
                            for (int e = 0; e < d; ++e) dqt[e] += attn_scale * da * ks[e];
                        }
                    }
                }
            }
            double wdw = 0.0;
            for (int j = 0; j < topk; ++j) if (ir[j] >= 0) wdw += wr[j] * dwj[j];
            double* dsr = dscore + ((size_t)b * nQ + c) * topk;
            for (int j = 0; j < topk; ++j) dsr[j] = (ir[j] >= 0) ? wr[j] * (dwj[j] - wdw) : 0.0;
            free(a); free(p); free(dp); free(oj);
        }
    }

    /* Key side: dk and dv of each selected key chunk gather every (query
     * chunk, slot) that retrieved it, in ascending query-chunk order. */
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int kappa = 0; kappa < nP; ++kappa) {
            if (kmask && !kmask[(size_t)b * nP + kappa]) continue;
            size_t row0 = (size_t)b * Lp + (size_t)kappa * S;
            const double* kc = k + row0 * H * d;
            const double* vc = v + row0 * H * d;
            double* dkc = dk + row0 * H * d;
            double* dvc = dv + row0 * H * d;
            double* a = (double*)malloc(sizeof(double) * (size_t)S);
            double* p = (double*)malloc(sizeof(double) * (size_t)S);
            double* dp = (double*)malloc(sizeof(double) * (size_t)S);
            double* oj = (double*)malloc(sizeof(double) * (size_t)d);
            for (int c = 0; c < nQ; ++c) {
                const int32_t* ir = idx + ((size_t)b * nQ + c) * topk;
                const double* wr = w + ((size_t)b * nQ + c) * topk;
                for (int j = 0; j < topk; ++j) {
                    if (ir[j] != kappa) continue;
                    for (int t = 0; t < S; ++t) {
                        size_t tok = (size_t)b * Lq + (size_t)c * S + t;
                        for (int h = 0; h < H; ++h) {
                            const double* qt = q + (tok * H + h) * d;
                            const double* gt = dout + (tok * H + h) * d;
                            double lse = attend_one(S, H, d, attn_scale, qt, kc, vc, h, a, oj);
                            double delta = 0.0;         /* dO_t . O_t^j */
                            for (int e = 0; e < d; ++e) delta += gt[e] * oj[e];
                            for (int s = 0; s < S; ++s) {
                                const double* vs = vc + ((size_t)s * H + h) * d;
                                double g = 0.0;
                                for (int e = 0; e < d; ++e) g += gt[e] * vs[e];
                                p[s] = exp(a[s] - lse);
                                dp[s] = wr[j] * g;
                            }
                            for (int s = 0; s < S; ++s) {
                                double da = p[s] * (dp[s] - wr[j] * delta);
                                double* dks = dkc + ((size_t)s * H + h) * d;
                                double* dvs = dvc + ((size_t)s * H + h) * d;
                                for (int e = 0; e < d; ++e) {
                                    dks[e] += attn_scale * da * qt[e];
                                    dvs[e] += p[s] * wr[j] * gt[e];
                                }
                            }
                        }
                    }
                }
            }
            free(a); free(p); free(dp); free(oj);
        }
    }
}

/* Number of OpenMP threads the oracle will use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif

/* ---------------------------------------------------------------------- */
/* Landmark gradients ([P1] sections 1 and 3: the relevance scores take    */
/* part in next-token prediction, so the retriever that produces the       */
/* landmarks learns from the loss; [P2] Cmt 1: r = sigma * l_{c-1} . l_k). */
/* For every valid slot (b, c, j) with chunk kappa:                        */
/*   dl[b][c-1]   += sigma * dr[b][c][j] * l[b][kappa]                     */
/*   dl[b][kappa] += sigma * dr[b][c][j] * l[b][c-1]                       */
/*   lm, dl [B, nC, D]; idx, dr [B, nC, topk]; dl is overwritten.          */
/* ---------------------------------------------------------------------- */
void oracle_landmark_bwd(int B, int nC, int D, int topk, double score_scale, const double* lm,
                         const int32_t* idx, const double* dr, double* dl)
{
    memset(dl, 0, sizeof(double) * (size_t)B * nC * D);
    for (int b = 0; b < B; ++b) {
        for (int c = 1; c < nC; ++c) {
            const double* lt = lm + ((size_t)b * nC + (c - 1)) * D;
            double* dlt = dl + ((size_t)b * nC + (c - 1)) * D;
            for (int j = 0; j < topk; ++j) {
                int kappa = idx[((size_t)b * nC + c) * topk + j];
                if (kappa < 0 || kappa >= nC) continue;
                double g = score_scale * dr[((size_t)b * nC + c) * topk + j];
                const double* lk = lm + ((size_t)b * nC + kappa) * D;
                double* dlk = dl + ((size_t)b * nC + kappa) * D;
                for (int e = 0; e < D; ++e) {
                    dlt[e] += g * lk[e];
                    dlk[e] += g * lt[e];
                }
            }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Top-k under Gumbel noise ([P1] section 3.2: during training, noise is    */
/* added to the relevance scores before the top-k selection; the pages do  */
/* not say which scores the softmax then uses: here the clean ones).       */
/* The selection key is  fl32(fl32(fl32(s) * fl32(sigma)) + fl32(g))        */
/* evaluated in single precision exactly as written (no fused multiply-    */
/* add), so that the integer decision is taken in the same precision as on */
/* the GPU; ties go to the lower chunk index.  noise [B, nC, nC]: the noise */
/* for query chunk c and candidate kappa is noise[b][c][kappa].             */
/* ---------------------------------------------------------------------- */
typedef struct { float key; int kappa; double s; } ncand_t;

static int ncand_cmp(const void* a, const void* b)
{
    const ncand_t* x = (const ncand_t*)a;
    const ncand_t* y = (const ncand_t*)b;
    if (x->key > y->key) return -1;
    if (x->key < y->key) return 1;
    return (x->kappa > y->kappa) - (x->kappa < y->kappa);
}

int oracle_score_topk_noisy(int B, int nC, int D, int topk, int include_self, int off_by_one,
                            double score_scale, const double* lm, const float* noise,
                            int32_t* idx, double* score, double* weight)
{
    if (topk < 1 || topk > 64) return -1;
    volatile float sigma32 = (float)score_scale;
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < nC; ++c) {
            int32_t* ir = idx + ((size_t)b * nC + c) * topk;
            double* sr = score + ((size_t)b * nC + c) * topk;
            double* wr = weight + ((size_t)b * nC + c) * topk;
            int t = c - 1;
            int n = (t < 0) ? 0 : (include_self ? t + 1 : t);
            ncand_t* cand = (ncand_t*)malloc(sizeof(ncand_t) * (size_t)(n > 0 ? n : 1));
            const double* lt = lm + ((size_t)b * nC + (t < 0 ? 0 : t)) * D;
            for (int kappa = 0; kappa < n; ++kappa) {
                const double* lk = lm + ((size_t)b * nC + kappa) * D;
                double s = 0.0;
                for (int e = 0; e < D; ++e) s += lt[e] * lk[e];
                volatile float s32 = (float)s;
                volatile float r32 = s32 * sigma32;
                volatile float key = r32 + noise[((size_t)b * nC + c) * nC + kappa];
                cand[kappa].key = key;
                cand[kappa].kappa = kappa;
                cand[kappa].s = s;
            }
            qsort(cand, (size_t)n, sizeof(ncand_t), ncand_cmp);
            int m = n < topk ? n : topk;
            double r[64];
            for (int j = 0; j < topk; ++j) { ir[j] = -1; sr[j] = 0.0; wr[j] = 0.0; }
            for (int j = 0; j < m; ++j) {
                ir[j] = cand[j].kappa;
                r[j] = cand[j].s * score_scale;
                sr[j] = r[j];
            }
            oracle_weights_from_scores(m, r, off_by_one, wr);
            free(cand);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Sliding-window self-attention ([P1] section 1: DRT combines top-k past  */
/* chunks with fixed-size sliding-window self-attention; section 4.1.2:    */
/* the window is 512 tokens; the GCA modules come after the attention      */
/* modules of a layer).  Reading: token t of a sequence attends to the     */
/* keys s with max(0, t - W + 1) <= s <= t (itself included), softmax of   */
/* attn_scale * q_t . k_s per head, no other mask.                         */
/* Layouts: q, k, v, o, dout, dq, dk, dv [B, L, H, d]; lse [B, L, H].      */
/* ---------------------------------------------------------------------- */

/* Forward: o_t = sum_s p_ts v_s with p_ts = exp(a_ts - lse_t),
 * a_ts = attn_scale q_t . k_s, lse_t = ln sum_s exp(a_ts). */
void oracle_swa_fwd(int B, int L, int H, int d, int W, double attn_scale, const double* q,
                    const double* k, const double* v, double* o, double* lse)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double* a = (double*)malloc(sizeof(double) * (size_t)(W > 0 ? W : 1));
            for (int t = 0; t < L; ++t) {
                const int s0 = t - W + 1 > 0 ? t - W + 1 : 0;
                const double* qt = q + (((size_t)b * L + t) * H + h) * d;
                double m = -INFINITY;
                for (int s = s0; s <= t; ++s) {
                    const double* ks = k + (((size_t)b * L + s) * H + h) * d;
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e) acc += qt[e] * ks[e];
                    a[s - s0] = attn_scale * acc;
                    if (a[s - s0] > m) m = a[s - s0];
                }
                double l = 0.0;
                for (int s = s0; s <= t; ++s) l += exp(a[s - s0] - m);
                double* ot = o + (((size_t)b * L + t) * H + h) * d;
                for (int e = 0; e < d; ++e) ot[e] = 0.0;
                for (int s = s0; s <= t; ++s) {
                    const double p = exp(a[s - s0] - m) / l;
                    const double* vs = v + (((size_t)b * L + s) * H + h) * d;
                    for (int e = 0; e < d; ++e) ot[e] += p * vs[e];
                }
                lse[((size_t)b * L + t) * H + h] = m + log(l);
            }
            free(a);
        }
    }
}

/* Backward of oracle_swa_fwd for an upstream gradient dout:
 *   delta_t = dout_t . o_t,  dp_ts = dout_t . v_s,  ds_ts = p_ts (dp_ts - delta_t),
 *   dq_t = attn_scale sum_s ds_ts k_s,  dk_s = attn_scale sum_t ds_ts q_t,
 *   dv_s = sum_t p_ts dout_t.
 * p and o are recomputed here from q, k, v (nothing is taken from a forward). */
void oracle_swa_bwd(int B, int L, int H, int d, int W, double attn_scale, const double* q,
                    const double* k, const double* v, const double* dout, double* dq, double* dk,
                    double* dv)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double* p = (double*)malloc(sizeof(double) * (size_t)(W > 0 ? W : 1));
            double* ot = (double*)malloc(sizeof(double) * (size_t)d);
            for (int t = 0; t < L; ++t) {
                size_t ix = (((size_t)b * L + t) * H + h) * d;
                for (int e = 0; e < d; ++e) { dk[ix + e] = 0.0; dv[ix + e] = 0.0; }
            }
            for (int t = 0; t < L; ++t) {
                const int s0 = t - W + 1 > 0 ? t - W + 1 : 0;
                const double* qt = q + (((size_t)b * L + t) * H + h) * d;
                const double* gt = dout + (((size_t)b * L + t) * H + h) * d;
                double m = -INFINITY;
                for (int s = s0; s <= t; ++s) {
                    const double* ks = k + (((size_t)b * L + s) * H + h) * d;
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e) acc += qt[e] * ks[e];
                    p[s - s0] = attn_scale * acc;
                    if (p[s - s0] > m) m = p[s - s0];
                }
                double l = 0.0;
                for (int s = s0; s <= t; ++s) { p[s - s0] = exp(p[s - s0] - m); l += p[s - s0]; }
                for (int s = s0; s <= t; ++s) p[s - s0] /= l;
                for (int e = 0; e < d; ++e) ot[e] = 0.0;
                for (int s = s0; s <= t; ++s) {
                    const double* vs = v + (((size_t)b * L + s) * H + h) * d;
                    for (int e = 0; e < d; ++e) ot[e] += p[s - s0] * vs[e];
                }
                double delta = 0.0;
                for (int e = 0; e < d; ++e) delta += gt[e] * ot[e];
                double* dqt = dq + (((size_t)b * L + t) * H + h) * d;
                for (int e = 0; e < d; ++e) dqt[e] = 0.0;
                for (int s = s0; s <= t; ++s) {
                    const size_t is = (((size_t)b * L + s) * H + h) * d;
                    double dp = 0.0;
                    for (int e = 0; e < d; ++e) dp += gt[e] * v[is + e];
                    const double ds = p[s - s0] * (dp - delta);
                    for (int e = 0; e < d; ++e) {
                        dqt[e] += attn_scale * ds * k[is + e];
                        dk[is + e] += attn_scale * ds * qt[e];
                        dv[is + e] += p[s - s0] * gt[e];
                    }
                }
            }
            free(ot);
            free(p);
        }
    }
}
