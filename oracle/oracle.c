/*
 * Reference oracle for exact scaled-dot-product attention: TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously-correct fp64 CPU code.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the library under test never does, and
 * this file shares no code, header or constant with it.
 *
 * Sources (web pages, cited by title and section):
 *   [FA1-review]  "[논문 리뷰] FlashAttention: Fast and Memory-Efficient Exact Attention with
 *                 IO-Awareness" (osehyeon.github.io) - "Standard Attention Implementation"
 *                 (Algorithm 0), "Tilting" (softmax decomposition m, f, l) and Algorithm 1.
 *   [IO-essay]    "Flash Attention IO-awareness principle" (hrletsgo.me) - sections on
 *                 standard attention (S = QK^T / sqrt(d)), tiling/online softmax, recomputation.
 *   [Triton-FA2]  "Triton 06: Flash Attention v2" (wonbeomjang.kr) - "개선 3" (causal mask
 *                 offs_m >= offs_n, i.e. key index <= query index) and "Backward 구현" /
 *                 "Forward/Backward 전체 흐름 요약" (Delta, dV, dK, dQ equations).
 *
 * Conventions (one head; row-major; N rows, d columns):
 *   S_ij = scale * sum_k Q_ik K_jk ; causal: S_ij = -inf for j > i ;
 *   P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i) with m_i = max_j S_ij ;
 *   O = P V ;  lse_i = m_i + ln sum_j exp(S_ij - m_i)  (natural log of the scaled logits).
 * Backward is the gradient of L = sum(dO o O):
 *   dV = P^T dO ; dP = dO V^T ; Delta_i = sum_j P_ij dP_ij ; dS = P o (dP - Delta) ;
 *   dQ = scale dS K ; dK = scale dS^T Q.
 *
 * Every function returns 0 on success and a negative value on bad arguments or when memory
 * cannot be allocated.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ENOMEM (-2)
#define ORACLE_EINVAL (-1)

static int key_valid(int causal, long i, long j) { return !causal || j <= i; }

/* ---------------------------------------------------------------------------------------
 * Algorithm 0 ([FA1-review], "Standard Attention Implementation"), one head.
 * Step 1 materialises S = scale * Q K^T (N x N), step 2 P = softmax(S) row by row,
 * step 3 O = P V.  Masked entries are -inf before the softmax.  lse is returned per row.
 * If P_out is not NULL the N x N matrix P is copied there.
 * ------------------------------------------------------------------------------------- */
int oracle_attention_fwd_head(int N, int d, double scale, int causal, const double* Q,
                              const double* K, const double* V, double* O, double* lse,
                              double* P_out)
{
    if (N < 1 || d < 1 || !Q || !K || !V || !O || !lse) return ORACLE_EINVAL;
    const long n = N;
    double* S = (double*)malloc(sizeof(double) * n * n);
    double* Kt = (double*)malloc(sizeof(double) * n * d);
    if (!S || !Kt) { free(S); free(Kt); return ORACLE_ENOMEM; }
    /* K^T so that row i of S accumulates over k with a contiguous inner loop over j. */
    for (long j = 0; j < n; ++j)
        for (int k = 0; k < d; ++k) Kt[(long)k * n + j] = K[j * d + k];

    for (long i = 0; i < n; ++i) {
        double* Si = S + i * n;
        for (long j = 0; j < n; ++j) Si[j] = 0.0;
        for (int k = 0; k < d; ++k) {
            const double qik = Q[i * d + k];
            const double* Ktk = Kt + (long)k * n;
            for (long j = 0; j < n; ++j) Si[j] += qik * Ktk[j];
        }
        for (long j = 0; j < n; ++j) Si[j] = key_valid(causal, i, j) ? scale * Si[j] : -INFINITY;
        /* softmax of row i: m(x), f(x) = exp(x - m(x)), l(x) = sum f(x), f / l */
        double m = -INFINITY;
        for (long j = 0; j < n; ++j) if (Si[j] > m) m = Si[j];
        double l = 0.0;
        for (long j = 0; j < n; ++j) { Si[j] = exp(Si[j] - m); l += Si[j]; }
        for (long j = 0; j < n; ++j) Si[j] /= l;
        lse[i] = m + log(l);
        /* O_i = sum_j P_ij V_j */
        double* Oi = O + i * d;
        for (int c = 0; c < d; ++c) Oi[c] = 0.0;
        for (long j = 0; j < n; ++j) {
            const double p = Si[j];
            const double* Vj = V + j * d;
            for (int c = 0; c < d; ++c) Oi[c] += p * Vj[c];
        }
    }
    if (P_out) memcpy(P_out, S, sizeof(double) * n * n);
    free(S);
    free(Kt);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Backward of Algorithm 0 for one head, recomputing its own P from Q, K (never from any
 * library output).  Equations as listed in [Triton-FA2] "Forward/Backward 전체 흐름 요약",
 * written in natural-log form with a materialised P and dP.
 * Optional outputs: O and lse of the forward, Delta (per row).
 * ------------------------------------------------------------------------------------- */
int oracle_attention_bwd_head(int N, int d, double scale, int causal, const double* Q,
                              const double* K, const double* V, const double* dO, double* dQ,
                              double* dK, double* dV, double* O_out, double* lse_out,
                              double* delta_out)
{
    if (N < 1 || d < 1 || !Q || !K || !V || !dO || !dQ || !dK || !dV) return ORACLE_EINVAL;
    const long n = N;
    double* P = (double*)malloc(sizeof(double) * n * n);
    double* dP = (double*)malloc(sizeof(double) * n * n);
    double* T = (double*)malloc(sizeof(double) * n * d); /* transposes of K, then V */
    double* O = (double*)malloc(sizeof(double) * n * d);
    double* lse = (double*)malloc(sizeof(double) * n);
    if (!P || !dP || !T || !O || !lse) {
        free(P); free(dP); free(T); free(O); free(lse);
        return ORACLE_ENOMEM;
    }
    int rc = oracle_attention_fwd_head(N, d, scale, causal, Q, K, V, O, lse, P);
    if (rc) { free(P); free(dP); free(T); free(O); free(lse); return rc; }

    /* dP = dO V^T (masked entries are irrelevant: P is exactly 0 there) */
    for (long j = 0; j < n; ++j)
        for (int k = 0; k < d; ++k) T[(long)k * n + j] = V[j * d + k];
    for (long i = 0; i < n; ++i) {
        double* r = dP + i * n;
        for (long j = 0; j < n; ++j) r[j] = 0.0;
        for (int k = 0; k < d; ++k) {
            const double a = dO[i * d + k];
            const double* Tk = T + (long)k * n;
            for (long j = 0; j < n; ++j) r[j] += a * Tk[j];
        }
    }
    /* dV = P^T dO */
    for (long j = 0; j < n * d; ++j) dV[j] = 0.0;
    for (long i = 0; i < n; ++i)
        for (long j = 0; j < n; ++j) {
            const double p = P[i * n + j];
            if (p == 0.0) continue;
            double* dVj = dV + j * d;
            const double* dOi = dO + i * d;
            for (int c = 0; c < d; ++c) dVj[c] += p * dOi[c];
        }
    /* Delta_i = sum_j P_ij dP_ij ; dS = P o (dP - Delta) stored over dP */
    for (long i = 0; i < n; ++i) {
        double delta = 0.0;
        for (long j = 0; j < n; ++j) delta += P[i * n + j] * dP[i * n + j];
        if (delta_out) delta_out[i] = delta;
        for (long j = 0; j < n; ++j) dP[i * n + j] = P[i * n + j] * (dP[i * n + j] - delta);
    }
    /* dQ = scale dS K ; dK = scale dS^T Q */
    for (long i = 0; i < n * d; ++i) { dQ[i] = 0.0; dK[i] = 0.0; }
    for (long i = 0; i < n; ++i)
        for (long j = 0; j < n; ++j) {
            const double ds = dP[i * n + j];
            if (ds == 0.0) continue;
            double* dQi = dQ + i * d;
            double* dKj = dK + j * d;
            const double* Kj = K + j * d;
            const double* Qi = Q + i * d;
            for (int c = 0; c < d; ++c) { dQi[c] += ds * Kj[c]; dKj[c] += ds * Qi[c]; }
        }
    for (long i = 0; i < n * d; ++i) { dQ[i] *= scale; dK[i] *= scale; }
    if (O_out) memcpy(O_out, O, sizeof(double) * n * d);
    if (lse_out) memcpy(lse_out, lse, sizeof(double) * n);
    free(P); free(dP); free(T); free(O); free(lse);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Algorithm 1 of [FA1-review] (tiled, K/V blocks outer, Q blocks inner), one head, in fp64.
 * Used only to check that the tiled online-softmax update reaches the Algorithm 0 result
 * ("exact attention", [IO-essay] tiling section).  Block sizes Br x Bc are free parameters;
 * T_r = ceil(N/Br), T_c = ceil(N/Bc) and the last blocks may be ragged.
 * Reading for the causal mask, which Algorithm 1 does not state: masked entries of S_ij are
 * -inf; a block row whose entries are all masked contributes nothing (m, l, O unchanged).
 * The scaled, normalised O update of step 12 is used as written once its garbled exponent
 * is read as exp(m~_ij - m_new).
 * ------------------------------------------------------------------------------------- */
int oracle_attention_fwd_tiled_head(int N, int d, double scale, int causal, int Br, int Bc,
                                    const double* Q, const double* K, const double* V,
                                    double* O, double* lse)
{
    if (N < 1 || d < 1 || Br < 1 || Bc < 1 || !Q || !K || !V || !O || !lse) return ORACLE_EINVAL;
    const long n = N;
    double* l = (double*)malloc(sizeof(double) * n);
    double* m = (double*)malloc(sizeof(double) * n);
    double* Sij = (double*)malloc(sizeof(double) * (long)Br * Bc);
    double* PV = (double*)malloc(sizeof(double) * (long)d);
    if (!l || !m || !Sij || !PV) { free(l); free(m); free(Sij); free(PV); return ORACLE_ENOMEM; }
    for (long i = 0; i < n * d; ++i) O[i] = 0.0;           /* step 2 */
    for (long i = 0; i < n; ++i) { l[i] = 0.0; m[i] = -INFINITY; }
    const long Tr = (n + Br - 1) / Br, Tc = (n + Bc - 1) / Bc; /* step 3 */
    for (long jb = 0; jb < Tc; ++jb) {                        /* step 5 */
        const long j0 = jb * Bc, j1 = (j0 + Bc < n) ? j0 + Bc : n;
        for (long ib = 0; ib < Tr; ++ib) {                    /* step 7 */
            const long i0 = ib * Br, i1 = (i0 + Br < n) ? i0 + Br : n;
            for (long i = i0; i < i1; ++i) {
                double* s = Sij + (i - i0) * Bc;
                /* step 9: S_ij = Q_i K_j^T (scaled, masked) */
                for (long j = j0; j < j1; ++j) {
                    double acc = 0.0;
                    for (int k = 0; k < d; ++k) acc += Q[i * d + k] * K[j * d + k];
                    s[j - j0] = key_valid(causal, i, j) ? scale * acc : -INFINITY;
                }
                /* step 10: m~ = rowmax, P~ = exp(S - m~), l~ = rowsum(P~) */
                double mt = -INFINITY;
                for (long j = j0; j < j1; ++j) if (s[j - j0] > mt) mt = s[j - j0];
                if (mt == -INFINITY) continue; /* fully masked block row */
                double lt = 0.0;
                for (long j = j0; j < j1; ++j) { s[j - j0] = exp(s[j - j0] - mt); lt += s[j - j0]; }
                /* step 11 */
                const double mnew = (m[i] > mt) ? m[i] : mt;
                const double a_old = exp(m[i] - mnew), a_new = exp(mt - mnew);
                const double lnew = a_old * l[i] + a_new * lt;
                /* step 12: O_i <- diag(l_new)^-1 (diag(l_i) e^{m_i - m_new} O_i + e^{m~ - m_new} P~ V_j) */
                for (int c = 0; c < d; ++c) PV[c] = 0.0;
                for (long j = j0; j < j1; ++j) {
                    const double p = s[j - j0];
                    for (int c = 0; c < d; ++c) PV[c] += p * V[j * d + c];
                }
                for (int c = 0; c < d; ++c)
                    O[i * d + c] = (l[i] * a_old * O[i * d + c] + a_new * PV[c]) / lnew;
                /* step 13 */
                l[i] = lnew;
                m[i] = mnew;
            }
        }
    }
    for (long i = 0; i < n; ++i) lse[i] = m[i] + log(l[i]);
    free(l); free(m); free(Sij); free(PV);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Sampled mode for heads too long to materialise (Algorithm 0 restricted to rows).
 * For each listed query row i: the full row S_i. (length N) is formed, then
 * O_i, lse_i, Delta_i = sum_j P_ij dP_ij and dQ_i = scale sum_j dS_ij K_j.
 * For each listed key row j: dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij Q_i, which
 * needs, for every query row i that sees key j, the row statistics lse_i and Delta_i;
 * those rows are each formed in full exactly as above.  Rows are split across nthreads.
 * ------------------------------------------------------------------------------------- */
typedef struct {
    int N, d, causal;
    double scale;
    const double *Q, *K, *V, *dO;
    int nk;
    const int* krows;
    long i_begin, i_end;
    double *dK_acc, *dV_acc; /* nk x d partials owned by this worker */
    double *s, *dp;          /* scratch rows of length N */
    int rc;
} rows_job;

/* Full row statistics of query row i: fills s (probabilities P_i.), dp (dP_i.) and returns
 * lse_i and Delta_i.  Masked entries get P = 0. */
static void row_stats(int N, int d, double scale, int causal, const double* Q, const double* K,
                      const double* V, const double* dO, long i, double* s, double* dp,
                      double* lse_i, double* delta_i)
{
    const double* qi = Q + i * d;
    const double* gi = dO + i * d;
    double m = -INFINITY;
    for (long j = 0; j < N; ++j) {
        if (!key_valid(causal, i, j)) { s[j] = -INFINITY; dp[j] = 0.0; continue; }
        double acc = 0.0, accp = 0.0;
        const double* kj = K + j * d;
        const double* vj = V + j * d;
        for (int c = 0; c < d; ++c) { acc += qi[c] * kj[c]; accp += gi[c] * vj[c]; }
        s[j] = scale * acc;
        dp[j] = accp;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < N; ++j) { s[j] = exp(s[j] - m); l += s[j]; }
    double delta = 0.0;
    for (long j = 0; j < N; ++j) { s[j] /= l; delta += s[j] * dp[j]; }
    *lse_i = m + log(l);
    *delta_i = delta;
}

static void* rows_worker(void* arg)
{
    rows_job* jb = (rows_job*)arg;
    const int d = jb->d;
    for (long i = jb->i_begin; i < jb->i_end; ++i) {
        int any = 0;
        for (int r = 0; r < jb->nk; ++r) any |= key_valid(jb->causal, i, jb->krows[r]);
        if (!any) continue;
        double lse_i, delta_i;
        row_stats(jb->N, d, jb->scale, jb->causal, jb->Q, jb->K, jb->V, jb->dO, i, jb->s, jb->dp,
                  &lse_i, &delta_i);
        for (int r = 0; r < jb->nk; ++r) {
            const long j = jb->krows[r];
            if (!key_valid(jb->causal, i, j)) continue;
            const double p = jb->s[j];
            const double ds = p * (jb->dp[j] - delta_i);
            for (int c = 0; c < d; ++c) {
                jb->dV_acc[(long)r * d + c] += p * jb->dO[i * d + c];
                jb->dK_acc[(long)r * d + c] += ds * jb->Q[i * d + c];
            }
        }
    }
    return NULL;
}

int oracle_attention_rows_head(int N, int d, double scale, int causal, const double* Q,
                               const double* K, const double* V, const double* dO, int nq,
                               const int* qrows, double* O_rows, double* lse_rows,
                               double* delta_rows, double* dQ_rows, int nk, const int* krows,
                               double* dK_rows, double* dV_rows, int nthreads)
{
    if (N < 1 || d < 1 || nq < 0 || nk < 0 || !Q || !K || !V || !dO) return ORACLE_EINVAL;
    for (int r = 0; r < nq; ++r) if (qrows[r] < 0 || qrows[r] >= N) return ORACLE_EINVAL;
    for (int r = 0; r < nk; ++r) if (krows[r] < 0 || krows[r] >= N) return ORACLE_EINVAL;
    double* s = (double*)malloc(sizeof(double) * N);
    double* dp = (double*)malloc(sizeof(double) * N);
    if (!s || !dp) { free(s); free(dp); return ORACLE_ENOMEM; }
    for (int r = 0; r < nq; ++r) {
        const long i = qrows[r];
        double lse_i, delta_i;
        row_stats(N, d, scale, causal, Q, K, V, dO, i, s, dp, &lse_i, &delta_i);
        if (lse_rows) lse_rows[r] = lse_i;
        if (delta_rows) delta_rows[r] = delta_i;
        double* o = O_rows ? O_rows + (long)r * d : NULL;
        double* g = dQ_rows ? dQ_rows + (long)r * d : NULL;
        for (int c = 0; c < d; ++c) { if (o) o[c] = 0.0; if (g) g[c] = 0.0; }
        for (long j = 0; j < N; ++j) {
            if (s[j] == 0.0) continue; /* masked (or underflowed) entry contributes nothing */
            const double p = s[j], ds = s[j] * (dp[j] - delta_i);
            for (int c = 0; c < d; ++c) {
                if (o) o[c] += p * V[j * d + c];
                if (g) g[c] += ds * K[j * d + c];
            }
        }
        if (g) for (int c = 0; c < d; ++c) g[c] *= scale;
    }
    free(s);
    free(dp);
    if (nk == 0) return 0;

    if (nthreads < 1) nthreads = 1;
    long first = 0;
    if (causal) { /* rows before the smallest key index never see any listed key */
        first = krows[0];
        for (int r = 1; r < nk; ++r) if (krows[r] < first) first = krows[r];
    }
    const long span = N - first;
    if (nthreads > span) nthreads = (int)span;
    rows_job* jobs = (rows_job*)calloc(nthreads, sizeof(rows_job));
    pthread_t* th = (pthread_t*)calloc(nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return ORACLE_ENOMEM; }
    int rc = 0;
    /* Under a causal mask row i costs about i*d: split rows so each worker gets equal area. */
    for (int t = 0; t < nthreads; ++t) {
        rows_job* jb = &jobs[t];
        jb->N = N; jb->d = d; jb->causal = causal; jb->scale = scale;
        jb->Q = Q; jb->K = K; jb->V = V; jb->dO = dO; jb->nk = nk; jb->krows = krows;
        double f0 = (double)t / nthreads, f1 = (double)(t + 1) / nthreads;
        if (causal) {
            const double a = (double)first * first, b = (double)N * N;
            jb->i_begin = (long)sqrt(a + f0 * (b - a));
            jb->i_end = (t == nthreads - 1) ? N : (long)sqrt(a + f1 * (b - a));
        } else {
            jb->i_begin = first + (long)(f0 * span);
            jb->i_end = (t == nthreads - 1) ? N : first + (long)(f1 * span);
        }
        if (jb->i_begin < first) jb->i_begin = first;
        jb->dK_acc = (double*)calloc((size_t)nk * d, sizeof(double));
        jb->dV_acc = (double*)calloc((size_t)nk * d, sizeof(double));
        jb->s = (double*)malloc(sizeof(double) * N);
        jb->dp = (double*)malloc(sizeof(double) * N);
        if (!jb->dK_acc || !jb->dV_acc || !jb->s || !jb->dp) rc = ORACLE_ENOMEM;
    }
    if (!rc) {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&th[t], NULL, rows_worker, &jobs[t]) != 0) { rows_worker(&jobs[t]); th[t] = 0; }
            else started++;
        }
        for (int t = 0; t < nthreads; ++t) if (th[t]) pthread_join(th[t], NULL);
        (void)started;
        for (int r = 0; r < nk; ++r)
            for (int c = 0; c < d; ++c) {
                double gk = 0.0, gv = 0.0;
                for (int t = 0; t < nthreads; ++t) {
                    gk += jobs[t].dK_acc[(long)r * d + c];
                    gv += jobs[t].dV_acc[(long)r * d + c];
                }
                if (dK_rows) dK_rows[(long)r * d + c] = scale * gk;
                if (dV_rows) dV_rows[(long)r * d + c] = gv;
            }
    }
    for (int t = 0; t < nthreads; ++t) {
        free(jobs[t].dK_acc); free(jobs[t].dV_acc); free(jobs[t].s); free(jobs[t].dp);
    }
    free(jobs);
    free(th);
    return rc;
}

/* ---------------------------------------------------------------------------------------
 * Algorithm 0 and its backward for one head with Nq query rows and Nk key rows (Nq != Nk
 * allowed).  [IO-essay] places the kernel under chunked prefill: a chunk of the last Nq
 * queries of a sequence attends to all Nk keys of the sequence so far, with the causal mask
 * inside the chunk.  So the causal mask is aligned to the bottom-right corner:
 *   key j is visible to query i  iff  j <= i + (Nk - Nq),
 * which is the square mask of [Triton-FA2] "개선 3" when Nq == Nk.
 * A query row that sees no key (Nq > Nk, or Nk == 0) has an empty softmax: its P row is 0,
 * O_i = 0 and lse_i = log(0) = -inf, and it contributes no gradient.
 * dO == NULL computes the forward only (dQ, dK, dV, delta are then ignored).
 * ------------------------------------------------------------------------------------- */
int oracle_attention_rect_head(int Nq, int Nk, int d, double scale, int causal,
                               const double* Q, const double* K, const double* V,
                               const double* dO, double* O, double* lse, double* delta,
                               double* dQ, double* dK, double* dV)
{
    if (Nq < 0 || Nk < 0 || d < 1 || !O || !lse) return ORACLE_EINVAL;
    if (dO && (!dQ || !dK || !dV)) return ORACLE_EINVAL;
    const long nq = Nq, nk = Nk, off = (long)Nk - (long)Nq;
    double* P = (double*)malloc(sizeof(double) * (nq * nk + 1));
    double* dP = dO ? (double*)malloc(sizeof(double) * (nq * nk + 1)) : NULL;
    if (!P || (dO && !dP)) { free(P); free(dP); return ORACLE_ENOMEM; }
    /* S = scale Q K^T with the mask, then P = softmax(S) row by row */
    for (long i = 0; i < nq; ++i) {
        double* Pi = P + i * nk;
        double m = -INFINITY;
        for (long j = 0; j < nk; ++j) {
            if (causal && j > i + off) { Pi[j] = -INFINITY; continue; }
            double sij = 0.0;
            for (int c = 0; c < d; ++c) sij += Q[i * d + c] * K[j * d + c];
            Pi[j] = scale * sij;
            if (Pi[j] > m) m = Pi[j];
        }
        if (m == -INFINITY) { /* no visible key */
            for (long j = 0; j < nk; ++j) Pi[j] = 0.0;
            lse[i] = -INFINITY;
        } else {
            double l = 0.0;
            for (long j = 0; j < nk; ++j) { Pi[j] = exp(Pi[j] - m); l += Pi[j]; }
            for (long j = 0; j < nk; ++j) Pi[j] /= l;
            lse[i] = m + log(l);
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (long j = 0; j < nk; ++j) acc += Pi[j] * V[j * d + c];
            O[i * d + c] = acc;
        }
    }
    if (dO) {
        /* dP = dO V^T ; Delta_i = sum_j P_ij dP_ij ; dS = P o (dP - Delta) */
        for (long i = 0; i < nq; ++i) {
            double dl = 0.0;
            for (long j = 0; j < nk; ++j) {
                double a = 0.0;
                for (int c = 0; c < d; ++c) a += dO[i * d + c] * V[j * d + c];
                dP[i * nk + j] = a;
                dl += P[i * nk + j] * a;
            }
            if (delta) delta[i] = dl;
            for (long j = 0; j < nk; ++j) dP[i * nk + j] = P[i * nk + j] * (dP[i * nk + j] - dl);
        }
        /* dV = P^T dO ; dK = scale dS^T Q ; dQ = scale dS K  (sums over i and j, row by row) */
        for (long x = 0; x < nk * d; ++x) { dV[x] = 0.0; dK[x] = 0.0; }
        for (long i = 0; i < nq; ++i) {
            double* dQi = dQ + i * d;
            for (int c = 0; c < d; ++c) dQi[c] = 0.0;
            for (long j = 0; j < nk; ++j) {
                const double p = P[i * nk + j], ds = dP[i * nk + j];
                for (int c = 0; c < d; ++c) {
                    dV[j * d + c] += p * dO[i * d + c];
                    dK[j * d + c] += ds * Q[i * d + c];
                    dQi[c] += ds * K[j * d + c];
                }
            }
        }
        for (long x = 0; x < nk * d; ++x) dK[x] *= scale;
        for (long x = 0; x < nq * d; ++x) dQ[x] *= scale;
    }
    free(P);
    free(dP);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Batched drivers: heads are independent; one head per worker thread at a time.
 * Arrays are [BH, N, d] (lse and delta [BH, N]), contiguous.
 * ------------------------------------------------------------------------------------- */
typedef struct {
    int bwd, BH, N, d, causal;
    double scale;
    const double *Q, *K, *V, *dO;
    double *O, *lse, *dQ, *dK, *dV, *delta;
    int next; /* next head to take */
    pthread_mutex_t mu;
    int rc;
} batch_job;

static void* batch_worker(void* arg)
{
    batch_job* jb = (batch_job*)arg;
    const long hs = (long)jb->N * jb->d;
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        const int h = jb->next++;
        pthread_mutex_unlock(&jb->mu);
        if (h >= jb->BH) break;
        int rc;
        if (!jb->bwd) {
            rc = oracle_attention_fwd_head(jb->N, jb->d, jb->scale, jb->causal, jb->Q + h * hs,
                                           jb->K + h * hs, jb->V + h * hs, jb->O + h * hs,
                                           jb->lse + (long)h * jb->N, NULL);
        } else {
            rc = oracle_attention_bwd_head(
                jb->N, jb->d, jb->scale, jb->causal, jb->Q + h * hs, jb->K + h * hs,
                jb->V + h * hs, jb->dO + h * hs, jb->dQ + h * hs, jb->dK + h * hs, jb->dV + h * hs,
                jb->O ? jb->O + h * hs : NULL, jb->lse ? jb->lse + (long)h * jb->N : NULL,
                jb->delta ? jb->delta + (long)h * jb->N : NULL);
        }
        if (rc) {
            pthread_mutex_lock(&jb->mu);
            jb->rc = rc;
            pthread_mutex_unlock(&jb->mu);
        }
    }
    return NULL;
}

static int run_batch(batch_job* jb, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > jb->BH) nthreads = jb->BH;
    pthread_mutex_init(&jb->mu, NULL);
    pthread_t* th = (pthread_t*)calloc(nthreads, sizeof(pthread_t));
    if (!th) return ORACLE_ENOMEM;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, batch_worker, jb) != 0) th[t] = 0;
    batch_worker(jb); /* the calling thread helps too, and guarantees progress */
    for (int t = 0; t < nthreads; ++t) if (th[t]) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&jb->mu);
    return jb->rc;
}

int oracle_attention_fwd(int BH, int N, int d, double scale, int causal, const double* Q,
                         const double* K, const double* V, double* O, double* lse, int nthreads)
{
    if (BH < 1) return ORACLE_EINVAL;
    batch_job jb;
    memset(&jb, 0, sizeof jb);
    jb.BH = BH; jb.N = N; jb.d = d; jb.causal = causal; jb.scale = scale;
    jb.Q = Q; jb.K = K; jb.V = V; jb.O = O; jb.lse = lse;
    return run_batch(&jb, nthreads - 1);
}

int oracle_attention_bwd(int BH, int N, int d, double scale, int causal, const double* Q,
                         const double* K, const double* V, const double* dO, double* dQ,
                         double* dK, double* dV, double* O, double* lse, double* delta,
                         int nthreads)
{
    if (BH < 1) return ORACLE_EINVAL;
    batch_job jb;
    memset(&jb, 0, sizeof jb);
    jb.bwd = 1; jb.BH = BH; jb.N = N; jb.d = d; jb.causal = causal; jb.scale = scale;
    jb.Q = Q; jb.K = K; jb.V = V; jb.dO = dO; jb.dQ = dQ; jb.dK = dK; jb.dV = dV;
    jb.O = O; jb.lse = lse; jb.delta = delta;
    return run_batch(&jb, nthreads - 1);
}
