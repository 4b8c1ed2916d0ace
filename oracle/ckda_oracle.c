/*
 * ckda_oracle.c -- plain fp64 CPU oracle for the Complex KDA (CKDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * reference that the CUDA path is checked against.  Only the test-suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load it; the
 * library path never does.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (one head, one sequence), in the order the pages state it:
 *
 *   H_t = (I - beta_t k_t k_t^T) Diag(alpha_t) H_{t-1} + beta_t k_t v_t^T
 *   o_t = H_t^T q_t
 *
 *   - "Complex KDA" discussion slides, frame "CKDA keeps the original
 *     gate--delta--readout structure" (the recurrence and the readout of the
 *     UPDATED state; H_t is n x d_v, rows are key channels).
 *   - "Complex KDA: Understanding and Enhancing the Expressivity of Kimi Delta
 *     Attention", App. B.2, Eq. (9): A(x_t) = (I - beta k k^T) Diag(alpha),
 *     B(x_t) = beta k v^T.
 *   - "Kimi Delta Attention: a bounded case study", worked case A/B: the same
 *     update written as three steps -- per-channel decay S' = Diag(a) S
 *     (row i scaled by a_i), read  v_hat = S'^T k, correct
 *     S = S' + beta k (v - v_hat)^T.  This oracle follows those three steps
 *     literally and then reads out o_t = S^T (scale * q_t).
 *
 * `scale` multiplies q before the readout; the pages use no scale (1.0).
 * The oracle does not renormalise k: it consumes exactly the values given.
 *
 * Layouts (row-major, contiguous, the same as the C-ABI of the library):
 *   q, k, alpha : [B, H, T, dk]      v, o : [B, H, T, dv]      beta : [B, H, T]
 *   h0, hT      : [N, H, dk, dv]     N = B (dense) or num_seqs (packed)
 *   cu_seqlens  : [num_seqs + 1] token offsets into T when B == 1 (packed
 *                 variable-length sequences), or NULL for dense [B, H, T].
 *   h0 == NULL means a zero initial state; hT == NULL means "do not store".
 *
 * Parallelism: independent (sequence, head) pairs run on separate OpenMP
 * threads (same paper, App. B.2 "Heads and layers": heads have separate
 * states).  Every pair is computed token by token, in order.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One token of the recurrence on a state S[dk][dv] (row i = key channel i).
 * Worked case A/B order: decay, read, correct; then the readout of the
 * updated state.  `pred` is scratch of length dv. */
static void ckda_token(double *S, int dk, int dv,
                       const double *q, const double *k, const double *v,
                       const double *alpha, double beta, double scale,
                       double *o, double *pred)
{
    /* (1) per-channel decay: S' = Diag(alpha) S  -- row i times alpha_i */
    for (int i = 0; i < dk; ++i) {
        double a = alpha[i];
        double *row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) row[j] *= a;
    }
    /* (2) read: v_hat = S'^T k */
    for (int j = 0; j < dv; ++j) pred[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        double ki = k[i];
        const double *row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) pred[j] += row[j] * ki;
    }
    /* (3) compare and correct: S = S' + beta k (v - v_hat)^T */
    for (int i = 0; i < dk; ++i) {
        double bk = beta * k[i];
        double *row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) row[j] += bk * (v[j] - pred[j]);
    }
    /* (4) readout of the updated state: o = S^T (scale q) */
    if (o) {
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            double qi = scale * q[i];
            const double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) o[j] += row[j] * qi;
        }
    }
}

/* Runs one (sequence, head) pair over tokens [t0, t0 + len) of the [B,H,T,.]
 * arrays at batch index b and head h. */
static void ckda_pair(const double *q, const double *k, const double *v,
                      const double *alpha, const double *beta,
                      const double *h0, double *o, double *hT,
                      int b, int h, int t0, int len,
                      int H, int T, int dk, int dv, double scale, size_t state_idx)
{
    size_t state_elems = (size_t)dk * dv;
    double *S = (double *)malloc(state_elems * sizeof(double));
    double *pred = (double *)malloc((size_t)dv * sizeof(double));
    if (!S || !pred) { free(S); free(pred); return; }
    if (h0) memcpy(S, h0 + state_idx * state_elems, state_elems * sizeof(double));
    else memset(S, 0, state_elems * sizeof(double));

    size_t base = ((size_t)b * H + h) * (size_t)T;
    for (int t = t0; t < t0 + len; ++t) {
        size_t row = base + (size_t)t;
        ckda_token(S, dk, dv,
                   q + row * dk, k + row * dk, v + row * dv,
                   alpha + row * dk, beta[row], scale,
                   o ? o + row * dv : NULL, pred);
    }
    if (hT) memcpy(hT + state_idx * state_elems, S, state_elems * sizeof(double));
    free(S);
    free(pred);
}

/* Returns 0 on success, -1 on an argument error.  nthreads <= 0 uses the
 * OpenMP default. */
int ckda_oracle_fwd(const double *q, const double *k, const double *v,
                    const double *alpha, const double *beta, const double *h0,
                    double *o, double *hT, const int32_t *cu_seqlens, int num_seqs,
                    int B, int H, int T, int dk, int dv, double scale, int nthreads)
{
    if (!q || !k || !v || !alpha || !beta) return -1;
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1) return -1;
    int N = B;
    if (cu_seqlens) {
        if (B != 1 || num_seqs < 1) return -1;
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return -1;
        for (int s = 0; s < num_seqs; ++s)
            if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
        N = num_seqs;
    }
    long pairs = (long)N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long p = 0; p < pairs; ++p) {
        int n = (int)(p / H), h = (int)(p % H);
        int b = cu_seqlens ? 0 : n;
        int t0 = cu_seqlens ? cu_seqlens[n] : 0;
        int len = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : T;
        ckda_pair(q, k, v, alpha, beta, h0, o, hT, b, h, t0, len,
                  H, T, dk, dv, scale, (size_t)n * H + h);
    }
    (void)nthreads;
    return 0;
}

/* One decode step on a resident state [B, H, dk, dv], updated in place.
 * q, k, alpha: [B, H, dk]; v, o: [B, H, dv]; beta: [B, H]. */
int ckda_oracle_decode_step(const double *q, const double *k, const double *v,
                            const double *alpha, const double *beta, double *state,
                            double *o, int B, int H, int dk, int dv, double scale,
                            int nthreads)
{
    if (!q || !k || !v || !alpha || !beta || !state) return -1;
    if (B < 1 || H < 1 || dk < 1 || dv < 1) return -1;
    long pairs = (long)B * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (long p = 0; p < pairs; ++p) {
        double *pred = (double *)malloc((size_t)dv * sizeof(double));
        if (!pred) continue;
        ckda_token(state + (size_t)p * dk * dv, dk, dv,
                   q + (size_t)p * dk, k + (size_t)p * dk, v + (size_t)p * dv,
                   alpha + (size_t)p * dk, beta[p], scale,
                   o ? o + (size_t)p * dv : NULL, pred);
        free(pred);
    }
    (void)nthreads;
    return 0;
}

/* Gradients of one (sequence, head) pair by reverse-mode differentiation of
 * the token steps of ckda_token, taken in reverse order.  The loss is
 * L = sum_t <o_t, do_t> + <H_T, dhT>.  Every state S_0 .. S_len of the pair is
 * kept.
 *
 * Forward step t:  G = Diag(alpha) S_t,  p = G^T k,  u = beta (v - p),
 *                  S_{t+1} = G + k u^T,  o = S_{t+1}^T (scale q).
 * Reverse step t, with D = dL/dS_{t+1} (starting from dhT, or 0):
 *   D += (scale q) do^T;         dq = scale S_{t+1} do
 *   du = D^T k;                  dk = D u
 *   dbeta = <du, v - p>;         dv = beta du;      dp = -beta du
 *   dk += G dp;                  dG = D + k dp^T
 *   dalpha_i = sum_j dG_ij (S_t)_ij;                D = Diag(alpha) dG
 * and dh0 = D at the end. */
static int ckda_pair_bwd(const double *q, const double *k, const double *v,
                         const double *alpha, const double *beta, const double *h0,
                         const double *dout, const double *dhT, double *dq, double *dkk,
                         double *dvv, double *dal, double *dbe, double *dh0,
                         long row0, int len, int dk, int dv, double scale, size_t sidx)
{
    const size_t nn = (size_t)dk * dv;
    double *S = (double *)malloc((size_t)(len + 1) * nn * sizeof(double));
    double *D = (double *)malloc(nn * sizeof(double));
    double *G = (double *)malloc(nn * sizeof(double));
    double *vec = (double *)malloc((size_t)4 * dv * sizeof(double));
    if (!S || !D || !G || !vec) { free(S); free(D); free(G); free(vec); return -1; }
    double *p = vec, *u = vec + dv, *du = vec + 2 * dv, *dp = vec + 3 * dv;
    for (size_t e = 0; e < nn; ++e) S[e] = h0 ? h0[sidx + e] : 0.0;
    for (int t = 0; t < len; ++t) {
        const size_t r = (size_t)(row0 + t);
        const double *St = S + (size_t)t * nn;
        double *Sn = S + (size_t)(t + 1) * nn;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += k[r * dk + i] * alpha[r * dk + i] * St[(size_t)i * dv + j];
            p[j] = acc;
            u[j] = beta[r] * (v[r * dv + j] - acc);
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                Sn[(size_t)i * dv + j] = alpha[r * dk + i] * St[(size_t)i * dv + j] + k[r * dk + i] * u[j];
    }
    for (size_t e = 0; e < nn; ++e) D[e] = dhT ? dhT[sidx + e] : 0.0;
    for (int t = len - 1; t >= 0; --t) {
        const size_t r = (size_t)(row0 + t);
        const double *St = S + (size_t)t * nn, *Sn = S + (size_t)(t + 1) * nn;
        const double *qt = q + r * dk, *kt = k + r * dk, *at = alpha + r * dk;
        const double *vt = v + r * dv, *dot = dout + r * dv;
        const double bt = beta[r];
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                D[(size_t)i * dv + j] += scale * qt[i] * dot[j];
                acc += Sn[(size_t)i * dv + j] * dot[j];
            }
            dq[r * dk + i] = scale * acc;
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] = at[i] * St[(size_t)i * dv + j];
        double dbeta = 0.0;
        for (int j = 0; j < dv; ++j) {
            double pj = 0.0, dj = 0.0;
            for (int i = 0; i < dk; ++i) {
                pj += kt[i] * G[(size_t)i * dv + j];
                dj += kt[i] * D[(size_t)i * dv + j];
            }
            p[j] = pj;
            u[j] = bt * (vt[j] - pj);
            du[j] = dj;
            dbeta += dj * (vt[j] - pj);
            dvv[r * dv + j] = bt * dj;
            dp[j] = -bt * dj;
        }
        dbe[r] = dbeta;
        for (int i = 0; i < dk; ++i) {
            double gk = 0.0, ga = 0.0;
            for (int j = 0; j < dv; ++j) {
                const size_t e = (size_t)i * dv + j;
                gk += D[e] * u[j] + G[e] * dp[j];
                const double dG = D[e] + kt[i] * dp[j];
                ga += dG * St[e];
                D[e] = at[i] * dG;
            }
            dkk[r * dk + i] = gk;
            dal[r * dk + i] = ga;
        }
    }
    if (dh0)
        for (size_t e = 0; e < nn; ++e) dh0[sidx + e] = D[e];
    free(S); free(D); free(G); free(vec);
    return 0;
}

/* The backward of ckda_oracle_fwd: gradients of L = sum <o, do> + <hT, dhT>
 * (dhT may be NULL: zero) with respect to q, k, v, alpha, beta ([.., T, .]
 * layouts as the forward) and h0 (dh0 may be NULL: not stored). */
int ckda_oracle_bwd(const double *q, const double *k, const double *v, const double *alpha,
                    const double *beta, const double *h0, const double *dout,
                    const double *dhT, double *dq, double *dkk, double *dvv, double *dal,
                    double *dbe, double *dh0, const int32_t *cu_seqlens, int num_seqs,
                    int B, int H, int T, int dk, int dv, double scale, int nthreads)
{
    if (!q || !k || !v || !alpha || !beta || !dout || !dq || !dkk || !dvv || !dal || !dbe)
        return -1;
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1) return -1;
    int N = B;
    if (cu_seqlens) {
        if (B != 1 || num_seqs < 1) return -1;
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return -1;
        for (int s = 0; s < num_seqs; ++s)
            if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
        N = num_seqs;
    }
    long pairs = (long)N * H;
    int fail = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
#endif
    for (long pp = 0; pp < pairs; ++pp) {
        int n = (int)(pp / H), h = (int)(pp % H);
        int t0 = cu_seqlens ? cu_seqlens[n] : 0;
        int len = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : T;
        long row0 = cu_seqlens ? (long)h * T + t0 : ((long)n * H + h) * T;
        size_t sidx = ((size_t)n * H + h) * (size_t)dk * dv;
        fail |= ckda_pair_bwd(q, k, v, alpha, beta, h0, dout, dhT, dq, dkk, dvv, dal, dbe, dh0,
                              row0, len, dk, dv, scale, sidx) != 0;
    }
    (void)nthreads;
    return fail ? -2 : 0;
}

/* Input preparation, per token (row) of dk channels, in the paper's
 * parameterisation ("Complex KDA" discussion slides, backup frame "practical
 * gates differ from exact theoretical endpoints"; paper App. E-G.1):
 *
 *   r = tanh(a / 2),   s = +1 if r >= 0 else -1,
 *   alpha = s [eps + (1 - eps) |r|],   eps = e^-5,
 *   beta  = 2 sigma(b) = 2 / (1 + e^-b),
 *
 * and the unit-norm keys the recurrence assumes (paper Sec. 2: ||k_t|| = 1),
 * here k / sqrt(sum_i k_i^2 + norm_eps) per token; q likewise when
 * normalize_q is set, else copied.  Arrays are [rows, dk] (q, k, a) and
 * [rows] (b); q_raw / q may be NULL together. */
int ckda_oracle_prep(const double *q_raw, const double *k_raw, const double *a_raw,
                     const double *b_raw, double *q, double *k, double *alpha,
                     double *beta, long rows, int dk, int normalize_q, double norm_eps)
{
    if (!k_raw || !a_raw || !b_raw || !k || !alpha || !beta) return -1;
    if ((q_raw == NULL) != (q == NULL)) return -1;
    if (rows < 0 || dk < 1) return -1;
    const double eps = exp(-5.0);
    for (long t = 0; t < rows; ++t) {
        const double *kr = k_raw + (size_t)t * dk;
        double ss = 0.0;
        for (int i = 0; i < dk; ++i) ss += kr[i] * kr[i];
        double inv = 1.0 / sqrt(ss + norm_eps);
        for (int i = 0; i < dk; ++i) k[(size_t)t * dk + i] = kr[i] * inv;
        if (q_raw) {
            const double *qr = q_raw + (size_t)t * dk;
            double qi = 1.0;
            if (normalize_q) {
                double sq = 0.0;
                for (int i = 0; i < dk; ++i) sq += qr[i] * qr[i];
                qi = 1.0 / sqrt(sq + norm_eps);
            }
            for (int i = 0; i < dk; ++i) q[(size_t)t * dk + i] = qr[i] * qi;
        }
        for (int i = 0; i < dk; ++i) {
            double r = tanh(a_raw[(size_t)t * dk + i] / 2.0);
            double sgn = r >= 0.0 ? 1.0 : -1.0;
            alpha[(size_t)t * dk + i] = sgn * (eps + (1.0 - eps) * fabs(r));
        }
        beta[t] = 2.0 / (1.0 + exp(-b_raw[t]));
    }
    return 0;
}

/*
 * Backward of ckda_oracle_prep: from the raw inputs and the gradients of a
 * loss with respect to the prepared q, k, alpha, beta, the gradients with
 * respect to q_raw, k_raw, a_raw and b_raw, all fp64 (any pointer of the q
 * side may be NULL together with q_raw).
 *
 * Normalisation (unit keys, paper Sec. 2; the same norm_eps as the forward):
 *   k = x / n with n = sqrt(sum_i x_i^2 + norm_eps), so
 *   dk_raw_j = sum_i dk_i dk_i/dx_j = (dk_j - k_j (k . dk)) / n.
 * Gates ("Complex KDA" discussion slides, backup frame "practical gates differ
 * from exact theoretical endpoints"):
 *   alpha = s [e^-5 + (1 - e^-5) |r|], r = tanh(a / 2).  The sign s is
 *   piecewise constant and carries no gradient; |r| takes the subgradient 0 at
 *   r = 0.  For r != 0, s sign(r) = 1 and d|r|/da = sign(r) (1 - r^2) / 2, so
 *   dalpha/da = (1 - e^-5) (1 - r^2) / 2, and 0 at r = 0.
 *   beta = 2 sigma(b), so dbeta/db = 2 sigma(b) (1 - sigma(b)).
 */
int ckda_oracle_prep_bwd(const double *q_raw, const double *k_raw, const double *a_raw,
                         const double *b_raw, const double *dq, const double *dk,
                         const double *dalpha, const double *dbeta, double *dq_raw,
                         double *dk_raw, double *da_raw, double *db_raw, long rows, int n,
                         int normalize_q, double norm_eps)
{
    if (!k_raw || !a_raw || !b_raw || !dk || !dalpha || !dbeta) return -1;
    if (!dk_raw || !da_raw || !db_raw) return -1;
    if ((q_raw == NULL) != (dq == NULL) || (q_raw == NULL) != (dq_raw == NULL)) return -1;
    if (rows < 0 || n < 1) return -1;
    const double eps = exp(-5.0);
    for (long t = 0; t < rows; ++t) {
        const size_t o = (size_t)t * n;
        /* keys */
        double ss = 0.0;
        for (int i = 0; i < n; ++i) ss += k_raw[o + i] * k_raw[o + i];
        double nrm = sqrt(ss + norm_eps);
        double dot = 0.0;
        for (int i = 0; i < n; ++i) dot += (k_raw[o + i] / nrm) * dk[o + i];
        for (int i = 0; i < n; ++i)
            dk_raw[o + i] = (dk[o + i] - (k_raw[o + i] / nrm) * dot) / nrm;
        /* queries */
        if (q_raw) {
            if (normalize_q) {
                double sq = 0.0;
                for (int i = 0; i < n; ++i) sq += q_raw[o + i] * q_raw[o + i];
                double qn = sqrt(sq + norm_eps);
                double qd = 0.0;
                for (int i = 0; i < n; ++i) qd += (q_raw[o + i] / qn) * dq[o + i];
                for (int i = 0; i < n; ++i)
                    dq_raw[o + i] = (dq[o + i] - (q_raw[o + i] / qn) * qd) / qn;
            } else {
                for (int i = 0; i < n; ++i) dq_raw[o + i] = dq[o + i];
            }
        }
        /* decay gate */
        for (int i = 0; i < n; ++i) {
            double r = tanh(a_raw[o + i] / 2.0);
            double g = r == 0.0 ? 0.0 : (1.0 - eps) * (1.0 - r * r) / 2.0;
            da_raw[o + i] = dalpha[o + i] * g;
        }
        /* write strength */
        double sg = 1.0 / (1.0 + exp(-b_raw[t]));
        db_raw[t] = dbeta[t] * 2.0 * sg * (1.0 - sg);
    }
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int ckda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
