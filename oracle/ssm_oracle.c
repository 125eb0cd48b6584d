/*
 * Plain fp64 CPU oracle for the selective state-space (S6) scan, its scalar-A
 * multi-head (SSD) form and the single-token decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library; the two meet only in the seeded input generators.
 *
 * Every routine is the sequential definition, one time step after another, in
 * double precision, with no blocking, chunking or reordering:
 *
 *   - "Mamba 논문 리뷰: 선형 시간복잡도로 Transformer에 도전하는 Selective State
 *     Space Model" (tildalice.io), section "Δ의 직관적 이해": the discretised
 *     recurrence h_t = exp(Δ_t A) h_{t-1} + Δ_t B_t x_t (the simplified B̄ = ΔB),
 *     section "Selection Mechanism": Δ_t = softplus(s_Δ(x_t)), and the
 *     block diagram / reference class in section "Mamba 블록 아키텍처": readout
 *     y_t = C_t h_t after the update, then the gate y·SiLU(z).
 *   - "[yongggg's] Mamba: Linear-Time Sequence Modeling with Selective State
 *     Spaces (Review)", section "State Space Model": the D skip term D·x.
 *   - "Mamba-2: 상태 공간 기반 시퀀스 모델" (obsidian-dorae222.pages.dev),
 *     sections "1-세미분리 행렬" and "멀티-헤드 구조": one independent SSM per
 *     head with a scalar decay per head and B, C shared by the heads of a group.
 *
 * Readings where the pages are silent or garbled (all listed in the design
 * notes): Δ is per channel; B̄ = ΔB (the simplified form; the zero-order-hold form
 * (exp(ΔA) - I) A^-1 B of section "이산화" on request); y = (C·h + D·x)·silu(z); the initial state
 * is zero unless given; softplus(v) = log(1 + e^v) evaluated in the overflow-
 * free form max(v,0) + log1p(exp(-|v|)).
 *
 * Layouts (row-major, last index fastest):
 *   scan   : x, delta, z, y (B,L,D); Bm, Cm (B,L,N); A (D,N); Dv, bias (D);
 *            h0, h_final (B,D,N)
 *   ssd    : x, z, y (B,L,H,P); delta (B,L,H); A, Dv, bias (H);
 *            Bm, Cm (B,L,G,N); h0, h_final (B,H,P,N)
 *   decode : state (B,D,N) updated in place; x, delta, z, y (B,D); Bm, Cm (B,N);
 *            A (D,N); Dv, bias (D)
 * Nullable pointers: Dv, z, bias, h0, h_final (scan/ssd); Dv, z, bias (decode).
 * Return value: 0 on success, -1 on a bad size, -2 on allocation failure.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(v) = log(1 + e^v), written so that neither branch overflows. */
static double softplus_f64(double v)
{
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

/* SiLU(z) = z * sigmoid(z). */
static double silu_f64(double z)
{
    return z / (1.0 + exp(-z));
}

static double step_size(double raw, const double *bias, int64_t c, int softplus)
{
    double v = raw + (bias ? bias[c] : 0.0);
    return softplus ? softplus_f64(v) : v;
}

/* Input coefficient of the discretised recurrence for one state with diagonal entry a:
 *   Euler (the simplified form, tildalice "Δ의 직관적 이해"):  dl
 *   zero-order hold (tildalice "이산화"):  (exp(dl a) - 1) / a, whose limit as a -> 0
 *   is dl; B̄ x = coefficient * B * x. */
static double input_coef(double dl, double a, int zoh)
{
    if (!zoh || a == 0.0) return dl;
    return expm1(dl * a) / a;
}

int oracle_scan_f64(int64_t nb, int64_t L, int64_t D, int64_t N,
                    const double *x, const double *delta, const double *A,
                    const double *Bm, const double *Cm, const double *Dv,
                    const double *z, const double *bias, int softplus, int zoh,
                    const double *h0, double *y, double *h_final, int nthreads)
{
    if (nb < 0 || L < 0 || D < 0 || N < 1) return -1;
    int64_t chains = nb * D;
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : failed)
    for (int64_t c = 0; c < chains; ++c) {
        int64_t b = c / D, d = c % D;
        double *h = (double *)malloc((size_t)N * sizeof(double));
        if (!h) { failed |= 1; continue; }
        for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            int64_t bt = b * L + t;
            double xv = x[bt * D + d];
            double dl = step_size(delta[bt * D + d], bias, d, softplus);
            /* state update: h <- exp(dl*A) h + coef*B_t*x_t (coef = dl, or the ZOH one) */
            for (int64_t n = 0; n < N; ++n)
                h[n] = exp(dl * A[d * N + n]) * h[n] +
                       input_coef(dl, A[d * N + n], zoh) * Bm[bt * N + n] * xv;
            /* readout after the update, then the D skip and the gate */
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) acc += Cm[bt * N + n] * h[n];
            double out = acc + (Dv ? Dv[d] : 0.0) * xv;
            if (z) out *= silu_f64(z[bt * D + d]);
            y[bt * D + d] = out;
        }
        if (h_final)
            for (int64_t n = 0; n < N; ++n) h_final[(b * D + d) * N + n] = h[n];
        free(h);
    }
    return failed ? -2 : 0;
}

/* Derivatives of the ZOH input coefficient c(dl, a) = (exp(dl a) - 1) / a:
 *   dc/d(dl) = exp(dl a)
 *   dc/da    = dl^2 (v e^v - e^v + 1) / v^2 with v = dl a, whose power series is
 *              dl^2 sum_{j>=0} (j+1) v^j / (j+2)!  (used for |v| < 1e-2, where the closed
 *              form cancels; six terms leave an error below 2e-16 relative). */
static double zoh_dc_da(double dl, double a)
{
    double v = dl * a;
    if (fabs(v) < 1e-2) {
        double s = 0.0, f = 1.0, pw = 1.0;      /* f = (j+2)! */
        for (int j = 0; j < 6; ++j) {
            f *= (double)(j + 2);
            s += (double)(j + 1) * pw / f;
            pw *= v;
        }
        return dl * dl * s;
    }
    return (dl * exp(v) - expm1(v) / a) / a;
}

static double sigmoid_f64(double v)
{
    return 1.0 / (1.0 + exp(-v));
}

/*
 * Gradients of the scan above (reverse-mode, the adjoint of the recurrence).  The
 * pages ask for the backward pass of the selective scan to rebuild the states instead
 * of storing them (tildalice review, section "Hardware-Aware 병렬 알고리즘", item
 * "역전파 시 재계산"; yongggg review, section "하드웨어 인식 알고리즘"); the
 * oracle has no memory limit and keeps every h_t of one (b, d) chain, then walks
 * back in time:
 *   lam      = dLoss/dh_t, starting from gh_final (or 0)
 *   g_yr     = gy_t silu(z_t)                 (gradient of C.h + D x)
 *   gz_t     = gy_t (C.h_t + D x_t) silu'(z_t), silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   gC_t,n  += g_yr h_t,n       gD += g_yr x_t       gx_t = g_yr D
 *   lam_n   += g_yr C_t,n
 *   with h_t,n = a h_{t-1},n + c B_t,n x_t,  a = exp(dl A_n),  c = dl (Euler) or
 *   (exp(dl A_n) - 1)/A_n (ZOH):
 *   gB_t,n  += lam_n c x_t      gx_t += lam_n c B_t,n
 *   gdl_t   += lam_n (h_{t-1},n a A_n + B_t,n x_t dc/d(dl))
 *   gA_n    += lam_n (h_{t-1},n a dl + B_t,n x_t dc/dA)
 *   lam_n    = lam_n a            (now dLoss/dh_{t-1})
 *   gdelta_t = gdl_t softplus'(v) = gdl_t sigmoid(v), v = delta_t + bias (or gdl_t
 *              without softplus);  gbias += gdelta_t;  gh0 = lam at t = -1.
 * gB, gC are summed over d; gA, gD, gbias over b (and t).  Outputs gz, gD, gbias, gh0
 * are nullable.  gh_final (B,D,N) is nullable (zero).
 */
int oracle_scan_bwd_f64(int64_t nb, int64_t L, int64_t D, int64_t N,
                        const double *x, const double *delta, const double *A,
                        const double *Bm, const double *Cm, const double *Dv,
                        const double *z, const double *bias, int softplus, int zoh,
                        const double *h0, const double *gy, const double *gh_final,
                        double *gx, double *gdelta, double *gA, double *gB, double *gC,
                        double *gD, double *gz, double *gbias, double *gh0, int nthreads)
{
    if (nb < 0 || L < 0 || D < 0 || N < 1) return -1;
    if (nthreads < 1) nthreads = 1;
    memset(gA, 0, (size_t)(D * N) * sizeof(double));
    memset(gB, 0, (size_t)(nb * L * N) * sizeof(double));
    memset(gC, 0, (size_t)(nb * L * N) * sizeof(double));
    if (gD) memset(gD, 0, (size_t)D * sizeof(double));
    if (gbias) memset(gbias, 0, (size_t)D * sizeof(double));
    int failed = 0;
    for (int64_t b = 0; b < nb; ++b) {
        /* channels of one batch row in parallel; gB/gC of this row are summed over d
         * from per-thread copies, in channel order within a thread */
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
        {
            double *hs = (double *)malloc((size_t)((L + 1) * N) * sizeof(double));
            double *lam = (double *)malloc((size_t)N * sizeof(double));
            double *pB = (double *)calloc((size_t)(L * N), sizeof(double));
            double *pC = (double *)calloc((size_t)(L * N), sizeof(double));
            int ok = hs && lam && pB && pC;
            if (!ok) failed |= 1;
#pragma omp for schedule(static)
            for (int64_t d = 0; d < D; ++d) {
                if (!ok) continue;
                const double *Ad = A + d * N;
                double Dd = Dv ? Dv[d] : 0.0;
                /* forward, keeping h_{-1} .. h_{L-1} in hs[0 .. L] */
                for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
                for (int64_t t = 0; t < L; ++t) {
                    int64_t bt = b * L + t;
                    double xv = x[bt * D + d];
                    double dl = step_size(delta[bt * D + d], bias, d, softplus);
                    for (int64_t n = 0; n < N; ++n)
                        hs[(t + 1) * N + n] = exp(dl * Ad[n]) * hs[t * N + n] +
                                              input_coef(dl, Ad[n], zoh) * Bm[bt * N + n] * xv;
                }
                /* backward */
                for (int64_t n = 0; n < N; ++n)
                    lam[n] = gh_final ? gh_final[(b * D + d) * N + n] : 0.0;
                double gD_acc = 0.0, gbias_acc = 0.0;
                for (int64_t t = L - 1; t >= 0; --t) {
                    int64_t bt = b * L + t;
                    double xv = x[bt * D + d];
                    double v = delta[bt * D + d] + (bias ? bias[d] : 0.0);
                    double dl = softplus ? softplus_f64(v) : v;
                    const double *ht = hs + (t + 1) * N, *hp = hs + t * N;
                    double g_yr = gy[bt * D + d];
                    if (z) {
                        double zv = z[bt * D + d], sg = sigmoid_f64(zv);
                        double yr = Dd * xv;
                        for (int64_t n = 0; n < N; ++n) yr += Cm[bt * N + n] * ht[n];
                        if (gz) gz[bt * D + d] = g_yr * yr * sg * (1.0 + zv * (1.0 - sg));
                        g_yr *= zv * sg;
                    }
                    double gxv = g_yr * Dd, gdl = 0.0;
                    gD_acc += g_yr * xv;
                    for (int64_t n = 0; n < N; ++n) {
                        double an = Ad[n], a = exp(dl * an), c = input_coef(dl, an, zoh);
                        double Bn = Bm[bt * N + n];
                        pC[t * N + n] += g_yr * ht[n];
                        lam[n] += g_yr * Cm[bt * N + n];
                        pB[t * N + n] += lam[n] * c * xv;
                        gxv += lam[n] * c * Bn;
                        double dc_ddl = zoh ? a : 1.0;
                        double dc_da = zoh ? (an == 0.0 ? 0.5 * dl * dl : zoh_dc_da(dl, an)) : 0.0;
                        gdl += lam[n] * (hp[n] * a * an + Bn * xv * dc_ddl);
                        gA[d * N + n] += lam[n] * (hp[n] * a * dl + Bn * xv * dc_da);
                        lam[n] *= a;
                    }
                    double gv = softplus ? gdl * sigmoid_f64(v) : gdl;
                    gx[bt * D + d] = gxv;
                    gdelta[bt * D + d] = gv;
                    gbias_acc += gv;
                }
                if (gD) gD[d] += gD_acc;
                if (gbias) gbias[d] += gbias_acc;
                if (gh0)
                    for (int64_t n = 0; n < N; ++n) gh0[(b * D + d) * N + n] = lam[n];
            }
#pragma omp critical
            if (ok) {
                for (int64_t i = 0; i < L * N; ++i) {
                    gB[b * L * N + i] += pB[i];
                    gC[b * L * N + i] += pC[i];
                }
            }
            free(hs); free(lam); free(pB); free(pC);
        }
    }
    return failed ? -2 : 0;
}

int oracle_ssd_f64(int64_t nb, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                   const double *x, const double *delta, const double *A,
                   const double *Bm, const double *Cm, const double *Dv,
                   const double *z, const double *bias, int softplus,
                   const double *h0, double *y, double *h_final, int nthreads)
{
    if (nb < 0 || L < 0 || H < 1 || P < 1 || G < 1 || N < 1 || H % G) return -1;
    int64_t heads_per_group = H / G;
    int64_t chains = nb * H;
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : failed)
    for (int64_t c = 0; c < chains; ++c) {
        int64_t b = c / H, hd = c % H, g = hd / heads_per_group;
        /* matrix state S (P x N) of head hd */
        double *S = (double *)malloc((size_t)(P * N) * sizeof(double));
        if (!S) { failed |= 1; continue; }
        for (int64_t i = 0; i < P * N; ++i) S[i] = h0 ? h0[(b * H + hd) * P * N + i] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            int64_t bt = b * L + t;
            double dl = step_size(delta[bt * H + hd], bias, hd, softplus);
            double decay = exp(dl * A[hd]);
            const double *Bt = Bm + (bt * G + g) * N;
            const double *Ct = Cm + (bt * G + g) * N;
            for (int64_t p = 0; p < P; ++p) {
                double xv = x[(bt * H + hd) * P + p];
                double *Sp = S + p * N;
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    Sp[n] = decay * Sp[n] + dl * xv * Bt[n];
                    acc += Ct[n] * Sp[n];
                }
                double out = acc + (Dv ? Dv[hd] : 0.0) * xv;
                if (z) out *= silu_f64(z[(bt * H + hd) * P + p]);
                y[(bt * H + hd) * P + p] = out;
            }
        }
        if (h_final)
            for (int64_t i = 0; i < P * N; ++i) h_final[(b * H + hd) * P * N + i] = S[i];
        free(S);
    }
    return failed ? -2 : 0;
}

int oracle_decode_f64(int64_t nb, int64_t D, int64_t N, double *state,
                      const double *x, const double *delta, const double *A,
                      const double *Bm, const double *Cm, const double *Dv,
                      const double *z, const double *bias, int softplus, int zoh,
                      double *y, int nthreads)
{
    if (nb < 0 || D < 0 || N < 1) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t c = 0; c < nb * D; ++c) {
        int64_t b = c / D, d = c % D;
        double xv = x[c];
        double dl = step_size(delta[c], bias, d, softplus);
        double *h = state + c * N;
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            h[n] = exp(dl * A[d * N + n]) * h[n] + input_coef(dl, A[d * N + n], zoh) * Bm[b * N + n] * xv;
            acc += Cm[b * N + n] * h[n];
        }
        double out = acc + (Dv ? Dv[d] : 0.0) * xv;
        if (z) out *= silu_f64(z[c]);
        y[c] = out;
    }
    return 0;
}

/* One token of the multi-head scalar-A recurrence (the SSD form's decode step): per
 * batch b and head hd (group g = hd / (H / G)), with dl = step(delta[b,hd]):
 *   S[p,n] <- exp(dl A[hd]) S[p,n] + dl x[b,hd,p] B[b,g,n]   (state updated in place)
 *   y[b,hd,p] = sum_n C[b,g,n] S[p,n] + D[hd] x[b,hd,p], times silu(z) if given.
 * Layouts: state (B,H,P,N); x, z, y (B,H,P); delta (B,H); Bm, Cm (B,G,N); A, Dv, bias (H). */
int oracle_ssd_decode_f64(int64_t nb, int64_t H, int64_t P, int64_t G, int64_t N, double *state,
                          const double *x, const double *delta, const double *A,
                          const double *Bm, const double *Cm, const double *Dv,
                          const double *z, const double *bias, int softplus, double *y,
                          int nthreads)
{
    if (nb < 0 || H < 1 || P < 1 || G < 1 || N < 1 || H % G) return -1;
    if (nthreads < 1) nthreads = 1;
    int64_t heads_per_group = H / G;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t c = 0; c < nb * H; ++c) {
        int64_t b = c / H, hd = c % H, g = hd / heads_per_group;
        double dl = step_size(delta[c], bias, hd, softplus);
        double decay = exp(dl * A[hd]);
        const double *Bt = Bm + (b * G + g) * N;
        const double *Ct = Cm + (b * G + g) * N;
        for (int64_t p = 0; p < P; ++p) {
            double xv = x[c * P + p];
            double *Sp = state + (c * P + p) * N;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                Sp[n] = decay * Sp[n] + dl * xv * Bt[n];
                acc += Ct[n] * Sp[n];
            }
            double out = acc + (Dv ? Dv[hd] : 0.0) * xv;
            if (z) out *= silu_f64(z[c * P + p]);
            y[c * P + p] = out;
        }
    }
    return 0;
}

/* Causal depthwise convolution along time, then SiLU (tildalice review, section
 * "Mamba 블록 아키텍처" and its reference class: a depthwise Conv1D of kernel K with
 * K - 1 steps of left padding, cropped to L, followed by SiLU):
 *   pre[b,t,d] = bias[d] + sum_{k=0}^{K-1} w[d,k] x[b, t-(K-1)+k, d]
 *   out[b,t,d] = silu(pre) (or pre when silu == 0)
 * x at t < 0 comes from x_prev (B, K-1, D) (the K-1 inputs just before this call, oldest
 * first) or is zero.  Layouts: x, out (B,L,D); w (D,K); bias (D). */
int oracle_conv1d_f64(int64_t nb, int64_t L, int64_t D, int64_t K, const double *x,
                      const double *w, const double *bias, const double *x_prev, int silu,
                      double *out, int nthreads)
{
    if (nb < 0 || L < 0 || D < 0 || K < 1) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t c = 0; c < nb * D; ++c) {
        int64_t b = c / D, d = c % D;
        for (int64_t t = 0; t < L; ++t) {
            double acc = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t s = t - (K - 1) + k;
                double xv;
                if (s >= 0) xv = x[(b * L + s) * D + d];
                else xv = x_prev ? x_prev[(b * (K - 1) + (K - 1 + s)) * D + d] : 0.0;
                acc += w[d * K + k] * xv;
            }
            out[(b * L + t) * D + d] = silu ? silu_f64(acc) : acc;
        }
    }
    return 0;
}

/* Helper exposed for the pins: the scalar softplus used above. */
double oracle_softplus_f64(double v) { return softplus_f64(v); }

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
