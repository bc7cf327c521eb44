/*
 * Float64 CPU oracle for the selective-scan hot path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA library never
 * links, includes or calls it, and this file shares no code with it.
 *
 * Every function below is the plain sequential definition, evaluated in
 * double precision from the exact values the GPU is given (fp32, or bf16
 * widened exactly to fp32 by the caller). There is no blocking, no
 * reassociation and no fast-math: build with -O2 -ffp-contract=off.
 *
 * Sources (web pages on the selective scan):
 *   [SSK]  "Selective-scan CUDA kernels" (persus.netlify.app), opening
 *          paragraphs: the recurrence h[t] = a[t]*h[t-1] + b[t] and its
 *          affine-pair scan form.
 *   [S6]   "POPCORNBENCH FW-GLM-5-1 l2_p30" (arjun-banerjee.github.io),
 *          forward-pass derivation: dA = exp(delta*A), dB = delta*B_t,
 *          x_db = x*dB, h = dA*h + x_db, y_t = sum_n h*C_t, y + x*D; the
 *          layouts x,delta,y (B,L,D), B_t,C_t (B,L,N), A (D,N), D (D);
 *          softplus on delta via log(1 + exp(v)); h starts at zero.
 *   [ARM]  "ARM-Scan - Optimized Mamba Selective-Scan Kernel"
 *          (krithiksama.me), Approach and What broke: forward and reverse
 *          recurrences share the discretisation, and the fused result must
 *          equal the two scans run independently.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - h[-1] = 0 for the affine scan; h starts at 0 for S6 ([S6]). A scan
 *     continued from an earlier segment starts from that segment's last
 *     state h0 instead.
 *   - softplus uses threshold 20: v > 20 returns v (PyTorch's default).
 *   - the reverse recurrence applies dA and dBx of the same time index:
 *     h_rev[t] = dA[t]*h_rev[t+1] + dBx[t], i.e. the forward scan of the
 *     time-reversed inputs, read back in original order.
 *   - in the bidirectional output each direction carries its own D*x term.
 *   - state in/out (forward only): h0 (B, D, N) replaces the zero state
 *     before t = 0, and h_last (B, D, N) is the state after t = L-1; running
 *     [0, L1) and then [L1, L) from the first run's h_last is the same loop
 *     as running [0, L) in one go.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* ------------------------------------------------------------------ affine */

/* [SSK] h[t] = a[t]*h[t-1] + b[t], with h[-1] = h0 (the reading for a
 * scan continued from an earlier segment: h0 is that segment's last state). */
void oracle_affine_state_f64(const float *a, const float *b, double h0, double *h, int64_t n)
{
    double state = h0;
    for (int64_t t = 0; t < n; ++t) {
        state = (double)a[t] * state + (double)b[t];
        h[t] = state;
    }
}

/* [SSK] h[t] = a[t]*h[t-1] + b[t], with h[-1] = 0. */
void oracle_affine_f64(const float *a, const float *b, double *h, int64_t n)
{
    oracle_affine_state_f64(a, b, 0.0, h, n);
}

/* ------------------------------------------------------------------ S6 */

/* [S6] softplus(v) = log(1 + exp(v)); v > 20 returns v. */
double oracle_softplus_f64(double v)
{
    if (v > 20.0)
        return v;
    return log1p(exp(v));
}

typedef struct {
    const float *x, *delta, *Bt, *Ct, *A, *Dskip;
    int64_t B, L, D, N;
    int softplus;
    int bidir;
    const int64_t *chans;   /* channel c = b*D + d; NULL means all B*D */
    int64_t nchan;
    const double *h0;       /* (B, D, N) state before t = 0; NULL: zeros */
    double *hlast;          /* (B, D, N) state after t = L-1; NULL: not kept */
    double *out;            /* chans != NULL: (nchan, L); else (B, L, D) */
    int64_t begin, end;     /* range of channel slots this worker owns */
} s6_job;

/* One (b, d) channel, every state n, every step t ([S6] forward pass).
 * Writes y[t] for t in [0, L) with stride `ystride`.
 * With `bidir`, adds the reverse recurrence ([ARM]) over the same dA, dBx. */
static void s6_channel(const s6_job *j, int64_t b, int64_t d, double *h,
                       double *y, int64_t ystride)
{
    const int64_t L = j->L, D = j->D, N = j->N;
    const double Dd = (double)j->Dskip[d];

    /* forward: t = 0 .. L-1, from h0 (zeros unless given) */
    for (int64_t n = 0; n < N; ++n)
        h[n] = j->h0 ? j->h0[(b * D + d) * N + n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t xi = (b * L + t) * D + d;   /* x[b, t, d] */
        const int64_t bi = (b * L + t) * N;       /* B_t[b, t, :] */
        double dl = (double)j->delta[xi];
        if (j->softplus)
            dl = oracle_softplus_f64(dl);
        const double xv = (double)j->x[xi];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double dA = exp(dl * (double)j->A[d * N + n]);
            const double dB = dl * (double)j->Bt[bi + n];
            const double x_db = xv * dB;
            h[n] = dA * h[n] + x_db;
            acc += h[n] * (double)j->Ct[bi + n];
        }
        y[t * ystride] = acc + xv * Dd;
    }
    if (j->hlast)
        for (int64_t n = 0; n < N; ++n)
            j->hlast[(b * D + d) * N + n] = h[n];
    if (!j->bidir)
        return;

    /* reverse: t = L-1 .. 0, h_rev[t] = dA[t]*h_rev[t+1] + dBx[t] */
    for (int64_t n = 0; n < N; ++n)
        h[n] = 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t xi = (b * L + t) * D + d;
        const int64_t bi = (b * L + t) * N;
        double dl = (double)j->delta[xi];
        if (j->softplus)
            dl = oracle_softplus_f64(dl);
        const double xv = (double)j->x[xi];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double dA = exp(dl * (double)j->A[d * N + n]);
            const double dB = dl * (double)j->Bt[bi + n];
            const double x_db = xv * dB;
            h[n] = dA * h[n] + x_db;
            acc += h[n] * (double)j->Ct[bi + n];
        }
        y[t * ystride] += acc + xv * Dd;
    }
}

static void *s6_worker(void *arg)
{
    const s6_job *j = (const s6_job *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    if (!h)
        return (void *)1;
    for (int64_t s = j->begin; s < j->end; ++s) {
        const int64_t c = j->chans ? j->chans[s] : s;
        const int64_t b = c / j->D, d = c % j->D;
        if (j->chans)
            s6_channel(j, b, d, h, j->out + s * j->L, 1);
        else
            s6_channel(j, b, d, h, j->out + b * j->L * j->D + d, j->D);
    }
    free(h);
    return NULL;
}

/* Splits the independent (b, d) channels over `threads` POSIX threads.
 * The per-channel loop is the same whatever the split. Returns 0 on success. */
static int s6_run(s6_job base, int threads)
{
    const int64_t total = base.chans ? base.nchan : base.B * base.D;
    if (total <= 0 || base.L <= 0)
        return 0;
    if (threads < 1)
        threads = 1;
    if (threads > total)
        threads = (int)total;
    if (threads == 1) {
        base.begin = 0;
        base.end = total;
        return s6_worker(&base) ? -1 : 0;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    s6_job *jobs = (s6_job *)malloc(sizeof(s6_job) * (size_t)threads);
    if (!tid || !jobs) {
        free(tid);
        free(jobs);
        return -1;
    }
    int rc = 0, started = 0;
    for (int i = 0; i < threads; ++i) {
        jobs[i] = base;
        jobs[i].begin = total * i / threads;
        jobs[i].end = total * (i + 1) / threads;
        if (pthread_create(&tid[i], NULL, s6_worker, &jobs[i]) != 0) {
            rc = -1;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret)
            rc = -1;
    }
    free(tid);
    free(jobs);
    return rc;
}

/* [S6] forward pass over all channels; y is (B, L, D) float64. */
int oracle_s6_fwd_f64(const float *x, const float *delta, const float *Bt,
                      const float *Ct, const float *A, const float *Dskip,
                      double *y, int64_t B, int64_t L, int64_t D, int64_t N,
                      int softplus, int threads)
{
    s6_job j = {x, delta, Bt, Ct, A, Dskip, B, L, D, N, softplus, 0,
                NULL, 0, NULL, NULL, y, 0, 0};
    return s6_run(j, threads);
}

/* [S6] forward pass from the state h0 (NULL: zeros), also returning the
 * state after the last step in h_last (NULL: not returned); h0 and h_last
 * are (B, D, N) float64, y is (B, L, D). */
int oracle_s6_fwd_state_f64(const float *x, const float *delta, const float *Bt,
                            const float *Ct, const float *A, const float *Dskip,
                            const double *h0, double *y, double *h_last,
                            int64_t B, int64_t L, int64_t D, int64_t N,
                            int softplus, int threads)
{
    s6_job j = {x, delta, Bt, Ct, A, Dskip, B, L, D, N, softplus, 0,
                NULL, 0, h0, h_last, y, 0, 0};
    return s6_run(j, threads);
}

/* [ARM] forward plus reverse recurrence over shared dA, dBx; y is (B, L, D). */
int oracle_s6_bidir_f64(const float *x, const float *delta, const float *Bt,
                        const float *Ct, const float *A, const float *Dskip,
                        double *y, int64_t B, int64_t L, int64_t D, int64_t N,
                        int softplus, int threads)
{
    s6_job j = {x, delta, Bt, Ct, A, Dskip, B, L, D, N, softplus, 1,
                NULL, 0, NULL, NULL, y, 0, 0};
    return s6_run(j, threads);
}

/* Selected channels only (c = b*D + d); out is (nchan, L) float64.
 * Used to check full-size GPU outputs channel by channel. */
int oracle_s6_channels_f64(const float *x, const float *delta, const float *Bt,
                           const float *Ct, const float *A, const float *Dskip,
                           int64_t B, int64_t L, int64_t D, int64_t N,
                           int softplus, int bidir, const int64_t *chans,
                           int64_t nchan, double *out, int threads)
{
    for (int64_t i = 0; i < nchan; ++i)
        if (chans[i] < 0 || chans[i] >= B * D)
            return -2;
    s6_job j = {x, delta, Bt, Ct, A, Dskip, B, L, D, N, softplus, bidir,
                chans, nchan, NULL, NULL, out, 0, 0};
    return s6_run(j, threads);
}


/* ------------------------------------------------------------------ backward */

/* Reverse-mode derivative of the forward pass from h0 (the scope table's
 * "next" row; the pages give only the forward pass, so this is the exact
 * derivative of that definition, taken step by step in reverse order) for the
 * scalar loss  sum_{b,t,d} dy*y + sum_{b,d,n} dh_last*h_last.
 * Forward per (b, d), as above:  dl = sp(v) or v;  dA = exp(dl*A[d,n]);
 *   h_t = dA*h_{t-1} + dl*B_t*x;  y_t = sum_n h_t*C_t + D*x.
 * Reverse, with g[n] the gradient reaching h_t from later steps (starting
 * from dh_last) and lam = g + dy_t*C_t the whole gradient of h_t:
 *   dC_t += dy_t*h_t;  dD += dy_t*x;  dx_t = dy_t*D + sum_n lam*dl*B_t;
 *   ddl_t = sum_n lam*(B_t*x + h_{t-1}*dA*A);  dA_param += lam*h_{t-1}*dA*dl;
 *   dB_t += lam*dl*x;  g = lam*dA (the gradient of h_{t-1});  dh0 = final g.
 *   dv = ddl * sigmoid(v) under softplus (v > 20: ddl).
 * dx, ddelta: (B, L, D); dA: (D, N); dBt, dCt: (B, L, N); dDskip: (D,);
 * dh0: (B, D, N) or NULL; h0, dh_last: (B, D, N) or NULL (zeros). */
typedef struct {
    const float *x, *delta, *Bt, *Ct, *A, *Dskip, *dy;
    const double *h0, *dh_last;
    int64_t B, L, D, N;
    int softplus;
    double *dx, *ddelta, *dA, *dBt, *dCt, *dDskip, *dh0;
    int64_t b0, b1;          /* batch range of this worker */
    double *dA_part, *dD_part; /* this worker's sums over its batch range */
} s6_bwd_job;

static void *s6_bwd_worker(void *arg)
{
    s6_bwd_job *j = (s6_bwd_job *)arg;
    const int64_t L = j->L, D = j->D, N = j->N;
    double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N));  /* h_{-1} .. h_{L-1} */
    double *dAs = (double *)malloc(sizeof(double) * (size_t)(L * N));
    double *dls = (double *)malloc(sizeof(double) * (size_t)L);
    double *g = (double *)malloc(sizeof(double) * (size_t)N);
    if (!hs || !dAs || !dls || !g) {
        free(hs); free(dAs); free(dls); free(g);
        return (void *)1;
    }
    for (int64_t b = j->b0; b < j->b1; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const double Dd = (double)j->Dskip[d];
            /* forward, keeping every state and every dA */
            for (int64_t n = 0; n < N; ++n)
                hs[n] = j->h0 ? j->h0[(b * D + d) * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t xi = (b * L + t) * D + d, bi = (b * L + t) * N;
                double dl = (double)j->delta[xi];
                if (j->softplus)
                    dl = oracle_softplus_f64(dl);
                dls[t] = dl;
                const double xv = (double)j->x[xi];
                for (int64_t n = 0; n < N; ++n) {
                    const double dA = exp(dl * (double)j->A[d * N + n]);
                    dAs[t * N + n] = dA;
                    hs[(t + 1) * N + n] = dA * hs[t * N + n] + dl * (double)j->Bt[bi + n] * xv;
                }
            }
            /* reverse */
            for (int64_t n = 0; n < N; ++n)
                g[n] = j->dh_last ? j->dh_last[(b * D + d) * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                const int64_t xi = (b * L + t) * D + d, bi = (b * L + t) * N;
                const double gy = (double)j->dy[xi], xv = (double)j->x[xi], dl = dls[t];
                double gx = gy * Dd, gdl = 0.0;
                j->dD_part[d] += gy * xv;
                for (int64_t n = 0; n < N; ++n) {
                    const double Bv = (double)j->Bt[bi + n], Cv = (double)j->Ct[bi + n];
                    const double ht = hs[(t + 1) * N + n], hprev = hs[t * N + n];
                    const double dA = dAs[t * N + n], An = (double)j->A[d * N + n];
                    const double lam = g[n] + gy * Cv;
                    j->dCt[bi + n] += gy * ht;
                    gx += lam * dl * Bv;
                    gdl += lam * (Bv * xv + hprev * dA * An);
                    j->dA_part[d * N + n] += lam * hprev * dA * dl;
                    j->dBt[bi + n] += lam * dl * xv;
                    g[n] = lam * dA;
                }
                j->dx[xi] = gx;
                if (j->softplus) {
                    const double v = (double)j->delta[xi];
                    gdl = v > 20.0 ? gdl : gdl / (1.0 + exp(-v));
                }
                j->ddelta[xi] = gdl;
            }
            if (j->dh0)
                for (int64_t n = 0; n < N; ++n)
                    j->dh0[(b * D + d) * N + n] = g[n];
        }
    }
    free(hs); free(dAs); free(dls); free(g);
    return NULL;
}

/* Splits the batch over `threads` workers; each keeps its own dA and dDskip
 * sums, added in worker order at the end. Returns 0 on success. */
int oracle_s6_bwd_f64(const float *x, const float *delta, const float *Bt,
                      const float *Ct, const float *A, const float *Dskip,
                      const double *h0, const float *dy, const double *dh_last,
                      int64_t B, int64_t L, int64_t D, int64_t N, int softplus,
                      double *dx, double *ddelta, double *dA, double *dBt,
                      double *dCt, double *dDskip, double *dh0, int threads)
{
    if (B <= 0 || L < 0 || D <= 0 || N <= 0)
        return 0;
    if (threads < 1)
        threads = 1;
    if (threads > B)
        threads = (int)B;
    for (int64_t i = 0; i < B * L * N; ++i)
        dBt[i] = dCt[i] = 0.0;
    s6_bwd_job *jobs = (s6_bwd_job *)calloc((size_t)threads, sizeof(s6_bwd_job));
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    double *parts = (double *)calloc((size_t)threads * (size_t)(D * N + D), sizeof(double));
    if (!jobs || !tid || !parts) {
        free(jobs); free(tid); free(parts);
        return -1;
    }
    int rc = 0, started = 0;
    for (int i = 0; i < threads; ++i) {
        s6_bwd_job jb = {x, delta, Bt, Ct, A, Dskip, dy, h0, dh_last, B, L, D, N, softplus,
                         dx, ddelta, dA, dBt, dCt, dDskip, dh0,
                         B * i / threads, B * (i + 1) / threads,
                         parts + (size_t)i * (size_t)(D * N + D),
                         parts + (size_t)i * (size_t)(D * N + D) + D * N};
        jobs[i] = jb;
        if (threads == 1) {
            if (s6_bwd_worker(&jobs[0]))
                rc = -1;
            started = 0;
            break;
        }
        if (pthread_create(&tid[i], NULL, s6_bwd_worker, &jobs[i]) != 0) {
            rc = -1;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret)
            rc = -1;
    }
    for (int64_t k = 0; k < D * N; ++k) {
        double s = 0.0;
        for (int i = 0; i < threads; ++i)
            s += parts[(size_t)i * (size_t)(D * N + D) + k];
        dA[k] = s;
    }
    for (int64_t k = 0; k < D; ++k) {
        double s = 0.0;
        for (int i = 0; i < threads; ++i)
            s += parts[(size_t)i * (size_t)(D * N + D) + D * N + k];
        dDskip[k] = s;
    }
    free(jobs); free(tid); free(parts);
    return rc;
}
