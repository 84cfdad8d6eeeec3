/*
 * ssm_oracle.c -- fp64 CPU oracle for the selective-scan linear recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, strictly
 * sequential definition of what the GPU library computes.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header or constant with the CUDA path.
 *
 * Sources (web pages, by title and section):
 *   [P1] "scan output is different between sequential and parallel
 *        versions" (alxndrTL/mamba.py issue 26): the shape API of
 *        selective_scan / selective_scan_seq -- x, delta (Bs,L,ED),
 *        A (ED,N), B, C (Bs,L,N), D (ED) -> y (Bs,L,ED) -- and the
 *        sequential form selective_scan_seq that this file writes out.
 *   [P2] "Some questions of Bi-Mamba2 and Hydra" (Hprairie/Bi-Mamba2
 *        issue 1): the chunked scalar-decay scan's argument list
 *        (x, dt, A, B, C, chunk_size, D, ...) and the bidirectional
 *        reading: a forward and a backward SSM that share their weights,
 *        summed, plus the skip term D x counted once.
 *
 * The recurrence itself is not printed on the pages; the plainest reading
 * that they support (Mamba zero-order-hold discretisation) is used:
 *
 *   diagonal A, per (b, e, n):
 *     h_t[n] = exp(delta_t * A[e,n]) * h_{t-1}[n] + delta_t * B_t[n] * x_t
 *     y_t    = sum_n C_t[n] * h_t[n] + D[e] * x_t,          h_{-1} = 0
 *
 *   scalar A per head (SSD form), per (b, h), state H_t in R^{P x N}:
 *     H_t[p][n] = exp(dt_t * A_h) * H_{t-1}[p][n] + dt_t * x_t[p] * B_t[n]
 *     y_t[p]    = sum_n H_t[p][n] * C_t[n] + D_h * x_t[p],   H_{-1} = 0
 *
 *   bidirectional: y = F(x) + flip(F(flip(x))) + D x, where F is the SSD
 *   recurrence above without the D term and flip reverses the time axis
 *   of x, dt, B and C together.  D x is added once.
 *
 * Options of the chunked scan's argument list in [P2] (dt_bias,
 * dt_softplus, dt_limit, z, initial and final states), applied to both
 * scans with their plainest reading (the Mamba convention):
 *   delta <- delta + dt_bias[channel or head]          (if a bias is given)
 *   delta <- log(1 + exp(delta))                        (if dt_softplus)
 *   delta <- min(max(delta, dt_min), dt_max)            (if dt_limit)
 *   y     <- y * z / (1 + exp(-z))   (silu gate, after D x; if z is given)
 *   h_{-1} = h0 instead of 0; h_final = h_{L-1}        (if given / asked)
 * State I/O is defined for the single-direction scans only.
 *
 * Groups of B, C (ngroups in the chunked scan's interface): B, C have shape
 * (Bs, L, G, N) and head h reads group h / (H / G); G = 1 is one group
 * shared by all heads.
 *
 * Gradients (the backward passes [P2] names): reverse mode written out by
 * hand for the diagonal scan and for the SSD scan, the latter also with its
 * options (dz, ddt_bias and the initial state's gradient besides dx, ddt,
 * dA, dB, dC, dD).
 *
 * All arrays are dense row-major (last index fastest) fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* The delta (dt) seen by the recurrence, after the optional preprocessing. */
static double prep_delta(double d, const double *bias, int64_t k, int softplus, int limit,
                         double dmin, double dmax) {
    if (bias) d += bias[k];
    if (softplus) d = log1p(exp(d));
    if (limit) d = fmin(fmax(d, dmin), dmax);
    return d;
}

/* silu gate: z * sigmoid(z). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Diagonal selective scan, sequential over t for every (b, e) channel.
 * x, delta, y, z: (Bs, L, ED); A: (ED, N); B, C: (Bs, L, N); D, dt_bias:
 * (ED) or NULL; h0, h_final: (Bs, ED, N) or NULL.
 * Channels listed in [c_begin, c_end) of the flattened (b, e) index are
 * computed; the rest of y is left untouched (lets a caller time a sample).
 */
void oracle_diag_scan_ex_range(const double *x, const double *delta, const double *A,
                               const double *B, const double *C, const double *D,
                               double *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                               const double *dt_bias, int dt_softplus, int dt_limit,
                               double dt_min, double dt_max, const double *z,
                               const double *h0, double *h_final, int64_t c_begin,
                               int64_t c_end, int nthreads) {
    set_threads(nthreads);
    if (c_end > Bs * ED) c_end = Bs * ED;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = c_begin; c < c_end; ++c) {
        const int64_t b = c / ED, e = c % ED;
        double *h = (double *)calloc((size_t)N, sizeof(double));
        if (h0)
            for (int64_t n = 0; n < N; ++n) h[n] = h0[(b * ED + e) * N + n];
        for (int64_t t = 0; t < L; ++t) {
            const int64_t i = (b * L + t) * ED + e;   /* x, delta, y */
            const int64_t r = (b * L + t) * N;        /* B, C row     */
            const double dl = prep_delta(delta[i], dt_bias, e, dt_softplus, dt_limit, dt_min,
                                         dt_max);
            const double xv = x[i];
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(dl * A[e * N + n]);
                h[n] = a * h[n] + dl * B[r + n] * xv;
                acc += C[r + n] * h[n];
            }
            const double out = acc + (D ? D[e] * xv : 0.0);
            y[i] = z ? out * silu(z[i]) : out;
        }
        if (h_final)
            for (int64_t n = 0; n < N; ++n) h_final[(b * ED + e) * N + n] = h[n];
        free(h);
    }
}

void oracle_diag_scan_range(const double *x, const double *delta, const double *A,
                            const double *B, const double *C, const double *D, double *y,
                            int64_t Bs, int64_t L, int64_t ED, int64_t N, int64_t c_begin,
                            int64_t c_end, int nthreads) {
    oracle_diag_scan_ex_range(x, delta, A, B, C, D, y, Bs, L, ED, N, NULL, 0, 0, 0.0, 0.0, NULL,
                              NULL, NULL, c_begin, c_end, nthreads);
}

void oracle_diag_scan(const double *x, const double *delta, const double *A,
                      const double *B, const double *C, const double *D,
                      double *y, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                      int nthreads) {
    oracle_diag_scan_range(x, delta, A, B, C, D, y, Bs, L, ED, N, 0, Bs * ED,
                           nthreads);
}

/*
 * One direction of the SSD recurrence for a single (b, h), written into
 * y (accumulating).  `rev` = 0 walks t = 0..L-1; `rev` = 1 walks the
 * flipped sequence, i.e. t = L-1..0, which is F applied to flip(inputs)
 * and flipped back.  `dth` is this head's preprocessed dt, (L).
 * x, y: (Bs, L, H, P); B, C: (Bs, L, G, N), group g.  `state` (P x N) holds the
 * entering state on entry and the final state on return.
 */
static void ssd_one_direction(const double *x, const double *dth, double Ah,
                              const double *B, const double *C, double *y,
                              int64_t b, int64_t h, int64_t L, int64_t H,
                              int64_t P, int64_t N, int64_t G, int64_t g, int rev,
                              double *state) {
    for (int64_t k = 0; k < L; ++k) {
        const int64_t t = rev ? (L - 1 - k) : k;
        const double d = dth[t];
        const double a = exp(d * Ah);
        const double *xt = x + ((b * L + t) * H + h) * P;
        const double *Bt = B + ((b * L + t) * G + g) * N;
        const double *Ct = C + ((b * L + t) * G + g) * N;
        double *yt = y + ((b * L + t) * H + h) * P;
        for (int64_t p = 0; p < P; ++p) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double *s = state + p * N + n;
                *s = a * (*s) + d * xt[p] * Bt[n];
                acc += (*s) * Ct[n];
            }
            yt[p] += acc;
        }
    }
}

/*
 * Scalar-per-head (SSD) scan, optionally bidirectional, for the (b, h)
 * pairs in [u_begin, u_end) of the flattened index u = b * H + h.
 * x, y, z: (Bs, L, H, P); dt: (Bs, L, H); A_head, D, dt_bias: (H) (D and
 * dt_bias may be NULL); B, C: (Bs, L, G, N), G dividing H;
 * h0, h_final: (Bs, H, P, N) or NULL (single direction only).
 */
void oracle_ssd_scan_ex_range(const double *x, const double *dt, const double *A_head,
                              const double *B, const double *C, const double *D, double *y,
                              int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                              int64_t G, int bidirectional, const double *dt_bias, int dt_softplus,
                              int dt_limit, double dt_min, double dt_max, const double *z,
                              const double *h0, double *h_final, int64_t u_begin,
                              int64_t u_end, int nthreads) {
    set_threads(nthreads);
    if (u_end > Bs * H) u_end = Bs * H;
    if (bidirectional && (h0 || h_final)) return;   /* not defined */
    if (G < 1 || H % G != 0) return;                 /* heads split evenly into groups */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = u_begin; u < u_end; ++u) {
        const int64_t b = u / H, h = u % H;
        const int64_t g = h / (H / G);   /* this head's group of B, C */
        double *state = (double *)malloc((size_t)(P * N) * sizeof(double));
        /* this head's preprocessed dt */
        double *dtp = (double *)malloc((size_t)L * sizeof(double));
        for (int64_t t = 0; t < L; ++t)
            dtp[t] = prep_delta(dt[(b * L + t) * H + h], dt_bias, h, dt_softplus, dt_limit, dt_min,
                                dt_max);
        for (int64_t t = 0; t < L; ++t) {
            const int64_t o = ((b * L + t) * H + h) * P;
            for (int64_t p = 0; p < P; ++p)
                y[o + p] = D ? D[h] * x[o + p] : 0.0;
        }
        for (int64_t i = 0; i < P * N; ++i) state[i] = h0 ? h0[u * P * N + i] : 0.0;
        ssd_one_direction(x, dtp, A_head[h], B, C, y, b, h, L, H, P, N, G, g, 0, state);
        if (h_final)
            for (int64_t i = 0; i < P * N; ++i) h_final[u * P * N + i] = state[i];
        if (bidirectional) {
            memset(state, 0, (size_t)(P * N) * sizeof(double));
            ssd_one_direction(x, dtp, A_head[h], B, C, y, b, h, L, H, P, N, G, g, 1, state);
        }
        if (z) {
            for (int64_t t = 0; t < L; ++t) {
                const int64_t o = ((b * L + t) * H + h) * P;
                for (int64_t p = 0; p < P; ++p) y[o + p] *= silu(z[o + p]);
            }
        }
        free(dtp);
        free(state);
    }
}

void oracle_ssd_scan_range(const double *x, const double *dt,
                           const double *A_head, const double *B,
                           const double *C, const double *D, double *y,
                           int64_t Bs, int64_t L, int64_t H, int64_t P,
                           int64_t N, int bidirectional, int64_t u_begin,
                           int64_t u_end, int nthreads) {
    oracle_ssd_scan_ex_range(x, dt, A_head, B, C, D, y, Bs, L, H, P, N, 1, bidirectional, NULL, 0, 0,
                             0.0, 0.0, NULL, NULL, NULL, u_begin, u_end, nthreads);
}

void oracle_ssd_scan(const double *x, const double *dt, const double *A_head,
                     const double *B, const double *C, const double *D,
                     double *y, int64_t Bs, int64_t L, int64_t H, int64_t P,
                     int64_t N, int bidirectional, int nthreads) {
    oracle_ssd_scan_range(x, dt, A_head, B, C, D, y, Bs, L, H, P, N,
                          bidirectional, 0, Bs * H, nthreads);
}

/*
 * Gradients of the diagonal scan (reverse mode, written out by hand) for the
 * channels in [c_begin, c_end) of the flattened (b, e) index, given dy,
 * the gradient of the loss with respect to y.  With a_t[n] = exp(delta_t A[e,n])
 * the adjoint of the state obeys the reverse-time recurrence
 *   g_t[n] = dy_t C_t[n] + a_{t+1}[n] g_{t+1}[n],   g_L = 0,
 * and, with h_{t-1} the state entering step t,
 *   dx_t     = sum_n g_t[n] delta_t B_t[n] + D[e] dy_t
 *   ddelta_t = sum_n g_t[n] (A[e,n] a_t[n] h_{t-1}[n] + B_t[n] x_t)
 *   dA[e,n]  = sum_{b,t} g_t[n] delta_t a_t[n] h_{t-1}[n]
 *   dB_t[n]  = sum_e g_t[n] delta_t x_t,    dC_t[n] = sum_e dy_t h_t[n]
 *   dD[e]    = sum_{b,t} dy_t x_t.
 * dx, ddelta: (Bs, L, ED) overwritten for the channels done; dA (ED, N),
 * dB, dC (Bs, L, N) and dD (ED) are ACCUMULATED into (the caller zeroes
 * them); dD may be NULL.
 */
/* The diagonal scan's gradients for the channels [c_begin, c_end), from
 * initial states h0 (Bs, ED, N) or zero; dh0 (same shape, optional) gets the
 * gradient with respect to h0: a_0 g_0, what g holds when the walk ends. */
static void diag_bwd_core(const double *x, const double *delta, const double *A,
                          const double *B, const double *C, const double *D, const double *dy,
                          double *dx, double *ddelta, double *dA, double *dB, double *dC,
                          double *dD, int64_t Bs, int64_t L, int64_t ED, int64_t N,
                          int64_t c_begin, int64_t c_end, const double *h0, double *dh0) {
    if (c_end > Bs * ED) c_end = Bs * ED;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = c_begin; c < c_end; ++c) {
        const int64_t b = c / ED, e = c % ED;
        /* forward: the states h_t (t = -1 .. L-1), row t + 1 of hist */
        double *hist = (double *)calloc((size_t)((L + 1) * N), sizeof(double));
        if (h0)
            for (int64_t n = 0; n < N; ++n) hist[n] = h0[c * N + n];
        double *g = (double *)calloc((size_t)N, sizeof(double));
        double *lA = (double *)calloc((size_t)N, sizeof(double));
        double *lB = (double *)calloc((size_t)(L * N), sizeof(double));
        double *lC = (double *)calloc((size_t)(L * N), sizeof(double));
        double lD = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const int64_t i = (b * L + t) * ED + e, r = (b * L + t) * N;
            for (int64_t n = 0; n < N; ++n)
                hist[(t + 1) * N + n] = exp(delta[i] * A[e * N + n]) * hist[t * N + n] +
                                        delta[i] * B[r + n] * x[i];
        }
        /* reverse */
        for (int64_t t = L - 1; t >= 0; --t) {
            const int64_t i = (b * L + t) * ED + e, r = (b * L + t) * N;
            const double dl = delta[i], xv = x[i], gy = dy[i];
            double sdx = 0.0, sdd = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(A[e * N + n] * dl);
                const double hprev = hist[t * N + n];
                g[n] += gy * C[r + n];                 /* g now holds g_t[n] */
                sdx += g[n] * dl * B[r + n];
                sdd += g[n] * (A[e * N + n] * a * hprev + B[r + n] * xv);
                lA[n] += g[n] * dl * a * hprev;
                lB[t * N + n] += g[n] * dl * xv;
                lC[t * N + n] += gy * hist[(t + 1) * N + n];
                g[n] *= a;                             /* a_t g_t, carried to step t - 1 */
            }
            dx[i] = sdx + (D ? D[e] * gy : 0.0);
            ddelta[i] = sdd;
            lD += gy * xv;
        }
        if (dh0)
            for (int64_t n = 0; n < N; ++n) dh0[c * N + n] = g[n];
#pragma omp critical
        {
            for (int64_t n = 0; n < N; ++n) dA[e * N + n] += lA[n];
            for (int64_t k = 0; k < L * N; ++k) {
                dB[b * L * N + k] += lB[k];
                dC[b * L * N + k] += lC[k];
            }
            if (dD) dD[e] += lD;
        }
        free(hist);
        free(g);
        free(lA);
        free(lB);
        free(lC);
    }
}

void oracle_diag_scan_bwd_range(const double *x, const double *delta, const double *A,
                                const double *B, const double *C, const double *D,
                                const double *dy, double *dx, double *ddelta, double *dA,
                                double *dB, double *dC, double *dD, int64_t Bs, int64_t L,
                                int64_t ED, int64_t N, int64_t c_begin, int64_t c_end,
                                int nthreads) {
    set_threads(nthreads);
    diag_bwd_core(x, delta, A, B, C, D, dy, dx, ddelta, dA, dB, dC, dD, Bs, L, ED, N, c_begin,
                  c_end, NULL, NULL);
}

/*
 * Gradients of the diagonal scan with its options, by the same chain rule
 * as oracle_ssd_scan_bwd_ex: with v = delta + dt_bias[e], s = softplus(v)
 * (or v), delta_seen = clamp(s) (or s), u = scan(delta_seen) + D x and
 * y = u silu(z) (or u); g = dy silu(z) enters the plain gradients (run from
 * h0), dz = dy u silu'(z), ddelta = d delta_seen * [lo < s < hi] * sig(v),
 * ddt_bias[e] = sum over (b, t) of ddelta, dh0 = the gradient of h0.
 * delta: (Bs, L, ED) before the preprocessing; z, dz like x; h0, dh0
 * (Bs, ED, N).  Outputs are overwritten; dz, ddt_bias, dh0 may be NULL.
 */
void oracle_diag_scan_bwd_ex(const double *x, const double *delta, const double *A,
                             const double *B, const double *C, const double *D,
                             const double *dy, double *dx, double *ddelta, double *dA,
                             double *dB, double *dC, double *dD, int64_t Bs, int64_t L,
                             int64_t ED, int64_t N, const double *dt_bias, int dt_softplus,
                             int dt_limit, double dt_min, double dt_max, const double *z,
                             const double *h0, double *dz, double *ddt_bias, double *dh0,
                             int nthreads) {
    set_threads(nthreads);
    const int64_t nx = Bs * L * ED;
    double *dse = (double *)malloc((size_t)nx * sizeof(double));
    double *chain = (double *)malloc((size_t)nx * sizeof(double));
    double *g = (double *)malloc((size_t)nx * sizeof(double));
    for (int64_t i = 0; i < nx; ++i) {
        const double w = delta[i] + (dt_bias ? dt_bias[i % ED] : 0.0);
        double sv = w, fac = 1.0;
        if (dt_softplus) {
            sv = log1p(exp(w));
            fac = 1.0 / (1.0 + exp(-w));            /* softplus' = sigmoid */
        }
        if (dt_limit) {
            if (sv < dt_min || sv > dt_max) fac = 0.0;  /* clamped: no gradient */
            sv = fmin(fmax(sv, dt_min), dt_max);
        }
        dse[i] = sv;
        chain[i] = fac;
    }
    if (z) {
        double *u = (double *)malloc((size_t)nx * sizeof(double));
        oracle_diag_scan_ex_range(x, dse, A, B, C, D, u, Bs, L, ED, N, NULL, 0, 0, 0.0, 0.0,
                                  NULL, h0, NULL, 0, Bs * ED, nthreads);
        for (int64_t i = 0; i < nx; ++i) {
            const double sgm = 1.0 / (1.0 + exp(-z[i]));
            g[i] = dy[i] * z[i] * sgm;
            if (dz) dz[i] = dy[i] * u[i] * sgm * (1.0 + z[i] * (1.0 - sgm));  /* silu' */
        }
        free(u);
    } else {
        memcpy(g, dy, (size_t)nx * sizeof(double));
    }
    memset(dA, 0, (size_t)(ED * N) * sizeof(double));
    memset(dB, 0, (size_t)(Bs * L * N) * sizeof(double));
    memset(dC, 0, (size_t)(Bs * L * N) * sizeof(double));
    if (dD) memset(dD, 0, (size_t)ED * sizeof(double));
    diag_bwd_core(x, dse, A, B, C, D, g, dx, ddelta, dA, dB, dC, dD, Bs, L, ED, N, 0, Bs * ED, h0,
                  dh0);
    if (ddt_bias) memset(ddt_bias, 0, (size_t)ED * sizeof(double));
    for (int64_t i = 0; i < nx; ++i) {
        ddelta[i] *= chain[i];                 /* through the clamp and the softplus */
        if (ddt_bias) ddt_bias[i % ED] += ddelta[i];
    }
    free(dse);
    free(chain);
    free(g);
}

/* Gradients of the chunked scalar-decay scan (the SSD form above) for an
 * upstream gradient dy of y, written out by hand in reverse mode -- the
 * quantities the chunked backward pass named in "Some questions of Bi-Mamba2
 * and Hydra" (Bi-Mamba2 issue 1) returns: dx, ddt, dA, dB, dC, dD.  Per
 * (b, h) and direction, walking k = 0 .. L-1 over t = k (forward) or
 * t = L-1-k (reversed), with H_k the P x N state after walk step k and
 * a_k = exp(dt_t A_h):
 *   H_k = a_k H_{k-1} + dt_t x_t B_t^T,   y_t += H_k C_t   (+ D_h x_t once)
 * the adjoint of H_k is
 *   Gb_k = dy_t C_t^T + a_{k+1} Gb_{k+1},   Gb_L = 0,
 * and
 *   dx_t[p]   += dt_t sum_n Gb_k[p,n] B_t[n]          (+ D_h dy_t[p] once)
 *   dB_t[n]   += dt_t sum_p Gb_k[p,n] x_t[p]          (summed over the heads of a group)
 *   dC_t[n]   += sum_p dy_t[p] H_k[p,n]               (likewise)
 *   ddt_t     += sum_{p,n} Gb_k[p,n] (x_t[p] B_t[n] + A_h a_k H_{k-1}[p,n])
 *   dA_h      += sum_k dt_t a_k sum_{p,n} Gb_k[p,n] H_{k-1}[p,n]
 *   dD_h      += sum_t dy_t . x_t                      (once).
 * B, C, dB, dC: (Bs, L, G, N), head h reads group h / (H / G).  All outputs
 * are ACCUMULATED into (the caller zeroes them); dD may be NULL.  The loop
 * over batch rows is the parallel one (a batch row's heads share its dB, dC).
 * With an initial state H_{-1} = init (P x N, or NULL for zero), the walk
 * starts from it, and the gradient of the loss with respect to it is
 * a_0 Gb_0 -- what gb holds when the reverse walk ends (copied to d_init).
 */
static void ssd_bwd_one_direction(const double *x, const double *dt, double Ah,
                                  const double *B, const double *C, const double *dy,
                                  double *dx, double *ddt, double *dAh, double *dB, double *dC,
                                  int64_t b, int64_t h, int64_t L, int64_t H, int64_t P,
                                  int64_t N, int64_t G, int64_t g, int rev, double *hist,
                                  double *gb, const double *init, double *d_init) {
    const int64_t PN = P * N;
    /* forward: hist row k + 1 holds H_k; row 0 is the initial state */
    for (int64_t i = 0; i < PN; ++i) hist[i] = init ? init[i] : 0.0;
    for (int64_t k = 0; k < L; ++k) {
        const int64_t t = rev ? L - 1 - k : k;
        const double dtv = dt[(b * L + t) * H + h], a = exp(dtv * Ah);
        const double *xr = x + ((b * L + t) * H + h) * P;
        const double *br = B + ((b * L + t) * G + g) * N;
        for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n)
                hist[(k + 1) * PN + p * N + n] = a * hist[k * PN + p * N + n] + dtv * xr[p] * br[n];
    }
    /* reverse */
    for (int64_t i = 0; i < PN; ++i) gb[i] = 0.0;
    for (int64_t k = L - 1; k >= 0; --k) {
        const int64_t t = rev ? L - 1 - k : k;
        const double dtv = dt[(b * L + t) * H + h], a = exp(dtv * Ah);
        const double *xr = x + ((b * L + t) * H + h) * P;
        const double *gy = dy + ((b * L + t) * H + h) * P;
        const double *br = B + ((b * L + t) * G + g) * N;
        const double *cr = C + ((b * L + t) * G + g) * N;
        double *dxr = dx + ((b * L + t) * H + h) * P;
        double *dbr = dB + ((b * L + t) * G + g) * N;
        double *dcr = dC + ((b * L + t) * G + g) * N;
        const double *hk = hist + (k + 1) * PN, *hprev = hist + k * PN;
        double sdt = 0.0, sda = 0.0;
        for (int64_t p = 0; p < P; ++p) {
            double sx = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double *gpn = gb + p * N + n;
                *gpn += gy[p] * cr[n];                 /* Gb_k */
                sx += *gpn * br[n];
                dbr[n] += dtv * *gpn * xr[p];
                dcr[n] += gy[p] * hk[p * N + n];
                sdt += *gpn * xr[p] * br[n];
                sda += *gpn * hprev[p * N + n];
                *gpn *= a;                             /* a_k Gb_k, carried to step k - 1 */
            }
            dxr[p] += dtv * sx;
        }
        ddt[(b * L + t) * H + h] += sdt + Ah * a * sda;
        *dAh += dtv * a * sda;
    }
    if (d_init)
        for (int64_t i = 0; i < PN; ++i) d_init[i] = gb[i];
}

/* The plain scan's gradients, from an initial state h0 (Bs, H, P, N) or
 * zero, with dh0 (same shape) the gradient with respect to it when given. */
static void ssd_bwd_core(const double *x, const double *dt, const double *A_head,
                         const double *B, const double *C, const double *D, const double *dy,
                         double *dx, double *ddt, double *dA, double *dB, double *dC,
                         double *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                         int64_t G, int bidirectional, const double *h0, double *dh0) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < Bs; ++b) {
        double *hist = (double *)malloc((size_t)((L + 1) * P * N) * sizeof(double));
        double *gb = (double *)malloc((size_t)(P * N) * sizeof(double));
        double *lA = (double *)calloc((size_t)H, sizeof(double));
        double *lD = (double *)calloc((size_t)H, sizeof(double));
        for (int64_t h = 0; h < H; ++h) {
            const int64_t hg = h / (H / G);   /* the head's group of B, C */
            const int64_t u = b * H + h;
            for (int dir = 0; dir < (bidirectional ? 2 : 1); ++dir)
                ssd_bwd_one_direction(x, dt, A_head[h], B, C, dy, dx, ddt, &lA[h], dB, dC, b, h,
                                      L, H, P, N, G, hg, dir, hist, gb,
                                      (dir == 0 && h0) ? h0 + u * P * N : NULL,
                                      (dir == 0 && dh0) ? dh0 + u * P * N : NULL);
            for (int64_t t = 0; t < L; ++t)
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t i = ((b * L + t) * H + h) * P + p;
                    if (D) dx[i] += D[h] * dy[i];
                    lD[h] += dy[i] * x[i];
                }
        }
#pragma omp critical
        {
            for (int64_t h = 0; h < H; ++h) {
                dA[h] += lA[h];
                if (dD) dD[h] += lD[h];
            }
        }
        free(hist);
        free(gb);
        free(lA);
        free(lD);
    }
}

void oracle_ssd_scan_bwd(const double *x, const double *dt, const double *A_head,
                         const double *B, const double *C, const double *D, const double *dy,
                         double *dx, double *ddt, double *dA, double *dB, double *dC,
                         double *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                         int64_t G, int bidirectional, int nthreads) {
    set_threads(nthreads);
    if (G < 1 || H % G != 0) return;
    ssd_bwd_core(x, dt, A_head, B, C, D, dy, dx, ddt, dA, dB, dC, dD, Bs, L, H, P, N, G,
                 bidirectional, NULL, NULL);
}

/*
 * Gradients of the scan with its options ("Some questions of Bi-Mamba2 and
 * Hydra": the chunked backward returns dz, ddt_bias and the initial
 * states' gradient besides dx, ddt, dA, dB, dC, dD).  With
 *   v = dt + dt_bias,  s = softplus(v) (or v),  dte = clamp(s, lo, hi) (or s),
 *   u = scan(dte) + D x,  y = u * silu(z) (or u),
 * the chain rule gives, with g = dy * silu(z):
 *   dz    = dy * u * silu'(z),   silu'(z) = sig(z) (1 + z (1 - sig(z)))
 *   (dx, d dte, dA, dB, dC, dD, dh0) = the plain scan's gradients for g,
 *                                        run from h0
 *   ddt   = d dte * [lo < s < hi] * sig(v)   (each factor if its option is on)
 *   ddt_bias[h] = sum over (b, t) of ddt.
 * dt: (Bs, L, H) before the preprocessing; z, dz: like x; h0, dh0:
 * (Bs, H, P, N), single direction only.  Outputs are overwritten; dz,
 * ddt_bias, dh0 may be NULL when the matching option is off.
 */
void oracle_ssd_scan_bwd_ex(const double *x, const double *dt, const double *A_head,
                            const double *B, const double *C, const double *D, const double *dy,
                            double *dx, double *ddt, double *dA, double *dB, double *dC,
                            double *dD, int64_t Bs, int64_t L, int64_t H, int64_t P, int64_t N,
                            int64_t G, int bidirectional, const double *dt_bias, int dt_softplus,
                            int dt_limit, double dt_min, double dt_max, const double *z,
                            const double *h0, double *dz, double *ddt_bias, double *dh0,
                            int nthreads) {
    set_threads(nthreads);
    if (G < 1 || H % G != 0 || (bidirectional && (h0 || dh0))) return;
    const int64_t nt = Bs * L * H, nx = nt * P;
    double *dte = (double *)malloc((size_t)nt * sizeof(double));
    double *chain = (double *)malloc((size_t)nt * sizeof(double));
    double *g = (double *)malloc((size_t)nx * sizeof(double));
    for (int64_t i = 0; i < nt; ++i) {
        const double v = dt[i] + (dt_bias ? dt_bias[i % H] : 0.0);
        double s = v, f = 1.0;
        if (dt_softplus) {
            s = log1p(exp(v));
            f = 1.0 / (1.0 + exp(-v));
        }
        if (dt_limit) {
            if (s < dt_min || s > dt_max) f = 0.0;
            s = fmin(fmax(s, dt_min), dt_max);
        }
        dte[i] = s;
        chain[i] = f;
    }
    if (z) {
        /* the ungated output u, from the same preprocessed dt and h0 */
        double *u = (double *)malloc((size_t)nx * sizeof(double));
        oracle_ssd_scan_ex_range(x, dte, A_head, B, C, D, u, Bs, L, H, P, N, G, bidirectional,
                                 NULL, 0, 0, 0.0, 0.0, NULL, h0, NULL, 0, Bs * H, nthreads);
        for (int64_t i = 0; i < nx; ++i) {
            const double sg = 1.0 / (1.0 + exp(-z[i]));
            g[i] = dy[i] * z[i] * sg;
            if (dz) dz[i] = dy[i] * u[i] * sg * (1.0 + z[i] * (1.0 - sg));
        }
        free(u);
    } else {
        memcpy(g, dy, (size_t)nx * sizeof(double));
    }
    memset(dx, 0, (size_t)nx * sizeof(double));
    memset(ddt, 0, (size_t)nt * sizeof(double));
    memset(dA, 0, (size_t)H * sizeof(double));
    memset(dB, 0, (size_t)(Bs * L * G * N) * sizeof(double));
    memset(dC, 0, (size_t)(Bs * L * G * N) * sizeof(double));
    if (dD) memset(dD, 0, (size_t)H * sizeof(double));
    ssd_bwd_core(x, dte, A_head, B, C, D, g, dx, ddt, dA, dB, dC, dD, Bs, L, H, P, N, G,
                 bidirectional, h0, dh0);
    if (ddt_bias) memset(ddt_bias, 0, (size_t)H * sizeof(double));
    for (int64_t i = 0; i < nt; ++i) {
        ddt[i] *= chain[i];                    /* through the clamp and the softplus */
        if (ddt_bias) ddt_bias[i % H] += ddt[i];
    }
    free(dte);
    free(chain);
    free(g);
}
