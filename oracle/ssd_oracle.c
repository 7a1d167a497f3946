/*
 * fp64 CPU oracle of the SSD selective-state recurrence.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may build, load or call this
 * file.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (page "Mamba-2架构与LaCT并行计算技术解析", §1.1, the state
 * equations; zero initial state per the note under them; heads independent
 * per §1.2):
 *
 *     delta_t = softplus(raw_t + delta_init)
 *     H_t     = exp(-delta_t) * H_{t-1} + delta_t * x_t B_t^T      (H is P x N)
 *     y_t     = H_t C_t
 *
 * one head and one sequence at a time, token by token, with no chunking: the
 * chunked (semiseparable) evaluation of page "长序列 Mamba 多卡训练算力和显存
 * 怎么同时省" §一 is an exact reformulation of this loop, so the loop itself is
 * the definition the GPU path is held to.  Packed sequences (the cu_seqlens
 * boundaries of that page's §三) restart from their own initial state.
 *
 * The page writes the state as B_t^T x_t and the output as C_t H_t (state
 * N x P); the P x N orientation used here is its transpose and gives the same
 * y.  Heads map to B/C groups as h / (H / G).
 *
 * The backward pass is plain reverse-mode differentiation of the same loop:
 * with G_t = dL/dH_t,
 *     G_t       = dy_t C_t^T + exp(-delta_{t+1}) G_{t+1}   (G after the end = dL/dH_final)
 *     dC_t     += H_t^T dy_t                  (summed over the heads of a group)
 *     dx_t      = delta_t G_t B_t
 *     dB_t     += delta_t G_t^T x_t           (summed over the heads of a group)
 *     ddelta_t  = <G_t, x_t B_t^T> - exp(-delta_t) <G_t, H_{t-1}>
 *     draw_t    = ddelta_t * sigmoid(raw_t + delta_init)
 *     dH_init   = exp(-delta_0) G_0
 * The forward states are recomputed from checkpoints kept every CKPT tokens
 * (the per-segment recomputation idea of that page's §4.1).
 *
 * Layouts (row-major, tokens packed back to back):
 *   x, y, dy, dx  [T][H][P]      raw, draw  [T][H]
 *   Bm, Cm, dB, dC [T][G][N]     h0, hT, dhT, dh0  [nseq][H][P][N]
 *   cu            [nseq + 1], cu[0] = 0, cu[nseq] = T, non-decreasing
 * Every function returns 0 on success and a negative code on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 256

static double softplus(double z) {
    /* log(1 + e^z) without overflow */
    return (z > 0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

static double sigmoid(double z) {
    if (z >= 0) return 1.0 / (1.0 + exp(-z));
    double e = exp(z);
    return e / (1.0 + e);
}

static int check_args(int64_t T, int H, int P, int N, int G, int nseq, const int64_t* cu) {
    if (T < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || nseq <= 0 || !cu) return -1;
    if (H % G) return -2;
    if (cu[0] != 0 || cu[nseq] != T) return -3;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return -4;
    return 0;
}

int ssd_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One head of one sequence, forward. */
static void fwd_head(int64_t t0, int64_t len, int h, int H, int P, int N, int G,
                     const double* x, const double* raw, const double* Bm, const double* Cm,
                     double delta_init, const double* h0, double* y, double* hT, double* S) {
    const int g = h / (H / G);
    if (h0) memcpy(S, h0, sizeof(double) * P * N);
    else memset(S, 0, sizeof(double) * P * N);
    for (int64_t t = t0; t < t0 + len; ++t) {
        const double d = softplus(raw[t * H + h] + delta_init);
        const double a = exp(-d);
        const double* xt = x + (t * H + h) * P;
        const double* bt = Bm + (t * G + g) * N;
        const double* ct = Cm + (t * G + g) * N;
        double* yt = y + (t * H + h) * P;
        for (int p = 0; p < P; ++p) {
            double* row = S + (int64_t)p * N;
            const double dx = d * xt[p];
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                row[n] = a * row[n] + dx * bt[n];
                acc += row[n] * ct[n];
            }
            yt[p] = acc;
        }
    }
    if (hT) memcpy(hT, S, sizeof(double) * P * N);
}

int ssd_oracle_forward(int64_t T, int H, int P, int N, int G, int nseq, const int64_t* cu,
                       const double* x, const double* raw, const double* Bm, const double* Cm,
                       double delta_init, const double* h0, double* y, double* hT, int nthreads) {
    int rc = check_args(T, H, P, N, G, nseq, cu);
    if (rc) return rc;
    if (!x || !raw || !Bm || !Cm || !y) return -5;
    const int64_t npairs = (int64_t)nseq * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* S = (double*)malloc(sizeof(double) * P * N);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t k = 0; k < npairs; ++k) {
            const int s = (int)(k / H), h = (int)(k % H);
            const int64_t off = ((int64_t)s * H + h) * P * N;
            fwd_head(cu[s], cu[s + 1] - cu[s], h, H, P, N, G, x, raw, Bm, Cm, delta_init,
                     h0 ? h0 + off : NULL, y, hT ? hT + off : NULL, S);
        }
        free(S);
    }
    return 0;
}

/* One head of one sequence, backward.  dB/dC contributions go to the
 * caller's (thread-private) accumulators dBacc/dCacc [T][G][N]. */
static void bwd_head(int64_t t0, int64_t len, int h, int H, int P, int N, int G,
                     const double* x, const double* raw, const double* Bm, const double* Cm,
                     double delta_init, const double* h0, const double* dy, const double* dhT,
                     double* dx, double* draw, double* dBacc, double* dCacc, double* dh0,
                     double* ckpt, double* seg, double* Gs, double* gb) {
    const int g = h / (H / G);
    const int64_t PN = (int64_t)P * N;
    /* forward sweep: keep the state entering every CKPT-token block */
    double* cur = seg; /* scratch, first slot */
    if (h0) memcpy(cur, h0, sizeof(double) * PN);
    else memset(cur, 0, sizeof(double) * PN);
    for (int64_t i = 0; i < len; ++i) {
        const int64_t t = t0 + i;
        if (i % CKPT == 0) memcpy(ckpt + (i / CKPT) * PN, cur, sizeof(double) * PN);
        const double d = softplus(raw[t * H + h] + delta_init);
        const double a = exp(-d);
        const double* xt = x + (t * H + h) * P;
        const double* bt = Bm + (t * G + g) * N;
        for (int p = 0; p < P; ++p)
            for (int n = 0; n < N; ++n)
                cur[p * N + n] = a * cur[p * N + n] + d * xt[p] * bt[n];
    }
    /* reverse sweep */
    if (dhT) memcpy(Gs, dhT, sizeof(double) * PN);
    else memset(Gs, 0, sizeof(double) * PN);
    const int64_t nblk = (len + CKPT - 1) / CKPT;
    for (int64_t b = nblk - 1; b >= 0; --b) {
        const int64_t ia = b * CKPT;
        const int64_t ib = (ia + CKPT < len) ? ia + CKPT : len;
        /* seg[j] = state before token ia + j; seg[ib - ia] = state after ib - 1 */
        memcpy(seg, ckpt + b * PN, sizeof(double) * PN);
        for (int64_t i = ia; i < ib; ++i) {
            const int64_t t = t0 + i;
            const double d = softplus(raw[t * H + h] + delta_init);
            const double a = exp(-d);
            const double* xt = x + (t * H + h) * P;
            const double* bt = Bm + (t * G + g) * N;
            const double* prv = seg + (i - ia) * PN;
            double* nxt = seg + (i - ia + 1) * PN;
            for (int p = 0; p < P; ++p)
                for (int n = 0; n < N; ++n)
                    nxt[p * N + n] = a * prv[p * N + n] + d * xt[p] * bt[n];
        }
        for (int64_t i = ib - 1; i >= ia; --i) {
            const int64_t t = t0 + i;
            const double z = raw[t * H + h] + delta_init;
            const double d = softplus(z);
            const double a = exp(-d);
            const double* xt = x + (t * H + h) * P;
            const double* bt = Bm + (t * G + g) * N;
            const double* ct = Cm + (t * G + g) * N;
            const double* dyt = dy + (t * H + h) * P;
            const double* Hprev = seg + (i - ia) * PN;
            const double* Ht = seg + (i - ia + 1) * PN;
            double* dBt = dBacc + (t * G + g) * N;
            double* dCt = dCacc + (t * G + g) * N;
            /* G_t = dy_t C_t^T + (carried exp(-delta_{t+1}) G_{t+1}) */
            for (int p = 0; p < P; ++p)
                for (int n = 0; n < N; ++n) Gs[p * N + n] += dyt[p] * ct[n];
            /* dC_t += H_t^T dy_t ; dB_t += delta_t G_t^T x_t */
            for (int p = 0; p < P; ++p)
                for (int n = 0; n < N; ++n) {
                    dCt[n] += Ht[p * N + n] * dyt[p];
                    dBt[n] += d * Gs[p * N + n] * xt[p];
                }
            /* dx_t = delta_t G_t B_t ; <G_t, x_t B_t^T> = x_t . (G_t B_t) */
            double xgb = 0.0, gh = 0.0;
            for (int p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int n = 0; n < N; ++n) {
                    acc += Gs[p * N + n] * bt[n];
                    gh += Gs[p * N + n] * Hprev[p * N + n];
                }
                gb[p] = acc;
                xgb += xt[p] * acc;
            }
            for (int p = 0; p < P; ++p) dx[(t * H + h) * P + p] = d * gb[p];
            const double ddelta = xgb - a * gh;
            draw[t * H + h] = ddelta * sigmoid(z);
            for (int64_t k = 0; k < PN; ++k) Gs[k] *= a;
        }
    }
    if (dh0) memcpy(dh0, Gs, sizeof(double) * PN);
}

int ssd_oracle_backward(int64_t T, int H, int P, int N, int G, int nseq, const int64_t* cu,
                        const double* x, const double* raw, const double* Bm, const double* Cm,
                        double delta_init, const double* h0, const double* dy, const double* dhT,
                        double* dx, double* draw, double* dB, double* dC, double* dh0,
                        int nthreads) {
    int rc = check_args(T, H, P, N, G, nseq, cu);
    if (rc) return rc;
    if (!x || !raw || !Bm || !Cm || !dy || !dx || !draw || !dB || !dC) return -5;
    int64_t maxlen = 0;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] - cu[s] > maxlen) maxlen = cu[s + 1] - cu[s];
    const int64_t PN = (int64_t)P * N;
    const int64_t nBC = T * G * N;
    memset(dB, 0, sizeof(double) * nBC);
    memset(dC, 0, sizeof(double) * nBC);
    const int64_t npairs = (int64_t)nseq * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* ckpt = (double*)malloc(sizeof(double) * PN * ((maxlen + CKPT - 1) / CKPT + 1));
        double* seg = (double*)malloc(sizeof(double) * PN * (CKPT + 1));
        double* Gs = (double*)malloc(sizeof(double) * PN);
        double* gb = (double*)malloc(sizeof(double) * P);
        double* dBacc = (double*)calloc((size_t)nBC, sizeof(double));
        double* dCacc = (double*)calloc((size_t)nBC, sizeof(double));
        if (!ckpt || !seg || !Gs || !gb || !dBacc || !dCacc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp barrier
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t k = 0; k < npairs; ++k) {
            if (failed) continue;
            const int s = (int)(k / H), h = (int)(k % H);
            const int64_t off = ((int64_t)s * H + h) * PN;
            bwd_head(cu[s], cu[s + 1] - cu[s], h, H, P, N, G, x, raw, Bm, Cm, delta_init,
                     h0 ? h0 + off : NULL, dy, dhT ? dhT + off : NULL, dx, draw, dBacc, dCacc,
                     dh0 ? dh0 + off : NULL, ckpt, seg, Gs, gb);
        }
#ifdef _OPENMP
#pragma omp critical
#endif
        {
            if (dBacc && dCacc)
                for (int64_t i = 0; i < nBC; ++i) {
                    dB[i] += dBacc[i];
                    dC[i] += dCacc[i];
                }
        }
        free(ckpt); free(seg); free(Gs); free(gb); free(dBacc); free(dCacc);
    }
    return failed ? -6 : 0;
}

/* softplus in fp64, exported so the tests can pin it to the page's printed
 * value for delta_init = -4.6. */
double ssd_oracle_softplus(double z) { return softplus(z); }
