/*
 * oracle.c -- plain, slow, fp64 CPU oracle of the selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (per (batch b, channel d) row, in time order):
 *
 *   delta_t = softplus(delta_raw_t + bias_d)      (or the raw sum when
 *                                                   softplus == 0)
 *   for every state n:
 *     h_n <- exp(delta_t * A_dn) * h_n + delta_t * B_bnt * u_t
 *   y_t   = sum_n C_bnt * h_n + D_d * u_t
 *   out_t = y_t * z_t * sigmoid(z_t)               (no gate when z is NULL)
 *
 * Source of the recurrence: the scan loop quoted in the Hacker News thread
 * on the "Triển khai Mamba trong một tệp PyTorch" page (vi.news.hada.io,
 * topic 12448) and its Korean original "PyTorch 한 파일에서의 Mamba 구현"
 * (news.hada.io, topic 12448): state = deltaA[:, :, i] * state +
 * deltaB_u[:, :, i]; y = einsum(state, C[:, i, :], 'b d_in n, b n -> b d_in').
 * The pages name "deltaA" and "deltaB_u" without printing them; we read
 * them as deltaA = exp(delta * A) (zero-order hold) and deltaB_u =
 * delta * B * u (Euler), the plainest reading of the names.  Softplus,
 * the D skip and the silu gate follow the selective SSM layer described
 * on the "Mamba SSM 架构" page (toolpotion.ai) and the "Mamba 7.9.1"
 * article (lpnh.cn, section 2.2: parameters become functions of the
 * input).  Initial state is zero (the quoted loop starts from a zero
 * state).  Layouts: u/delta/z/out [Bsz][Dch][L]; B/C [Bsz][N][L];
 * A [Dch][N]; D, delta_bias [Dch]; h [Bsz][Dch][N].
 *
 * Backward (oracle_scan_bwd) stores the whole fp64 state trajectory of a
 * row and applies the chain rule to the loop above, walking time in
 * reverse (the adjoint of a forward linear recurrence is a reverse-time
 * recurrence; cf. the "mamba.py" page (gittoolsai.com), performance TODO
 * list: the backward of its parallel scan runs the same scan on
 * time-flipped arrays).
 *
 * oracle_step is the one-token recurrent ("RNN form") update used for
 * decoding ("mamba.py" page, update of 2024-01-17 on the step function;
 * "Mamba 7.9.1" article, section 6.2 on streaming with a carried state).
 *
 * oracle_scan_fwd_blelloch evaluates the same scan in Blelloch's
 * up-sweep/down-sweep order over the pairs (a_t, b_t) with the operator
 * (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) ("mamba.py" page, overview:
 * pscan.py is a Blelloch parallel scan), so that the sequential oracle can
 * be checked against an independent evaluation order.
 *
 * Parallelism: rows are spread over host threads (pthreads); nothing else.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef int64_t i64;

static double softplus_or_raw(double x, int softplus) {
    if (!softplus) return x;
    /* softplus(x) = log(1 + e^x), written in the overflow-free form */
    return fmax(x, 0.0) + log1p(exp(-fabs(x)));
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------ */
/* thread pool over rows                                               */
/* ------------------------------------------------------------------ */

typedef void (*row_fn)(void* ctx, i64 row, int tid);

typedef struct {
    row_fn fn;
    void* ctx;
    i64 nrows;
    int tid;
    int nthreads;
} job_t;

static void* job_main(void* p) {
    job_t* j = (job_t*)p;
    for (i64 r = j->tid; r < j->nrows; r += j->nthreads) j->fn(j->ctx, r, j->tid);
    return NULL;
}

static void run_rows(row_fn fn, void* ctx, i64 nrows, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || nrows <= 1) {
        for (i64 r = 0; r < nrows; ++r) fn(ctx, r, 0);
        return;
    }
    pthread_t th[256];
    job_t jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (job_t){fn, ctx, nrows, t, nthreads};
        pthread_create(&th[t], NULL, job_main, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* forward: sequential recurrence                                      */
/* ------------------------------------------------------------------ */

typedef struct {
    const double *u, *delta, *A, *B, *C, *D, *z, *bias, *h0;
    int softplus;
    i64 Bsz, Dch, L, N;
    double *out, *h_last;
} fwd_ctx;

static void fwd_row(void* p, i64 row, int tid) {
    (void)tid;
    fwd_ctx* c = (fwd_ctx*)p;
    const i64 L = c->L, N = c->N, Dch = c->Dch;
    const i64 b = row / Dch, d = row % Dch;
    const double* u = c->u + row * L;
    const double* dr = c->delta + row * L;
    const double* z = c->z ? c->z + row * L : NULL;
    const double* Bb = c->B + b * N * L;
    const double* Cb = c->C + b * N * L;
    const double* A = c->A + d * N;
    const double Dd = c->D ? c->D[d] : 0.0;
    const double bias = c->bias ? c->bias[d] : 0.0;
    double h[1024];
    for (i64 n = 0; n < N; ++n) h[n] = c->h0 ? c->h0[row * N + n] : 0.0;
    for (i64 t = 0; t < L; ++t) {
        const double dt = softplus_or_raw(dr[t] + bias, c->softplus);
        double y = 0.0;
        for (i64 n = 0; n < N; ++n) {
            const double dA = exp(dt * A[n]);
            const double dBu = dt * Bb[n * L + t] * u[t];
            h[n] = dA * h[n] + dBu;
            y += Cb[n * L + t] * h[n];
        }
        y += Dd * u[t];
        if (z) y = y * z[t] * sigmoid(z[t]);
        c->out[row * L + t] = y;
    }
    if (c->h_last)
        for (i64 n = 0; n < N; ++n) c->h_last[row * N + n] = h[n];
}

/* h0 (nullable, [Bsz][Dch][N]) is the state before t = 0; NULL = zeros. */
int oracle_scan_fwd(const double* u, const double* delta, const double* A, const double* B,
                    const double* C, const double* D, const double* z, const double* delta_bias,
                    int softplus, i64 Bsz, i64 Dch, i64 L, i64 N, const double* h0, double* out,
                    double* h_last, int nthreads) {
    if (N > 1024 || N < 1 || L < 0 || Bsz < 0 || Dch < 0) return 1;
    fwd_ctx c = {u, delta, A, B, C, D, z, delta_bias, h0, softplus, Bsz, Dch, L, N, out, h_last};
    run_rows(fwd_row, &c, Bsz * Dch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* forward in Blelloch order                                           */
/* ------------------------------------------------------------------ */

/* In-place exclusive-then-inclusive Blelloch scan over pairs (a[i], b[i])
 * of length m (power of two), combining earlier o later as
 * (a1, b1) o (a2, b2) = (a1*a2, a2*b1 + b2).  On return b[i] is the
 * inclusive composition of elements 0..i applied to a zero start. */
static void blelloch_pairs(double* a, double* b, double* ea, double* eb, i64 m) {
    memcpy(ea, a, sizeof(double) * m);
    memcpy(eb, b, sizeof(double) * m);
    /* up-sweep: node at k holds the composition of its subtree */
    for (i64 s = 1; s < m; s <<= 1)
        for (i64 k = 2 * s - 1; k < m; k += 2 * s) {
            const double a1 = ea[k - s], b1 = eb[k - s], a2 = ea[k], b2 = eb[k];
            ea[k] = a1 * a2;
            eb[k] = a2 * b1 + b2;
        }
    /* down-sweep: turn the tree into an exclusive scan (identity = (1, 0)) */
    ea[m - 1] = 1.0;
    eb[m - 1] = 0.0;
    for (i64 s = m >> 1; s >= 1; s >>= 1)
        for (i64 k = 2 * s - 1; k < m; k += 2 * s) {
            const double la = ea[k - s], lb = eb[k - s]; /* left subtree total */
            const double pa = ea[k], pb = eb[k];         /* prefix before subtree */
            ea[k - s] = pa;
            eb[k - s] = pb;
            ea[k] = pa * la;
            eb[k] = la * pb + lb;
        }
    /* inclusive = exclusive o own element */
    for (i64 i = 0; i < m; ++i) {
        b[i] = a[i] * eb[i] + b[i];
        a[i] = ea[i] * a[i];
    }
}

typedef struct {
    fwd_ctx f;
    double* scratch; /* per thread: 4*m + m (y) doubles */
    i64 m;
} blel_ctx;

static void blel_row(void* p, i64 row, int tid) {
    blel_ctx* c = (blel_ctx*)p;
    fwd_ctx* f = &c->f;
    const i64 L = f->L, N = f->N, Dch = f->Dch, m = c->m;
    const i64 b = row / Dch, d = row % Dch;
    double* a = c->scratch + (size_t)tid * 5 * m;
    double* bb = a + m;
    double* ea = bb + m;
    double* eb = ea + m;
    double* y = eb + m;
    const double* u = f->u + row * L;
    const double* dr = f->delta + row * L;
    const double bias = f->bias ? f->bias[d] : 0.0;
    for (i64 t = 0; t < L; ++t) y[t] = 0.0;
    for (i64 n = 0; n < N; ++n) {
        const double An = f->A[d * N + n];
        for (i64 t = 0; t < m; ++t) {
            if (t < L) {
                const double dt = softplus_or_raw(dr[t] + bias, f->softplus);
                a[t] = exp(dt * An);
                bb[t] = dt * f->B[(b * N + n) * L + t] * u[t];
            } else {
                a[t] = 1.0;
                bb[t] = 0.0;
            }
        }
        /* a nonzero initial state enters as a leading element (1, h0) */
        if (f->h0) bb[0] += a[0] * f->h0[row * N + n];
        blelloch_pairs(a, bb, ea, eb, m);
        for (i64 t = 0; t < L; ++t) y[t] += f->C[(b * N + n) * L + t] * bb[t];
        if (f->h_last) f->h_last[row * N + n] = L ? bb[L - 1] : (f->h0 ? f->h0[row * N + n] : 0.0);
    }
    const double Dd = f->D ? f->D[d] : 0.0;
    for (i64 t = 0; t < L; ++t) {
        double v = y[t] + Dd * u[t];
        if (f->z) {
            const double zz = f->z[row * L + t];
            v = v * zz * sigmoid(zz);
        }
        f->out[row * L + t] = v;
    }
}

int oracle_scan_fwd_blelloch(const double* u, const double* delta, const double* A,
                             const double* B, const double* C, const double* D, const double* z,
                             const double* delta_bias, int softplus, i64 Bsz, i64 Dch, i64 L,
                             i64 N, const double* h0, double* out, double* h_last, int nthreads) {
    if (L < 1) return 1;
    i64 m = 1;
    while (m < L) m <<= 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    blel_ctx c;
    c.f = (fwd_ctx){u, delta, A, B, C, D, z, delta_bias, h0, softplus, Bsz, Dch, L, N, out, h_last};
    c.m = m;
    c.scratch = (double*)malloc(sizeof(double) * 5 * m * nthreads);
    if (!c.scratch) return 2;
    run_rows(blel_row, &c, Bsz * Dch, nthreads);
    free(c.scratch);
    return 0;
}

/* ------------------------------------------------------------------ */
/* backward                                                            */
/* ------------------------------------------------------------------ */

/*
 * Given g = dL/dout, for each row (chain rule through the forward above):
 *   s   = sigmoid(z),  gate = z*s,  y = sum_n C h + D u (pre-gate)
 *   dz  = g * y * s * (1 + z*(1 - s));     yhat = g * gate
 *   dD += yhat * u;    du = yhat * D
 *   lam_t[n] = yhat_t C_t[n] + a_{t+1}[n] lam_{t+1}[n]   (reverse time)
 *   dC_t[n] += yhat_t h_t[n]                  (summed over d)
 *   dB_t[n] += lam_t[n] delta_t u_t           (summed over d)
 *   du_t    += sum_n lam_t[n] delta_t B_t[n]
 *   ddelta_t = sum_n lam_t[n] (h_{t-1}[n] a_t[n] A[n] + B_t[n] u_t)
 *   dA[n]   += sum_{b,t} lam_t[n] h_{t-1}[n] a_t[n] delta_t
 *   ddelta_raw = ddelta * sigmoid(delta_raw + bias)   (if softplus)
 *   dbias   += sum_{b,t} ddelta_raw
 * Row work is spread over threads by channel d; dB and dC sums over d go
 * into per-thread buffers added in thread order at the end.
 */
typedef struct {
    const double *u, *delta, *A, *B, *C, *D, *z, *bias, *dy;
    int softplus;
    i64 Bsz, Dch, L, N;
    double *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *dbias;
    double* tbuf;   /* per thread: 2 * Bsz*N*L (dB, dC) */
    double* hbuf;   /* per thread: (L+1)*N trajectory + L*N a + 2L */
    int nthreads;
} bwd_ctx;

static void bwd_channel(void* p, i64 d, int tid) {
    bwd_ctx* c = (bwd_ctx*)p;
    const i64 L = c->L, N = c->N, Dch = c->Dch, Bsz = c->Bsz;
    double* tdB = c->tbuf + (size_t)tid * 2 * Bsz * N * L;
    double* tdC = tdB + Bsz * N * L;
    double* H = c->hbuf + (size_t)tid * ((L + 1) * N + L * N + 3 * L);
    double* Aa = H + (L + 1) * N; /* a_t[n] */
    double* dts = Aa + L * N;     /* delta_t */
    double* yhat = dts + L;
    double* xs = yhat + L;        /* delta_raw + bias */
    const double* A = c->A + d * N;
    const double Dd = c->D ? c->D[d] : 0.0;
    const double bias = c->bias ? c->bias[d] : 0.0;
    double dA_acc[1024];
    double lam[1024];
    for (i64 n = 0; n < N; ++n) dA_acc[n] = 0.0;
    double dD_acc = 0.0, dbias_acc = 0.0;
    for (i64 b = 0; b < Bsz; ++b) {
        const i64 row = b * Dch + d;
        const double* u = c->u + row * L;
        const double* dr = c->delta + row * L;
        const double* z = c->z ? c->z + row * L : NULL;
        const double* g = c->dy + row * L;
        const double* Bb = c->B + b * N * L;
        const double* Cb = c->C + b * N * L;
        /* forward, keeping H[t+1][n] = h_t[n], H[0] = 0 */
        for (i64 n = 0; n < N; ++n) H[n] = 0.0;
        for (i64 t = 0; t < L; ++t) {
            xs[t] = dr[t] + bias;
            const double dt = softplus_or_raw(xs[t], c->softplus);
            dts[t] = dt;
            double y = Dd * u[t];
            for (i64 n = 0; n < N; ++n) {
                const double a = exp(dt * A[n]);
                Aa[t * N + n] = a;
                H[(t + 1) * N + n] = a * H[t * N + n] + dt * Bb[n * L + t] * u[t];
                y += Cb[n * L + t] * H[(t + 1) * N + n];
            }
            if (z) {
                const double s = sigmoid(z[t]);
                yhat[t] = g[t] * z[t] * s;
                c->dz[row * L + t] = g[t] * y * s * (1.0 + z[t] * (1.0 - s));
            } else {
                yhat[t] = g[t];
            }
        }
        /* reverse */
        for (i64 n = 0; n < N; ++n) lam[n] = 0.0;
        for (i64 t = L - 1; t >= 0; --t) {
            const double dt = dts[t];
            double du_t = yhat[t] * Dd;
            double ddt = 0.0;
            dD_acc += yhat[t] * u[t];
            for (i64 n = 0; n < N; ++n) {
                const double a_next = (t + 1 < L) ? Aa[(t + 1) * N + n] : 0.0;
                lam[n] = yhat[t] * Cb[n * L + t] + a_next * lam[n];
                const double h_t = H[(t + 1) * N + n];
                const double h_prev = H[t * N + n];
                const double a_t = Aa[t * N + n];
                const double Bt = Bb[n * L + t];
                tdC[(b * N + n) * L + t] += yhat[t] * h_t;
                tdB[(b * N + n) * L + t] += lam[n] * dt * u[t];
                du_t += lam[n] * dt * Bt;
                ddt += lam[n] * (h_prev * a_t * A[n] + Bt * u[t]);
                dA_acc[n] += lam[n] * h_prev * a_t * dt;
            }
            c->du[row * L + t] = du_t;
            const double ddraw = c->softplus ? ddt * sigmoid(xs[t]) : ddt;
            c->ddelta[row * L + t] = ddraw;
            dbias_acc += ddraw;
        }
    }
    for (i64 n = 0; n < N; ++n) c->dA[d * N + n] = dA_acc[n];
    if (c->dD) c->dD[d] = dD_acc;
    if (c->dbias) c->dbias[d] = dbias_acc;
}

int oracle_scan_bwd(const double* u, const double* delta, const double* A, const double* B,
                    const double* C, const double* D, const double* z, const double* delta_bias,
                    int softplus, i64 Bsz, i64 Dch, i64 L, i64 N, const double* dy, double* du,
                    double* ddelta, double* dA, double* dB, double* dC, double* dD, double* dz,
                    double* ddelta_bias, int nthreads) {
    if (N > 1024 || N < 1 || L < 1 || Bsz < 1 || Dch < 1) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > Dch) nthreads = (int)Dch;
    if (nthreads > 256) nthreads = 256;
    const size_t bcn = (size_t)Bsz * N * L;
    bwd_ctx c = {u, delta, A, B, C, D, z, delta_bias, dy, softplus, Bsz, Dch, L, N,
                 du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, NULL, NULL, nthreads};
    c.tbuf = (double*)calloc((size_t)nthreads * 2 * bcn, sizeof(double));
    c.hbuf = (double*)malloc((size_t)nthreads * ((L + 1) * N + L * N + 3 * L) * sizeof(double));
    if (!c.tbuf || !c.hbuf) {
        free(c.tbuf);
        free(c.hbuf);
        return 2;
    }
    run_rows(bwd_channel, &c, Dch, nthreads);
    for (size_t i = 0; i < bcn; ++i) {
        double sb = 0.0, sc = 0.0;
        for (int t = 0; t < nthreads; ++t) {
            sb += c.tbuf[(size_t)t * 2 * bcn + i];
            sc += c.tbuf[(size_t)t * 2 * bcn + bcn + i];
        }
        dB[i] = sb;
        dC[i] = sc;
    }
    free(c.tbuf);
    free(c.hbuf);
    return 0;
}

/* ------------------------------------------------------------------ */
/* one-token step                                                      */
/* ------------------------------------------------------------------ */

typedef struct {
    double* h;
    const double *u, *delta, *A, *B, *C, *D, *z, *bias;
    int softplus;
    i64 Bsz, Dch, N;
    double* y;
} step_ctx;

static void step_row(void* p, i64 row, int tid) {
    (void)tid;
    step_ctx* c = (step_ctx*)p;
    const i64 N = c->N, Dch = c->Dch;
    const i64 b = row / Dch, d = row % Dch;
    const double dt = softplus_or_raw(c->delta[row] + (c->bias ? c->bias[d] : 0.0), c->softplus);
    double y = 0.0;
    for (i64 n = 0; n < N; ++n) {
        double* hn = c->h + row * N + n;
        *hn = exp(dt * c->A[d * N + n]) * *hn + dt * c->B[b * N + n] * c->u[row];
        y += c->C[b * N + n] * *hn;
    }
    y += (c->D ? c->D[d] : 0.0) * c->u[row];
    if (c->z) y = y * c->z[row] * sigmoid(c->z[row]);
    c->y[row] = y;
}

/* h [Bsz][Dch][N] in/out; u, delta, z, y [Bsz][Dch]; B, C [Bsz][N] */
int oracle_step(double* h, const double* u, const double* delta, const double* A,
                const double* B, const double* C, const double* D, const double* z,
                const double* delta_bias, int softplus, i64 Bsz, i64 Dch, i64 N, double* y,
                int nthreads) {
    if (N < 1 || Bsz < 0 || Dch < 0) return 1;
    step_ctx c = {h, u, delta, A, B, C, D, z, delta_bias, softplus, Bsz, Dch, N, y};
    run_rows(step_row, &c, Bsz * Dch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* causal depthwise conv1d + silu (the step that produces u)           */
/* ------------------------------------------------------------------ */
/*
 * The block that feeds the scan: a depthwise causal convolution of width K
 * (d_conv = 4 in the "Mamba 7.9.1" article, section 4.1; mamba-minimal uses
 * a torch.nn.Conv1d there, "mamba.py" page, resources section), then silu:
 *
 *   c_t = bias_d + sum_{k=0..K-1} w[d][k] x_{t-(K-1)+k}    (x_s = 0 for s < 0)
 *   u_t = c_t sigmoid(c_t)                                 (c_t when silu == 0)
 *
 * Backward, with g = dL/du:  gc_t = g_t silu'(c_t) (or g_t);
 *   dx_s = sum_k w[d][k] gc_{s+(K-1)-k};  dw[d][k] = sum_{b,t} gc_t x_{t-(K-1)+k};
 *   dbias_d = sum_{b,t} gc_t.
 * Layouts: x, u, g, dx [Bsz][Dch][L]; w, dw [Dch][K]; bias, dbias [Dch].
 */
typedef struct {
    const double *x, *w, *bias, *g;
    int silu;
    i64 Bsz, Dch, L, K;
    double *u, *dx, *dw, *dbias;
} conv_ctx;

static double conv_pre(const conv_ctx* c, const double* xr, i64 d, i64 t) {
    double s = c->bias ? c->bias[d] : 0.0;
    for (i64 k = 0; k < c->K; ++k) {
        const i64 src = t - (c->K - 1) + k;
        if (src >= 0) s += c->w[d * c->K + k] * xr[src];
    }
    return s;
}

static void conv_fwd_row(void* p, i64 row, int tid) {
    (void)tid;
    conv_ctx* c = (conv_ctx*)p;
    const i64 d = row % c->Dch, L = c->L;
    const double* xr = c->x + row * L;
    for (i64 t = 0; t < L; ++t) {
        const double v = conv_pre(c, xr, d, t);
        c->u[row * L + t] = c->silu ? v * sigmoid(v) : v;
    }
}

int oracle_conv1d_silu(const double* x, const double* w, const double* bias, int silu, i64 Bsz,
                       i64 Dch, i64 L, i64 K, double* u, int nthreads) {
    if (K < 1 || Bsz < 0 || Dch < 0 || L < 0) return 1;
    conv_ctx c = {x, w, bias, NULL, silu, Bsz, Dch, L, K, u, NULL, NULL, NULL};
    run_rows(conv_fwd_row, &c, Bsz * Dch, nthreads);
    return 0;
}

static void conv_bwd_channel(void* p, i64 d, int tid) {
    (void)tid;
    conv_ctx* c = (conv_ctx*)p;
    const i64 L = c->L, K = c->K;
    double* gc = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double db = 0.0;
    for (i64 k = 0; k < K; ++k) c->dw[d * K + k] = 0.0;
    for (i64 b = 0; b < c->Bsz; ++b) {
        const i64 row = b * c->Dch + d;
        const double* xr = c->x + row * L;
        for (i64 t = 0; t < L; ++t) {
            const double v = conv_pre(c, xr, d, t);
            const double s = sigmoid(v);
            gc[t] = c->silu ? c->g[row * L + t] * s * (1.0 + v * (1.0 - s)) : c->g[row * L + t];
            db += gc[t];
            for (i64 k = 0; k < K; ++k) {
                const i64 src = t - (K - 1) + k;
                if (src >= 0) c->dw[d * K + k] += gc[t] * xr[src];
            }
        }
        for (i64 s = 0; s < L; ++s) {
            double acc = 0.0;
            for (i64 k = 0; k < K; ++k) {
                const i64 t = s + (K - 1) - k;
                if (t < L) acc += c->w[d * K + k] * gc[t];
            }
            c->dx[row * L + s] = acc;
        }
    }
    if (c->dbias) c->dbias[d] = db;
    free(gc);
}

int oracle_conv1d_silu_bwd(const double* x, const double* w, const double* bias, int silu,
                           const double* g, i64 Bsz, i64 Dch, i64 L, i64 K, double* dx,
                           double* dw, double* dbias, int nthreads) {
    if (K < 1 || Bsz < 0 || Dch < 0 || L < 0) return 1;
    conv_ctx c = {x, w, bias, g, silu, Bsz, Dch, L, K, NULL, dx, dw, dbias};
    run_rows(conv_bwd_channel, &c, Dch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* input projection: x_proj then dt_proj, producing delta_raw, B, C    */
/* ------------------------------------------------------------------ */
/*
 * The projections that feed the scan ("PyTorch 한 파일에서의 Mamba 구현",
 * news.hada.io topic 12448, and its Vietnamese edition, comment thread:
 * x_proj has no bias, so x_proj and dt_proj compose into one projection and
 * dt_proj's bias is the one the scan adds to delta_raw).  With R = dt_rank,
 * N states and M = R + 2N projected features per token:
 *
 *   xdbl[b][t][m]  = sum_{k < Dch} Wx[m][k] u[b][k][t]          (m < M)
 *   delta[b][d][t] = sum_{r < R}   Wdt[d][r] xdbl[b][t][r]
 *   B[b][n][t]     = xdbl[b][t][R + n],   C[b][n][t] = xdbl[b][t][R + N + n]
 *
 * Layouts: u, delta [Bsz][Dch][L]; Wx [M][Dch]; Wdt [Dch][R]; B, C [Bsz][N][L].
 * One job per (b, t) token.
 */
typedef struct {
    const double *u, *Wx, *Wdt;
    i64 Bsz, Dch, L, R, N;
    double *delta, *B, *C;
} xproj_ctx;

static void xproj_token(void* p, i64 bt, int tid) {
    (void)tid;
    const xproj_ctx* c = (const xproj_ctx*)p;
    const i64 b = bt / c->L, t = bt % c->L, M = c->R + 2 * c->N;
    const double* ub = c->u + b * c->Dch * c->L;
    double* x = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
    for (i64 m = 0; m < M; ++m) {
        double s = 0.0;
        for (i64 k = 0; k < c->Dch; ++k) s += c->Wx[m * c->Dch + k] * ub[k * c->L + t];
        x[m] = s;
    }
    for (i64 d = 0; d < c->Dch; ++d) {
        double s = 0.0;
        for (i64 r = 0; r < c->R; ++r) s += c->Wdt[d * c->R + r] * x[r];
        c->delta[(b * c->Dch + d) * c->L + t] = s;
    }
    for (i64 n = 0; n < c->N; ++n) {
        c->B[(b * c->N + n) * c->L + t] = x[c->R + n];
        c->C[(b * c->N + n) * c->L + t] = x[c->R + c->N + n];
    }
    free(x);
}

int oracle_xproj(const double* u, const double* Wx, const double* Wdt, i64 Bsz, i64 Dch, i64 L,
                 i64 R, i64 N, double* delta, double* B, double* C, int nthreads) {
    if (Bsz < 0 || Dch < 0 || L < 0 || R < 0 || N < 0) return 1;
    xproj_ctx c = {u, Wx, Wdt, Bsz, Dch, L, R, N, delta, B, C};
    run_rows(xproj_token, &c, Bsz * L, nthreads);
    return 0;
}
