/*
 * ssm_oracle.c -- float64 CPU oracle for the selective state space scan (S6).
 *
 * TEST INFRASTRUCTURE ONLY. This file defines what the CUDA path must compute.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * build, load or call it. It shares no code, header, table or helper with the
 * CUDA library, and the CUDA library never links or calls it.
 *
 * Everything is plain float64 C with no fast-math, no blocking and no
 * reordering: each function is the textbook loop, written so that it can be
 * checked against the pages by eye.
 *
 * Sources (page title, then section):
 *  - "State Space Models -- Mamba, S4, and Beyond", section "Mamba (S6 --
 *    Selective State Space)", method `_selective_scan`: discretize with the
 *    per-token step, dA = exp(delta * A), dB = delta * B, then the sequential
 *    loop h = dA * h + dB * u; y = C . h; output y + D * u.
 *  - "Mamba: State Space Models Challenge Transformers", section "Selective
 *    Scan Algorithm" (`selective_scan(x, delta, A, B, C, D)`, A of shape
 *    [D, N]) and section "Mamba's Innovation: Selection" (`delta =
 *    softplus(delta)`; the block output is gated as y * silu(z)).
 *  - "State-space models (Mamba, S4)", section "The Convolution View"
 *    (h_k = Abar h_{k-1} + Bbar x_k, starting from h_0 = 0; the output reads
 *    the updated state) and section "Worked Example: 2D SSM Step".
 *  - "State Space Models and Mamba", section "Mamba: Selective State Spaces"
 *    (Delta_t = softplus(Linear(x_t))).
 *
 * Readings taken where the pages are silent or disagree:
 *  - Bbar is the first-order form delta * B (every code listing uses it).
 *  - y_t reads the state after the update at t.
 *  - delta_bias, when given, is added to delta before the optional softplus,
 *    whether or not softplus is on.
 *  - D and z are optional; the gate multiplies after the D skip.
 *  - softplus(v) = log(1 + exp(v)), evaluated in the overflow-free form
 *    max(v, 0) + log1p(exp(-|v|)), with no threshold.
 *  - silu(z) = z / (1 + exp(-z)).
 *
 * Layouts (row-major, contiguous):
 *   x, delta, z, out : [batch, L, dim]      B, C : [batch, L, N]
 *   A : [dim, N]    D, delta_bias : [dim]   h0, final_state : [batch, dim, N]
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* softplus(v) = log(1 + e^v). */
double oracle_softplus(double v) { return fmax(v, 0.0) + log1p(exp(-fabs(v))); }

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * phi(z) = (e^z - 1) / z, with phi(0) = 1: the exact zero-order-hold input
 * matrix of a diagonal state is Bbar = A^-1 (e^{A dt} - 1) B = dt * phi(dt A) * B
 * ("State-space models (Mamba, S4)", section "From Continuous to Discrete: The
 * Key Step": the exact solution for an input held constant over the step; and
 * its flashcard Bbar = (A^-1 (e^{A Delta} - I)) B). expm1 keeps it accurate as
 * z -> 0, where it tends to 1 and the first-order form dt * B is recovered.
 */
double oracle_phi(double z) { return z == 0.0 ? 1.0 : expm1(z) / z; }

/*
 * phi'(z), the derivative of phi, needed by the gradient of the zero-order-hold
 * Bbar with respect to A. Since phi(z) = integral_0^1 e^{zs} ds,
 *   phi'(z) = integral_0^1 s e^{zs} ds = sum_{k>=0} z^k / (k! (k + 2))
 *           = (e^z (z - 1) + 1) / z^2                     (z != 0),
 * with phi'(0) = 1/2. The closed form cancels badly for small |z|, so the
 * series (terms below 1e-19 after k = 20 when |z| <= 1) is summed there and the
 * closed form used elsewhere.
 */
double oracle_phi_prime(double z)
{
    if (fabs(z) <= 1.0) {
        double term = 1.0, sum = 0.0;   /* term = z^k / k! */
        for (int k = 0; k <= 24; ++k) {
            sum += term / (k + 2);
            term *= z / (k + 1);
        }
        return sum;
    }
    return (exp(z) * (z - 1.0) + 1.0) / (z * z);
}

/*
 * The recurrence with the discretized parameters given directly, one channel:
 *   h[n] <- Abar[t,n] * h[n] + Bbar[t,n] * x[t]
 *   y[t]  = sum_n C[t,n] * h[n]           (h after the update)
 * h holds h0 on entry and the last state on exit. No D, no gate: this is the
 * core of "The Convolution View" and of the worked 2-D example.
 */
void oracle_recurrence(int64_t L, int64_t N, const double* Abar, const double* Bbar,
                       const double* C, const double* x, double* h, double* y)
{
    for (int64_t t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            h[n] = Abar[t * N + n] * h[n] + Bbar[t * N + n] * x[t];
            acc += C[t * N + n] * h[n];
        }
        y[t] = acc;
    }
}

typedef struct {
    int64_t batch, L, dim, N;
    const double *x, *delta, *A, *B, *C, *D, *z, *delta_bias, *h0;
    int delta_softplus;
    int zoh;                      /* exact zero-order-hold Bbar instead of dt * B */
    double *out, *final_state;
    int64_t chan_begin, chan_end; /* channel = b * dim + d */
} scan_job;

/* One (b, d) channel of the selective scan, straight from the definition. */
static void scan_channel(const scan_job* j, int64_t b, int64_t d, double* h)
{
    const int64_t L = j->L, dim = j->dim, N = j->N;
    for (int64_t n = 0; n < N; ++n)
        h[n] = j->h0 ? j->h0[(b * dim + d) * N + n] : 0.0;

    for (int64_t t = 0; t < L; ++t) {
        const int64_t e = (b * L + t) * dim + d; /* element (b, t, d) */
        const double xv = j->x[e];

        double dt = j->delta[e];
        if (j->delta_bias) dt += j->delta_bias[d];
        if (j->delta_softplus) dt = oracle_softplus(dt);

        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double dA = exp(dt * j->A[d * N + n]);          /* Abar */
            const double dBx = dt * j->B[(b * L + t) * N + n] * xv  /* Bbar x */
                               * (j->zoh ? oracle_phi(dt * j->A[d * N + n]) : 1.0);
            h[n] = dA * h[n] + dBx;
            acc += j->C[(b * L + t) * N + n] * h[n];
        }
        double y = acc;
        if (j->D) y += j->D[d] * xv;
        if (j->z) y *= oracle_silu(j->z[e]);
        j->out[e] = y;
    }
    if (j->final_state)
        for (int64_t n = 0; n < N; ++n) j->final_state[(b * dim + d) * N + n] = h[n];
}

static void* scan_worker(void* arg)
{
    const scan_job* j = (const scan_job*)arg;
    double* h = (double*)malloc((size_t)j->N * sizeof(double));
    if (!h) return (void*)1;
    for (int64_t c = j->chan_begin; c < j->chan_end; ++c)
        scan_channel(j, c / j->dim, c % j->dim, h);
    free(h);
    return NULL;
}

/*
 * Full selective scan over [batch, L, dim] with an N-wide diagonal state per
 * channel. h0 may be NULL (zero initial state, as on the pages); D, z,
 * delta_bias and final_state may be NULL. Channels are independent, so they
 * are split across nthreads POSIX threads; each channel is one sequential loop.
 * Returns 0, or -1 on bad arguments / thread failure.
 */
static int scan_run(int64_t batch, int64_t L, int64_t dim, int64_t N, const double* x,
                    const double* delta, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* delta_bias,
                    int delta_softplus, int zoh, const double* h0, double* out,
                    double* final_state, int nthreads);

int oracle_selective_scan(int64_t batch, int64_t L, int64_t dim, int64_t N,
                          const double* x, const double* delta, const double* A,
                          const double* B, const double* C, const double* D,
                          const double* z, const double* delta_bias, int delta_softplus,
                          const double* h0, double* out, double* final_state, int nthreads)
{
    return scan_run(batch, L, dim, N, x, delta, A, B, C, D, z, delta_bias, delta_softplus, 0,
                    h0, out, final_state, nthreads);
}

/* The same scan with the exact zero-order-hold Bbar = dt * phi(dt A) * B. */
int oracle_selective_scan_zoh(int64_t batch, int64_t L, int64_t dim, int64_t N,
                              const double* x, const double* delta, const double* A,
                              const double* B, const double* C, const double* D,
                              const double* z, const double* delta_bias, int delta_softplus,
                              const double* h0, double* out, double* final_state, int nthreads)
{
    return scan_run(batch, L, dim, N, x, delta, A, B, C, D, z, delta_bias, delta_softplus, 1,
                    h0, out, final_state, nthreads);
}

static int scan_run(int64_t batch, int64_t L, int64_t dim, int64_t N, const double* x,
                    const double* delta, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* delta_bias,
                    int delta_softplus, int zoh, const double* h0, double* out,
                    double* final_state, int nthreads)
{
    if (batch < 0 || L < 0 || dim < 0 || N <= 0) return -1;
    if (!x || !delta || !A || !B || !C || !out) return -1;
    const int64_t nchan = batch * dim;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nchan) nthreads = nchan > 0 ? (int)nchan : 1;

    scan_job jobs[256];
    pthread_t tid[256];
    for (int i = 0; i < nthreads; ++i) {
        scan_job* j = &jobs[i];
        j->batch = batch; j->L = L; j->dim = dim; j->N = N;
        j->x = x; j->delta = delta; j->A = A; j->B = B; j->C = C; j->D = D; j->z = z;
        j->delta_bias = delta_bias; j->h0 = h0; j->delta_softplus = delta_softplus;
        j->zoh = zoh;
        j->out = out; j->final_state = final_state;
        j->chan_begin = nchan * i / nthreads;
        j->chan_end = nchan * (i + 1) / nthreads;
    }
    if (nthreads == 1) return scan_worker(&jobs[0]) ? -1 : 0;
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tid[i], NULL, scan_worker, &jobs[i]) != 0) { rc = -1; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void* r = NULL;
        pthread_join(tid[i], &r);
        if (r) rc = -1;
    }
    return rc;
}

/*
 * One recurrent generation step ("State-space models (Mamba, S4)", section
 * "Training vs Inference Modes": keep h_{k-1}, take x_k, update the state,
 * read out y_k; O(1) per token). It is exactly one t-iteration of the scan
 * above on a persisted state, updated in place.
 *   state : [batch, dim, N]   x, delta, z, out : [batch, dim]   B, C : [batch, N]
 */
static int state_update_run(int64_t batch, int64_t dim, int64_t N, double* state,
                            const double* x, const double* delta, const double* A,
                            const double* B, const double* C, const double* D, const double* z,
                            const double* delta_bias, int delta_softplus, int zoh, double* out);

int oracle_state_update(int64_t batch, int64_t dim, int64_t N, double* state,
                        const double* x, const double* delta, const double* A,
                        const double* B, const double* C, const double* D,
                        const double* z, const double* delta_bias, int delta_softplus,
                        double* out)
{
    return state_update_run(batch, dim, N, state, x, delta, A, B, C, D, z, delta_bias,
                            delta_softplus, 0, out);
}

/* The same step with the exact zero-order-hold Bbar. */
int oracle_state_update_zoh(int64_t batch, int64_t dim, int64_t N, double* state,
                            const double* x, const double* delta, const double* A,
                            const double* B, const double* C, const double* D,
                            const double* z, const double* delta_bias, int delta_softplus,
                            double* out)
{
    return state_update_run(batch, dim, N, state, x, delta, A, B, C, D, z, delta_bias,
                            delta_softplus, 1, out);
}

static int state_update_run(int64_t batch, int64_t dim, int64_t N, double* state,
                            const double* x, const double* delta, const double* A,
                            const double* B, const double* C, const double* D, const double* z,
                            const double* delta_bias, int delta_softplus, int zoh, double* out)
{
    if (batch < 0 || dim < 0 || N <= 0) return -1;
    if (!state || !x || !delta || !A || !B || !C || !out) return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t e = b * dim + d;
            const double xv = x[e];
            double dt = delta[e];
            if (delta_bias) dt += delta_bias[d];
            if (delta_softplus) dt = oracle_softplus(dt);
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double* h = &state[e * N + n];
                *h = exp(dt * A[d * N + n]) * (*h) + dt * B[b * N + n] * xv
                     * (zoh ? oracle_phi(dt * A[d * N + n]) : 1.0);
                acc += C[b * N + n] * (*h);
            }
            double y = acc;
            if (D) y += D[d] * xv;
            if (z) y *= oracle_silu(z[e]);
            out[e] = y;
        }
    }
    return 0;
}

/*
 * Causal depthwise 1-D convolution followed by SiLU: the input stage of the
 * Mamba block ("State Space Models -- Mamba, S4, and Beyond", section "Mamba
 * (S6 -- Selective State Space)", MambaBlock: nn.Conv1d with kernel_size =
 * d_conv, padding = d_conv - 1, groups = d_inner, the output cut to seq_len,
 * then silu; "State-space models (Mamba, S4)", the block diagram's
 * "Conv1D + SiLU"). Conv1d is a cross-correlation over the left-padded input,
 * so for every batch row b, channel d and token t:
 *   pre[t] = bias[d] + sum_{k=0..K-1} w[d,k] * x[t - (K-1) + k]   (x = 0 before t = 0)
 *   u[t]   = silu(pre[t])
 * Layouts: x, u [batch, L, dim]; w [dim, K]; bias [dim] or NULL (zero).
 */
void oracle_causal_conv1d_silu(int64_t batch, int64_t L, int64_t dim, int64_t K,
                               const double* x, const double* w, const double* bias, double* u)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t t = 0; t < L; ++t)
            for (int64_t d = 0; d < dim; ++d) {
                double pre = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t s = t - (K - 1) + k;
                    if (s >= 0) pre += w[d * K + k] * x[(b * L + s) * dim + d];
                }
                u[(b * L + t) * dim + d] = oracle_silu(pre);
            }
}

/*
 * Gradients of the input stage above for a loss with dLoss/du = du (the chain
 * rule on its loop, in the same order). With s(p) = 1 / (1 + e^-p) and
 * silu'(p) = s(p) (1 + p (1 - s(p))):
 *   dpre[t]      = du[t] silu'(pre[t])
 *   dx[t-(K-1)+k] += dpre[t] w[d,k]        (the taps that read that token)
 *   dw[d,k]      += dpre[t] x[t-(K-1)+k]   (over batch rows and tokens)
 *   dbias[d]     += dpre[t]
 * Outputs are overwritten; dw and dbias may be NULL. Layouts as the forward.
 */
void oracle_causal_conv1d_silu_bwd(int64_t batch, int64_t L, int64_t dim, int64_t K,
                                   const double* x, const double* w, const double* bias,
                                   const double* du, double* dx, double* dw, double* dbias)
{
    for (int64_t i = 0; i < batch * L * dim; ++i) dx[i] = 0.0;
    if (dw) for (int64_t i = 0; i < dim * K; ++i) dw[i] = 0.0;
    if (dbias) for (int64_t i = 0; i < dim; ++i) dbias[i] = 0.0;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t t = 0; t < L; ++t)
            for (int64_t d = 0; d < dim; ++d) {
                double pre = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t s = t - (K - 1) + k;
                    if (s >= 0) pre += w[d * K + k] * x[(b * L + s) * dim + d];
                }
                const double sg = 1.0 / (1.0 + exp(-pre));
                const double dpre = du[(b * L + t) * dim + d] * sg * (1.0 + pre * (1.0 - sg));
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t s = t - (K - 1) + k;
                    if (s < 0) continue;
                    dx[(b * L + s) * dim + d] += dpre * w[d * K + k];
                    if (dw) dw[d * K + k] += dpre * x[(b * L + s) * dim + d];
                }
                if (dbias) dbias[d] += dpre;
            }
}

/*
 * Gradients of the selective scan (the reverse-mode derivative of
 * oracle_selective_scan, from the chain rule on its loop; the pages ask that
 * gradients flow through the discretization: "State Space Models -- Mamba, S4,
 * and Beyond", section "Verification Checklist", and "State-space models
 * (Mamba, S4)", section "Training vs Inference Modes": training runs the scan
 * in parallel and backpropagates through it).
 *
 * Given dout = dLoss/dout [batch, L, dim] and, optionally, dh_final =
 * dLoss/dfinal_state [batch, dim, N], with per token (one channel)
 *   v = delta + bias,  dt = softplus(v) or v,  a[n] = exp(dt A[n]),
 *   h[n] = a[n] hp[n] + dt x B[n]   (hp: the state before the token),
 *   y = sum_n C[n] h[n] + D x,      out = y * silu(z)  (or y),
 * the reverse sweep carries G[n] = dLoss/dh[n] from the last token back:
 *   dy     = dout * silu(z)                      dz = dout * y * silu'(z)
 *   G[n]   = a_next[n] G_next[n] + dy C[n]       (a_next G_next = dh_final at the end)
 *   dC[n] += dy h[n]          dB[n] += G[n] dt x        dx = dy D + dt sum_n G[n] B[n]
 *   ddt    = sum_n G[n] (x B[n] + A[n] a[n] hp[n])     dA[n] += G[n] dt a[n] hp[n]
 *   ddelta = ddt * sigmoid(v) (softplus) or ddt;  dbias += ddelta;  dD += dy x
 *   dh0[n] = a_0[n] G_0[n]
 * dB and dC sum over channels d (B, C are shared by all channels); dA, dD and
 * dbias sum over batch rows and tokens. Optional outputs may be NULL; dD, dz,
 * dbias are only defined when D, z, delta_bias were given.
 *
 * With the exact zero-order hold (oracle_selective_scan_bwd_zoh) the input term
 * is dt phi(dt A[n]) B[n] x = (e^{dt A[n]} - 1)/A[n] B[n] x; its derivative in
 * dt is a[n] B[n] x (phi(z) + z phi'(z) = e^z) and in A[n] is
 * dt^2 phi'(dt A[n]) B[n] x, so with p[n] = phi(dt A[n]):
 *   dB[n] += G[n] dt p[n] x    dx = dy D + dt sum_n G[n] p[n] B[n]
 *   ddt    = sum_n G[n] (a[n] x B[n] + A[n] a[n] hp[n])
 *   dA[n] += G[n] (dt a[n] hp[n] + dt^2 phi'(dt A[n]) B[n] x)
 *
 * Channels are split across threads; each thread sums its own dA, dD, dbias,
 * dB and dC and the partial sums are added in thread order (deterministic for a
 * given thread count). Returns 0, or -1 on bad arguments / allocation failure.
 */
typedef struct {
    int64_t batch, L, dim, N;
    const double *x, *delta, *A, *B, *C, *D, *z, *delta_bias, *h0, *dout, *dh_final;
    int delta_softplus;
    int zoh;                                      /* exact zero-order-hold Bbar */
    double *dx, *ddelta, *dz, *dh0;               /* per channel: written directly */
    double *dA, *dB, *dC, *dD, *dbias;            /* this thread's partial sums */
    int64_t chan_begin, chan_end;
    int failed;
} bwd_job;

static double oracle_sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

static void bwd_channel(bwd_job* j, int64_t b, int64_t d, double* hp, double* dtv, double* yv,
                        double* G)
{
    const int64_t L = j->L, dim = j->dim, N = j->N;
    const double* Ad = j->A + d * N;                              /* A[d, :] */
    const double* h0c = j->h0 ? j->h0 + (b * dim + d) * N : NULL; /* h0[b, d, :] */
    const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;
    /* forward sweep: keep the state before every token, dt and y (pre-gate) */
    double* h = hp + L * N;   /* running state (the slot after the last token) */
    for (int64_t n = 0; n < N; ++n) h[n] = h0c ? h0c[n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t e = (b * L + t) * dim + d;
        const double* Bt = j->B + (b * L + t) * N;
        const double* Ct = j->C + (b * L + t) * N;
        const double v = j->delta[e] + bias;
        const double dt = j->delta_softplus ? oracle_softplus(v) : v;
        dtv[t] = dt;
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            hp[t * N + n] = h[n];
            const double p = j->zoh ? oracle_phi(dt * Ad[n]) : 1.0;
            h[n] = exp(dt * Ad[n]) * h[n] + dt * p * Bt[n] * j->x[e];
            acc += Ct[n] * h[n];
        }
        yv[t] = acc + (j->D ? j->D[d] * j->x[e] : 0.0);
    }
    /* reverse sweep */
    for (int64_t n = 0; n < N; ++n) G[n] = j->dh_final ? j->dh_final[(b * dim + d) * N + n] : 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t e = (b * L + t) * dim + d;
        const double* Bt = j->B + (b * L + t) * N;
        const double* Ct = j->C + (b * L + t) * N;
        const double xv = j->x[e], dt = dtv[t];
        double dy = j->dout[e];
        if (j->z) {
            const double s = oracle_sigmoid(j->z[e]);
            if (j->dz) j->dz[e] = j->dout[e] * yv[t] * s * (1.0 + j->z[e] * (1.0 - s));
            dy *= j->z[e] * s;
        }
        double dx = j->D ? dy * j->D[d] : 0.0;
        if (j->D) j->dD[d] += dy * xv;
        double ddt = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double a = exp(dt * Ad[n]);
            const double p = j->zoh ? oracle_phi(dt * Ad[n]) : 1.0;   /* Bbar = dt p B */
            const double hprev = hp[t * N + n];
            const double ht = a * hprev + dt * p * Bt[n] * xv;
            const double g = G[n] + dy * Ct[n];           /* dLoss/dh_t */
            j->dC[(b * L + t) * N + n] += dy * ht;
            j->dB[(b * L + t) * N + n] += g * dt * p * xv;
            dx += g * dt * p * Bt[n];
            ddt += g * ((j->zoh ? a : 1.0) * xv * Bt[n] + Ad[n] * a * hprev);
            j->dA[d * N + n] += g * (dt * a * hprev
                                     + (j->zoh ? dt * dt * oracle_phi_prime(dt * Ad[n]) * Bt[n] * xv
                                               : 0.0));
            G[n] = a * g;                                  /* carried to the token before */
        }
        const double dd = j->delta_softplus ? ddt * oracle_sigmoid(j->delta[e] + bias) : ddt;
        if (j->ddelta) j->ddelta[e] = dd;
        if (j->delta_bias) j->dbias[d] += dd;
        if (j->dx) j->dx[e] = dx;
    }
    if (j->dh0)
        for (int64_t n = 0; n < N; ++n) j->dh0[(b * dim + d) * N + n] = G[n];
}

static void* bwd_worker(void* arg)
{
    bwd_job* j = (bwd_job*)arg;
    const int64_t L = j->L, N = j->N;
    double* hp = (double*)malloc((size_t)((L + 1) * N + 2 * L + N) * sizeof(double));
    if (!hp) { j->failed = 1; return NULL; }
    double* dtv = hp + (L + 1) * N;
    double* yv = dtv + L;
    double* G = yv + L;
    for (int64_t c = j->chan_begin; c < j->chan_end; ++c)
        bwd_channel(j, c / j->dim, c % j->dim, hp, dtv, yv, G);
    free(hp);
    return NULL;
}

static int bwd_run(int64_t batch, int64_t L, int64_t dim, int64_t N, const double* x,
                   const double* delta, const double* A, const double* B, const double* C,
                   const double* D, const double* z, const double* delta_bias,
                   int delta_softplus, int zoh, const double* h0, const double* dout,
                   const double* dh_final, double* dx, double* ddelta, double* dA, double* dB,
                   double* dC, double* dD, double* dz, double* ddelta_bias, double* dh0,
                   int nthreads);

int oracle_selective_scan_bwd(int64_t batch, int64_t L, int64_t dim, int64_t N,
                              const double* x, const double* delta, const double* A,
                              const double* B, const double* C, const double* D,
                              const double* z, const double* delta_bias, int delta_softplus,
                              const double* h0, const double* dout, const double* dh_final,
                              double* dx, double* ddelta, double* dA, double* dB, double* dC,
                              double* dD, double* dz, double* ddelta_bias, double* dh0,
                              int nthreads)
{
    return bwd_run(batch, L, dim, N, x, delta, A, B, C, D, z, delta_bias, delta_softplus, 0, h0,
                   dout, dh_final, dx, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dh0, nthreads);
}

/* The gradients of the scan with the exact zero-order-hold Bbar. */
int oracle_selective_scan_bwd_zoh(int64_t batch, int64_t L, int64_t dim, int64_t N,
                                  const double* x, const double* delta, const double* A,
                                  const double* B, const double* C, const double* D,
                                  const double* z, const double* delta_bias, int delta_softplus,
                                  const double* h0, const double* dout, const double* dh_final,
                                  double* dx, double* ddelta, double* dA, double* dB, double* dC,
                                  double* dD, double* dz, double* ddelta_bias, double* dh0,
                                  int nthreads)
{
    return bwd_run(batch, L, dim, N, x, delta, A, B, C, D, z, delta_bias, delta_softplus, 1, h0,
                   dout, dh_final, dx, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dh0, nthreads);
}

static int bwd_run(int64_t batch, int64_t L, int64_t dim, int64_t N, const double* x,
                   const double* delta, const double* A, const double* B, const double* C,
                   const double* D, const double* z, const double* delta_bias,
                   int delta_softplus, int zoh, const double* h0, const double* dout,
                   const double* dh_final, double* dx, double* ddelta, double* dA, double* dB,
                   double* dC, double* dD, double* dz, double* ddelta_bias, double* dh0,
                   int nthreads)
{
    if (batch < 0 || L < 0 || dim < 0 || N <= 0) return -1;
    if (!x || !delta || !A || !B || !C || !dout) return -1;
    const int64_t nchan = batch * dim;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    if ((int64_t)nthreads > nchan) nthreads = nchan > 0 ? (int)nchan : 1;
    const size_t nA = (size_t)(dim * N), nBC = (size_t)(batch * L * N), nd = (size_t)dim;
    const size_t per = nA + 2 * nBC + 2 * nd;   /* dA, dB, dC, dD, dbias */
    double* part = (double*)calloc((size_t)nthreads * per, sizeof(double));
    if (!part) return -1;

    bwd_job jobs[64];
    pthread_t tid[64];
    for (int i = 0; i < nthreads; ++i) {
        bwd_job* j = &jobs[i];
        j->batch = batch; j->L = L; j->dim = dim; j->N = N;
        j->x = x; j->delta = delta; j->A = A; j->B = B; j->C = C; j->D = D; j->z = z;
        j->delta_bias = delta_bias; j->h0 = h0; j->dout = dout; j->dh_final = dh_final;
        j->delta_softplus = delta_softplus;
        j->zoh = zoh;
        j->dx = dx; j->ddelta = ddelta; j->dz = dz; j->dh0 = dh0;
        double* p = part + (size_t)i * per;
        j->dA = p; j->dB = p + nA; j->dC = p + nA + nBC; j->dD = p + nA + 2 * nBC;
        j->dbias = p + nA + 2 * nBC + nd;
        j->chan_begin = nchan * i / nthreads;
        j->chan_end = nchan * (i + 1) / nthreads;
        j->failed = 0;
    }
    int rc = 0;
    if (nthreads == 1) {
        bwd_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tid[i], NULL, bwd_worker, &jobs[i]) != 0) { rc = -1; break; }
            ++started;
        }
        for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    }
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].failed) rc = -1;
    /* partial sums, added in thread order */
    if (dA) for (size_t k = 0; k < nA; ++k) dA[k] = 0.0;
    if (dB) for (size_t k = 0; k < nBC; ++k) dB[k] = 0.0;
    if (dC) for (size_t k = 0; k < nBC; ++k) dC[k] = 0.0;
    if (dD) for (size_t k = 0; k < nd; ++k) dD[k] = 0.0;
    if (ddelta_bias) for (size_t k = 0; k < nd; ++k) ddelta_bias[k] = 0.0;
    for (int i = 0; i < nthreads; ++i) {
        const bwd_job* j = &jobs[i];
        if (dA) for (size_t k = 0; k < nA; ++k) dA[k] += j->dA[k];
        if (dB) for (size_t k = 0; k < nBC; ++k) dB[k] += j->dB[k];
        if (dC) for (size_t k = 0; k < nBC; ++k) dC[k] += j->dC[k];
        if (dD && D) for (size_t k = 0; k < nd; ++k) dD[k] += j->dD[k];
        if (ddelta_bias && delta_bias) for (size_t k = 0; k < nd; ++k) ddelta_bias[k] += j->dbias[k];
    }
    free(part);
    return rc;
}

/*
 * The SSD layer of Mamba-2 ("Mamba: State Space Models Challenge Transformers",
 * section "Mamba-2: Improved Architecture": a multi-head structure with
 * n_heads heads of d_head channels and a d_state-wide state per channel; "State
 * Space Models and Mamba", section "Mamba 2 and Hybrid Architectures": the SSM
 * recast as a structured matrix multiplication, dual to attention). The pages
 * give the block as a stub; the readings
 * taken here are the plainest ones the selective scan supports:
 *  - each head hd has one scalar decay A[hd] (a multiple of the identity, the
 *    structure that makes the layer a masked matrix product) and one step
 *    dt[b,t,hd] shared by its P channels;
 *  - B, C rows of width N are shared by the heads of a group: head hd reads
 *    group g = hd / (H / G) (consecutive heads share a group; G divides H);
 *  - dt = dt_raw + dt_bias (if given), then softplus if asked, as in the scan;
 *  - D is per head; there is no gate inside the layer.
 * Per batch row b, head hd, token t, channel p < P and state n < N:
 *   a = exp(dt A[hd]);   h[p][n] <- a h[p][n] + dt x[b,t,hd,p] B[b,t,g,n]
 *   y[b,t,hd,p] = sum_n C[b,t,g,n] h[p][n] + D[hd] x[b,t,hd,p]
 * Layouts (row-major): x, y [batch, L, H, P]; dt [batch, L, H]; A, D, dt_bias [H];
 * B, C [batch, L, G, N]; h0, final_state [batch, H, P, N]. h0, D, dt_bias and
 * final_state may be NULL. Threads split the (b, hd) pairs. Returns 0, or -1 on
 * bad arguments or a failed allocation / thread.
 */
typedef struct {
    int64_t batch, L, H, P, G, N;
    const double *x, *dt, *A, *B, *C, *D, *dt_bias, *h0;
    int dt_softplus;
    double *y, *final_state;
    int64_t begin, end;   /* pairs b * H + hd */
} ssd_job;

static void* ssd_worker(void* arg)
{
    const ssd_job* j = (const ssd_job*)arg;
    const int64_t L = j->L, H = j->H, P = j->P, G = j->G, N = j->N;
    double* h = (double*)malloc((size_t)(P * N) * sizeof(double));
    if (!h) return (void*)1;
    for (int64_t pair = j->begin; pair < j->end; ++pair) {
        const int64_t b = pair / H, hd = pair % H, g = hd / (H / G);
        for (int64_t i = 0; i < P * N; ++i) h[i] = j->h0 ? j->h0[pair * P * N + i] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double dt = j->dt[(b * L + t) * H + hd];
            if (j->dt_bias) dt += j->dt_bias[hd];
            if (j->dt_softplus) dt = oracle_softplus(dt);
            const double a = exp(dt * j->A[hd]);
            const double* Bt = j->B + ((b * L + t) * G + g) * N;
            const double* Ct = j->C + ((b * L + t) * G + g) * N;
            for (int64_t p = 0; p < P; ++p) {
                const int64_t e = ((b * L + t) * H + hd) * P + p;   /* x[b, t, hd, p] */
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    h[p * N + n] = a * h[p * N + n] + dt * j->x[e] * Bt[n];
                    acc += Ct[n] * h[p * N + n];
                }
                j->y[e] = acc + (j->D ? j->D[hd] * j->x[e] : 0.0);
            }
        }
        if (j->final_state)
            for (int64_t i = 0; i < P * N; ++i) j->final_state[pair * P * N + i] = h[i];
    }
    free(h);
    return NULL;
}

int oracle_ssd(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
               const double* x, const double* dt, const double* A, const double* B,
               const double* C, const double* D, const double* dt_bias, int dt_softplus,
               const double* h0, double* y, double* final_state, int nthreads)
{
    if (batch < 0 || L < 0 || H <= 0 || P <= 0 || G <= 0 || N <= 0 || H % G != 0) return -1;
    if (!x || !dt || !A || !B || !C || !y) return -1;
    const int64_t npairs = batch * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > npairs) nthreads = npairs > 0 ? (int)npairs : 1;
    ssd_job jobs[256];
    pthread_t tid[256];
    for (int i = 0; i < nthreads; ++i) {
        ssd_job* j = &jobs[i];
        j->batch = batch; j->L = L; j->H = H; j->P = P; j->G = G; j->N = N;
        j->x = x; j->dt = dt; j->A = A; j->B = B; j->C = C; j->D = D; j->dt_bias = dt_bias;
        j->h0 = h0; j->dt_softplus = dt_softplus; j->y = y; j->final_state = final_state;
        j->begin = npairs * i / nthreads;
        j->end = npairs * (i + 1) / nthreads;
    }
    if (nthreads == 1) return ssd_worker(&jobs[0]) ? -1 : 0;
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tid[i], NULL, ssd_worker, &jobs[i]) != 0) { rc = -1; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void* r = NULL;
        pthread_join(tid[i], &r);
        if (r) rc = -1;
    }
    return rc;
}
