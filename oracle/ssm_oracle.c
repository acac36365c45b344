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
            const double dBx = dt * j->B[(b * L + t) * N + n] * xv; /* Bbar x */
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
int oracle_selective_scan(int64_t batch, int64_t L, int64_t dim, int64_t N,
                          const double* x, const double* delta, const double* A,
                          const double* B, const double* C, const double* D,
                          const double* z, const double* delta_bias, int delta_softplus,
                          const double* h0, double* out, double* final_state, int nthreads)
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
int oracle_state_update(int64_t batch, int64_t dim, int64_t N, double* state,
                        const double* x, const double* delta, const double* A,
                        const double* B, const double* C, const double* D,
                        const double* z, const double* delta_bias, int delta_softplus,
                        double* out)
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
                *h = exp(dt * A[d * N + n]) * (*h) + dt * B[b * N + n] * xv;
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
