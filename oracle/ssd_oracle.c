/*
 * fp64 CPU oracle for the Mamba-2 state-space-duality (SSD) scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code with the CUDA kernels.
 *
 * What it computes (sources: "Mamba-Family State-Space Model Kernels on a
 * Programmable CGLA", section III.A "Mamba-2 Layer with Three Kernel Shapes"
 * -- Step-3 updates the recurrent state h sequentially, the transition A_c is
 * an input-dependent diagonal; and "Compiler-First State Space Duality and
 * Portable O(1) Autoregressive Caching", abstract -- diagonal per-head
 * dynamics, fixed-size chunking):
 *
 *   for every (b, h), with g = h / (H / G) and h_{-1} = init (or 0):
 *     abar_t = exp(dt_t * A_h)
 *     h_t[p][n] = abar_t * h_{t-1}[p][n] + dt_t * B_t[n] * x_t[p]
 *     y_t[p]    = sum_n C_t[n] * h_t[p][n] + D_h * x_t[p]
 *   final = h_{L-1}
 *
 * The state is an N x P matrix stored [P][N] (N fastest), matching the
 * "N x d matrix-vector product per chunk" of section III.C of the CGLA page.
 * y uses the updated state; D multiplies the raw x; dt is used as given.
 *
 * Layouts (row-major, contiguous):
 *   x  [b][L][H][P]   dt [b][L][H]   A [H]   B, C [b][L][G][N]   D [H]
 *   init, final [b][H][P][N]         y [b][L][H][P]
 *
 * oracle_scan_seq     -- the recurrence above, token by token.
 * oracle_step         -- one token of the same recurrence, state in place.
 * oracle_scan_chunked -- the same result computed by the SSD chunk steps in
 *                        the order the CGLA page names them (Step-1 intra-chunk
 *                        GEMM1 -> mask -> GEMM2; chunk state; Step-3 sequential
 *                        inter-chunk recurrence; off-diagonal output), used
 *                        only to expose per-chunk intermediates to tests.
 *
 * Parity pins (tests/test_oracle_pins.py): quadratic dual form on tiny inputs,
 * A = 0 prefix sum, constant-decay geometric series, x = 0 pure decay,
 * a hand-derived worked example, chunk-size invariance, split/resume
 * invariance, linearity.  The pages print no SSD input/output values, so no
 * pin comes from the pages themselves.
 *
 * All arithmetic is double precision with libm exp(); threads only split
 * independent (b, h) pairs, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *x, *dt, *A, *B, *C, *D, *init;
    double *y, *fin;
    double *state_io;         /* oracle_step: state in place */
    double *chunk_states;     /* chunked: S_c  [b][nc][H][P][N] (nullable) */
    double *chunk_prev;       /* chunked: H_{c-1} [b][nc][H][P][N] (nullable) */
    int64_t batch, L, H, P, N, G, Q;
    int kind;                 /* 0 seq, 1 step, 2 chunked */
    int64_t next_unit;        /* shared work counter */
    pthread_mutex_t mu;
    int err;
} job_t;

static int64_t take_unit(job_t *j) {
    pthread_mutex_lock(&j->mu);
    int64_t u = j->next_unit++;
    pthread_mutex_unlock(&j->mu);
    return u;
}

/* One (b, h) pair, token by token. */
static void seq_unit(job_t *j, int64_t b, int64_t h, double *s) {
    const int64_t L = j->L, H = j->H, P = j->P, N = j->N, G = j->G;
    const int64_t g = h / (H / G);
    const double Dh = j->D ? j->D[h] : 0.0;
    if (j->init) memcpy(s, j->init + (b * H + h) * P * N, sizeof(double) * P * N);
    else memset(s, 0, sizeof(double) * P * N);
    for (int64_t t = 0; t < L; ++t) {
        const int64_t bt = b * L + t;
        const double dtv = j->dt[bt * H + h];
        const double abar = exp(dtv * j->A[h]);
        const double *Bt = j->B + (bt * G + g) * N;
        const double *Ct = j->C + (bt * G + g) * N;
        const double *xt = j->x + (bt * H + h) * P;
        double *yt = j->y + (bt * H + h) * P;
        for (int64_t p = 0; p < P; ++p) {
            double *row = s + p * N;
            const double dx = dtv * xt[p];
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                row[n] = abar * row[n] + dx * Bt[n];
                acc += Ct[n] * row[n];
            }
            yt[p] = acc + Dh * xt[p];
        }
    }
    if (j->fin) memcpy(j->fin + (b * H + h) * P * N, s, sizeof(double) * P * N);
}

/* One decode step for one (b, h): the t = 0 iteration of seq_unit with the
 * state read from and written back to state_io. */
static void step_unit(job_t *j, int64_t b, int64_t h) {
    const int64_t H = j->H, P = j->P, N = j->N, G = j->G;
    const int64_t g = h / (H / G);
    const double Dh = j->D ? j->D[h] : 0.0;
    const double dtv = j->dt[b * H + h];
    const double abar = exp(dtv * j->A[h]);
    const double *Bt = j->B + (b * G + g) * N;
    const double *Ct = j->C + (b * G + g) * N;
    const double *xt = j->x + (b * H + h) * P;
    double *yt = j->y + (b * H + h) * P;
    double *s = j->state_io + (b * H + h) * P * N;
    for (int64_t p = 0; p < P; ++p) {
        double *row = s + p * N;
        const double dx = dtv * xt[p];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            row[n] = abar * row[n] + dx * Bt[n];
            acc += Ct[n] * row[n];
        }
        yt[p] = acc + Dh * xt[p];
    }
}

/* One (b, h) pair by chunks of Q tokens (the last chunk may be shorter).
 * work: a[Q] chunk-local inclusive cumsum of dt*A, Sc[P*N], Hp[P*N]. */
static void chunked_unit(job_t *j, int64_t b, int64_t h, double *Hs, double *a,
                         double *Sc) {
    const int64_t L = j->L, H = j->H, P = j->P, N = j->N, G = j->G, Q = j->Q;
    const int64_t g = h / (H / G);
    const int64_t nc = (L + Q - 1) / Q;
    const double Dh = j->D ? j->D[h] : 0.0;
    if (j->init) memcpy(Hs, j->init + (b * H + h) * P * N, sizeof(double) * P * N);
    else memset(Hs, 0, sizeof(double) * P * N);
    for (int64_t c = 0; c < nc; ++c) {
        const int64_t c0 = c * Q;
        const int64_t len = (L - c0 < Q) ? (L - c0) : Q;
        /* chunk-local inclusive cumulative sum of dt*A */
        double run = 0.0;
        for (int64_t i = 0; i < len; ++i) {
            run += j->dt[(b * L + c0 + i) * H + h] * j->A[h];
            a[i] = run;
        }
        const double a_end = a[len - 1];
        /* expose the state entering this chunk */
        if (j->chunk_prev)
            memcpy(j->chunk_prev + ((b * nc + c) * H + h) * P * N, Hs,
                   sizeof(double) * P * N);
        /* outputs: Step-1 (GEMM1 C.B^T over N, mask, GEMM2 over s) plus the
         * off-diagonal term from the entering state and the D skip */
        for (int64_t ti = 0; ti < len; ++ti) {
            const int64_t bt = b * L + c0 + ti;
            const double *Ct = j->C + (bt * G + g) * N;
            double *yt = j->y + (bt * H + h) * P;
            const double *xt = j->x + (bt * H + h) * P;
            for (int64_t p = 0; p < P; ++p) yt[p] = 0.0;
            for (int64_t si = 0; si <= ti; ++si) {
                const int64_t bs = b * L + c0 + si;
                const double *Bs = j->B + (bs * G + g) * N;
                double cb = 0.0;
                for (int64_t n = 0; n < N; ++n) cb += Ct[n] * Bs[n];
                const double m = cb * exp(a[ti] - a[si]) * j->dt[bs * H + h];
                const double *xs = j->x + (bs * H + h) * P;
                for (int64_t p = 0; p < P; ++p) yt[p] += m * xs[p];
            }
            const double ea = exp(a[ti]);
            for (int64_t p = 0; p < P; ++p) {
                double off = 0.0;
                for (int64_t n = 0; n < N; ++n) off += Ct[n] * Hs[p * N + n];
                yt[p] += ea * off + Dh * xt[p];
            }
        }
        /* chunk state S_c = sum_s exp(a_end - a_s) dt_s x_s B_s^T */
        memset(Sc, 0, sizeof(double) * P * N);
        for (int64_t si = 0; si < len; ++si) {
            const int64_t bs = b * L + c0 + si;
            const double w = exp(a_end - a[si]) * j->dt[bs * H + h];
            const double *Bs = j->B + (bs * G + g) * N;
            const double *xs = j->x + (bs * H + h) * P;
            for (int64_t p = 0; p < P; ++p)
                for (int64_t n = 0; n < N; ++n) Sc[p * N + n] += w * xs[p] * Bs[n];
        }
        if (j->chunk_states)
            memcpy(j->chunk_states + ((b * nc + c) * H + h) * P * N, Sc,
                   sizeof(double) * P * N);
        /* Step-3: H_c = exp(a_end) H_{c-1} + S_c */
        const double de = exp(a_end);
        for (int64_t k = 0; k < P * N; ++k) Hs[k] = de * Hs[k] + Sc[k];
    }
    if (j->fin) memcpy(j->fin + (b * H + h) * P * N, Hs, sizeof(double) * P * N);
}

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    const int64_t units = j->batch * j->H;
    double *s = NULL, *a = NULL, *Sc = NULL;
    if (j->kind == 0) s = (double *)malloc(sizeof(double) * j->P * j->N);
    if (j->kind == 2) {
        s = (double *)malloc(sizeof(double) * j->P * j->N);
        a = (double *)malloc(sizeof(double) * j->Q);
        Sc = (double *)malloc(sizeof(double) * j->P * j->N);
    }
    if ((j->kind == 0 && !s) || (j->kind == 2 && (!s || !a || !Sc))) {
        pthread_mutex_lock(&j->mu);
        j->err = 1;
        pthread_mutex_unlock(&j->mu);
        free(s); free(a); free(Sc);
        return NULL;
    }
    for (;;) {
        const int64_t u = take_unit(j);
        if (u >= units) break;
        const int64_t b = u / j->H, h = u % j->H;
        if (j->kind == 0) seq_unit(j, b, h, s);
        else if (j->kind == 1) step_unit(j, b, h);
        else chunked_unit(j, b, h, s, a, Sc);
    }
    free(s); free(a); free(Sc);
    return NULL;
}

static int run(job_t *j, int nthreads) {
    if (j->batch <= 0 || j->H <= 0 || j->P <= 0 || j->N <= 0 || j->G <= 0 ||
        j->H % j->G != 0)
        return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    const int64_t units = j->batch * j->H;
    if (nthreads > units) nthreads = (int)units;
    j->next_unit = 0;
    j->err = 0;
    pthread_mutex_init(&j->mu, NULL);
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, j) != 0) break;
        started = i;
    }
    worker(j);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&j->mu);
    return j->err;
}

/* Returns 0 on success, nonzero on bad sizes or allocation failure. */
int oracle_scan_seq(const double *x, const double *dt, const double *A,
                    const double *B, const double *C, const double *D,
                    const double *init, int64_t batch, int64_t seqlen,
                    int64_t nheads, int64_t headdim, int64_t dstate,
                    int64_t ngroups, double *y, double *final_state,
                    int nthreads) {
    if (seqlen <= 0) return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.x = x; j.dt = dt; j.A = A; j.B = B; j.C = C; j.D = D; j.init = init;
    j.y = y; j.fin = final_state;
    j.batch = batch; j.L = seqlen; j.H = nheads; j.P = headdim; j.N = dstate;
    j.G = ngroups; j.kind = 0;
    return run(&j, nthreads);
}

int oracle_step(double *state, const double *x, const double *dt,
                const double *A, const double *B, const double *C,
                const double *D, int64_t batch, int64_t nheads, int64_t headdim,
                int64_t dstate, int64_t ngroups, double *y, int nthreads) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.x = x; j.dt = dt; j.A = A; j.B = B; j.C = C; j.D = D;
    j.state_io = state; j.y = y;
    j.batch = batch; j.L = 1; j.H = nheads; j.P = headdim; j.N = dstate;
    j.G = ngroups; j.kind = 1;
    return run(&j, nthreads);
}

int oracle_scan_chunked(const double *x, const double *dt, const double *A,
                        const double *B, const double *C, const double *D,
                        const double *init, int64_t batch, int64_t seqlen,
                        int64_t nheads, int64_t headdim, int64_t dstate,
                        int64_t ngroups, int64_t chunk, double *y,
                        double *final_state, double *chunk_states,
                        double *chunk_prev, int nthreads) {
    if (seqlen <= 0 || chunk <= 0) return 1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.x = x; j.dt = dt; j.A = A; j.B = B; j.C = C; j.D = D; j.init = init;
    j.y = y; j.fin = final_state;
    j.chunk_states = chunk_states; j.chunk_prev = chunk_prev;
    j.batch = batch; j.L = seqlen; j.H = nheads; j.P = headdim; j.N = dstate;
    j.G = ngroups; j.Q = chunk; j.kind = 2;
    return run(&j, nthreads);
}
