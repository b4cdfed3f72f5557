/*
 * Oracle for the SSD (structured state space duality) layer forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct CPU
 * definition that the GPU path is checked against. Nothing in the product
 * path links, loads or calls it; only tests/, the smoke check and the bench's
 * CPU-baseline leg do. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes: the selective state space recurrence with a
 * scalar-times-identity transition, run token by token in fp64:
 *
 *     a_t = exp(dt_t * A_h)                       (scalar per token and head)
 *     h_t = a_t * h_{t-1} + x_t (outer) B_t       (state, P x N per head)
 *     y_t = h_t . C_t + D_h * x_t                 (P outputs per head)
 *
 * Sources:
 *   - recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t^T h_t:
 *     "Mamba-2 状态空间对偶性理论", §1.2 (selective SSM definition);
 *     "Transformers是SSMs：通过结构化状态空间对偶性的广义模型和高效算法(一)",
 *     §3.1 (matrix transformation form of SSMs).
 *   - A_t restricted to a scalar times identity, one scalar per (token, head);
 *     multi-head with head dim P and shared dynamics across the P channels:
 *     "LLM(十一)——Mamba", §3.1.2 (SSD: scalar structured SSM, multi-head SSMs).
 *   - D skip connection y += D x: "LLM(十一)——Mamba", §1.2 (output equation,
 *     matrix D as skip connection).
 *   - initial state consumed before the first token and final state returned:
 *     "LLM(十一)——Mamba", §3.5.3 (the ssd listing takes initial_states and
 *     returns final_state; the initial state enters chunk 0 through the same
 *     exp(cumsum) decay as any earlier state, so it is decayed by the first
 *     token's a_t).
 *   - variable length: one packed row, no state carried across sequence
 *     boundaries: "LLM(十一)——Mamba", §3.7.3 (Variable Length). Each sequence
 *     starts from its own initial state (zero when none is given).
 *   - grouped B, C (a group of H/G consecutive heads shares B_t, C_t):
 *     "LLM(十一)——Mamba", §3.6 (multi-input / grouped-value head patterns).
 *   - optional input scaling by dt (ssd_oracle_f64_ex with scale_x_by_dt): the input term becomes
 *     dt_t * x_t (outer) B_t while the skip term keeps D_h * x_t. This is the discretization the
 *     full model keeps from Mamba ("LLM(十一)——Mamba" §3.5.4: the parameters are transformed
 *     before they enter the SSD code; "Transformers是SSMs (一)" §2.1, Remark 1), read as
 *     B-bar = dt * B; the pages do not print the formula itself.
 *
 * Layouts (all row-major, contiguous, fp64):
 *   x, y        (rows, H, P)   rows = batch*seqlen (dense) or total tokens
 *   dt          (rows, H)
 *   A, D        (H)            D may be NULL (no skip)
 *   B, C        (rows, G, N)
 *   init, final (nseq, H, P, N)  nseq = batch (dense) or number of segments;
 *                                init may be NULL (zero), final may be NULL
 *   cu_seqlens  (nseq + 1) int32 host array of segment starts, or NULL for a
 *               dense batch of `batch` rows of `seqlen` tokens.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int64_t H, P, N, G;
    int scale_x_by_dt;
    const double *x, *dt, *A, *B, *C, *D, *init;
    const int64_t *seq_start, *seq_len;
    int64_t nseq;
    double *y, *final_state;
    int64_t next_unit;            /* work counter over (sequence, head) */
    pthread_mutex_t lock;
} oracle_job;

/* One (sequence, head) pair: the plain token-by-token recurrence. */
static void run_unit(oracle_job *j, int64_t s, int64_t h, double *S)
{
    const int64_t H = j->H, P = j->P, N = j->N, G = j->G;
    const int64_t g = h / (H / G);
    const double A_h = j->A[h];
    const double D_h = j->D ? j->D[h] : 0.0;

    if (j->init)
        memcpy(S, j->init + ((s * H + h) * P) * N, sizeof(double) * P * N);
    else
        memset(S, 0, sizeof(double) * P * N);

    for (int64_t t = j->seq_start[s]; t < j->seq_start[s] + j->seq_len[s]; ++t) {
        const double dt_th = j->dt[t * H + h];
        const double a = exp(dt_th * A_h);
        const double in_scale = j->scale_x_by_dt ? dt_th : 1.0;
        const double *xt = j->x + (t * H + h) * P;
        const double *Bt = j->B + (t * G + g) * N;
        const double *Ct = j->C + (t * G + g) * N;
        double *yt = j->y + (t * H + h) * P;
        for (int64_t p = 0; p < P; ++p) {
            double *Sp = S + p * N;
            const double xp = xt[p];
            const double xin = in_scale * xp;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                Sp[n] = a * Sp[n] + xin * Bt[n];
                acc += Sp[n] * Ct[n];
            }
            yt[p] = acc + D_h * xp;
        }
    }
    if (j->final_state)
        memcpy(j->final_state + ((s * H + h) * P) * N, S, sizeof(double) * P * N);
}

static void *worker(void *arg)
{
    oracle_job *j = (oracle_job *)arg;
    double *S = (double *)malloc(sizeof(double) * j->P * j->N);
    if (!S) return (void *)1;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t u = j->next_unit++;
        pthread_mutex_unlock(&j->lock);
        if (u >= j->nseq * j->H) break;
        run_unit(j, u / j->H, u % j->H, S);
    }
    free(S);
    return NULL;
}

/* Number of threads the oracle uses when asked for "all cores". */
int ssd_oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 * nthreads <= 0 uses every online core. scale_x_by_dt != 0 selects the dt-scaled input term.
 */
int ssd_oracle_f64_ex(int64_t batch, int64_t seqlen, int64_t H, int64_t P, int64_t N, int64_t G,
                      const double *x, const double *dt, const double *A,
                      const double *B, const double *C, const double *D,
                      const double *init, const int32_t *cu_seqlens, int64_t nseq,
                      double *y, double *final_state, int scale_x_by_dt, int nthreads)
{
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return 1;
    if (!x || !dt || !A || !B || !C || !y) return 1;
    int64_t *start, *len;
    if (cu_seqlens) {
        if (batch != 1 || nseq <= 0) return 1;
        start = (int64_t *)malloc(sizeof(int64_t) * nseq);
        len = (int64_t *)malloc(sizeof(int64_t) * nseq);
        if (!start || !len) { free(start); free(len); return 2; }
        for (int64_t s = 0; s < nseq; ++s) {
            start[s] = cu_seqlens[s];
            len[s] = (int64_t)cu_seqlens[s + 1] - cu_seqlens[s];
            if (len[s] < 0 || cu_seqlens[s + 1] > seqlen) { free(start); free(len); return 1; }
        }
    } else {
        nseq = batch;
        start = (int64_t *)malloc(sizeof(int64_t) * (nseq > 0 ? nseq : 1));
        len = (int64_t *)malloc(sizeof(int64_t) * (nseq > 0 ? nseq : 1));
        if (!start || !len) { free(start); free(len); return 2; }
        for (int64_t s = 0; s < nseq; ++s) { start[s] = s * seqlen; len[s] = seqlen; }
    }

    oracle_job j;
    j.H = H; j.P = P; j.N = N; j.G = G;
    j.scale_x_by_dt = scale_x_by_dt;
    j.x = x; j.dt = dt; j.A = A; j.B = B; j.C = C; j.D = D; j.init = init;
    j.seq_start = start; j.seq_len = len; j.nseq = nseq;
    j.y = y; j.final_state = final_state;
    j.next_unit = 0;
    pthread_mutex_init(&j.lock, NULL);

    if (nthreads <= 0) nthreads = ssd_oracle_default_threads();
    if (nthreads > nseq * H) nthreads = (int)(nseq * H > 0 ? nseq * H : 1);
    int rc = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    if (!th) rc = 2;
    int started = 0;
    for (int i = 0; rc == 0 && i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &j) != 0) break;
        ++started;
    }
    if (rc == 0 && started == 0) worker(&j);   /* no threads available: run inline */
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret) rc = 2;
    }
    free(th);
    pthread_mutex_destroy(&j.lock);
    free(start);
    free(len);
    return rc;
}

/* The recurrence without input scaling. */
int ssd_oracle_f64(int64_t batch, int64_t seqlen, int64_t H, int64_t P, int64_t N, int64_t G,
                   const double *x, const double *dt, const double *A,
                   const double *B, const double *C, const double *D,
                   const double *init, const int32_t *cu_seqlens, int64_t nseq,
                   double *y, double *final_state, int nthreads)
{
    return ssd_oracle_f64_ex(batch, seqlen, H, P, N, G, x, dt, A, B, C, D, init, cu_seqlens, nseq, y,
                             final_state, 0, nthreads);
}
