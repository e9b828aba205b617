/*
 * ssd_oracle.c -- plain sequential CPU oracle for the selective-SSM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load this library.  It shares no
 * code, header, table or constant with the CUDA library, and the CUDA library
 * never calls it.
 *
 * What it follows
 *   [vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링 (blog.secrett2633.cloud),
 *     section "논문 핵심 내용": the selective SSM (S6) in which Delta, B and C
 *     depend on the input; Mamba replaces attention by a linear recurrence.
 *   [vllm] vLLM Mamba2 SSD 커널 웜업 (blog.secrett2633.cloud, PR 39822),
 *     section "mamba_mixer2.py 변경 사항 (핵심)": the kernel call takes
 *     dt_bias, dt_softplus=True, dt_limit=(0, inf), D, per-head A, grouped
 *     B and C of shape [seqlen, ngroups, dstate], x of shape
 *     [seqlen, nheads, headdim] and states of shape [batch, nheads, headdim,
 *     dstate].
 *
 * The recurrence, evaluated token by token in fp64 with no chunking:
 *   delta_t = clamp(softplus(dt[t,h] + dt_bias[h]), dt_min, dt_max)
 *   s[p,n] <- exp(delta_t * A[h]) * s[p,n] + delta_t * x[t,h,p] * B[t,g,n]
 *   y[t,h,p] = sum_n C[t,g,n] * s[p,n] + D[h] * x[t,h,p]
 * with g = h / (nheads / ngroups) (consecutive heads share a group).  After
 * the last token of every chunk the running state is emitted.
 *
 * The chunk metadata is the plain per-token definition: token i of sequence r
 * sits at absolute position pos = num_computed[r] + (i - cu_seqlens[r]); it
 * opens a new chunk iff it is the first new token of r or pos % chunk_size == 0
 * ([vLLM] Mamba (SSM) page, section "청크 메타데이터 계산": every chunk holds
 * tokens of one sequence only, and the state can be taken out every chunk_size
 * tokens).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* softplus(v) = log(1 + exp(v)), written so that neither branch overflows. */
static double oracle_softplus(double v) {
    return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
}

/* delta for one (token, head); the clamp is dt_limit from the kernel call. */
static double oracle_delta(double dt, double bias, int dt_softplus,
                           double dt_min, double dt_max) {
    double d = dt + bias;
    if (dt_softplus) d = oracle_softplus(d);
    if (d < dt_min) d = dt_min;
    if (d > dt_max) d = dt_max;
    return d;
}

double oracle_delta_value(double dt, double bias, int dt_softplus,
                          double dt_min, double dt_max) {
    return oracle_delta(dt, bias, dt_softplus, dt_min, dt_max);
}

typedef struct {
    int64_t T;
    int32_t S, H, P, N, G, K;
    const double *x, *dt, *B, *C, *A, *D, *dt_bias;
    int dt_softplus;
    double dt_min, dt_max;
    const int32_t *cu_seqlens;
    const int32_t *chunk_of_end_token; /* [T]: k if token t ends chunk k, else -1 */
    const double *init_states;         /* [S,H,P,N] or NULL */
    const uint8_t *has_init;           /* [S] or NULL */
    double *y;                          /* [T,H,P] */
    double *chunk_states;               /* [K,H,P,N] or NULL */
    double *final_states;               /* [S,H,P,N] or NULL */
    int32_t nthreads;
    int32_t tid;
} oracle_job;

/* One (sequence r, head h) unit: the recurrence over r's tokens in order. */
static void oracle_run_unit(const oracle_job *j, int32_t r, int32_t h, double *s) {
    const int32_t P = j->P, N = j->N, H = j->H, G = j->G;
    const int32_t g = h / (H / G);
    const size_t PN = (size_t)P * N;
    const size_t state_off = (size_t)h * PN;
    if (j->init_states && j->has_init && j->has_init[r])
        memcpy(s, j->init_states + (size_t)r * H * PN + state_off, PN * sizeof(double));
    else
        memset(s, 0, PN * sizeof(double));
    const double Ah = j->A[h];
    const double Dh = j->D ? j->D[h] : 0.0;
    const double bias = j->dt_bias ? j->dt_bias[h] : 0.0;
    for (int64_t t = j->cu_seqlens[r]; t < j->cu_seqlens[r + 1]; ++t) {
        const double delta = oracle_delta(j->dt[t * H + h], bias, j->dt_softplus,
                                          j->dt_min, j->dt_max);
        const double decay = exp(delta * Ah);
        const double *xt = j->x + ((size_t)t * H + h) * P;
        const double *Bt = j->B + ((size_t)t * G + g) * N;
        const double *Ct = j->C + ((size_t)t * G + g) * N;
        double *yt = j->y + ((size_t)t * H + h) * P;
        for (int32_t p = 0; p < P; ++p) {
            double *sp = s + (size_t)p * N;
            const double dx = delta * xt[p];
            double acc = 0.0;
            for (int32_t n = 0; n < N; ++n) {
                sp[n] = decay * sp[n] + dx * Bt[n];
                acc += Ct[n] * sp[n];
            }
            yt[p] = acc + Dh * xt[p];
        }
        const int32_t k = j->chunk_of_end_token ? j->chunk_of_end_token[t] : -1;
        if (k >= 0 && j->chunk_states)
            memcpy(j->chunk_states + (size_t)k * H * PN + state_off, s, PN * sizeof(double));
    }
    if (j->final_states)
        memcpy(j->final_states + (size_t)r * H * PN + state_off, s, PN * sizeof(double));
}

static void *oracle_worker(void *arg) {
    const oracle_job *j = (const oracle_job *)arg;
    double *s = (double *)malloc((size_t)j->P * j->N * sizeof(double));
    if (!s) return (void *)1;
    const int64_t units = (int64_t)j->S * j->H;
    for (int64_t u = j->tid; u < units; u += j->nthreads)
        oracle_run_unit(j, (int32_t)(u / j->H), (int32_t)(u % j->H), s);
    free(s);
    return NULL;
}

/*
 * Varlen prefill over packed sequences.  Sequence r owns tokens
 * [cu_seqlens[r], cu_seqlens[r+1]); chunk k owns [cu_chunk_seqlens[k],
 * cu_chunk_seqlens[k+1]).  Returns 0 on success, a negative code on bad
 * arguments.  Work is split over (sequence, head) units across nthreads
 * POSIX threads; units are independent, so the arithmetic does not depend
 * on the thread count.
 */
int oracle_ssd_prefill(int64_t T, int32_t S, int32_t H, int32_t P, int32_t N, int32_t G,
                       const double *x, const double *dt, const double *B, const double *C,
                       const double *A, const double *D, const double *dt_bias,
                       int32_t dt_softplus, double dt_min, double dt_max,
                       const int32_t *cu_seqlens, int32_t K, const int32_t *cu_chunk_seqlens,
                       const double *init_states, const uint8_t *has_init,
                       double *y, double *chunk_states, double *final_states,
                       int32_t nthreads) {
    if (T < 0 || S < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[S] != T) return -2;
    for (int32_t r = 0; r < S; ++r)
        if (cu_seqlens[r + 1] < cu_seqlens[r]) return -2;
    int32_t *end_chunk = NULL;
    if (K > 0) {
        if (!cu_chunk_seqlens || cu_chunk_seqlens[0] != 0 || cu_chunk_seqlens[K] != T) return -3;
        end_chunk = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int32_t));
        if (!end_chunk) return -4;
        for (int64_t t = 0; t < T; ++t) end_chunk[t] = -1;
        for (int32_t k = 0; k < K; ++k) {
            if (cu_chunk_seqlens[k + 1] <= cu_chunk_seqlens[k]) { free(end_chunk); return -3; }
            end_chunk[cu_chunk_seqlens[k + 1] - 1] = k;
        }
    }
    if (nthreads < 1) nthreads = 1;
    oracle_job *jobs = (oracle_job *)malloc((size_t)nthreads * sizeof(oracle_job));
    pthread_t *th = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); free(end_chunk); return -4; }
    oracle_job base = {T, S, H, P, N, G, K, x, dt, B, C, A, D, dt_bias, dt_softplus,
                       dt_min, dt_max, cu_seqlens, end_chunk, init_states, has_init,
                       y, chunk_states, final_states, nthreads, 0};
    int rc = 0;
    for (int32_t i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].tid = i;
        if (i > 0 && pthread_create(&th[i], NULL, oracle_worker, &jobs[i]) != 0) { rc = -5; nthreads = i; break; }
    }
    if (oracle_worker(&jobs[0]) != NULL) rc = -4;
    for (int32_t i = 1; i < nthreads; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -4;
    }
    free(jobs); free(th); free(end_chunk);
    return rc;
}

/*
 * Chunk metadata by the per-token definition (see the file header).  Writes
 * cu_chunk_seqlens[K+1], seq_idx[K], last_chunk_indices[S] and
 * chunk_block_col[K] (absolute position of the chunk's last token divided by
 * chunk_size).  last_chunk_indices[r] is the number of chunks of sequences
 * 0..r minus one, which is r's last chunk when r has new tokens.  Returns K,
 * or -1 on bad arguments, or -2 if max_chunks is too small.
 */
int32_t oracle_chunk_metadata(int32_t S, int32_t chunk_size, const int32_t *cu_seqlens,
                              const int32_t *num_computed, int32_t max_chunks,
                              int32_t *cu_chunk_seqlens, int32_t *seq_idx,
                              int32_t *last_chunk_indices, int32_t *chunk_block_col) {
    if (S < 0 || chunk_size < 1 || cu_seqlens[0] != 0) return -1;
    int32_t k = 0;
    for (int32_t r = 0; r < S; ++r) {
        if (cu_seqlens[r + 1] < cu_seqlens[r]) return -1;
        const int64_t nc = num_computed ? num_computed[r] : 0;
        if (nc < 0) return -1;
        for (int32_t i = cu_seqlens[r]; i < cu_seqlens[r + 1]; ++i) {
            const int64_t pos = nc + (i - cu_seqlens[r]);
            const int opens = (i == cu_seqlens[r]) || (pos % chunk_size == 0);
            if (opens) {
                if (k >= max_chunks) return -2;
                cu_chunk_seqlens[k] = i;
                seq_idx[k] = r;
                ++k;
            }
            /* the chunk that holds token i is k-1; its last token so far is i */
            chunk_block_col[k - 1] = (int32_t)(pos / chunk_size);
        }
        last_chunk_indices[r] = k - 1;
    }
    cu_chunk_seqlens[k] = cu_seqlens[S];
    return k;
}

/*
 * Mamba1 selective scan (S6), per-channel state.
 *
 * What it follows
 *   [vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링, section "논문 핵심 내용":
 *     S6 makes Delta, B and C functions of the input, where S4 kept them
 *     fixed; the state of each channel is a vector of dstate values.
 *   [vllm] vLLM Mamba2 SSD 커널 웜업, section "vllm/config/model.py 변경 사항":
 *     Mamba1 has no chunk of its own; the default chunk size (2048) is the
 *     granularity at which states are taken out for prefix caching.
 * Readings where the pages are silent (the Mamba paper's S6): A is a real
 * [channels, dstate] matrix (one decay rate per channel and state index),
 * Delta is per (token, channel) with the same softplus/clamp as Mamba2, B and
 * C are [T, G, dstate] shared by the channels of a group (G = 1 in Mamba1),
 * D and dt_bias are per channel.  Evaluated token by token in fp64:
 *   delta = clamp(softplus(dt[t,d] + dt_bias[d]), dt_min, dt_max)
 *   s[d,n] <- exp(delta * A[d,n]) * s[d,n] + delta * x[t,d] * B[t,g,n]
 *   y[t,d] = sum_n C[t,g,n] * s[d,n] + D[d] * x[t,d],   g = d / (channels / G)
 * and the running state of every channel is emitted after the last token of
 * every chunk.
 */
typedef struct {
    int64_t T;
    int32_t S, Dc, N, G;
    const double *x, *dt, *B, *C, *A, *Dskip, *dt_bias;
    int dt_softplus;
    double dt_min, dt_max;
    const int32_t *cu_seqlens;
    const int32_t *chunk_of_end_token;
    const double *init_states; /* [S,Dc,N] or NULL */
    const uint8_t *has_init;
    double *y;                 /* [T,Dc] */
    double *chunk_states;      /* [K,Dc,N] or NULL */
    double *final_states;      /* [S,Dc,N] or NULL */
    int32_t nthreads, tid;
} oracle_m1_job;

static void oracle_m1_unit(const oracle_m1_job *j, int32_t r, int32_t d, double *s) {
    const int32_t N = j->N, Dc = j->Dc, G = j->G;
    const int32_t g = d / (Dc / G);
    const size_t off = (size_t)d * N;
    if (j->init_states && j->has_init && j->has_init[r])
        memcpy(s, j->init_states + (size_t)r * Dc * N + off, (size_t)N * sizeof(double));
    else
        memset(s, 0, (size_t)N * sizeof(double));
    const double *Ad = j->A + off;
    const double Dd = j->Dskip ? j->Dskip[d] : 0.0;
    const double bias = j->dt_bias ? j->dt_bias[d] : 0.0;
    for (int64_t t = j->cu_seqlens[r]; t < j->cu_seqlens[r + 1]; ++t) {
        const double delta = oracle_delta(j->dt[t * Dc + d], bias, j->dt_softplus, j->dt_min, j->dt_max);
        const double xt = j->x[t * Dc + d];
        const double *Bt = j->B + ((size_t)t * G + g) * N;
        const double *Ct = j->C + ((size_t)t * G + g) * N;
        double acc = 0.0;
        for (int32_t n = 0; n < N; ++n) {
            s[n] = exp(delta * Ad[n]) * s[n] + delta * xt * Bt[n];
            acc += Ct[n] * s[n];
        }
        j->y[t * Dc + d] = acc + Dd * xt;
        const int32_t k = j->chunk_of_end_token ? j->chunk_of_end_token[t] : -1;
        if (k >= 0 && j->chunk_states)
            memcpy(j->chunk_states + (size_t)k * Dc * N + off, s, (size_t)N * sizeof(double));
    }
    if (j->final_states)
        memcpy(j->final_states + (size_t)r * Dc * N + off, s, (size_t)N * sizeof(double));
}

static void *oracle_m1_worker(void *arg) {
    const oracle_m1_job *j = (const oracle_m1_job *)arg;
    double *s = (double *)malloc((size_t)j->N * sizeof(double));
    if (!s) return (void *)1;
    const int64_t units = (int64_t)j->S * j->Dc;
    for (int64_t u = j->tid; u < units; u += j->nthreads)
        oracle_m1_unit(j, (int32_t)(u / j->Dc), (int32_t)(u % j->Dc), s);
    free(s);
    return NULL;
}

/* Varlen Mamba1 scan; arguments and return codes as oracle_ssd_prefill, with
 * x, dt [T,Dc], A [Dc,N], D and dt_bias [Dc], states [.,Dc,N]. */
int oracle_mamba1_prefill(int64_t T, int32_t S, int32_t Dc, int32_t N, int32_t G,
                          const double *x, const double *dt, const double *B, const double *C,
                          const double *A, const double *Dskip, const double *dt_bias,
                          int32_t dt_softplus, double dt_min, double dt_max,
                          const int32_t *cu_seqlens, int32_t K, const int32_t *cu_chunk_seqlens,
                          const double *init_states, const uint8_t *has_init,
                          double *y, double *chunk_states, double *final_states, int32_t nthreads) {
    if (T < 0 || S < 0 || Dc <= 0 || N <= 0 || G <= 0 || Dc % G != 0) return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[S] != T) return -2;
    for (int32_t r = 0; r < S; ++r)
        if (cu_seqlens[r + 1] < cu_seqlens[r]) return -2;
    int32_t *end_chunk = NULL;
    if (K > 0) {
        if (!cu_chunk_seqlens || cu_chunk_seqlens[0] != 0 || cu_chunk_seqlens[K] != T) return -3;
        end_chunk = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int32_t));
        if (!end_chunk) return -4;
        for (int64_t t = 0; t < T; ++t) end_chunk[t] = -1;
        for (int32_t k = 0; k < K; ++k) {
            if (cu_chunk_seqlens[k + 1] <= cu_chunk_seqlens[k]) { free(end_chunk); return -3; }
            end_chunk[cu_chunk_seqlens[k + 1] - 1] = k;
        }
    }
    if (nthreads < 1) nthreads = 1;
    oracle_m1_job *jobs = (oracle_m1_job *)malloc((size_t)nthreads * sizeof(oracle_m1_job));
    pthread_t *th = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); free(end_chunk); return -4; }
    oracle_m1_job base = {T, S, Dc, N, G, x, dt, B, C, A, Dskip, dt_bias, dt_softplus, dt_min, dt_max,
                          cu_seqlens, end_chunk, init_states, has_init, y, chunk_states, final_states,
                          nthreads, 0};
    int rc = 0;
    for (int32_t i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].tid = i;
        if (i > 0 && pthread_create(&th[i], NULL, oracle_m1_worker, &jobs[i]) != 0) { rc = -5; nthreads = i; break; }
    }
    if (oracle_m1_worker(&jobs[0]) != NULL) rc = -4;
    for (int32_t i = 1; i < nthreads; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -4;
    }
    free(jobs); free(th); free(end_chunk);
    return rc;
}
