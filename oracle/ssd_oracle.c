/*
 * ssd_oracle.c -- plain fp64 CPU oracle for the Mamba-2 SSD forward pass and
 * its reverse mode (gradients, at the end of the file).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [disconfirmai] "Jane Street ML Engineers Map Mamba-2 Recurrent State
 *       Computation to Tensor Cores with cuTile" -- paragraph on the
 *       fixed-size hidden state (Mamba-2 as a state-space model whose state
 *       update can be done chunkwise) and paragraph on the jump formula
 *       h(t+T) = h(t) + B X^T with decay folded in through log-space sums.
 *   [devotd] devotd.net news page on the Mamba-2 cuTile forward kernels,
 *       section 1 (recurrent model with a fixed-size hidden state, chunking)
 *       and section 2 (chunk_cumsum: decay rate x time interval accumulated
 *       inside a chunk; fwd_pass_state: chunk-start states and the state
 *       after the last chunk; compute_out: output from the chunk-start state).
 *
 * What is computed is the definition, token by token, never the chunked
 * algorithm.  Per (batch b, head h), with group g = h / (H/G) and the hidden
 * state hs[n][p] (N x P, the "B X^T" orientation of the jump formula):
 *
 *     a          = exp(dt[b,t,h] * A[h])
 *     hs[n][p]   = a * hs[n][p] + B[b,t,g,n] * dt[b,t,h] * x[b,t,h,p]
 *     y[b,t,h,p] = sum_n C[b,t,g,n] * hs[n][p] + D[h] * x[b,t,h,p]
 *
 * Inputs x, B, C are bfloat16 bit patterns; dt, A, D and the states are
 * float32.  Every input is widened exactly to double; all arithmetic is
 * double with libm exp/exp2.  States are exchanged in the (P, N) orientation
 * (state[p][n] = hs[n][p]).
 *
 * Parallelism: one task per (batch, head) unit, spread over POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define LOG2E_D 1.4426950408889634073599246810018921

/* bfloat16 bit pattern -> double (exact: bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t v) {
    uint32_t u = ((uint32_t)v) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size;
} dims_t;

static int64_t nchunks_of(const dims_t* d) {
    return (d->seqlen + d->chunk_size - 1) / d->chunk_size;
}

/* ---------------------------------------------------------------- threads */

typedef void (*unit_fn)(void* ctx, int64_t unit_index);

typedef struct {
    unit_fn fn;
    void* ctx;
    int64_t nunits;
    int64_t next;
    pthread_mutex_t lock;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        int64_t u = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (u >= p->nunits) break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

/* Runs fn(ctx, u) for u in [0, nunits) on nthreads threads (<= 0: all
 * online cores).  Returns the number of threads used. */
static int run_units(unit_fn fn, void* ctx, int64_t nunits, int nthreads) {
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > nunits) nthreads = (int)(nunits > 0 ? nunits : 1);
    pool_t pool;
    pool.fn = fn;
    pool.ctx = ctx;
    pool.nunits = nunits;
    pool.next = 0;
    pthread_mutex_init(&pool.lock, NULL);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, pool_worker, &pool) == 0) ++started;
        else break;
    }
    if (started == 0) pool_worker(&pool); /* no thread could start: run inline */
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&pool.lock);
    return started > 0 ? started : 1;
}

/* ------------------------------------------------------- recurrence core */

/*
 * Runs the recurrence for one (b, h) over tokens [t0, t1), starting from the
 * state hs (N x P, updated in place).  If y is non-NULL, writes y rows
 * y[(t - t0) * P + p].  C/D may be NULL when y is NULL.
 */
/*
 * Input-side options of a whole Mamba-2 layer around the scan.  The pages
 * take dt as given and D as one weight per head; these are the plainest
 * readings of the steps a layer adds on either side, applied per token:
 *
 *     dt <- dt + dt_bias[h]                      (dt_bias non-NULL)
 *     dt <- log(1 + exp(dt))                     (dt_softplus)
 *     dt <- min(max(dt, dt_min), dt_max)         (dt_limit)
 *     skip term D[h][p] x[p]                     (D_per_channel: D is (H, P))
 *     y  <- y * z / (1 + exp(-z))                (z non-NULL, x's layout, bf16)
 */
typedef struct {
    const float* dt_bias;
    int dt_softplus, dt_limit;
    double dt_min, dt_max;
    int D_per_channel;
    const uint16_t* z;
} opts_t;

typedef struct {
    const dims_t* d;
    const uint16_t *x, *B, *C;
    const float *dt, *A, *D;
    const opts_t* opt; /* NULL: dt, D and y as they are */
} inputs_t;

/* log(1 + exp(v)) without overflow: for v > 0 it is v + log(1 + exp(-v)). */
static double softplus_d(double v) {
    return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
}

static double effective_dt(const opts_t* o, int64_t h, double v) {
    if (o == NULL) return v;
    if (o->dt_bias != NULL) v += (double)o->dt_bias[h];
    if (o->dt_softplus) v = softplus_d(v);
    if (o->dt_limit) v = fmin(fmax(v, o->dt_min), o->dt_max);
    return v;
}

static void recur_tokens(const inputs_t* in, int64_t b, int64_t h, int64_t t0, int64_t t1,
                         double* hs, double* y) {
    const dims_t* d = in->d;
    const int64_t H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups;
    const int64_t g = h / (H / G);
    const double A = (double)in->A[h];
    const opts_t* opt = in->opt;
    const int d_per_p = (opt != NULL && opt->D_per_channel);
    const uint16_t* z = (opt != NULL) ? opt->z : NULL;
    double* xv = (double*)malloc(sizeof(double) * (size_t)P);
    double* bv = (double*)malloc(sizeof(double) * (size_t)N);
    double* cv = (double*)malloc(sizeof(double) * (size_t)N);
    for (int64_t t = t0; t < t1; ++t) {
        const double dt = effective_dt(opt, h, (double)in->dt[(b * d->seqlen + t) * H + h]);
        const double a = exp(dt * A);
        const uint16_t* xr = in->x + ((b * d->seqlen + t) * H + h) * P;
        const uint16_t* br = in->B + ((b * d->seqlen + t) * G + g) * N;
        for (int64_t p = 0; p < P; ++p) xv[p] = bf16_to_double(xr[p]);
        for (int64_t n = 0; n < N; ++n) bv[n] = bf16_to_double(br[n]);
        for (int64_t n = 0; n < N; ++n) {
            const double bdt = bv[n] * dt;
            double* row = hs + n * P;
            for (int64_t p = 0; p < P; ++p) row[p] = a * row[p] + bdt * xv[p];
        }
        if (y != NULL) {
            const uint16_t* cr = in->C + ((b * d->seqlen + t) * G + g) * N;
            for (int64_t n = 0; n < N; ++n) cv[n] = bf16_to_double(cr[n]);
            double* yr = y + (t - t0) * P;
            for (int64_t p = 0; p < P; ++p) {
                const double Dp = (in->D == NULL) ? 0.0 : (double)in->D[d_per_p ? h * P + p : h];
                yr[p] = Dp * xv[p];
            }
            for (int64_t n = 0; n < N; ++n) {
                const double c = cv[n];
                const double* row = hs + n * P;
                for (int64_t p = 0; p < P; ++p) yr[p] += c * row[p];
            }
            if (z != NULL) {
                const uint16_t* zr = z + ((b * d->seqlen + t) * H + h) * P;
                for (int64_t p = 0; p < P; ++p) {
                    const double zv = bf16_to_double(zr[p]);
                    yr[p] *= zv / (1.0 + exp(-zv));
                }
            }
        }
    }
    free(xv);
    free(bv);
    free(cv);
}

/* state (P,N) float/double layout <-> working state hs (N,P) double */
static void load_state_f32(double* hs, const float* st, int64_t P, int64_t N) {
    for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) hs[n * P + p] = (double)st[p * N + n];
}
static void store_state(double* dst, const double* hs, int64_t P, int64_t N) {
    for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) dst[p * N + n] = hs[n * P + p];
}

/* ------------------------------------------------------------ forward */

typedef struct {
    inputs_t in;
    const float* init;       /* (batch, H, P, N) or NULL */
    const int64_t* units;    /* unit u -> b * H + h */
    double* y;               /* per unit (L, P) */
    double* final_state;     /* per unit (P, N) or NULL */
    double* chunk_starts;    /* per unit (nc, P, N) or NULL */
} fwd_ctx_t;

static void fwd_unit(void* vctx, int64_t u) {
    fwd_ctx_t* c = (fwd_ctx_t*)vctx;
    const dims_t* d = c->in.d;
    const int64_t H = d->nheads, P = d->headdim, N = d->dstate, L = d->seqlen;
    const int64_t b = c->units[u] / H, h = c->units[u] % H;
    const int64_t Q = d->chunk_size, nc = nchunks_of(d);
    double* hs = (double*)calloc((size_t)(N * P), sizeof(double));
    if (c->init != NULL) load_state_f32(hs, c->init + (b * H + h) * P * N, P, N);
    double* y = c->y + u * L * P;
    for (int64_t ci = 0; ci < nc; ++ci) {
        const int64_t t0 = ci * Q, t1 = (t0 + Q < L) ? t0 + Q : L;
        if (c->chunk_starts != NULL) store_state(c->chunk_starts + (u * nc + ci) * P * N, hs, P, N);
        recur_tokens(&c->in, b, h, t0, t1, hs, y + t0 * P);
    }
    if (c->final_state != NULL) store_state(c->final_state + u * P * N, hs, P, N);
    free(hs);
}

/*
 * ssd_oracle_forward: y, the state before every chunk and the final state,
 * for the listed (batch, head) units, by the token-by-token recurrence.
 * Returns the number of threads used, or -1 on bad arguments.
 */
int ssd_oracle_forward(const uint16_t* x, const float* dt, const float* A, const uint16_t* B,
                       const uint16_t* C, const float* D, const float* init,
                       int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                       int64_t ngroups, int64_t dstate, int64_t chunk_size,
                       const int64_t* units, int64_t nunits,
                       double* y, double* final_state, double* chunk_starts, int nthreads) {
    if (!x || !dt || !A || !B || !C || !units || !y) return -1;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 ||
        chunk_size <= 0 || nheads % ngroups != 0 || nunits <= 0)
        return -1;
    dims_t d = {batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size};
    fwd_ctx_t ctx = {{&d, x, B, C, dt, A, D, NULL}, init, units, y, final_state, chunk_starts};
    return run_units(fwd_unit, &ctx, nunits, nthreads);
}

/*
 * ssd_oracle_forward_opts: ssd_oracle_forward with the input-side options
 * (see opts_t): dt_bias (H) or NULL, dt_softplus, dt_limit with [dt_min,
 * dt_max], D_per_channel (D is (H, P)), z (x's layout, bf16) or NULL.
 */
int ssd_oracle_forward_opts(const uint16_t* x, const float* dt, const float* A, const uint16_t* B,
                            const uint16_t* C, const float* D, const float* init,
                            int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                            int64_t ngroups, int64_t dstate, int64_t chunk_size,
                            const float* dt_bias, int dt_softplus, int dt_limit, double dt_min, double dt_max,
                            int D_per_channel, const uint16_t* z,
                            const int64_t* units, int64_t nunits,
                            double* y, double* final_state, double* chunk_starts, int nthreads) {
    if (!x || !dt || !A || !B || !C || !units || !y) return -1;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 ||
        chunk_size <= 0 || nheads % ngroups != 0 || nunits <= 0)
        return -1;
    if (dt_limit && !(dt_min <= dt_max)) return -1;
    dims_t d = {batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size};
    opts_t o = {dt_bias, dt_softplus, dt_limit, dt_min, dt_max, D_per_channel, z};
    fwd_ctx_t ctx = {{&d, x, B, C, dt, A, D, &o}, init, units, y, final_state, chunk_starts};
    return run_units(fwd_unit, &ctx, nunits, nthreads);
}

/* ------------------------------------------------------- chunk states */

typedef struct {
    inputs_t in;
    const int64_t* units;
    double* S; /* per unit (nc, P, N) */
} cst_ctx_t;

static void cst_unit(void* vctx, int64_t u) {
    cst_ctx_t* c = (cst_ctx_t*)vctx;
    const dims_t* d = c->in.d;
    const int64_t H = d->nheads, P = d->headdim, N = d->dstate, L = d->seqlen;
    const int64_t b = c->units[u] / H, h = c->units[u] % H;
    const int64_t Q = d->chunk_size, nc = nchunks_of(d);
    double* hs = (double*)malloc(sizeof(double) * (size_t)(N * P));
    for (int64_t ci = 0; ci < nc; ++ci) {
        const int64_t t0 = ci * Q, t1 = (t0 + Q < L) ? t0 + Q : L;
        memset(hs, 0, sizeof(double) * (size_t)(N * P));
        recur_tokens(&c->in, b, h, t0, t1, hs, NULL);
        store_state(c->S + (u * nc + ci) * P * N, hs, P, N);
    }
    free(hs);
}

/*
 * ssd_oracle_chunk_states: for every chunk, the state reached by running the
 * recurrence over that chunk alone from a zero state (the chunk's own
 * contribution, which the jump formula writes as one product of the stacked
 * b and x vectors once the decay weights are folded in).
 */
int ssd_oracle_chunk_states(const uint16_t* x, const float* dt, const float* A, const uint16_t* B,
                            int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                            int64_t ngroups, int64_t dstate, int64_t chunk_size,
                            const int64_t* units, int64_t nunits, double* S, int nthreads) {
    if (!x || !dt || !A || !B || !units || !S) return -1;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 ||
        chunk_size <= 0 || nheads % ngroups != 0 || nunits <= 0)
        return -1;
    dims_t d = {batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size};
    cst_ctx_t ctx = {{&d, x, B, NULL, dt, A, NULL, NULL}, units, S};
    return run_units(cst_unit, &ctx, nunits, nthreads);
}

/* --------------------------------------------------------- chunk scan */

typedef struct {
    inputs_t in;
    const float* states; /* full (batch, nc, H, P, N) */
    const int64_t* units;
    double* y;           /* per unit (L, P) */
} csc_ctx_t;

static void csc_unit(void* vctx, int64_t u) {
    csc_ctx_t* c = (csc_ctx_t*)vctx;
    const dims_t* d = c->in.d;
    const int64_t H = d->nheads, P = d->headdim, N = d->dstate, L = d->seqlen;
    const int64_t b = c->units[u] / H, h = c->units[u] % H;
    const int64_t Q = d->chunk_size, nc = nchunks_of(d);
    double* hs = (double*)malloc(sizeof(double) * (size_t)(N * P));
    double* y = c->y + u * L * P;
    for (int64_t ci = 0; ci < nc; ++ci) {
        const int64_t t0 = ci * Q, t1 = (t0 + Q < L) ? t0 + Q : L;
        load_state_f32(hs, c->states + ((b * nc + ci) * H + h) * P * N, P, N);
        recur_tokens(&c->in, b, h, t0, t1, hs, y + t0 * P);
    }
    free(hs);
}

/*
 * ssd_oracle_chunk_scan: outputs when every chunk starts from the given
 * chunk-start state (compute_out's role: output of the chunk from its start
 * state plus the chunk's own tokens and the skip term).
 */
int ssd_oracle_chunk_scan(const uint16_t* x, const float* dt, const float* A, const uint16_t* B,
                          const uint16_t* C, const float* D, const float* states,
                          int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                          int64_t ngroups, int64_t dstate, int64_t chunk_size,
                          const int64_t* units, int64_t nunits, double* y, int nthreads) {
    if (!x || !dt || !A || !B || !C || !states || !units || !y) return -1;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 ||
        chunk_size <= 0 || nheads % ngroups != 0 || nunits <= 0)
        return -1;
    dims_t d = {batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size};
    csc_ctx_t ctx = {{&d, x, B, C, dt, A, D, NULL}, states, units, y};
    return run_units(csc_unit, &ctx, nunits, nthreads);
}

/* ------------------------------------------------------- dA cumsum */

/*
 * ssd_oracle_dA_cumsum: per (b, h, chunk c, position i), the inclusive sum
 * over j <= i of dt[b, cQ+j, h] * A[h], times log2(e) ([devotd] section 2,
 * the chunk_cumsum kernel: product of decay rate and time interval,
 * accumulated inside the chunk, kept in base-2 log units).  Positions past
 * the end of the sequence contribute zero.  Also returns dt itself in the
 * same (b, H, nc, Q) layout (zero past the end).
 */
int ssd_oracle_dA_cumsum(const float* dt, const float* A, int64_t batch, int64_t seqlen,
                         int64_t nheads, int64_t chunk_size, double* cs, double* dt_t) {
    if (!dt || !A || !cs) return -1;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || chunk_size <= 0) return -1;
    const int64_t Q = chunk_size, nc = (seqlen + Q - 1) / Q, H = nheads;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t c = 0; c < nc; ++c) {
                double run = 0.0;
                for (int64_t i = 0; i < Q; ++i) {
                    const int64_t t = c * Q + i;
                    const double v = (t < seqlen) ? (double)dt[(b * seqlen + t) * H + h] : 0.0;
                    run += v * (double)A[h];
                    const int64_t o = ((b * H + h) * nc + c) * Q + i;
                    cs[o] = run * LOG2E_D;
                    if (dt_t != NULL) dt_t[o] = v;
                }
            }
    return 0;
}

/* ---------------------------------------------------- state passing */

/*
 * ssd_oracle_state_passing: the sequential hop across chunks
 * ([devotd] section 2, fwd_pass_state; [disconfirmai] jump formula):
 *     h_0 = init (or 0);  states[c] = h_c;
 *     h_{c+1} = 2^(cs[b,h,c,Q-1]) * h_c + S[c];   final = h_nc
 * S and states are (batch, nc, H, P, N); cs is (batch, H, nc, Q) in log2
 * units; init/final are (batch, H, P, N).
 */
int ssd_oracle_state_passing(const float* S, const float* cs, const float* init,
                             int64_t batch, int64_t nchunks, int64_t nheads, int64_t headdim,
                             int64_t dstate, int64_t chunk_size, double* states,
                             double* final_state) {
    if (!S || !cs || !states) return -1;
    if (batch <= 0 || nchunks <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || chunk_size <= 0)
        return -1;
    const int64_t H = nheads, PN = headdim * dstate, nc = nchunks, Q = chunk_size;
    double* hcur = (double*)malloc(sizeof(double) * (size_t)PN);
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t e = 0; e < PN; ++e)
                hcur[e] = (init != NULL) ? (double)init[(b * H + h) * PN + e] : 0.0;
            for (int64_t c = 0; c < nc; ++c) {
                const double decay = exp2((double)cs[((b * H + h) * nc + c) * Q + (Q - 1)]);
                const int64_t o = ((b * nc + c) * H + h) * PN;
                for (int64_t e = 0; e < PN; ++e) {
                    states[o + e] = hcur[e];
                    hcur[e] = decay * hcur[e] + (double)S[o + e];
                }
            }
            if (final_state != NULL)
                for (int64_t e = 0; e < PN; ++e) final_state[(b * H + h) * PN + e] = hcur[e];
        }
    free(hcur);
    return 0;
}

/* ------------------------------------------------------------ backward */

/*
 * Reverse mode of the recurrence (the pages describe no backward pass; this
 * is the adjoint of the forward definition above, derived here).  For a
 * scalar loss with dy = dLoss/dy (x's layout) and dfinal = dLoss/dfinal
 * ((P, N) per unit, or zero), let lam_t = dLoss/dhs_t, the gradient with
 * respect to the state after token t (N x P).  Going backward in time:
 *
 *     lam_{L-1} = dfinal + C_{L-1} dy_{L-1}^T
 *     lam_t     = a_{t+1} lam_{t+1} + C_t dy_t^T,      a_t = exp(dt_t A)
 *
 * and, per token t (hs_{t-1} the state before token t, hs_{-1} = init):
 *
 *     dx_t[p]  = dt_t sum_n B_t[n] lam_t[n][p] + D dy_t[p]
 *     dB_t[n] += dt_t sum_p lam_t[n][p] x_t[p]           (this head's share)
 *     dC_t[n] += sum_p hs_t[n][p] dy_t[p]                 (this head's share)
 *     ddt_t    = A a_t <lam_t, hs_{t-1}> + sum_{n,p} lam_t[n][p] B_t[n] x_t[p]
 *     dA      += dt_t a_t <lam_t, hs_{t-1}>
 *     dD      += sum_p x_t[p] dy_t[p]
 *     dinit    = a_0 lam_0
 *
 * The states hs_t are recomputed segment by segment from checkpoints taken
 * in a first forward sweep (a memory bound for the oracle, not part of the
 * method).
 */
typedef struct {
    inputs_t in;
    const float* init;      /* (batch, H, P, N) or NULL */
    const uint16_t* dy;     /* (batch, L, H, P) bf16 */
    const float* dfinal;    /* (batch, H, P, N) or NULL */
    const int64_t* units;
    double *dx, *dB, *dC, *ddt, *dA, *dD, *dinit; /* per unit: (L,P) (L,N) (L,N) (L) (1) (1) (P,N) */
    double* ddt_direct; /* per unit (L) or NULL: the second term of ddt alone, <lam_t, B_t x_t^T> */
    /* Scales, each NULL or per unit in the layout of its gradient: the sum of the magnitudes of the
     * products the gradient adds up (dx: dt sum_n |B lam| + |D dy|; dB: dt sum_p |lam x|; dC:
     * sum_p |hs dy|; ddt: |A| a sum |lam hs_prev| + sum |lam B x|; dA: sum_t dt a sum |lam hs_prev|;
     * dD: sum_t sum_p |x dy|; dinit: the adjoint's terms |C_t dy_t^T| and |dfinal|, each decayed to
     * the start as lam is). */
    double *dx_s, *dB_s, *dC_s, *ddt_s, *dA_s, *dD_s, *dinit_s;
} bwd_ctx_t;

static void bwd_unit(void* vctx, int64_t u) {
    bwd_ctx_t* c = (bwd_ctx_t*)vctx;
    const dims_t* d = c->in.d;
    const int64_t H = d->nheads, P = d->headdim, N = d->dstate, L = d->seqlen, G = d->ngroups;
    const int64_t b = c->units[u] / H, h = c->units[u] % H, g = h / (H / G);
    const double A = (double)c->in.A[h];
    const double Dh = (c->in.D == NULL) ? 0.0 : (double)c->in.D[h];
    int64_t K = 16;
    while (K * K < L) ++K; /* checkpoint spacing about sqrt(L) */
    const int64_t nseg = (L + K - 1) / K, NP = N * P;
    double* ck = (double*)calloc((size_t)(nseg * NP), sizeof(double));   /* state before each segment */
    double* seg = (double*)malloc(sizeof(double) * (size_t)((K + 1) * NP)); /* states through a segment */
    double* lam = (double*)calloc((size_t)NP, sizeof(double));
    double* lam_abs = (double*)calloc((size_t)NP, sizeof(double)); /* the same over |terms| (dinit's scale) */
    double* xv = (double*)malloc(sizeof(double) * (size_t)P);
    double* yv = (double*)malloc(sizeof(double) * (size_t)P);
    double* bv = (double*)malloc(sizeof(double) * (size_t)N);
    double* cv = (double*)malloc(sizeof(double) * (size_t)N);
    /* forward sweep: checkpoints */
    double* hs = seg;
    memset(hs, 0, sizeof(double) * (size_t)NP);
    if (c->init != NULL) load_state_f32(hs, c->init + (b * H + h) * P * N, P, N);
    for (int64_t s = 0; s < nseg; ++s) {
        const int64_t t0 = s * K, t1 = (t0 + K < L) ? t0 + K : L;
        memcpy(ck + s * NP, hs, sizeof(double) * (size_t)NP);
        recur_tokens(&c->in, b, h, t0, t1, hs, NULL);
    }
    /* backward sweep */
    if (c->dfinal != NULL) {
        load_state_f32(lam, c->dfinal + (b * H + h) * P * N, P, N);
        for (int64_t e = 0; e < NP; ++e) lam_abs[e] = fabs(lam[e]);
    }
    double dA = 0.0, dD = 0.0, dA_abs = 0.0, dD_abs = 0.0;
    double* dx = c->dx + u * L * P;
    double* dB = c->dB + u * L * N;
    double* dC = c->dC + u * L * N;
    double* ddt = c->ddt + u * L;
    for (int64_t s = nseg - 1; s >= 0; --s) {
        const int64_t t0 = s * K, t1 = (t0 + K < L) ? t0 + K : L;
        memcpy(seg, ck + s * NP, sizeof(double) * (size_t)NP);
        for (int64_t t = t0; t < t1; ++t) { /* seg[i + 1] = state after token t0 + i */
            memcpy(seg + (t - t0 + 1) * NP, seg + (t - t0) * NP, sizeof(double) * (size_t)NP);
            recur_tokens(&c->in, b, h, t, t + 1, seg + (t - t0 + 1) * NP, NULL);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const double* hprev = seg + (t - t0) * NP;
            const double* hcur = seg + (t - t0 + 1) * NP;
            const double dtv = (double)c->in.dt[(b * L + t) * H + h];
            const double a = exp(dtv * A);
            const uint16_t* xr = c->in.x + ((b * L + t) * H + h) * P;
            const uint16_t* dyr = c->dy + ((b * L + t) * H + h) * P;
            const uint16_t* br = c->in.B + ((b * L + t) * G + g) * N;
            const uint16_t* cr = c->in.C + ((b * L + t) * G + g) * N;
            for (int64_t p = 0; p < P; ++p) { xv[p] = bf16_to_double(xr[p]); yv[p] = bf16_to_double(dyr[p]); }
            for (int64_t n = 0; n < N; ++n) { bv[n] = bf16_to_double(br[n]); cv[n] = bf16_to_double(cr[n]); }
            /* lam_t = (carried) + C_t dy_t^T */
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p) {
                    lam[n * P + p] += cv[n] * yv[p];
                    lam_abs[n * P + p] += fabs(cv[n] * yv[p]);
                }
            double xdy = 0.0, xdy_abs = 0.0;
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0, acc_abs = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    acc += bv[n] * lam[n * P + p];
                    acc_abs += fabs(bv[n] * lam[n * P + p]);
                }
                dx[t * P + p] = dtv * acc + Dh * yv[p];
                if (c->dx_s != NULL) c->dx_s[(u * L + t) * P + p] = dtv * acc_abs + fabs(Dh * yv[p]);
                xdy += xv[p] * yv[p];
                xdy_abs += fabs(xv[p] * yv[p]);
            }
            double inner = 0.0, direct = 0.0, inner_abs = 0.0, direct_abs = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double lx = 0.0, hy = 0.0, lx_abs = 0.0, hy_abs = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    lx += lam[n * P + p] * xv[p];
                    hy += hcur[n * P + p] * yv[p];
                    inner += lam[n * P + p] * hprev[n * P + p];
                    lx_abs += fabs(lam[n * P + p] * xv[p]);
                    hy_abs += fabs(hcur[n * P + p] * yv[p]);
                    inner_abs += fabs(lam[n * P + p] * hprev[n * P + p]);
                }
                dB[t * N + n] = dtv * lx;
                dC[t * N + n] = hy;
                if (c->dB_s != NULL) c->dB_s[(u * L + t) * N + n] = dtv * lx_abs;
                if (c->dC_s != NULL) c->dC_s[(u * L + t) * N + n] = hy_abs;
                direct += bv[n] * lx;
                direct_abs += fabs(bv[n]) * lx_abs;
            }
            ddt[t] = A * a * inner + direct;
            if (c->ddt_direct != NULL) c->ddt_direct[u * L + t] = direct;
            if (c->ddt_s != NULL) c->ddt_s[u * L + t] = fabs(A) * a * inner_abs + direct_abs;
            dA += dtv * a * inner;
            dA_abs += dtv * a * inner_abs;
            dD += xdy;
            dD_abs += xdy_abs;
            for (int64_t e = 0; e < NP; ++e) { /* carry to token t - 1 */
                lam[e] *= a;
                lam_abs[e] *= a;
            }
        }
    }
    c->dA[u] = dA;
    c->dD[u] = dD;
    if (c->dA_s != NULL) c->dA_s[u] = dA_abs;
    if (c->dD_s != NULL) c->dD_s[u] = dD_abs;
    store_state(c->dinit + u * P * N, lam, P, N);
    if (c->dinit_s != NULL) store_state(c->dinit_s + u * P * N, lam_abs, P, N);
    free(ck); free(seg); free(lam); free(lam_abs); free(xv); free(yv); free(bv); free(cv);
}

/*
 * ssd_oracle_backward: per listed (batch, head) unit, the gradients of a
 * scalar loss with respect to x (dx, (L, P)), this head's share of dB and dC
 * ((L, N); a group's gradient is the sum over its heads), dt (ddt, (L)), A
 * and D (this unit's share, one value each) and init (dinit, (P, N)), given
 * dy (x's layout, bf16) and dfinal ((batch, H, P, N) f32, or NULL = 0).
 * ddt_direct (per unit (L), or NULL) receives ddt's second term alone; each
 * of dx_s, dB_s, dC_s, ddt_s, dA_s, dD_s, dinit_s (NULL or the layout of its gradient)
 * receives the sum of the magnitudes of the products that gradient adds up
 * (the scale of its rounding error in any method that rounds the factors).
 * Returns the number of threads used, or -1 on bad arguments.
 */
int ssd_oracle_backward(const uint16_t* x, const float* dt, const float* A, const uint16_t* B,
                        const uint16_t* C, const float* D, const float* init, const uint16_t* dy,
                        const float* dfinal, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                        int64_t ngroups, int64_t dstate, const int64_t* units, int64_t nunits,
                        double* dx, double* dB, double* dC, double* ddt, double* dA, double* dD,
                        double* dinit, double* ddt_direct, double* dx_s, double* dB_s, double* dC_s,
                        double* ddt_s, double* dA_s, double* dD_s, double* dinit_s, int nthreads) {
    if (!x || !dt || !A || !B || !C || !dy || !units || !dx || !dB || !dC || !ddt || !dA || !dD || !dinit)
        return -1;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 ||
        nheads % ngroups != 0 || nunits <= 0)
        return -1;
    dims_t d = {batch, seqlen, nheads, headdim, ngroups, dstate, seqlen};
    bwd_ctx_t ctx = {{&d, x, B, C, dt, A, D, NULL}, init, dy, dfinal, units, dx, dB, dC, ddt, dA, dD, dinit,
                     ddt_direct, dx_s, dB_s, dC_s, ddt_s, dA_s, dD_s, dinit_s};
    return run_units(bwd_unit, &ctx, nunits, nthreads);
}
