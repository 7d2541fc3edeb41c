/*
 * ssd_oracle.c -- TEST INFRASTRUCTURE ONLY.  Plain, slow, fp64 CPU oracle of
 * the selective state-space recurrence that the SSD layer forward computes,
 * and (oracle_s6_scan, at the end) of the Mamba-1 selective scan with a
 * decay per channel and state.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  It shares no code, header or constant with the CUDA
 * library; it does not include include/ssd.h.
 *
 * What it computes (per sequence s, head h, channel p, state n), fp64:
 *
 *     a_t      = exp(dt_t * A_h)                        (ZOH decay, A-bar)
 *     h_t[p,n] = a_t * h_{t-1}[p,n] + dt_t * x_t[p] * B_t[g,n]
 *     y_t[p]   = sum_n C_t[g,n] * h_t[p,n] + D_h * x_t[p]
 *     final    = h after the last token of the sequence
 *
 * Sources:
 *  - recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t^T h_t:
 *    "Mamba-2는 왜 Transformer와 닮았는가" (bdev.io), section
 *    "문제: 선형 복잡도만으로는 충분하지 않다".
 *  - ZOH discretisation A-bar = exp(dt A), B-bar ~= dt B, and the skip term
 *    y = C h + D x: "20.1 상태 공간 모델 (SSM)" (sungeuns.github.io), sec. 1
 *    (연속에서 이산으로: SSM의 수학) and the selective-scan loop of sec. 5.
 *  - scalar A per head, B/C shared by the heads of a group (SSD restriction):
 *    "Transformers are SSMs Review" (dimensionstp.github.io), sec. 3-2 (3)
 *    and (5).
 *  - variable-length packing: the state is cut at every sequence boundary,
 *    same review, sec. 3-2 (6).
 *
 * Readings where the pages are silent: head h uses group floor(h*G/H); D is
 * one scalar per head (NULL means 0); init NULL means a zero state; the
 * output y_t sees the updated state h_t (the loop updates h before reading
 * it).
 *
 * Layouts (row-major, flattened token index bt = b*T + t, or the packed
 * token index when cu_seqlens is given):
 *   x  [ntok, H, P]   dt [ntok, H]   A [H]   B, C [ntok, G, N]   D [H]
 *   init/final [nseq, H, P, N]       y [ntok, H, P]
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *x, *dt, *A, *B, *C, *D, *init;
    const int64_t *seq_begin, *seq_end; /* token range of each sequence */
    int nseq, H, P, N, G;
    double *y, *final_states;
    int nthreads;
    int tid;
} scan_job;

/* One (sequence, head) unit: the plain token-by-token loop. */
static void scan_unit(const scan_job *J, int s, int h, double *state) {
    const int H = J->H, P = J->P, N = J->N, G = J->G;
    const int g = (int)(((int64_t)h * G) / H);
    const double Ah = J->A[h];
    const double Dh = J->D ? J->D[h] : 0.0;
    const size_t PN = (size_t)P * N;
    if (J->init)
        memcpy(state, J->init + ((size_t)s * H + h) * PN, PN * sizeof(double));
    else
        memset(state, 0, PN * sizeof(double));
    for (int64_t t = J->seq_begin[s]; t < J->seq_end[s]; ++t) {
        const double dtt = J->dt[t * H + h];
        const double a = exp(dtt * Ah);
        const double *xt = J->x + ((size_t)t * H + h) * P;
        const double *Bt = J->B + ((size_t)t * G + g) * N;
        const double *Ct = J->C + ((size_t)t * G + g) * N;
        double *yt = J->y + ((size_t)t * H + h) * P;
        for (int p = 0; p < P; ++p) {
            double *hp = state + (size_t)p * N;
            const double u = dtt * xt[p];
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                hp[n] = a * hp[n] + u * Bt[n];
                acc += Ct[n] * hp[n];
            }
            yt[p] = acc + Dh * xt[p];
        }
    }
    if (J->final_states)
        memcpy(J->final_states + ((size_t)s * H + h) * PN, state, PN * sizeof(double));
}

static void *scan_worker(void *arg) {
    const scan_job *J = (const scan_job *)arg;
    double *state = (double *)malloc((size_t)J->P * J->N * sizeof(double));
    if (!state) return (void *)1;
    const int64_t units = (int64_t)J->nseq * J->H;
    for (int64_t u = J->tid; u < units; u += J->nthreads)
        scan_unit(J, (int)(u / J->H), (int)(u % J->H), state);
    free(state);
    return NULL;
}

/*
 * Full-sequence oracle.  cu_seqlens == NULL: `batch` independent rows of
 * `seqlen` tokens (nseq = batch).  Otherwise batch must be 1 and the nseq
 * sequences are the packed ranges [cu_seqlens[s], cu_seqlens[s+1]).
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
int oracle_ssd_scan(const double *x, const double *dt, const double *A,
                    const double *B, const double *C, const double *D,
                    int batch, int seqlen, int H, int P, int N, int G,
                    const double *init, const int32_t *cu_seqlens, int nseq,
                    double *y, double *final_states, int nthreads) {
    if (!x || !dt || !A || !B || !C || !y) return -1;
    if (batch < 0 || seqlen < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return -1;
    if (cu_seqlens && (batch != 1 || nseq < 0)) return -1;
    if (!cu_seqlens) nseq = batch;
    if (nthreads < 1) nthreads = 1;
    int64_t *rng = (int64_t *)malloc(2 * (size_t)(nseq > 0 ? nseq : 1) * sizeof(int64_t));
    if (!rng) return -2;
    for (int s = 0; s < nseq; ++s) {
        if (cu_seqlens) {
            rng[s] = cu_seqlens[s];
            rng[nseq + s] = cu_seqlens[s + 1];
            if (rng[s] < 0 || rng[nseq + s] < rng[s] || rng[nseq + s] > seqlen) {
                free(rng);
                return -1;
            }
        } else {
            rng[s] = (int64_t)s * seqlen;
            rng[nseq + s] = (int64_t)(s + 1) * seqlen;
        }
    }
    scan_job *jobs = (scan_job *)calloc((size_t)nthreads, sizeof(scan_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(rng); free(jobs); free(th);
        return -2;
    }
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        scan_job J = {x, dt, A, B, C, D, init, rng, rng + nseq, nseq, H, P, N, G,
                      y, final_states, nthreads, i};
        jobs[i] = J;
    }
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, scan_worker, &jobs[i]) != 0) break;
        started = i;
    }
    if (scan_worker(&jobs[0]) != NULL) rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    /* threads that failed to start: run their share here */
    for (int i = started + 1; i < nthreads; ++i)
        if (scan_worker(&jobs[i]) != NULL) rc = -2;
    free(rng); free(jobs); free(th);
    return rc;
}

/*
 * One decode step, in place on `state` [batch, H, P, N]: one iteration of the
 * loop above for a single new token per batch row.
 *   x [batch, H, P]  dt [batch, H]  B, C [batch, G, N]  y [batch, H, P]
 */
int oracle_ssd_step(double *state, const double *x, const double *dt,
                    const double *A, const double *B, const double *C,
                    const double *D, int batch, int H, int P, int N, int G,
                    double *y) {
    if (!state || !x || !dt || !A || !B || !C || !y) return -1;
    if (batch < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return -1;
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < H; ++h) {
            const int g = (int)(((int64_t)h * G) / H);
            const double dtt = dt[(size_t)b * H + h];
            const double a = exp(dtt * A[h]);
            const double Dh = D ? D[h] : 0.0;
            const double *xt = x + ((size_t)b * H + h) * P;
            const double *Bt = B + ((size_t)b * G + g) * N;
            const double *Ct = C + ((size_t)b * G + g) * N;
            double *st = state + ((size_t)b * H + h) * P * N;
            for (int p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int n = 0; n < N; ++n) {
                    double *e = st + (size_t)p * N + n;
                    *e = a * *e + dtt * xt[p] * Bt[n];
                    acc += Ct[n] * *e;
                }
                y[((size_t)b * H + h) * P + p] = acc + Dh * xt[p];
            }
        }
    }
    return 0;
}

/*
 * Selective scan with a decay per (channel, state): the S6 layer of Mamba-1,
 * the sequential loop of "20.1 상태 공간 모델 (SSM)" (sungeuns.github.io),
 * sec. 5 (Selective SSM forward), with an optional initial state added.
 * Per batch row b, channel d in [0, Dm), state n in [0, N), fp64:
 *
 *     dA_t[d,n] = exp(dt_t[d] * A[d,n])                 (ZOH decay, A-bar)
 *     h_t[d,n]  = dA_t[d,n] * h_{t-1}[d,n] + dt_t[d] * B_t[n] * x_t[d]
 *     y_t[d]    = sum_n h_t[d,n] * C_t[n] + D[d] * x_t[d]
 *
 * The input term is dt B x (B-bar ~= dt B, the same section, sec. 1); y_t
 * reads the updated state, as the loop does.  B and C are shared by all
 * channels; dt is per channel.
 * Layouts: x, dt, y [batch, seqlen, Dm]; A [Dm, N]; B, C [batch, seqlen, N];
 * D [Dm] or NULL (0); init, final [batch, Dm, N] (init NULL: zero state).
 */
typedef struct {
    const double *x, *dt, *A, *B, *C, *D, *init;
    int batch, L, Dm, N;
    double *y, *final_states;
    int nthreads, tid;
} s6_job;

static void *s6_worker(void *arg) {
    const s6_job *J = (const s6_job *)arg;
    const int L = J->L, Dm = J->Dm, N = J->N;
    double *h = (double *)malloc((size_t)N * sizeof(double));
    if (!h) return (void *)1;
    const int64_t units = (int64_t)J->batch * Dm;
    for (int64_t u = J->tid; u < units; u += J->nthreads) {
        const int b = (int)(u / Dm), d = (int)(u % Dm);
        const double *Ad = J->A + (size_t)d * N;
        const double Dd = J->D ? J->D[d] : 0.0;
        for (int n = 0; n < N; ++n)
            h[n] = J->init ? J->init[((size_t)b * Dm + d) * N + n] : 0.0;
        for (int t = 0; t < L; ++t) {
            const size_t bt = (size_t)b * L + t;
            const double dtt = J->dt[bt * Dm + d];
            const double xt = J->x[bt * Dm + d];
            const double *Bt = J->B + bt * N;
            const double *Ct = J->C + bt * N;
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                const double dA = exp(dtt * Ad[n]);
                h[n] = dA * h[n] + dtt * Bt[n] * xt;
                acc += h[n] * Ct[n];
            }
            J->y[bt * Dm + d] = acc + Dd * xt;
        }
        if (J->final_states)
            memcpy(J->final_states + ((size_t)b * Dm + d) * N, h, (size_t)N * sizeof(double));
    }
    free(h);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
int oracle_s6_scan(const double *x, const double *dt, const double *A, const double *B,
                   const double *C, const double *D, int batch, int seqlen, int Dm, int N,
                   const double *init, double *y, double *final_states, int nthreads) {
    if (!x || !dt || !A || !B || !C || !y) return -1;
    if (batch < 0 || seqlen < 0 || Dm <= 0 || N <= 0) return -1;
    if (nthreads < 1) nthreads = 1;
    s6_job *jobs = (s6_job *)calloc((size_t)nthreads, sizeof(s6_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th);
        return -2;
    }
    for (int i = 0; i < nthreads; ++i) {
        s6_job J = {x, dt, A, B, C, D, init, batch, seqlen, Dm, N, y, final_states, nthreads, i};
        jobs[i] = J;
    }
    int rc = 0, started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, s6_worker, &jobs[i]) != 0) break;
        started = i;
    }
    if (s6_worker(&jobs[0]) != NULL) rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    for (int i = started + 1; i < nthreads; ++i)
        if (s6_worker(&jobs[i]) != NULL) rc = -2;
    free(jobs); free(th);
    return rc;
}

/*
 * Backward of the SSD layer (reverse-mode derivative of the recurrence at
 * the top of this file), fp64, single-threaded.  For a scalar loss L with
 * dL/dy = dy and dL/dfinal = dfinal (NULL: 0), with G_t = dL/dh_t:
 *
 *     G_{T-1} = dfinal + dy_{T-1} C_{T-1}^T;  G_{t-1} = a_t G_t + dy_{t-1} C_{t-1}^T
 *     dx_t[p] = dt_t sum_n G_t[p,n] B_t[n] + D dy_t[p]
 *     dB_t[n] += dt_t sum_p G_t[p,n] x_t[p]          (summed over the group's heads)
 *     dC_t[n] += sum_p dy_t[p] h_t[p,n]              (summed over the group's heads)
 *     ddt_t    = sum_{p,n} G_t[p,n] (A a_t h_{t-1}[p,n] + x_t[p] B_t[n])
 *     dA      += sum_t dt_t a_t sum_{p,n} G_t[p,n] h_{t-1}[p,n]
 *     dD      += sum_t sum_p dy_t[p] x_t[p]
 *     dinit    = a_0 G_0                               (= dL/dh_{-1})
 *
 * with a_t = exp(dt_t A), h_{-1} = init (or 0).  Batch mode only.  Layouts as
 * the forward: dy, dx [batch*seqlen, H, P]; ddt [batch*seqlen, H]; dB, dC
 * [batch*seqlen, G, N]; dA, dD [H]; dfinal, dinit [batch, H, P, N].  dD and
 * dinit may be NULL.  Returns 0, -1 (bad arguments) or -2 (allocation).
 */
int oracle_ssd_bwd(const double *x, const double *dt, const double *A, const double *B,
                   const double *C, const double *D, int batch, int seqlen, int H, int P, int N,
                   int G, const double *init, const double *dy, const double *dfinal,
                   double *dx, double *ddt, double *dA, double *dB, double *dC, double *dD,
                   double *dinit) {
    if (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dA || !dB || !dC) return -1;
    if (batch < 0 || seqlen < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return -1;
    const size_t PN = (size_t)P * N;
    const size_t ntok = (size_t)batch * seqlen;
    double *hs = (double *)malloc((size_t)(seqlen + 1) * PN * sizeof(double));
    double *Gs = (double *)malloc(PN * sizeof(double));
    if (!hs || !Gs) {
        free(hs); free(Gs);
        return -2;
    }
    memset(dA, 0, (size_t)H * sizeof(double));
    if (dD) memset(dD, 0, (size_t)H * sizeof(double));
    memset(dB, 0, ntok * G * N * sizeof(double));
    memset(dC, 0, ntok * G * N * sizeof(double));
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < H; ++h) {
            const int g = (int)(((int64_t)h * G) / H);
            const double Ah = A[h];
            const double Dh = D ? D[h] : 0.0;
            /* forward: hs[t + 1] = h_t, hs[0] = h_{-1} */
            for (size_t e = 0; e < PN; ++e)
                hs[e] = init ? init[((size_t)b * H + h) * PN + e] : 0.0;
            for (int t = 0; t < seqlen; ++t) {
                const size_t bt = (size_t)b * seqlen + t;
                const double dtt = dt[bt * H + h], a = exp(dtt * Ah);
                const double *xt = x + (bt * H + h) * P;
                const double *Bt = B + (bt * G + g) * N;
                for (int p = 0; p < P; ++p)
                    for (int n = 0; n < N; ++n)
                        hs[(t + 1) * PN + p * N + n] =
                            a * hs[t * PN + p * N + n] + dtt * xt[p] * Bt[n];
            }
            /* backward */
            for (size_t e = 0; e < PN; ++e)
                Gs[e] = dfinal ? dfinal[((size_t)b * H + h) * PN + e] : 0.0;
            for (int t = seqlen - 1; t >= 0; --t) {
                const size_t bt = (size_t)b * seqlen + t;
                const double dtt = dt[bt * H + h], a = exp(dtt * Ah);
                const double *xt = x + (bt * H + h) * P;
                const double *dyt = dy + (bt * H + h) * P;
                const double *Bt = B + (bt * G + g) * N;
                const double *Ct = C + (bt * G + g) * N;
                const double *ht = hs + (t + 1) * PN, *hp = hs + t * PN;
                for (int p = 0; p < P; ++p)
                    for (int n = 0; n < N; ++n) Gs[p * N + n] += dyt[p] * Ct[n];
                double s_h = 0.0, s_xb = 0.0;
                for (int p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n) {
                        const double gv = Gs[p * N + n];
                        acc += gv * Bt[n];
                        s_h += gv * hp[p * N + n];
                        s_xb += gv * xt[p] * Bt[n];
                    }
                    dx[(bt * H + h) * P + p] = dtt * acc + Dh * dyt[p];
                    if (dD) dD[h] += dyt[p] * xt[p];
                }
                for (int n = 0; n < N; ++n) {
                    double gb = 0.0, gc = 0.0;
                    for (int p = 0; p < P; ++p) {
                        gb += Gs[p * N + n] * xt[p];
                        gc += dyt[p] * ht[p * N + n];
                    }
                    dB[(bt * G + g) * N + n] += dtt * gb;
                    dC[(bt * G + g) * N + n] += gc;
                }
                ddt[bt * H + h] = Ah * a * s_h + s_xb;
                dA[h] += dtt * a * s_h;
                for (size_t e = 0; e < PN; ++e) Gs[e] *= a;
            }
            if (dinit) memcpy(dinit + ((size_t)b * H + h) * PN, Gs, PN * sizeof(double));
        }
    }
    free(hs);
    free(Gs);
    return 0;
}
