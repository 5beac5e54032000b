/*
 * gla_oracle.c -- plain, slow, double-precision CPU oracle for the Simple
 * Gated Linear Attention (Simple GLA) mixer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check of the entry module
 * and the CPU-baseline / reference leg of the benchmark use it. It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Source: "Beyond the KV cache: Training and serving i14's Laplace 3B linear
 * attention model on AWS Trainium2 with native PyTorch",
 *   - section "i14 and the Laplace 3B architecture", paragraph "GLA mixer"
 *     (the "GLA recurrent-state update equation" and the "GLA state-readout
 *     equation"): per head h a dk x dv state, S_t = lambda_h * S_{t-1} +
 *     k_t v_t^T with a fixed per-head decay lambda_h, read out by the query;
 *   - section "Engineering challenges", "Challenge 1: Using native PyTorch on
 *     Trainium for GLA" (the "Chunked GLA intra-chunk output" and "Chunked
 *     GLA state update" equations, Figure 3): masked linear attention inside
 *     a chunk plus the running state, and the state advanced by lambda^C;
 *   - "Challenge 3: Backward-pass unrolling for a sequential recurrence":
 *     gradients flow through every serial state update.
 *
 * The equations themselves are images that did not survive extraction. The
 * readings used here (all stated in the design notes):
 *   - readout after the update: o_t = scale * S_t^T q_t;
 *   - the scale multiplies the readout only; S and hT are unscaled;
 *   - lambda = exp(log_lambda[h]); lambda^0 = 1 even when lambda = 0;
 *   - S_0 = h0 (zero when h0 is NULL).
 *
 * Layouts: q, k, do, dq, dk [B,T,H,dk]; v, o, dv [B,T,H,dv];
 * h0, hT, dhT, dh0 [B,H,dk,dv]; decode q, k [N,H,dk], v, o [N,H,dv],
 * S [N,H,dk,dv]. Everything is double. Work is split over independent
 * (b, h) pairs with pthreads; nothing else is reordered.
 *
 * Parity pins live in the test suite: brute force against the recurrence,
 * lambda = 1 (causal linear attention) and lambda = 0 special cases, the
 * closed-form final state, chunk-size invariance, split-call invariance,
 * linearity, hand-worked fixtures and central finite differences.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- threads */
typedef void (*unit_fn)(void *ctx, long unit);

typedef struct {
    unit_fn fn;
    void *ctx;
    long n_units;
    long next;
    pthread_mutex_t lock;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        long u;
        pthread_mutex_lock(&p->lock);
        u = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (u >= p->n_units) break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_units(long n_units, int nthreads, unit_fn fn, void *ctx) {
    int nt = resolve_threads(nthreads);
    if (nt > n_units) nt = (int)(n_units > 0 ? n_units : 1);
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.n_units = n_units; p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    if (nt <= 1) {
        pool_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
        int started = 0;
        for (int i = 0; i < nt; ++i)
            if (pthread_create(&th[i], NULL, pool_worker, &p) == 0) ++started;
        if (started == 0) pool_worker(&p);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.lock);
}

int gla_oracle_threads(int nthreads) { return resolve_threads(nthreads); }

/* lambda^n with lambda^0 = 1 (also for lambda = 0). */
static double lam_pow(double lam, long n) {
    if (n == 0) return 1.0;
    return pow(lam, (double)n);
}

/* ------------------------------------------------------------ arguments */
typedef struct {
    const double *q, *k, *v, *log_lambda, *h0, *do_, *dhT;
    double scale;
    long B, T, H, dk, dv, chunk;
    double *o, *hT, *dq, *dk_out, *dv_out, *dh0;
} args_t;

#define QIDX(a, b, t, h, i) ((((b) * (a)->T + (t)) * (a)->H + (h)) * (a)->dk + (i))
#define VIDX(a, b, t, h, j) ((((b) * (a)->T + (t)) * (a)->H + (h)) * (a)->dv + (j))
#define SIDX(a, b, h) (((b) * (a)->H + (h)) * (a)->dk * (a)->dv)

/* ------------------------------------------------- O2: recurrent forward */
/* The recurrence as the "GLA mixer" paragraph states it, one token at a time:
 *   S_t = lambda * S_{t-1} + k_t v_t^T,   o_t = scale * S_t^T q_t.         */
static void fwd_recurrent_unit(void *ctx, long unit) {
    const args_t *a = (const args_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv;
    double lam = exp(a->log_lambda[h]);
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    if (a->h0) memcpy(S, a->h0 + SIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    for (long t = 0; t < a->T; ++t) {
        const double *kt = a->k + QIDX(a, b, t, h, 0);
        const double *vt = a->v + VIDX(a, b, t, h, 0);
        const double *qt = a->q + QIDX(a, b, t, h, 0);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j)
                S[i * dv + j] = lam * S[i * dv + j] + kt[i] * vt[j];
        if (a->o) {
            double *ot = a->o + VIDX(a, b, t, h, 0);
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
                ot[j] = a->scale * acc;
            }
        }
    }
    if (a->hT) memcpy(a->hT + SIDX(a, b, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S);
}

int gla_oracle_fwd_recurrent(const double *q, const double *k, const double *v,
                             const double *log_lambda, const double *h0, double scale,
                             long B, long T, long H, long dk, long dv,
                             double *o, double *hT, int nthreads) {
    if (!q || !k || !v || !log_lambda || B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    args_t a; memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.log_lambda = log_lambda; a.h0 = h0; a.scale = scale;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.o = o; a.hT = hT;
    run_units(B * H, nthreads, fwd_recurrent_unit, &a);
    return 0;
}

/* ---------------------------------------------- O1: brute-force quadratic */
/* Unrolling the recurrence from S_0 = h0 (0-based t):
 *   o_t = scale * ( lambda^(t+1) h0^T q_t + sum_{u<=t} lambda^(t-u) (q_t.k_u) v_u )
 *   hT  = lambda^T h0 + sum_u lambda^(T-1-u) k_u v_u^T.
 * O(T^2); for tiny inputs only.                                             */
static void fwd_quadratic_unit(void *ctx, long unit) {
    const args_t *a = (const args_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv;
    double lam = exp(a->log_lambda[h]);
    const double *H0 = a->h0 ? a->h0 + SIDX(a, b, h) : NULL;
    for (long t = 0; t < a->T; ++t) {
        const double *qt = a->q + QIDX(a, b, t, h, 0);
        double *ot = a->o + VIDX(a, b, t, h, 0);
        for (long j = 0; j < dv; ++j) ot[j] = 0.0;
        if (H0) {
            double w = lam_pow(lam, t + 1);
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += H0[i * dv + j] * qt[i];
                ot[j] += w * acc;
            }
        }
        for (long u = 0; u <= t; ++u) {
            const double *ku = a->k + QIDX(a, b, u, h, 0);
            const double *vu = a->v + VIDX(a, b, u, h, 0);
            double qk = 0.0;
            for (long i = 0; i < dk; ++i) qk += qt[i] * ku[i];
            double w = lam_pow(lam, t - u) * qk;
            for (long j = 0; j < dv; ++j) ot[j] += w * vu[j];
        }
        for (long j = 0; j < dv; ++j) ot[j] *= a->scale;
    }
    if (a->hT) {
        double *S = a->hT + SIDX(a, b, h);
        double w0 = lam_pow(lam, a->T);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) S[i * dv + j] = H0 ? w0 * H0[i * dv + j] : 0.0;
        for (long u = 0; u < a->T; ++u) {
            const double *ku = a->k + QIDX(a, b, u, h, 0);
            const double *vu = a->v + VIDX(a, b, u, h, 0);
            double w = lam_pow(lam, a->T - 1 - u);
            for (long i = 0; i < dk; ++i)
                for (long j = 0; j < dv; ++j) S[i * dv + j] += w * ku[i] * vu[j];
        }
    }
}

int gla_oracle_fwd_quadratic(const double *q, const double *k, const double *v,
                             const double *log_lambda, const double *h0, double scale,
                             long B, long T, long H, long dk, long dv,
                             double *o, double *hT, int nthreads) {
    if (!q || !k || !v || !log_lambda || !o || B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    args_t a; memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.log_lambda = log_lambda; a.h0 = h0; a.scale = scale;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.o = o; a.hT = hT;
    run_units(B * H, nthreads, fwd_quadratic_unit, &a);
    return 0;
}

/* ------------------------------------------------ O5: chunked forward */
/* The chunked form of "Challenge 1" with chunk length C (0-based position i
 * inside a chunk of Cc valid tokens, S_prev the state entering the chunk):
 *   o_i   = scale * ( lambda^(i+1) S_prev^T q_i
 *                     + sum_{j<=i} lambda^(i-j) (q_i.k_j) v_j )   [intra-chunk output]
 *   S_new = lambda^Cc S_prev + sum_{j<Cc} lambda^(Cc-1-j) k_j v_j^T [chunk state update]
 * It is an exact regrouping of the recurrence; it serves to pin the chunk
 * equations, not as the CUDA path's reference.                              */
static void fwd_chunked_unit(void *ctx, long unit) {
    const args_t *a = (const args_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv, C = a->chunk;
    double lam = exp(a->log_lambda[h]);
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    double *Sn = (double *)calloc((size_t)(dk * dv), sizeof(double));
    if (a->h0) memcpy(S, a->h0 + SIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    for (long c0 = 0; c0 < a->T; c0 += C) {
        long Cc = a->T - c0 < C ? a->T - c0 : C;
        for (long i = 0; i < Cc; ++i) {
            const double *qi = a->q + QIDX(a, b, c0 + i, h, 0);
            double *oi = a->o ? a->o + VIDX(a, b, c0 + i, h, 0) : NULL;
            if (!oi) break;
            double wi = lam_pow(lam, i + 1);
            for (long jv = 0; jv < dv; ++jv) {
                double acc = 0.0;
                for (long r = 0; r < dk; ++r) acc += S[r * dv + jv] * qi[r];
                oi[jv] = wi * acc;
            }
            for (long j = 0; j <= i; ++j) {
                const double *kj = a->k + QIDX(a, b, c0 + j, h, 0);
                const double *vj = a->v + VIDX(a, b, c0 + j, h, 0);
                double qk = 0.0;
                for (long r = 0; r < dk; ++r) qk += qi[r] * kj[r];
                double w = lam_pow(lam, i - j) * qk;
                for (long jv = 0; jv < dv; ++jv) oi[jv] += w * vj[jv];
            }
            for (long jv = 0; jv < dv; ++jv) oi[jv] *= a->scale;
        }
        double wC = lam_pow(lam, Cc);
        for (long r = 0; r < dk * dv; ++r) Sn[r] = wC * S[r];
        for (long j = 0; j < Cc; ++j) {
            const double *kj = a->k + QIDX(a, b, c0 + j, h, 0);
            const double *vj = a->v + VIDX(a, b, c0 + j, h, 0);
            double w = lam_pow(lam, Cc - 1 - j);
            for (long r = 0; r < dk; ++r)
                for (long jv = 0; jv < dv; ++jv) Sn[r * dv + jv] += w * kj[r] * vj[jv];
        }
        double *tmp = S; S = Sn; Sn = tmp;
    }
    if (a->hT) memcpy(a->hT + SIDX(a, b, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S); free(Sn);
}

int gla_oracle_fwd_chunked(const double *q, const double *k, const double *v,
                           const double *log_lambda, const double *h0, double scale,
                           long B, long T, long H, long dk, long dv, long chunk,
                           double *o, double *hT, int nthreads) {
    if (!q || !k || !v || !log_lambda || chunk <= 0 || B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    args_t a; memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.log_lambda = log_lambda; a.h0 = h0; a.scale = scale;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk; a.o = o; a.hT = hT;
    run_units(B * H, nthreads, fwd_chunked_unit, &a);
    return 0;
}

/* ---------------------------------------------------- O3: backward */
/* Loss L = sum_t <do_t, o_t> + <dhT, hT>. With G_t = dL/dS_t (all paths):
 *   forward pass :  dq_t = scale * S_t do_t
 *   reverse pass :  G_{T-1} = dhT + scale q_{T-1} do_{T-1}^T,
 *                   G_{t-1} = lambda G_t + scale q_{t-1} do_{t-1}^T,
 *                   dk_t = G_t v_t,  dv_t = G_t^T k_t,  dh0 = lambda G_0.
 * Two passes over the sequence; nothing is stored between them.            */
static void bwd_unit(void *ctx, long unit) {
    const args_t *a = (const args_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv;
    double lam = exp(a->log_lambda[h]);
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    /* forward pass: dq */
    if (a->h0) memcpy(S, a->h0 + SIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    for (long t = 0; t < a->T; ++t) {
        const double *kt = a->k + QIDX(a, b, t, h, 0);
        const double *vt = a->v + VIDX(a, b, t, h, 0);
        const double *dot = a->do_ + VIDX(a, b, t, h, 0);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j)
                S[i * dv + j] = lam * S[i * dv + j] + kt[i] * vt[j];
        if (a->dq) {
            double *dqt = a->dq + QIDX(a, b, t, h, 0);
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long j = 0; j < dv; ++j) acc += S[i * dv + j] * dot[j];
                dqt[i] = a->scale * acc;
            }
        }
    }
    /* reverse pass: dk, dv, dh0 (S is reused as G) */
    if (a->dhT) memcpy(S, a->dhT + SIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
    for (long t = a->T - 1; t >= 0; --t) {
        const double *qt = a->q + QIDX(a, b, t, h, 0);
        const double *kt = a->k + QIDX(a, b, t, h, 0);
        const double *vt = a->v + VIDX(a, b, t, h, 0);
        const double *dot = a->do_ + VIDX(a, b, t, h, 0);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) S[i * dv + j] += a->scale * qt[i] * dot[j];
        if (a->dk_out) {
            double *dkt = a->dk_out + QIDX(a, b, t, h, 0);
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long j = 0; j < dv; ++j) acc += S[i * dv + j] * vt[j];
                dkt[i] = acc;
            }
        }
        if (a->dv_out) {
            double *dvt = a->dv_out + VIDX(a, b, t, h, 0);
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += S[i * dv + j] * kt[i];
                dvt[j] = acc;
            }
        }
        for (long r = 0; r < dk * dv; ++r) S[r] *= lam;
    }
    if (a->dh0) memcpy(a->dh0 + SIDX(a, b, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S);
}

int gla_oracle_bwd(const double *q, const double *k, const double *v,
                   const double *log_lambda, const double *h0, double scale,
                   const double *do_, const double *dhT,
                   long B, long T, long H, long dk, long dv,
                   double *dq, double *dk_out, double *dv_out, double *dh0, int nthreads) {
    if (!q || !k || !v || !log_lambda || !do_ || B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    args_t a; memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.log_lambda = log_lambda; a.h0 = h0; a.scale = scale;
    a.do_ = do_; a.dhT = dhT;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    a.dq = dq; a.dk_out = dk_out; a.dv_out = dv_out; a.dh0 = dh0;
    run_units(B * H, nthreads, bwd_unit, &a);
    return 0;
}

/* ---------------------------------------------- O6: chunked backward */
/* The backward of the chunked form, chunk by chunk (G the gradient of the
 * state leaving the chunk; S_prev the state entering it):
 *   dq_i = scale*( lambda^(i+1) S_prev do_i + sum_{j<=i} lambda^(i-j) (do_i.v_j) k_j )
 *   dk_j = scale*sum_{i>=j} lambda^(i-j) (do_i.v_j) q_i + lambda^(Cc-1-j) G v_j
 *   dv_j = scale*sum_{i>=j} lambda^(i-j) (q_i.k_j) do_i + lambda^(Cc-1-j) G^T k_j
 *   G   <- lambda^Cc G + scale * sum_i lambda^(i+1) q_i do_i^T   (to the previous chunk)
 *   dh0  = G after the first chunk.
 * Pins the chunk-level backward equations against O3.                        */
static void bwd_chunked_unit(void *ctx, long unit) {
    const args_t *a = (const args_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv, C = a->chunk, T = a->T;
    double lam = exp(a->log_lambda[h]);
    long nck = (T + C - 1) / C;
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    double *Sn = (double *)calloc((size_t)(dk * dv), sizeof(double));
    /* chunk order: dq with the state entering each chunk */
    if (a->h0) memcpy(S, a->h0 + SIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    for (long c = 0; c < nck; ++c) {
        long c0 = c * C, Cc = T - c0 < C ? T - c0 : C;
        for (long i = 0; i < Cc && a->dq; ++i) {
            const double *doi = a->do_ + VIDX(a, b, c0 + i, h, 0);
            double *dqi = a->dq + QIDX(a, b, c0 + i, h, 0);
            double wi = lam_pow(lam, i + 1);
            for (long r = 0; r < dk; ++r) {
                double acc = 0.0;
                for (long jv = 0; jv < dv; ++jv) acc += S[r * dv + jv] * doi[jv];
                dqi[r] = wi * acc;
            }
            for (long j = 0; j <= i; ++j) {
                const double *vj = a->v + VIDX(a, b, c0 + j, h, 0);
                const double *kj = a->k + QIDX(a, b, c0 + j, h, 0);
                double dv_ = 0.0;
                for (long jv = 0; jv < dv; ++jv) dv_ += doi[jv] * vj[jv];
                double w = lam_pow(lam, i - j) * dv_;
                for (long r = 0; r < dk; ++r) dqi[r] += w * kj[r];
            }
            for (long r = 0; r < dk; ++r) dqi[r] *= a->scale;
        }
        double wC = lam_pow(lam, Cc);
        for (long r = 0; r < dk * dv; ++r) Sn[r] = wC * S[r];
        for (long j = 0; j < Cc; ++j) {
            const double *kj = a->k + QIDX(a, b, c0 + j, h, 0);
            const double *vj = a->v + VIDX(a, b, c0 + j, h, 0);
            double w = lam_pow(lam, Cc - 1 - j);
            for (long r = 0; r < dk; ++r)
                for (long jv = 0; jv < dv; ++jv) Sn[r * dv + jv] += w * kj[r] * vj[jv];
        }
        double *tmp = S; S = Sn; Sn = tmp;
    }
    /* reverse chunk order: dk, dv and the state gradient G */
    if (a->dhT) memcpy(S, a->dhT + SIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
    for (long c = nck - 1; c >= 0; --c) {
        long c0 = c * C, Cc = T - c0 < C ? T - c0 : C;
        for (long j = 0; j < Cc; ++j) {
            const double *kj = a->k + QIDX(a, b, c0 + j, h, 0);
            const double *vj = a->v + VIDX(a, b, c0 + j, h, 0);
            double wj = lam_pow(lam, Cc - 1 - j);
            if (a->dk_out) {
                double *dkj = a->dk_out + QIDX(a, b, c0 + j, h, 0);
                for (long r = 0; r < dk; ++r) {
                    double acc = 0.0;
                    for (long jv = 0; jv < dv; ++jv) acc += S[r * dv + jv] * vj[jv];
                    dkj[r] = wj * acc;
                }
                for (long i = j; i < Cc; ++i) {
                    const double *doi = a->do_ + VIDX(a, b, c0 + i, h, 0);
                    const double *qi = a->q + QIDX(a, b, c0 + i, h, 0);
                    double dv_ = 0.0;
                    for (long jv = 0; jv < dv; ++jv) dv_ += doi[jv] * vj[jv];
                    double w = a->scale * lam_pow(lam, i - j) * dv_;
                    for (long r = 0; r < dk; ++r) dkj[r] += w * qi[r];
                }
            }
            if (a->dv_out) {
                double *dvj = a->dv_out + VIDX(a, b, c0 + j, h, 0);
                for (long jv = 0; jv < dv; ++jv) {
                    double acc = 0.0;
                    for (long r = 0; r < dk; ++r) acc += S[r * dv + jv] * kj[r];
                    dvj[jv] = wj * acc;
                }
                for (long i = j; i < Cc; ++i) {
                    const double *doi = a->do_ + VIDX(a, b, c0 + i, h, 0);
                    const double *qi = a->q + QIDX(a, b, c0 + i, h, 0);
                    double qk = 0.0;
                    for (long r = 0; r < dk; ++r) qk += qi[r] * kj[r];
                    double w = a->scale * lam_pow(lam, i - j) * qk;
                    for (long jv = 0; jv < dv; ++jv) dvj[jv] += w * doi[jv];
                }
            }
        }
        double wC = lam_pow(lam, Cc);
        for (long r = 0; r < dk * dv; ++r) Sn[r] = wC * S[r];
        for (long i = 0; i < Cc; ++i) {
            const double *qi = a->q + QIDX(a, b, c0 + i, h, 0);
            const double *doi = a->do_ + VIDX(a, b, c0 + i, h, 0);
            double w = a->scale * lam_pow(lam, i + 1);
            for (long r = 0; r < dk; ++r)
                for (long jv = 0; jv < dv; ++jv) Sn[r * dv + jv] += w * qi[r] * doi[jv];
        }
        double *tmp = S; S = Sn; Sn = tmp;
    }
    if (a->dh0) memcpy(a->dh0 + SIDX(a, b, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S); free(Sn);
}

int gla_oracle_bwd_chunked(const double *q, const double *k, const double *v,
                           const double *log_lambda, const double *h0, double scale,
                           const double *do_, const double *dhT,
                           long B, long T, long H, long dk, long dv, long chunk,
                           double *dq, double *dk_out, double *dv_out, double *dh0, int nthreads) {
    if (!q || !k || !v || !log_lambda || !do_ || chunk <= 0 || B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    args_t a; memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.log_lambda = log_lambda; a.h0 = h0; a.scale = scale;
    a.do_ = do_; a.dhT = dhT; a.chunk = chunk;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    a.dq = dq; a.dk_out = dk_out; a.dv_out = dv_out; a.dh0 = dh0;
    run_units(B * H, nthreads, bwd_chunked_unit, &a);
    return 0;
}

/* ------------------------------------------------------- O4: decode */
/* One recurrent step per (n, h), as served ("Inference optimization on
 * Trainium2": one fixed state page per sequence, O(1) work per token):
 *   S <- lambda S + k v^T (in place),  o = scale * S^T q (after the update). */
typedef struct {
    const double *q, *k, *v, *log_lambda;
    double *S, *o;
    double scale;
    long N, H, dk, dv;
} dec_t;

static void decode_unit(void *ctx, long unit) {
    const dec_t *a = (const dec_t *)ctx;
    long h = unit % a->H, dk = a->dk, dv = a->dv;
    double lam = exp(a->log_lambda[h]);
    const double *q = a->q + unit * dk, *k = a->k + unit * dk, *v = a->v + unit * dv;
    double *S = a->S + unit * dk * dv, *o = a->o + unit * dv;
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) S[i * dv + j] = lam * S[i * dv + j] + k[i] * v[j];
    for (long j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (long i = 0; i < dk; ++i) acc += S[i * dv + j] * q[i];
        o[j] = a->scale * acc;
    }
}

int gla_oracle_decode(const double *q, const double *k, const double *v,
                      const double *log_lambda, double *S, double scale,
                      long N, long H, long dk, long dv, double *o, int nthreads) {
    if (!q || !k || !v || !log_lambda || !S || !o || N < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    dec_t a;
    a.q = q; a.k = k; a.v = v; a.log_lambda = log_lambda; a.S = S; a.o = o; a.scale = scale;
    a.N = N; a.H = H; a.dk = dk; a.dv = dv;
    run_units(N * H, nthreads, decode_unit, &a);
    return 0;
}

/* ---------------------------------------------------------- mixer epilogue
 * The per-head epilogue of the mixer, from the "GLA mixer" paragraph of the
 * same page (its equations are images that did not survive extraction):
 *   - self-augmentation: a gated copy of the value is added to the head's
 *     output; the gate is the sigmoid of the query-key dot product with a
 *     learned per-channel scaling a_h (aug_balance, zero at initialisation,
 *     which makes the copy a half-strength skip):
 *         u = o + sigmoid(sum_i q_i a_i k_i) v;
 *   - Head RMSNorm over the head's dv channels with a per-channel weight w_h
 *     (the grouping of heads into decay tiers is not given: each head is
 *     normalised on its own):  y = w * u / sqrt(mean(u^2) + eps);
 *   - the output gate SiLU(g) of the fused projection:  z = y * g * sigmoid(g).
 * o, v, g, z [NT,H,dv]; q, k [NT,H,dk]; a [H,dk] (NULL: 0); w [H,dv] (NULL: 1).
 */
typedef struct {
    const double *o, *q, *k, *v, *g, *a, *w;
    double eps;
    long H, dk, dv;
    double *z;
} epi_t;

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void epilogue_unit(void *ctx, long unit) {
    const epi_t *e = (const epi_t *)ctx;
    const long h = unit % e->H, dk = e->dk, dv = e->dv;
    const double *q = e->q + unit * dk, *k = e->k + unit * dk;
    const double *o = e->o + unit * dv, *v = e->v + unit * dv, *g = e->g + unit * dv;
    double *z = e->z + unit * dv;
    double dot = 0.0;
    for (long i = 0; i < dk; ++i) dot += q[i] * (e->a ? e->a[h * dk + i] : 0.0) * k[i];
    const double gate = sigmoid(dot);
    double ss = 0.0;
    for (long c = 0; c < dv; ++c) {
        const double u = o[c] + gate * v[c];
        z[c] = u;
        ss += u * u;
    }
    const double r = 1.0 / sqrt(ss / (double)dv + e->eps);
    for (long c = 0; c < dv; ++c) {
        const double w = e->w ? e->w[h * dv + c] : 1.0;
        z[c] = z[c] * r * w * (g[c] * sigmoid(g[c]));
    }
}

int gla_oracle_mixer_epilogue(const double *o, const double *q, const double *k, const double *v,
                              const double *g, const double *a, const double *w, double eps, long NT, long H,
                              long dk, long dv, double *z, int nthreads) {
    if (!o || !q || !k || !v || !g || !z || NT < 0 || H <= 0 || dk <= 0 || dv <= 0 || eps < 0.0) return 1;
    epi_t e;
    e.o = o; e.q = q; e.k = k; e.v = v; e.g = g; e.a = a; e.w = w; e.eps = eps;
    e.H = H; e.dk = dk; e.dv = dv; e.z = z;
    run_units(NT * H, nthreads, epilogue_unit, &e);
    return 0;
}

/* ------------------------------------------------- causal depthwise Conv1d
 * The token filter in front of the mixer: "Beyond the KV cache: Training and
 * serving i14's Laplace 3B linear attention model on AWS Trainium2 with
 * native PyTorch", section "i14 and the Laplace 3B architecture", paragraph
 * "Normalisation and convolution": after its LayerNorm, each token's residual
 * vector passes a depthwise causal Conv1d of width 4 with SiLU, a 4-gram
 * summary per position. No equation is printed; the reading, per channel c:
 *     y_t[c] = SiLU( sum_{i=0..3} w[c][i] x_{t-3+i}[c] + b[c] ).
 * Inputs before the call's first token come from the conv window: the last
 * four inputs of the sequence so far, oldest first (zero for a new sequence;
 * its oldest row is carried but never multiplied). The window after the call
 * holds the sequence's last four inputs. A 4 x D window per layer in fp32 is
 * what makes the per-sequence state add up to the 29.5 MB the page states.
 * x, y [B,T,D]; w [D,4]; b [D] (NULL: 0); win_in, win_out [B,4,D] (win_in
 * NULL: zeros; win_out NULL: not written).
 */
typedef struct {
    const double *x, *w, *b, *win_in;
    long T, D;
    double *y, *win_out;
} conv_t;

/* Input at position p of sequence bi, channel c; p < 0 reads the window. */
static double conv_input(const conv_t *a, long bi, long c, long p) {
    if (p >= 0) return a->x[(bi * a->T + p) * a->D + c];
    return a->win_in ? a->win_in[(bi * 4 + 4 + p) * a->D + c] : 0.0;   /* p = -1 is row 3 */
}

static void conv_unit(void *ctx, long unit) {   /* unit = b * D + c */
    const conv_t *a = (const conv_t *)ctx;
    const long bi = unit / a->D, c = unit % a->D, T = a->T, D = a->D;
    for (long t = 0; t < T; ++t) {
        double acc = a->b ? a->b[c] : 0.0;
        for (int i = 0; i < 4; ++i) acc += a->w[c * 4 + i] * conv_input(a, bi, c, t - 3 + i);
        a->y[(bi * T + t) * D + c] = acc * sigmoid(acc);
    }
    if (a->win_out)
        for (int r = 0; r < 4; ++r) a->win_out[(bi * 4 + r) * D + c] = conv_input(a, bi, c, T - 4 + r);
}

int gla_oracle_conv1d(const double *x, const double *w, const double *b, const double *win_in, long B, long T,
                      long D, double *y, double *win_out, int nthreads) {
    if (!x || !w || !y || B < 0 || T < 0 || D <= 0) return 1;
    conv_t a;
    a.x = x; a.w = w; a.b = b; a.win_in = win_in; a.T = T; a.D = D; a.y = y; a.win_out = win_out;
    run_units(B * D, nthreads, conv_unit, &a);
    return 0;
}

/* ------------------------------------------- O9: per-token (gated) decay */
/* The "next" variant of the same mixer with a data-dependent decay: the
 * pages run the mixer through flash-linear-attention's fused_chunk_simple_gla
 * ("Challenge 1") and list "Gated Linear Attention Transformers with
 * Hardware-Efficient Training" among their resources; in that form the
 * per-head decay is a per-token scalar per head, alpha_t = exp(g_t) with a
 * log-decay g_t <= 0 (g may be -inf: the state is then cleared):
 *   S_t = exp(g_t) S_{t-1} + k_t v_t^T,   o_t = scale * S_t^T q_t.
 * With g_t = log lambda_h for every t it is the fixed-decay recurrence.
 * g is [B,T,H] (decode: [N,H]).                                            */
typedef struct {
    const double *q, *k, *v, *g, *h0;
    double scale;
    long B, T, H, dk, dv, chunk;
    double *o, *hT;
} gated_t;

#define GQIDX(a, b, t, h, i) ((((b) * (a)->T + (t)) * (a)->H + (h)) * (a)->dk + (i))
#define GVIDX(a, b, t, h, j) ((((b) * (a)->T + (t)) * (a)->H + (h)) * (a)->dv + (j))
#define GGIDX(a, b, t, h) (((b) * (a)->T + (t)) * (a)->H + (h))
#define GSIDX(a, b, h) (((b) * (a)->H + (h)) * (a)->dk * (a)->dv)

/* exp of the summed log-decays of tokens u+1..t (an empty sum is 0, so the
 * weight of a token on itself is 1 even after a -inf gate). */
static double gated_weight(const gated_t *a, long b, long h, long u, long t) {
    double s = 0.0;
    for (long r = u + 1; r <= t; ++r) s += a->g[GGIDX(a, b, r, h)];
    return exp(s);
}

/* O9: the token recurrence with per-token decay. */
static void gated_recurrent_unit(void *ctx, long unit) {
    const gated_t *a = (const gated_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv;
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    if (a->h0) memcpy(S, a->h0 + GSIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    for (long t = 0; t < a->T; ++t) {
        double alpha = exp(a->g[GGIDX(a, b, t, h)]);
        const double *kt = a->k + GQIDX(a, b, t, h, 0);
        const double *vt = a->v + GVIDX(a, b, t, h, 0);
        const double *qt = a->q + GQIDX(a, b, t, h, 0);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j)
                S[i * dv + j] = alpha * S[i * dv + j] + kt[i] * vt[j];
        if (a->o) {
            double *ot = a->o + GVIDX(a, b, t, h, 0);
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
                ot[j] = a->scale * acc;
            }
        }
    }
    if (a->hT) memcpy(a->hT + GSIDX(a, b, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S);
}

/* O9, unrolled (tiny inputs only): with the decay of tokens u+1..t
 *   o_t = scale * ( d(-1,t) h0^T q_t + sum_{u<=t} d(u,t) (q_t.k_u) v_u ),
 *   hT  = d(-1,T-1) h0 + sum_u d(u,T-1) k_u v_u^T,   d(u,t) = exp(sum g_{u+1..t}). */
static void gated_quadratic_unit(void *ctx, long unit) {
    const gated_t *a = (const gated_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv;
    const double *H0 = a->h0 ? a->h0 + GSIDX(a, b, h) : NULL;
    for (long t = 0; t < a->T; ++t) {
        const double *qt = a->q + GQIDX(a, b, t, h, 0);
        double *ot = a->o + GVIDX(a, b, t, h, 0);
        for (long j = 0; j < dv; ++j) ot[j] = 0.0;
        if (H0) {
            double w = gated_weight(a, b, h, -1, t);
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += H0[i * dv + j] * qt[i];
                ot[j] += w * acc;
            }
        }
        for (long u = 0; u <= t; ++u) {
            const double *ku = a->k + GQIDX(a, b, u, h, 0);
            const double *vu = a->v + GVIDX(a, b, u, h, 0);
            double qk = 0.0;
            for (long i = 0; i < dk; ++i) qk += qt[i] * ku[i];
            double w = gated_weight(a, b, h, u, t) * qk;
            for (long j = 0; j < dv; ++j) ot[j] += w * vu[j];
        }
        for (long j = 0; j < dv; ++j) ot[j] *= a->scale;
    }
    if (a->hT) {
        double *S = a->hT + GSIDX(a, b, h);
        double w0 = gated_weight(a, b, h, -1, a->T - 1);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) S[i * dv + j] = H0 ? w0 * H0[i * dv + j] : 0.0;
        for (long u = 0; u < a->T; ++u) {
            const double *ku = a->k + GQIDX(a, b, u, h, 0);
            const double *vu = a->v + GVIDX(a, b, u, h, 0);
            double w = gated_weight(a, b, h, u, a->T - 1);
            for (long i = 0; i < dk; ++i)
                for (long j = 0; j < dv; ++j) S[i * dv + j] += w * ku[i] * vu[j];
        }
    }
}

/* O9 in chunks of C (0-based i, j inside a chunk of Cc tokens entering with
 * S_prev; d(j,i) the decay of the chunk's tokens j+1..i, d(-1,i) that of
 * tokens 0..i):
 *   o_i   = scale * ( d(-1,i) S_prev^T q_i + sum_{j<=i} d(j,i) (q_i.k_j) v_j )
 *   S_new = d(-1,Cc-1) S_prev + sum_j d(j,Cc-1) k_j v_j^T
 * With a constant gate it is the fixed-decay chunked form.                  */
static void gated_chunked_unit(void *ctx, long unit) {
    const gated_t *a = (const gated_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv, C = a->chunk;
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    double *Sn = (double *)calloc((size_t)(dk * dv), sizeof(double));
    if (a->h0) memcpy(S, a->h0 + GSIDX(a, b, h), sizeof(double) * (size_t)(dk * dv));
    for (long c0 = 0; c0 < a->T; c0 += C) {
        long Cc = a->T - c0 < C ? a->T - c0 : C;
        for (long i = 0; i < Cc && a->o; ++i) {
            const double *qi = a->q + GQIDX(a, b, c0 + i, h, 0);
            double *oi = a->o + GVIDX(a, b, c0 + i, h, 0);
            double wi = gated_weight(a, b, h, c0 - 1, c0 + i);
            for (long jv = 0; jv < dv; ++jv) {
                double acc = 0.0;
                for (long r = 0; r < dk; ++r) acc += S[r * dv + jv] * qi[r];
                oi[jv] = wi * acc;
            }
            for (long j = 0; j <= i; ++j) {
                const double *kj = a->k + GQIDX(a, b, c0 + j, h, 0);
                const double *vj = a->v + GVIDX(a, b, c0 + j, h, 0);
                double qk = 0.0;
                for (long r = 0; r < dk; ++r) qk += qi[r] * kj[r];
                double w = gated_weight(a, b, h, c0 + j, c0 + i) * qk;
                for (long jv = 0; jv < dv; ++jv) oi[jv] += w * vj[jv];
            }
            for (long jv = 0; jv < dv; ++jv) oi[jv] *= a->scale;
        }
        double wC = gated_weight(a, b, h, c0 - 1, c0 + Cc - 1);
        for (long r = 0; r < dk * dv; ++r) Sn[r] = wC * S[r];
        for (long j = 0; j < Cc; ++j) {
            const double *kj = a->k + GQIDX(a, b, c0 + j, h, 0);
            const double *vj = a->v + GVIDX(a, b, c0 + j, h, 0);
            double w = gated_weight(a, b, h, c0 + j, c0 + Cc - 1);
            for (long r = 0; r < dk; ++r)
                for (long jv = 0; jv < dv; ++jv) Sn[r * dv + jv] += w * kj[r] * vj[jv];
        }
        double *tmp = S; S = Sn; Sn = tmp;
    }
    if (a->hT) memcpy(a->hT + GSIDX(a, b, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S); free(Sn);
}

static int gated_run(unit_fn fn, const double *q, const double *k, const double *v, const double *g,
                     const double *h0, double scale, long B, long T, long H, long dk, long dv, long chunk,
                     double *o, double *hT, int nthreads) {
    if (!q || !k || !v || !g || B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    gated_t a; memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.g = g; a.h0 = h0; a.scale = scale;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk; a.o = o; a.hT = hT;
    run_units(B * H, nthreads, fn, &a);
    return 0;
}

int gla_oracle_fwd_gated(const double *q, const double *k, const double *v, const double *g,
                         const double *h0, double scale, long B, long T, long H, long dk, long dv,
                         double *o, double *hT, int nthreads) {
    return gated_run(gated_recurrent_unit, q, k, v, g, h0, scale, B, T, H, dk, dv, 0, o, hT, nthreads);
}

int gla_oracle_fwd_gated_quadratic(const double *q, const double *k, const double *v, const double *g,
                                   const double *h0, double scale, long B, long T, long H, long dk, long dv,
                                   double *o, double *hT, int nthreads) {
    if (!o) return 1;
    return gated_run(gated_quadratic_unit, q, k, v, g, h0, scale, B, T, H, dk, dv, 0, o, hT, nthreads);
}

int gla_oracle_fwd_gated_chunked(const double *q, const double *k, const double *v, const double *g,
                                 const double *h0, double scale, long B, long T, long H, long dk, long dv,
                                 long chunk, double *o, double *hT, int nthreads) {
    if (chunk <= 0) return 1;
    return gated_run(gated_chunked_unit, q, k, v, g, h0, scale, B, T, H, dk, dv, chunk, o, hT, nthreads);
}

/* O10: one serving step with per-token decay, per (n, h):
 *   S <- exp(g[n,h]) S + k v^T (in place),  o = scale * S^T q.             */
typedef struct {
    const double *q, *k, *v, *g;
    double *S, *o;
    double scale;
    long N, H, dk, dv;
} gdec_t;

static void gated_decode_unit(void *ctx, long unit) {
    const gdec_t *a = (const gdec_t *)ctx;
    long dk = a->dk, dv = a->dv;
    double alpha = exp(a->g[unit]);
    const double *q = a->q + unit * dk, *k = a->k + unit * dk, *v = a->v + unit * dv;
    double *S = a->S + unit * dk * dv, *o = a->o + unit * dv;
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) S[i * dv + j] = alpha * S[i * dv + j] + k[i] * v[j];
    for (long j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (long i = 0; i < dk; ++i) acc += S[i * dv + j] * q[i];
        o[j] = a->scale * acc;
    }
}

int gla_oracle_decode_gated(const double *q, const double *k, const double *v, const double *g,
                            double *S, double scale, long N, long H, long dk, long dv, double *o,
                            int nthreads) {
    if (!q || !k || !v || !g || !S || !o || N < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    gdec_t a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.S = S; a.o = o; a.scale = scale;
    a.N = N; a.H = H; a.dk = dk; a.dv = dv;
    run_units(N * H, nthreads, gated_decode_unit, &a);
    return 0;
}

/* --------------------------------------------- O11: gated backward */
/* Gradients of L = sum_t <do_t, o_t> + <dhT, hT> for the per-token decay
 * alpha_t = exp(g_t): with G_t = dL/dS_t (all paths),
 *   G_{T-1} = dhT + scale q_{T-1} do_{T-1}^T,
 *   G_{t-1} = alpha_t G_t + scale q_{t-1} do_{t-1}^T,
 *   dq_t = scale S_t do_t,  dk_t = G_t v_t,  dv_t = G_t^T k_t,
 *   dh0  = alpha_0 G_0,
 *   dg_t = alpha_t <G_t, S_{t-1}>      (dL/dalpha_t times dalpha_t/dg_t; S_{-1} = h0).
 * S_{t-1} is recomputed going backwards from states saved every
 * GATED_CKPT tokens in the forward pass (no division by alpha). g [B,T,H]. */
#define GATED_CKPT 64

typedef struct {
    const double *q, *k, *v, *g, *h0, *do_, *dhT;
    double scale;
    long B, T, H, dk, dv;
    double *dq, *dk_out, *dv_out, *dh0, *dg;
} gbwd_t;

#define GB_QIDX(a, b, t, h, i) ((((b) * (a)->T + (t)) * (a)->H + (h)) * (a)->dk + (i))
#define GB_VIDX(a, b, t, h, j) ((((b) * (a)->T + (t)) * (a)->H + (h)) * (a)->dv + (j))
#define GB_GIDX(a, b, t, h) (((b) * (a)->T + (t)) * (a)->H + (h))
#define GB_SIDX(a, b, h) (((b) * (a)->H + (h)) * (a)->dk * (a)->dv)

/* one forward step S <- alpha_t S + k_t v_t^T */
static void gbwd_step(const gbwd_t *a, long b, long h, long t, double *S) {
    long dk = a->dk, dv = a->dv;
    double alpha = exp(a->g[GB_GIDX(a, b, t, h)]);
    const double *kt = a->k + GB_QIDX(a, b, t, h, 0), *vt = a->v + GB_VIDX(a, b, t, h, 0);
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) S[i * dv + j] = alpha * S[i * dv + j] + kt[i] * vt[j];
}

static void gated_bwd_unit(void *ctx, long unit) {
    const gbwd_t *a = (const gbwd_t *)ctx;
    long b = unit / a->H, h = unit % a->H, dk = a->dk, dv = a->dv, T = a->T, n = dk * dv;
    long ncp = T / GATED_CKPT + 1;
    double *cp = (double *)calloc((size_t)(ncp * n), sizeof(double));   /* S_{c*CKPT - 1} */
    double *S = (double *)calloc((size_t)n, sizeof(double));
    double *blk = (double *)calloc((size_t)(GATED_CKPT * n), sizeof(double));
    double *G = (double *)calloc((size_t)n, sizeof(double));
    if (a->h0) memcpy(S, a->h0 + GB_SIDX(a, b, h), sizeof(double) * (size_t)n);
    /* forward: dq_t and the checkpoints */
    for (long t = 0; t < T; ++t) {
        if (t % GATED_CKPT == 0) memcpy(cp + (t / GATED_CKPT) * n, S, sizeof(double) * (size_t)n);
        gbwd_step(a, b, h, t, S);
        const double *dot = a->do_ + GB_VIDX(a, b, t, h, 0);
        double *dqt = a->dq + GB_QIDX(a, b, t, h, 0);
        for (long i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j) acc += S[i * dv + j] * dot[j];
            dqt[i] = a->scale * acc;
        }
    }
    /* reverse: G_t, dk, dv, dg, one checkpoint block at a time */
    if (a->dhT) memcpy(G, a->dhT + GB_SIDX(a, b, h), sizeof(double) * (size_t)n);
    long t = T - 1;
    for (long c = (T - 1) / GATED_CKPT; c >= 0 && T > 0; --c) {
        long t0 = c * GATED_CKPT, t1 = t0 + GATED_CKPT < T ? t0 + GATED_CKPT : T;
        /* blk[r] = S_{t0 + r - 1}, r = 0 .. t1 - t0 - 1 */
        memcpy(S, cp + c * n, sizeof(double) * (size_t)n);
        for (long r = 0; r < t1 - t0; ++r) {
            memcpy(blk + r * n, S, sizeof(double) * (size_t)n);
            gbwd_step(a, b, h, t0 + r, S);
        }
        for (; t >= t0; --t) {
            const double *qt = a->q + GB_QIDX(a, b, t, h, 0), *dot = a->do_ + GB_VIDX(a, b, t, h, 0);
            const double *kt = a->k + GB_QIDX(a, b, t, h, 0), *vt = a->v + GB_VIDX(a, b, t, h, 0);
            for (long i = 0; i < dk; ++i)
                for (long j = 0; j < dv; ++j) G[i * dv + j] += a->scale * qt[i] * dot[j];
            double *dkt = a->dk_out + GB_QIDX(a, b, t, h, 0), *dvt = a->dv_out + GB_VIDX(a, b, t, h, 0);
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long j = 0; j < dv; ++j) acc += G[i * dv + j] * vt[j];
                dkt[i] = acc;
            }
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += G[i * dv + j] * kt[i];
                dvt[j] = acc;
            }
            double alpha = exp(a->g[GB_GIDX(a, b, t, h)]);
            const double *Sp = blk + (t - t0) * n;
            double ip = 0.0;
            for (long r = 0; r < n; ++r) ip += G[r] * Sp[r];
            a->dg[GB_GIDX(a, b, t, h)] = alpha * ip;
            for (long r = 0; r < n; ++r) G[r] *= alpha;   /* now dL/dS_{t-1} minus its own readout */
        }
    }
    if (a->dh0) memcpy(a->dh0 + GB_SIDX(a, b, h), G, sizeof(double) * (size_t)n);
    free(cp); free(S); free(blk); free(G);
}

int gla_oracle_bwd_gated(const double *q, const double *k, const double *v, const double *g,
                         const double *h0, double scale, const double *do_, const double *dhT,
                         long B, long T, long H, long dk, long dv,
                         double *dq, double *dk_out, double *dv_out, double *dh0, double *dg, int nthreads) {
    if (!q || !k || !v || !g || !do_ || !dq || !dk_out || !dv_out || !dg || B < 0 || T < 0 || H <= 0 ||
        dk <= 0 || dv <= 0)
        return 1;
    gbwd_t a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.h0 = h0; a.do_ = do_; a.dhT = dhT; a.scale = scale;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    a.dq = dq; a.dk_out = dk_out; a.dv_out = dv_out; a.dh0 = dh0; a.dg = dg;
    run_units(B * H, nthreads, gated_bwd_unit, &a);
    return 0;
}
