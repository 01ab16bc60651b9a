/*
 * gla_oracle.c — plain, slow, fp64 CPU reference for Simple Gated Linear
 * Attention (Simple GLA).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * compared against.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the library never links, calls or falls back
 * to it, and it shares no code, header or table with the CUDA path.
 *
 * Citation key used below:
 *   [L3B]  the page "线性注意力模型如何实现固定推理状态" (Beyond the KV cache:
 *          training and serving i14's Laplace 3B linear attention model on AWS
 *          Trainium2).  Sections: "i14 与 Laplace 3B 架构" (GLA mixer: state
 *          update, state read-out, decay scheme) and "挑战 1" (chunked GLA:
 *          intra-chunk output and chunk state update, Figure 3).
 *   [RFB]  the blog page on recurrence-free pre-trained recurrent networks,
 *          §3.2 (the state update S_t = S_{t-1} + k_t v_t as a prefix sum).
 *
 * The formula images on [L3B] did not survive extraction; only their captions
 * and the surrounding prose did.  The readings taken here:
 *   - per head h a fixed scalar decay lambda_h = exp(log_decay[h]) in (0, 1];
 *   - state S (dk x dv) updated as  S_t = lambda * S_{t-1} + k_t^T v_t;
 *   - read-out after the update:     o_t = q_t S_t   (no extra scale);
 *   - chunk c of length L (local positions i, j):
 *       O_c = ((Q_c K_c^T) .* D) V_c + diag(lambda^(i+1)) Q_c S_{c-1},
 *             D_ij = lambda^(i-j) for j <= i, else 0
 *       S_c = lambda^L S_{c-1} + K_c^T diag(lambda^(L-1-j)) V_c.
 *
 * Layout (row-major, innermost last):
 *   q, k : [rows, H, dk]   float32 (exact copies of bf16 / fp32 inputs)
 *   v    : [rows, H, dv]   float32
 *   o    : [rows, H, dv]   float64 (written)
 *   h0,hT: [nseq, H, dk, dv] float64 (h0 may be NULL = zeros; hT may be NULL)
 * A sequence s occupies rows seq_start[s] .. seq_start[s]+seq_len[s]-1.  A
 * dense batch [B, T, ...] is the case seq_start[b] = b*T, seq_len[b] = T.
 *
 * units: optional list of (sequence, head) pairs (2*nunits int32) selecting
 * which chains to compute; NULL computes every chain.  Rows of o that belong to
 * chains not selected are left untouched.
 *
 * All entry points return 0 on success and -1 on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float *q, *k, *v;
    const double *log_decay;
    const double *h0;
    double *o, *hT;
    const int64_t *seq_start, *seq_len;
    int nseq, H, dk, dv;
    const int32_t *units;
    int nunits;
    int chunk;       /* used by the chunked form only */
    int form;        /* 0 recurrent, 1 quadratic, 2 chunked */
    int next_unit;   /* shared work counter */
    int error;
} job_t;

/* lambda^n for integer n >= 0, from the natural-log decay. */
static double decay_pow(double log_decay, double n) { return exp(n * log_decay); }

/*
 * Token-by-token recurrence for one (sequence, head) chain.
 * [L3B] §"i14 与 Laplace 3B 架构", GLA mixer: the per-token state update and
 * the state read-out.
 */
static void chain_recurrent(const job_t *J, int s, int h) {
    const int H = J->H, dk = J->dk, dv = J->dv;
    const double lam = exp(J->log_decay[h]);
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    if (J->h0) memcpy(S, J->h0 + ((size_t)s * H + h) * dk * dv, sizeof(double) * dk * dv);
    for (int64_t t = 0; t < J->seq_len[s]; ++t) {
        const int64_t row = J->seq_start[s] + t;
        const float *qt = J->q + ((size_t)row * H + h) * dk;
        const float *kt = J->k + ((size_t)row * H + h) * dk;
        const float *vt = J->v + ((size_t)row * H + h) * dv;
        double *ot = J->o + ((size_t)row * H + h) * dv;
        for (int j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            double *Si = S + (size_t)i * dv;
            const double ki = kt[i], qi = qt[i];
            for (int j = 0; j < dv; ++j) {
                Si[j] = lam * Si[j] + ki * (double)vt[j];   /* S_t = lam S_{t-1} + k_t^T v_t */
                ot[j] += qi * Si[j];                        /* o_t = q_t S_t                 */
            }
        }
    }
    if (J->hT) memcpy(J->hT + ((size_t)s * H + h) * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
}

/*
 * Quadratic (attention) form of the same map for one chain:
 *   o_i = sum_{j<=i} lambda^(i-j) (q_i . k_j) v_j + lambda^(i+1) q_i S_0
 *   S_T = lambda^T S_0 + sum_j lambda^(T-1-j) k_j^T v_j
 * Obtained by unrolling the [L3B] GLA-mixer recurrence; used to pin the
 * recurrence above.  Powers of lambda come from exp(n * log_decay) here, not
 * from repeated products, so the two forms round differently.
 */
static void chain_quadratic(const job_t *J, int s, int h) {
    const int H = J->H, dk = J->dk, dv = J->dv;
    const double ld = J->log_decay[h];
    const int64_t T = J->seq_len[s], r0 = J->seq_start[s];
    const double *S0 = J->h0 ? J->h0 + ((size_t)s * H + h) * dk * dv : NULL;
    for (int64_t i = 0; i < T; ++i) {
        const float *qi = J->q + ((size_t)(r0 + i) * H + h) * dk;
        double *oi = J->o + ((size_t)(r0 + i) * H + h) * dv;
        for (int c = 0; c < dv; ++c) oi[c] = 0.0;
        for (int64_t j = 0; j <= i; ++j) {
            const float *kj = J->k + ((size_t)(r0 + j) * H + h) * dk;
            const float *vj = J->v + ((size_t)(r0 + j) * H + h) * dv;
            double a = 0.0;
            for (int d = 0; d < dk; ++d) a += (double)qi[d] * (double)kj[d];
            a *= decay_pow(ld, (double)(i - j));
            for (int c = 0; c < dv; ++c) oi[c] += a * (double)vj[c];
        }
        if (S0) {
            const double g = decay_pow(ld, (double)(i + 1));
            for (int d = 0; d < dk; ++d)
                for (int c = 0; c < dv; ++c) oi[c] += g * (double)qi[d] * S0[(size_t)d * dv + c];
        }
    }
    if (J->hT) {
        double *ST = J->hT + ((size_t)s * H + h) * dk * dv;
        const double gT = decay_pow(ld, (double)T);
        for (size_t e = 0; e < (size_t)dk * dv; ++e) ST[e] = S0 ? gT * S0[e] : 0.0;
        for (int64_t j = 0; j < T; ++j) {
            const float *kj = J->k + ((size_t)(r0 + j) * H + h) * dk;
            const float *vj = J->v + ((size_t)(r0 + j) * H + h) * dv;
            const double g = decay_pow(ld, (double)(T - 1 - j));
            for (int d = 0; d < dk; ++d)
                for (int c = 0; c < dv; ++c) ST[(size_t)d * dv + c] += g * (double)kj[d] * (double)vj[c];
        }
    }
}

/*
 * Chunkwise form for one chain, chunk length C (the last chunk may be shorter).
 * [L3B] §"挑战 1": intra-chunk output = decay-masked linear attention plus the
 * carried state's contribution; then the chunk state update with the decay
 * accumulated over the chunk (Figure 3).  Used only to check that the chunked
 * and recurrent forms agree.
 */
static void chain_chunked(const job_t *J, int s, int h) {
    const int H = J->H, dk = J->dk, dv = J->dv, C = J->chunk;
    const double ld = J->log_decay[h];
    const int64_t T = J->seq_len[s], r0 = J->seq_start[s];
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *dS = (double *)calloc((size_t)dk * dv, sizeof(double));
    if (J->h0) memcpy(S, J->h0 + ((size_t)s * H + h) * dk * dv, sizeof(double) * dk * dv);
    for (int64_t c0 = 0; c0 < T; c0 += C) {
        const int64_t L = (T - c0 < C) ? (T - c0) : C;
        /* output of the chunk, using S = S_{c-1} */
        for (int64_t i = 0; i < L; ++i) {
            const float *qi = J->q + ((size_t)(r0 + c0 + i) * H + h) * dk;
            double *oi = J->o + ((size_t)(r0 + c0 + i) * H + h) * dv;
            for (int c = 0; c < dv; ++c) oi[c] = 0.0;
            for (int64_t j = 0; j <= i; ++j) {            /* ((Q K^T) .* D) V */
                const float *kj = J->k + ((size_t)(r0 + c0 + j) * H + h) * dk;
                const float *vj = J->v + ((size_t)(r0 + c0 + j) * H + h) * dv;
                double a = 0.0;
                for (int d = 0; d < dk; ++d) a += (double)qi[d] * (double)kj[d];
                a *= decay_pow(ld, (double)(i - j));
                for (int c = 0; c < dv; ++c) oi[c] += a * (double)vj[c];
            }
            const double g = decay_pow(ld, (double)(i + 1));   /* diag(lambda^(i+1)) Q S */
            for (int d = 0; d < dk; ++d)
                for (int c = 0; c < dv; ++c) oi[c] += g * (double)qi[d] * S[(size_t)d * dv + c];
        }
        /* S_c = lambda^L S_{c-1} + K^T diag(lambda^(L-1-j)) V */
        memset(dS, 0, sizeof(double) * dk * dv);
        for (int64_t j = 0; j < L; ++j) {
            const float *kj = J->k + ((size_t)(r0 + c0 + j) * H + h) * dk;
            const float *vj = J->v + ((size_t)(r0 + c0 + j) * H + h) * dv;
            const double g = decay_pow(ld, (double)(L - 1 - j));
            for (int d = 0; d < dk; ++d)
                for (int c = 0; c < dv; ++c) dS[(size_t)d * dv + c] += (double)kj[d] * g * (double)vj[c];
        }
        const double gL = decay_pow(ld, (double)L);
        for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = gL * S[e] + dS[e];
    }
    if (J->hT) memcpy(J->hT + ((size_t)s * H + h) * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
    free(dS);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int total = J->units ? J->nunits : J->nseq * J->H;
    for (;;) {
        const int u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
        if (u >= total) break;
        int s, h;
        if (J->units) { s = J->units[2 * u]; h = J->units[2 * u + 1]; }
        else { s = u / J->H; h = u % J->H; }
        if (s < 0 || s >= J->nseq || h < 0 || h >= J->H) { J->error = 1; continue; }
        if (J->form == 0) chain_recurrent(J, s, h);
        else if (J->form == 1) chain_quadratic(J, s, h);
        else chain_chunked(J, s, h);
    }
    return NULL;
}

static int run(job_t *J, int nthreads) {
    if (!J->q || !J->k || !J->v || !J->log_decay || !J->o || !J->seq_start || !J->seq_len) return -1;
    if (J->nseq < 0 || J->H <= 0 || J->dk <= 0 || J->dv <= 0) return -1;
    if (J->form == 2 && J->chunk <= 0) return -1;
    for (int s = 0; s < J->nseq; ++s)
        if (J->seq_len[s] < 0 || J->seq_start[s] < 0) return -1;
    J->next_unit = 0;
    J->error = 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads == 1) {
        worker(J);
    } else {
        pthread_t tid[512];
        int started = 0;
        for (int t = 0; t < nthreads; ++t)
            if (pthread_create(&tid[started], NULL, worker, J) == 0) ++started;
        if (started == 0) worker(J);
        for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    }
    return J->error ? -1 : 0;
}

#define JOB_INIT(FORM, CHUNK)                                                        \
    job_t J;                                                                         \
    memset(&J, 0, sizeof J);                                                         \
    J.q = q; J.k = k; J.v = v; J.log_decay = log_decay; J.h0 = h0; J.o = o;          \
    J.hT = hT; J.seq_start = seq_start; J.seq_len = seq_len; J.nseq = nseq; J.H = H; \
    J.dk = dk; J.dv = dv; J.units = units; J.nunits = nunits; J.form = (FORM);       \
    J.chunk = (CHUNK)

int gla_oracle_recurrent(const float *q, const float *k, const float *v, const double *log_decay,
                         const double *h0, double *o, double *hT, const int64_t *seq_start,
                         const int64_t *seq_len, int nseq, int H, int dk, int dv,
                         const int32_t *units, int nunits, int nthreads) {
    JOB_INIT(0, 0);
    return run(&J, nthreads);
}

int gla_oracle_quadratic(const float *q, const float *k, const float *v, const double *log_decay,
                         const double *h0, double *o, double *hT, const int64_t *seq_start,
                         const int64_t *seq_len, int nseq, int H, int dk, int dv,
                         const int32_t *units, int nunits, int nthreads) {
    JOB_INIT(1, 0);
    return run(&J, nthreads);
}

int gla_oracle_chunked(const float *q, const float *k, const float *v, const double *log_decay,
                       const double *h0, double *o, double *hT, const int64_t *seq_start,
                       const int64_t *seq_len, int nseq, int H, int dk, int dv, int chunk,
                       const int32_t *units, int nunits, int nthreads) {
    JOB_INIT(2, chunk);
    return run(&J, nthreads);
}

/*
 * One recurrent decode step for N independent sequences, each with H heads:
 *   state <- lambda * state + k^T v   (in place),   o = q state.
 * [L3B] §"i14 与 Laplace 3B 架构" (GLA mixer, O(1) inference per token) and
 * §"Trainium2 上的推理优化" (a fixed per-sequence state page read and written
 * once per generated token).
 *   q, k : [N, H, dk] float32;  v : [N, H, dv] float32
 *   state: [N, H, dk, dv] float64 (in/out);  o : [N, H, dv] float64
 */
typedef struct {
    const float *q, *k, *v;
    const double *log_decay;
    double *state, *o;
    int N, H, dk, dv, next;
} dec_t;

static void *dec_worker(void *arg) {
    dec_t *D = (dec_t *)arg;
    const int H = D->H, dk = D->dk, dv = D->dv;
    for (;;) {
        const int u = __atomic_fetch_add(&D->next, 1, __ATOMIC_RELAXED);
        if (u >= D->N * H) break;
        const int h = u % H;
        const double lam = exp(D->log_decay[h]);
        double *S = D->state + (size_t)u * dk * dv;
        const float *qt = D->q + (size_t)u * dk, *kt = D->k + (size_t)u * dk, *vt = D->v + (size_t)u * dv;
        double *ot = D->o + (size_t)u * dv;
        for (int j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                S[(size_t)i * dv + j] = lam * S[(size_t)i * dv + j] + (double)kt[i] * (double)vt[j];
                ot[j] += (double)qt[i] * S[(size_t)i * dv + j];
            }
    }
    return NULL;
}

int gla_oracle_decode_step(const float *q, const float *k, const float *v, const double *log_decay,
                           double *state, double *o, int N, int H, int dk, int dv, int nthreads) {
    if (!q || !k || !v || !log_decay || !state || !o || N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    dec_t D = {q, k, v, log_decay, state, o, N, H, dk, dv, 0};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    pthread_t tid[512];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tid[started], NULL, dec_worker, &D) == 0) ++started;
    dec_worker(&D);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    return 0;
}

/*
 * Backward (vector-Jacobian product) of the recurrence, for training.
 * [L3B] §"挑战 3" (the backward pass differentiates every sequential state
 * update of the recurrence); the page prints no backward formulas, so this is
 * the chain rule applied to the [L3B] GLA-mixer recurrence, one token at a
 * time, in reverse:
 *   given dO = dL/do_t and dhT = dL/dS_T (NULL = 0), with G = dL/dS_t,
 *   G_T = dhT;  for t = T .. 1:
 *       G     += q_t^T do_t                 (o_t = q_t S_t)
 *       dq_t   = do_t S_t^T
 *       dk_t   = v_t G^T,   dv_t = k_t G    (S_t = lam S_{t-1} + k_t^T v_t)
 *       G      = lam G                      (gradient reaching S_{t-1})
 *   dh0 = G.
 * The forward states S_t are replayed from checkpoints kept every kCkpt
 * tokens (the replay repeats the forward's own operations, so the replayed
 * states equal the stored ones bit for bit).
 *   do  : [rows, H, dv] float32;   dhT, dh0 : [nseq, H, dk, dv] float64
 *   dq, dk : [rows, H, dk] float64; dv : [rows, H, dv] float64
 */
typedef struct {
    const float *q, *k, *v, *dout;
    const double *log_decay, *h0, *dhT;
    double *dq, *dk, *dv, *dh0;
    const int64_t *seq_start, *seq_len;
    int nseq, H, dk_, dv_;
    const int32_t *units;
    int nunits, next_unit, error;
} bwd_t;

enum { kCkpt = 64 };

/* one forward token step on S (dk x dv): S = lam S + k^T v */
static void state_step(double *S, const float *kt, const float *vt, double lam, int dk, int dv) {
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] = lam * S[(size_t)i * dv + j] + (double)kt[i] * (double)vt[j];
}

static int chain_backward(const bwd_t *J, int s, int h) {
    const int H = J->H, dk = J->dk_, dv = J->dv_;
    const size_t sz = (size_t)dk * dv;
    const double lam = exp(J->log_decay[h]);
    const int64_t T = J->seq_len[s], r0 = J->seq_start[s];
    const int64_t nck = (T + kCkpt - 1) / kCkpt;
    double *ck = (double *)calloc((size_t)(nck > 0 ? nck : 1) * sz, sizeof(double)); /* S before block b */
    double *blk = (double *)malloc((size_t)kCkpt * sz * sizeof(double));             /* S_t inside a block */
    double *G = (double *)calloc(sz, sizeof(double));
    double *S = (double *)calloc(sz, sizeof(double));
    if (!ck || !blk || !G || !S) { free(ck); free(blk); free(G); free(S); return -1; }
    /* forward sweep: checkpoints of S_{b*kCkpt} (state before the block's first token) */
    if (J->h0) memcpy(S, J->h0 + ((size_t)s * H + h) * sz, sizeof(double) * sz);
    for (int64_t t = 0; t < T; ++t) {
        if (t % kCkpt == 0) memcpy(ck + (size_t)(t / kCkpt) * sz, S, sizeof(double) * sz);
        const int64_t row = r0 + t;
        state_step(S, J->k + ((size_t)row * H + h) * dk, J->v + ((size_t)row * H + h) * dv, lam, dk, dv);
    }
    free(S);
    if (J->dhT) memcpy(G, J->dhT + ((size_t)s * H + h) * sz, sizeof(double) * sz);
    /* reverse sweep, one block at a time (last block first) */
    for (int64_t b = nck - 1; b >= 0; --b) {
        const int64_t t0 = b * kCkpt, t1 = (t0 + kCkpt < T) ? t0 + kCkpt : T;
        /* replay the block: blk[u] = S_{t0+u} after the update at token t0+u */
        const double *prev = ck + (size_t)b * sz;
        for (int64_t t = t0; t < t1; ++t) {
            double *cur = blk + (size_t)(t - t0) * sz;
            memcpy(cur, prev, sizeof(double) * sz);
            const int64_t row = r0 + t;
            state_step(cur, J->k + ((size_t)row * H + h) * dk, J->v + ((size_t)row * H + h) * dv, lam, dk, dv);
            prev = cur;
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const int64_t row = r0 + t;
            const float *qt = J->q + ((size_t)row * H + h) * dk;
            const float *kt = J->k + ((size_t)row * H + h) * dk;
            const float *vt = J->v + ((size_t)row * H + h) * dv;
            const float *dot = J->dout + ((size_t)row * H + h) * dv;
            const double *St = blk + (size_t)(t - t0) * sz;
            double *dqt = J->dq + ((size_t)row * H + h) * dk;
            double *dkt = J->dk + ((size_t)row * H + h) * dk;
            double *dvt = J->dv + ((size_t)row * H + h) * dv;
            for (int i = 0; i < dk; ++i)               /* G += q_t^T do_t */
                for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] += (double)qt[i] * (double)dot[j];
            for (int i = 0; i < dk; ++i) {             /* dq_t = do_t S_t^T;  dk_t = v_t G^T */
                double aq = 0.0, ak = 0.0;
                for (int j = 0; j < dv; ++j) {
                    aq += (double)dot[j] * St[(size_t)i * dv + j];
                    ak += (double)vt[j] * G[(size_t)i * dv + j];
                }
                dqt[i] = aq;
                dkt[i] = ak;
            }
            for (int j = 0; j < dv; ++j) {             /* dv_t = k_t G */
                double a = 0.0;
                for (int i = 0; i < dk; ++i) a += (double)kt[i] * G[(size_t)i * dv + j];
                dvt[j] = a;
            }
            for (size_t e = 0; e < sz; ++e) G[e] *= lam;   /* to S_{t-1} */
        }
    }
    if (J->dh0) memcpy(J->dh0 + ((size_t)s * H + h) * sz, G, sizeof(double) * sz);
    free(ck);
    free(blk);
    free(G);
    return 0;
}

static void *bwd_worker(void *arg) {
    bwd_t *J = (bwd_t *)arg;
    const int total = J->units ? J->nunits : J->nseq * J->H;
    for (;;) {
        const int u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
        if (u >= total) break;
        int s, h;
        if (J->units) { s = J->units[2 * u]; h = J->units[2 * u + 1]; }
        else { s = u / J->H; h = u % J->H; }
        if (s < 0 || s >= J->nseq || h < 0 || h >= J->H) { J->error = 1; continue; }
        if (chain_backward(J, s, h) != 0) J->error = 1;
    }
    return NULL;
}

int gla_oracle_backward(const float *q, const float *k, const float *v, const float *dout,
                        const double *log_decay, const double *h0, const double *dhT, double *dq,
                        double *dk, double *dv, double *dh0, const int64_t *seq_start,
                        const int64_t *seq_len, int nseq, int H, int dk_, int dv_,
                        const int32_t *units, int nunits, int nthreads) {
    if (!q || !k || !v || !dout || !log_decay || !dq || !dk || !dv || !seq_start || !seq_len) return -1;
    if (nseq < 0 || H <= 0 || dk_ <= 0 || dv_ <= 0) return -1;
    for (int s = 0; s < nseq; ++s)
        if (seq_len[s] < 0 || seq_start[s] < 0) return -1;
    bwd_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.dout = dout; J.log_decay = log_decay; J.h0 = h0; J.dhT = dhT;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dh0 = dh0; J.seq_start = seq_start; J.seq_len = seq_len;
    J.nseq = nseq; J.H = H; J.dk_ = dk_; J.dv_ = dv_; J.units = units; J.nunits = nunits;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    pthread_t tid[512];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tid[started], NULL, bwd_worker, &J) == 0) ++started;
    bwd_worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    return J.error ? -1 : 0;
}

/*
 * Causal depthwise Conv1d of width 4 followed by SiLU, per channel
 * ([L3B] §"i14 与 Laplace 3B 架构", "归一化与卷积": every position of the
 * normalised residual stream gets a 4-token summary from a per-channel causal
 * convolution of width k = 4 with SiLU, before the QKVG projection).  The page
 * prints no formula; the reading taken here, for channel c at token t:
 *   z = b[c] + sum_{k=0..3} w[c][k] * x_{t-3+k}[c]       (w[c][3] meets x_t)
 *   y_t[c] = z / (1 + exp(-z))                           (SiLU)
 * where x before a sequence's first token comes from its conv state
 * (state[s][c][m] = x_{m-3}[c], m = 0..2, oldest first; NULL = zeros).  The
 * state after the sequence holds its last three inputs (earlier ones from the
 * incoming state when the sequence is shorter than three).
 *   x, y  : [rows, D] float32 in, float64 out;  w : [D, 4];  b : [D] or NULL
 *   state_in / state_out : [nseq, D, 3] float64 or NULL
 */
int gla_oracle_conv1d_silu(const float *x, const double *w, const double *b, const double *state_in,
                           double *state_out, double *y, const int64_t *seq_start, const int64_t *seq_len,
                           int nseq, int D) {
    if (!x || !w || !y || !seq_start || !seq_len || nseq < 0 || D <= 0) return -1;
    for (int s = 0; s < nseq; ++s) {
        if (seq_len[s] < 0 || seq_start[s] < 0) return -1;
        const int64_t r0 = seq_start[s], T = seq_len[s];
        for (int c = 0; c < D; ++c) {
            double hist[3];  /* x_{t-3}, x_{t-2}, x_{t-1} */
            for (int m = 0; m < 3; ++m) hist[m] = state_in ? state_in[((size_t)s * D + c) * 3 + m] : 0.0;
            for (int64_t t = 0; t < T; ++t) {
                const double xt = (double)x[(size_t)(r0 + t) * D + c];
                double z = b ? b[c] : 0.0;
                for (int k = 0; k < 3; ++k) z += w[(size_t)c * 4 + k] * hist[k];
                z += w[(size_t)c * 4 + 3] * xt;
                y[(size_t)(r0 + t) * D + c] = z / (1.0 + exp(-z));
                hist[0] = hist[1];
                hist[1] = hist[2];
                hist[2] = xt;
            }
            if (state_out)
                for (int m = 0; m < 3; ++m) state_out[((size_t)s * D + c) * 3 + m] = hist[m];
        }
    }
    return 0;
}

/*
 * Output gate ([L3B] §"i14 与 Laplace 3B 架构", "QKVG 投影": the fused projection
 * splits into q_t, k_t, v_t and a gate g_t of H x dv values per token, and the
 * gate acts after the mixer).  The page names the gate and where it acts but
 * prints no formula; the reading taken here is an elementwise product of the
 * mixer output o_t with a function of g_t:
 *   kind 0:  o'_t = o_t * g_t / (1 + exp(-g_t))      (swish / SiLU gate)
 *   kind 1:  o'_t = o_t * 1 / (1 + exp(-g_t))        (sigmoid gate)
 *   o, out : n float64 values (out may be o);  g : n float32 values
 */
int gla_oracle_output_gate(const double *o, const float *g, int kind, double *out, int64_t n) {
    if (!o || !g || !out || n < 0 || (kind != 0 && kind != 1)) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const double x = (double)g[i];
        const double sig = 1.0 / (1.0 + exp(-x));
        out[i] = o[i] * (kind == 0 ? x * sig : sig);
    }
    return 0;
}
