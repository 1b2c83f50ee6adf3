/*
 * FP64 token-by-token oracle for the gated delta rule of Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness yardstick for the CUDA library in
 * linear_attention_chunked_gb300/.  Only tests/, __graft_entry__.smoke() and the cpu_baseline /
 * reference legs of bench.py load it.  It shares no code, header, table or helper with the CUDA
 * path, and the CUDA path never calls it.
 *
 * What it computes (the plain definition, one token at a time, in double precision):
 *   per document n and head h, with S the [d_k x d_v] state (rows = key channels):
 *     S_0 = h0[n,h]  (zeros when h0 is NULL); reset at every cu_seqlens boundary
 *     for each token t of the document:
 *       q, k <- optional L2 norm over the d channels of the head: x / sqrt(sum x^2 + eps)
 *       g    <- g_t (g form) or -exp(A_log[h]) * softplus(a_t + dt_bias[h])   (raw form)
 *       S'   =  Diag(exp(g)) S
 *       u    =  v - S'^T k
 *       S    =  S' + beta k u^T          ( == (I - beta k k^T) Diag(exp g) S + beta k v^T )
 *       o_t  =  scale * S^T q
 *     ht[n,h] = S
 *   Source: the recurrence of Kimi Delta Attention as used by the chunked KDA training package
 *   described on the page "fix(cake_kda_det): gate-gradient accuracy of the GLM intra stage"
 *   (flashinfer PR #8909, summary: gate form g / raw, Q/K L2 norm off / fused, saved / replay
 *   backward), with the state recurrence S_t = (I - b k k^T) Diag(exp g) S_{t-1} + b k v^T,
 *   o_t = S_t^T q_t and the raw gate -exp(A_log) softplus(a + dt_bias).
 *
 * The backward is the reverse-mode adjoint of exactly that loop (tokens in reverse order), with
 * the state re-materialised from checkpoints every OR_SEG tokens.  Loss convention:
 *   L = sum(o * dO) + sum(ht * dht).
 *
 * Fragment algebra (page "perf(cake_kda): ... BF16x3 half-width transfer walk", flashinfer PR
 * #7176, summary: the transfer walk carries the FP32 state across fragment boundaries as
 * S_out = M * S_in + B):
 *   M_f = product over the fragment's tokens, later tokens on the left, of (I - b k k^T) Diag(e^g)
 *   B_f = the fragment's final state from S = 0
 *   C_f = the gradient at the fragment's first state with zero incoming end gradient (dht = 0).
 *
 * All arrays are dense row-major doubles:  q,k,v,g/a,dO,o,dq,dk,dv,dg [T,H,d];  beta,dbeta [T,H];
 * A_log [H];  dt_bias [H,d];  h0,ht,dht,dh0 [N,H,d,d].  cu_seqlens is a host int32 array [N+1].
 * Work is split over (document, head) chains on POSIX threads; every output element is written by
 * exactly one chain, and per-chain partial sums are reduced in a fixed order, so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_SEG 64 /* tokens between state checkpoints in the backward sweep */

typedef struct {
    int64_t T;
    int32_t N, H, d;
    const int32_t* cu;
    const double *q, *k, *v, *beta, *gin, *A_log, *dt_bias, *h0;
    int raw, l2n;
    double scale, eps;
    /* forward outputs */
    double *o, *ht;
    /* backward */
    const double *dO, *dht;
    double *dq, *dk, *dv, *dbeta, *dgin, *dh0;
    double *dA_log_part; /* [N*H]    per-chain partial of dA_log  */
    double *ddt_part;    /* [N*H*d]  per-chain partial of ddt_bias */
    /* scheduling */
    int64_t next;
    int mode; /* 0 forward, 1 backward */
    int status;
} job_t;

/* softplus(x) = log(1 + e^x), written so that it neither overflows nor loses the small tail */
static double softplus(double x) { return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x))); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Per-token quantities of one (token, head). */
typedef struct {
    double *q, *k, *v, *g; /* d each: normalised q, k; v; log gate */
    double qn, kn;         /* sqrt(|q|^2+eps), sqrt(|k|^2+eps) (1 when no L2 norm) */
    double beta;
} tok_t;

static void load_token(const job_t* J, int64_t t, int h, tok_t* x) {
    const int d = J->d;
    const int64_t base = (t * J->H + h) * (int64_t)d;
    double sq = 0.0, sk = 0.0;
    for (int c = 0; c < d; ++c) {
        x->q[c] = J->q[base + c];
        x->k[c] = J->k[base + c];
        x->v[c] = J->v[base + c];
        sq += x->q[c] * x->q[c];
        sk += x->k[c] * x->k[c];
    }
    x->qn = 1.0;
    x->kn = 1.0;
    if (J->l2n) {
        x->qn = sqrt(sq + J->eps);
        x->kn = sqrt(sk + J->eps);
        for (int c = 0; c < d; ++c) {
            x->q[c] /= x->qn;
            x->k[c] /= x->kn;
        }
    }
    for (int c = 0; c < d; ++c) {
        if (J->raw) {
            double a = J->gin[base + c] + J->dt_bias[(int64_t)h * d + c];
            x->g[c] = -exp(J->A_log[h]) * softplus(a);
        } else {
            x->g[c] = J->gin[base + c];
        }
    }
    x->beta = J->beta[t * J->H + h];
}

/* One forward token step on S (d x d, row = key channel).  Writes S' (decayed state) and u if asked. */
static void step_fwd(int d, double* S, const tok_t* x, double* Sp, double* u) {
    for (int i = 0; i < d; ++i) {
        double e = exp(x->g[i]);
        for (int j = 0; j < d; ++j) S[i * d + j] *= e;
    }
    if (Sp) memcpy(Sp, S, sizeof(double) * d * d);
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += S[i * d + j] * x->k[i];
        u[j] = x->v[j] - acc;
    }
    for (int i = 0; i < d; ++i) {
        double bk = x->beta * x->k[i];
        for (int j = 0; j < d; ++j) S[i * d + j] += bk * u[j];
    }
}

typedef struct {
    double *q, *k, *v, *g, *u, *Sp, *S, *dS, *dq, *dk, *du, *dSp, *ck, *seg;
} scratch_t;

static int scratch_alloc(scratch_t* s, int d) {
    size_t dd = (size_t)d * d;
    s->q = malloc(sizeof(double) * d * 9);
    s->S = malloc(sizeof(double) * dd * 4);
    s->seg = malloc(sizeof(double) * dd * OR_SEG);
    if (!s->q || !s->S || !s->seg) return -1;
    s->k = s->q + d; s->v = s->k + d; s->g = s->v + d; s->u = s->g + d;
    s->dq = s->u + d; s->dk = s->dq + d; s->du = s->dk + d; s->ck = s->du + d;
    s->Sp = s->S + dd; s->dS = s->Sp + dd; s->dSp = s->dS + dd;
    return 0;
}
static void scratch_free(scratch_t* s) { free(s->q); free(s->S); free(s->seg); }

static void chain_fwd(job_t* J, int n, int h, scratch_t* s) {
    const int d = J->d;
    const size_t dd = (size_t)d * d;
    tok_t x = {s->q, s->k, s->v, s->g, 1.0, 1.0, 0.0};
    double* S = s->S;
    if (J->h0) memcpy(S, J->h0 + ((size_t)n * J->H + h) * dd, sizeof(double) * dd);
    else memset(S, 0, sizeof(double) * dd);
    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        load_token(J, t, h, &x);
        step_fwd(d, S, &x, NULL, s->u);
        if (J->o) {
            double* o = J->o + (t * J->H + h) * (int64_t)d;
            for (int j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += S[i * d + j] * x.q[i];
                o[j] = J->scale * acc;
            }
        }
    }
    if (J->ht) memcpy(J->ht + ((size_t)n * J->H + h) * dd, S, sizeof(double) * dd);
}

static void chain_bwd(job_t* J, int n, int h, scratch_t* s) {
    const int d = J->d;
    const size_t dd = (size_t)d * d;
    const int64_t bos = J->cu[n], eos = J->cu[n + 1];
    const int64_t len = eos - bos;
    const int64_t nseg = (len + OR_SEG - 1) / OR_SEG;
    tok_t x = {s->q, s->k, s->v, s->g, 1.0, 1.0, 0.0};
    /* checkpoints: state before each segment */
    double* ck = malloc(sizeof(double) * dd * (nseg > 0 ? nseg : 1));
    if (!ck) { J->status = -1; return; }
    double* S = s->S;
    if (J->h0) memcpy(S, J->h0 + ((size_t)n * J->H + h) * dd, sizeof(double) * dd);
    else memset(S, 0, sizeof(double) * dd);
    for (int64_t sg = 0; sg < nseg; ++sg) {
        memcpy(ck + sg * dd, S, sizeof(double) * dd);
        int64_t t1 = bos + (sg + 1) * OR_SEG;
        if (t1 > eos) t1 = eos;
        for (int64_t t = bos + sg * OR_SEG; t < t1; ++t) {
            load_token(J, t, h, &x);
            step_fwd(d, S, &x, NULL, s->u);
        }
    }
    double* dS = s->dS;
    if (J->dht) memcpy(dS, J->dht + ((size_t)n * J->H + h) * dd, sizeof(double) * dd);
    else memset(dS, 0, sizeof(double) * dd);
    double dA = 0.0;
    double* ddt = J->ddt_part ? J->ddt_part + ((size_t)n * J->H + h) * d : NULL;
    if (ddt) memset(ddt, 0, sizeof(double) * d);
    for (int64_t sg = nseg - 1; sg >= 0; --sg) {
        int64_t t0 = bos + sg * OR_SEG, t1 = t0 + OR_SEG;
        if (t1 > eos) t1 = eos;
        /* re-materialise the states before every token of the segment */
        memcpy(S, ck + sg * dd, sizeof(double) * dd);
        for (int64_t t = t0; t < t1; ++t) {
            memcpy(s->seg + (t - t0) * dd, S, sizeof(double) * dd);
            load_token(J, t, h, &x);
            step_fwd(d, S, &x, NULL, s->u);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const int64_t base = (t * J->H + h) * (int64_t)d;
            memcpy(S, s->seg + (t - t0) * dd, sizeof(double) * dd); /* S_{t-1} */
            load_token(J, t, h, &x);
            step_fwd(d, S, &x, s->Sp, s->u); /* S = S_t, Sp = S'_t, u = u_t */
            const double* dO = J->dO + base;
            /* o_t = scale S_t^T q */
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int j = 0; j < d; ++j) acc += S[i * d + j] * dO[j];
                s->dq[i] = J->scale * acc;
                for (int j = 0; j < d; ++j) dS[i * d + j] += J->scale * x.q[i] * dO[j];
            }
            /* S_t = S' + beta k u^T,  u = v - S'^T k */
            double db = 0.0;
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int j = 0; j < d; ++j) acc += dS[i * d + j] * s->u[j];
                db += x.k[i] * acc;
                s->dk[i] = x.beta * acc;
            }
            for (int j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += dS[i * d + j] * x.k[i];
                s->du[j] = x.beta * acc;
            }
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int j = 0; j < d; ++j) acc += s->Sp[i * d + j] * s->du[j];
                s->dk[i] -= acc;
            }
            /* dS' = dS - k du^T ; dg_i = sum_j S'_ij dS'_ij ; dS_{t-1} = Diag(e^g) dS' */
            double* dgo = J->dgin + base;
            for (int i = 0; i < d; ++i) {
                double acc = 0.0, e = exp(x.g[i]);
                for (int j = 0; j < d; ++j) {
                    double v = dS[i * d + j] - x.k[i] * s->du[j];
                    acc += s->Sp[i * d + j] * v;
                    dS[i * d + j] = e * v;
                }
                dgo[i] = acc;
            }
            for (int j = 0; j < d; ++j) J->dv[base + j] = s->du[j];
            J->dbeta[t * J->H + h] = db;
            /* L2-norm backward: dx = (dx^ - x^ (x^ . dx^)) / sqrt(|x|^2 + eps) */
            double pq = 0.0, pk = 0.0;
            for (int c = 0; c < d; ++c) { pq += x.q[c] * s->dq[c]; pk += x.k[c] * s->dk[c]; }
            for (int c = 0; c < d; ++c) {
                if (J->l2n) {
                    J->dq[base + c] = (s->dq[c] - x.q[c] * pq) / x.qn;
                    J->dk[base + c] = (s->dk[c] - x.k[c] * pk) / x.kn;
                } else {
                    J->dq[base + c] = s->dq[c];
                    J->dk[base + c] = s->dk[c];
                }
            }
            /* raw gate chain: g = -exp(A_log) softplus(a + dt_bias) */
            if (J->raw) {
                const double eA = exp(J->A_log[h]);
                for (int c = 0; c < d; ++c) {
                    double dg = dgo[c];
                    dA += dg * x.g[c]; /* dg/dA_log = g */
                    double da = dg * (-eA) * sigmoid(J->gin[base + c] + J->dt_bias[(int64_t)h * d + c]);
                    dgo[c] = da;
                    if (ddt) ddt[c] += da;
                }
            }
        }
    }
    if (J->dA_log_part) J->dA_log_part[(size_t)n * J->H + h] = dA;
    if (J->dh0) memcpy(J->dh0 + ((size_t)n * J->H + h) * dd, dS, sizeof(double) * dd);
    free(ck);
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    scratch_t s;
    if (scratch_alloc(&s, J->d)) { J->status = -1; return NULL; }
    const int64_t total = (int64_t)J->N * J->H;
    for (;;) {
        int64_t i = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (i >= total) break;
        int n = (int)(i / J->H), h = (int)(i % J->H);
        if (J->mode == 0) chain_fwd(J, n, h, &s);
        else chain_bwd(J, n, h, &s);
    }
    scratch_free(&s);
    return NULL;
}

static int run(job_t* J, int nthreads) {
    if (J->N < 0 || J->H < 1 || J->d < 1) return -2;
    for (int n = 0; n < J->N; ++n)
        if (J->cu[n + 1] < J->cu[n]) return -3;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    J->next = 0;
    J->status = 0;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, worker, J) == 0) ++started; else break;
    worker(J);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    return J->status;
}

/* Forward: o [T,H,d] (nullable), ht [N,H,d,d] (nullable).  Returns 0 on success. */
int oracle_kda_fwd(int64_t T, int32_t N, int32_t H, int32_t d, const int32_t* cu_seqlens,
                   const double* q, const double* k, const double* v, const double* beta,
                   const double* g_or_a, const double* A_log, const double* dt_bias,
                   const double* h0, int raw, int l2n, double scale, double eps,
                   double* o, double* ht, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.T = T; J.N = N; J.H = H; J.d = d; J.cu = cu_seqlens;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.gin = g_or_a; J.A_log = A_log;
    J.dt_bias = dt_bias; J.h0 = h0; J.raw = raw; J.l2n = l2n; J.scale = scale; J.eps = eps;
    J.o = o; J.ht = ht; J.mode = 0;
    return run(&J, nthreads);
}

/* Backward of L = sum(o*dO) + sum(ht*dht).  dg_or_da receives dL/dg (g form) or dL/da (raw
 * form).  dA_log [H] and ddt_bias [H,d] are written only in raw form (nullable).  dh0 nullable. */
int oracle_kda_bwd(int64_t T, int32_t N, int32_t H, int32_t d, const int32_t* cu_seqlens,
                   const double* q, const double* k, const double* v, const double* beta,
                   const double* g_or_a, const double* A_log, const double* dt_bias,
                   const double* h0, int raw, int l2n, double scale, double eps,
                   const double* dO, const double* dht,
                   double* dq, double* dk, double* dv, double* dbeta, double* dg_or_da,
                   double* dA_log, double* ddt_bias, double* dh0, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.T = T; J.N = N; J.H = H; J.d = d; J.cu = cu_seqlens;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.gin = g_or_a; J.A_log = A_log;
    J.dt_bias = dt_bias; J.h0 = h0; J.raw = raw; J.l2n = l2n; J.scale = scale; J.eps = eps;
    J.dO = dO; J.dht = dht; J.dq = dq; J.dk = dk; J.dv = dv; J.dbeta = dbeta; J.dgin = dg_or_da;
    J.dh0 = dh0; J.mode = 1;
    double* part = NULL;
    if (raw) {
        part = calloc((size_t)N * H * (d + 1), sizeof(double));
        if (!part) return -1;
        J.dA_log_part = part;
        J.ddt_part = part + (size_t)N * H;
    }
    int rc = run(&J, nthreads);
    if (raw && rc == 0) {
        /* fixed-order reduction over documents */
        for (int h = 0; h < H; ++h) {
            double a = 0.0;
            for (int n = 0; n < N; ++n) a += J.dA_log_part[(size_t)n * H + h];
            if (dA_log) dA_log[h] = a;
            for (int c = 0; c < d; ++c) {
                double b = 0.0;
                for (int n = 0; n < N; ++n) b += J.ddt_part[((size_t)n * H + h) * d + c];
                if (ddt_bias) ddt_bias[(size_t)h * d + c] = b;
            }
        }
    }
    free(part);
    return rc;
}

/* Fragment summaries, one per (fragment, head); fragments are given as documents of cu_seqlens.
 * mode 0: M [F,H,d,d] = product of the fragment's (I - b k k^T) Diag(e^g), later tokens on the
 *         left; B [F,H,d,d] = final state of the fragment started from zero.
 * mode 1: C [F,H,d,d] = gradient at the fragment's first state for the loss sum(o*dO) with a
 *         zero end gradient.  M and the B slot are untouched in mode 1 except B_or_C = C. */
int oracle_fragment_summary(int64_t T, int32_t F, int32_t H, int32_t d, const int32_t* frag_cu,
                            const double* q, const double* k, const double* v, const double* beta,
                            const double* g_or_a, const double* A_log, const double* dt_bias,
                            int raw, int l2n, double scale, double eps, int mode,
                            const double* dO, double* M, double* B_or_C, int nthreads) {
    if (mode == 0) {
        /* M: run the state recurrence on X = I with v = 0, i.e. X <- (I - b k k^T) Diag(e^g) X */
        size_t dd = (size_t)d * d;
        double* eye = calloc((size_t)F * H * dd, sizeof(double));
        double* zv = calloc((size_t)T * H * d, sizeof(double));
        if (!eye || !zv) { free(eye); free(zv); return -1; }
        for (size_t f = 0; f < (size_t)F * H; ++f)
            for (int i = 0; i < d; ++i) eye[f * dd + (size_t)i * d + i] = 1.0;
        int rc = oracle_kda_fwd(T, F, H, d, frag_cu, q, k, zv, beta, g_or_a, A_log, dt_bias, eye,
                                raw, l2n, scale, eps, NULL, M, nthreads);
        free(eye);
        free(zv);
        if (rc) return rc;
        return oracle_kda_fwd(T, F, H, d, frag_cu, q, k, v, beta, g_or_a, A_log, dt_bias, NULL,
                              raw, l2n, scale, eps, NULL, B_or_C, nthreads);
    }
    /* C_f: dh0 of each fragment for L = sum(o*dO), dht = 0 (the other gradients are discarded) */
    size_t th = (size_t)T * H;
    double* junk = malloc(sizeof(double) * (th * (size_t)d * 4 + th));
    if (!junk) return -1;
    double* dq = junk;
    double* dk = dq + th * d;
    double* dv = dk + th * d;
    double* dg = dv + th * d;
    double* db = dg + th * d;
    int rc = oracle_kda_bwd(T, F, H, d, frag_cu, q, k, v, beta, g_or_a, A_log, dt_bias, NULL, raw,
                            l2n, scale, eps, dO, NULL, dq, dk, dv, db, dg, NULL, NULL, B_or_C,
                            nthreads);
    free(junk);
    return rc;
}

/* Transfer walk over fragments of documents.  doc_frag [N+1]: fragments of document n are
 * doc_frag[n] .. doc_frag[n+1]-1, in order.
 * forward (reverse == 0): S_in[first] = S0[n] (zeros when NULL); S_in[f+1] = M_f S_in[f] + B_f;
 *                         S_final[n] = M_last S_in[last] + B_last.
 * backward (reverse == 1): dS_end[last] = S0[n] (here: dht of the document, zeros when NULL);
 *                         dS_end[f-1] = M_f^T dS_end[f] + C_f;
 *                         S_final[n] = M_first^T dS_end[first] + C_first  (= dh0 of the document).
 * S_in [F,H,d,d] receives S_in[f] (forward) or dS_end[f] (backward). */
int oracle_transfer_walk(int32_t N, const int32_t* doc_frag, int32_t H, int32_t d,
                         const double* M, const double* B, const double* S0, int reverse,
                         double* S_in, double* S_final) {
    size_t dd = (size_t)d * d;
    double* cur = malloc(sizeof(double) * dd * 2);
    if (!cur) return -1;
    double* nxt = cur + dd;
    for (int n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) {
            if (S0) memcpy(cur, S0 + ((size_t)n * H + h) * dd, sizeof(double) * dd);
            else memset(cur, 0, sizeof(double) * dd);
            int f0 = doc_frag[n], f1 = doc_frag[n + 1];
            for (int s = 0; s < f1 - f0; ++s) {
                int f = reverse ? f1 - 1 - s : f0 + s;
                const double* Mf = M + ((size_t)f * H + h) * dd;
                const double* Bf = B + ((size_t)f * H + h) * dd;
                memcpy(S_in + ((size_t)f * H + h) * dd, cur, sizeof(double) * dd);
                for (int i = 0; i < d; ++i)
                    for (int j = 0; j < d; ++j) {
                        double acc = Bf[(size_t)i * d + j];
                        for (int l = 0; l < d; ++l) {
                            double m = reverse ? Mf[(size_t)l * d + i] : Mf[(size_t)i * d + l];
                            acc += m * cur[(size_t)l * d + j];
                        }
                        nxt[(size_t)i * d + j] = acc;
                    }
                memcpy(cur, nxt, sizeof(double) * dd);
            }
            if (S_final) memcpy(S_final + ((size_t)n * H + h) * dd, cur, sizeof(double) * dd);
        }
    }
    free(cur);
    return 0;
}
