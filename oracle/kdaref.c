/*
 * kdaref.c -- CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the libkda C-ABI
 * library or its Python binding) links, loads or calls this file.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no source, header, table or constant generator with the CUDA
 * library: every function below is written from the mathematics.
 *
 * What it computes
 * ----------------
 * KDA is the gated delta rule with a per-channel decay.  The Kimi-K3 code
 * audit (data/code-audit.json, finding "dual-kda-execution-regimes") names
 * its two execution regimes: a chunked form for training/prefill and a fused
 * recurrent form for one-token cached decoding.  Per sequence and head the
 * state S is a d_k x d_v matrix and, token by token,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T (scale * q_t)
 *
 * which, with S' = Diag(exp(g_t)) S_{t-1}, is the same as
 *
 *     u_t = beta_t (v_t - S'^T k_t),   S_t = S' + k_t u_t^T.
 *
 * The gate is g = -exp(A_log) * softplus(f + dt_bias) and beta = sigmoid(b).
 * The parameter names and shapes (A_log, dt_bias [96 x 128], b_proj per head,
 * the low-rank f projection) are those of K3_ARTIFACT_AUDIT.md section 4.1
 * (KDA tensor table) and section 5.1 (A_log / dt_bias statistics); beta as a
 * sigmoid of the raw gate, applied in fp32, is the point of finding 1 of the
 * Model-Optimizer review "[OMNIML-6079] [20/21] Add the Kimi-K3
 * expert-parallel adapter".
 *
 * Precision: the recurrence and the chunked form run in fp64.  The gate is an
 * fp32 specification (one fixed sequence of IEEE-754 binary32 operations) so
 * that a GPU implementation written independently from the same specification
 * must agree with it bit for bit.  Build with -ffp-contract=off and without
 * -ffast-math, or the specification is not what runs.
 *
 * Entry points (C ABI, all arrays row-major and contiguous):
 *   kdaref_exp_f32, kdaref_log1p_f32, kdaref_softplus_f32, kdaref_sigmoid_f32
 *   kdaref_gate_f32        -- the fp32 gate specification
 *   kdaref_recurrent       -- the fp64 token-by-token recurrence (the oracle)
 *   kdaref_recurrent_backward -- its reverse mode: gradients of q, k, v, g, beta, S0
 *   kdaref_chunked         -- the fp64 chunked (WY/UT) form, used to show the
 *                             chunked algorithm reaches the recurrence's result
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* fp32 gate specification                                                    */
/* ------------------------------------------------------------------------- */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* 2^e for e in [-126, 127], built from its bit pattern. */
static float pow2_normal(int e) { return bits_to_f32((uint32_t)(e + 127) << 23); }

/*
 * exp in binary32 by Cody-Waite range reduction (W. J. Cody and W. Waite,
 * "Software Manual for the Elementary Functions", 1980):
 *   n = nearest integer to x / ln 2,  r = x - n ln2  (|r| <= ln2/2),
 *   exp(x) = 2^n * exp(r),
 * with ln 2 split into a binary32 head and a binary32 tail, and exp(r) from
 * its Taylor series through r^7 (truncation < 6e-9 relative on |r| <= 0.347),
 * summed by Horner's rule with fused multiply-adds.  2^n is applied as two
 * exact power-of-two factors so that results in the subnormal range round
 * exactly once.
 */
float kdaref_exp_f32(float x)
{
    const float log2e = 0x1.715476p+0f;      /* binary32 nearest 1/ln 2 */
    const float ln2_hi = 0x1.62e43p-1f;      /* binary32 nearest ln 2 */
    const float ln2_lo = -0x1.05c61p-29f;    /* ln 2 - ln2_hi, rounded */
    const float round_shift = 0x1.8p23f;     /* 1.5 * 2^23 */
    const float c2 = 0x1.0p-1f, c3 = 0x1.555556p-3f, c4 = 0x1.555556p-5f;
    const float c5 = 0x1.111112p-7f, c6 = 0x1.6c16c2p-10f, c7 = 0x1.a01a02p-13f;

    if (x != x) return x;
    if (x > 88.75f) return INFINITY;
    if (x < -104.0f) return 0.0f;

    /* kf = nearest integer to x*log2e, computed exactly inside one fma. */
    float kf = fmaf(x, log2e, round_shift) - round_shift;
    /* The first reduction step is exact (the result has at most 24 bits). */
    float r = fmaf(kf, -ln2_hi, x);
    r = fmaf(kf, -ln2_lo, r);

    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);

    int n = (int)kf;          /* in [-150, 128] */
    int n1 = n / 2;           /* C division truncates toward zero */
    int n2 = n - n1;
    return (p * pow2_normal(n1)) * pow2_normal(n2);
}

/*
 * log1p in binary32 for y > -1.  u = 1 + y is split as u = 2^e m with
 * m in [sqrt(1/2), sqrt(2)].  With f = m - 1 (exact) and s = f / (2 + f),
 *   log m = 2 atanh(s) = 2s + s R(s^2),  R(z) = sum_{j>=1} 2 z^j / (2j+1)
 * (Abramowitz and Stegun 4.1.27), and since 2s = f - s f,
 *   log m = f - s (f - R).
 * |s| <= 0.1716, so R through z^5 leaves < 1e-10 relative error.  The rounding
 * of u = 1 + y is undone by c = (y - (u - 1)) / u, and e ln 2 is added with
 * ln 2 split in a head and a tail.
 */
float kdaref_log1p_f32(float y)
{
    const float ln2_hi = 0x1.62e43p-1f;
    const float ln2_lo = -0x1.05c61p-29f;
    const float sqrt2 = 0x1.6a09e6p+0f;
    const float p1 = 0x1.555556p-1f;   /* 2/3  */
    const float p2 = 0x1.99999ap-2f;   /* 2/5  */
    const float p3 = 0x1.24924ap-2f;   /* 2/7  */
    const float p4 = 0x1.c71c72p-3f;   /* 2/9  */
    const float p5 = 0x1.745d18p-3f;   /* 2/11 */

    if (y != y) return y;
    if (y == INFINITY) return y;
    if (y <= -1.0f) return (y == -1.0f) ? -INFINITY : NAN;

    float u = 1.0f + y;
    uint32_t ub = f32_to_bits(u);
    int e = (int)(ub >> 23) - 127;                 /* u is a normal number */
    float m = bits_to_f32((ub & 0x007fffffu) | 0x3f800000u);
    if (m > sqrt2) { m = m * 0.5f; e = e + 1; }
    float f = m - 1.0f;
    float c = (y - (u - 1.0f)) / u;

    float s = f / (2.0f + f);
    float z = s * s;
    float R = p5;
    R = fmaf(R, z, p4);
    R = fmaf(R, z, p3);
    R = fmaf(R, z, p2);
    R = fmaf(R, z, p1);
    R = R * z;
    float t = s * (f - R);
    float ef = (float)e;
    float lo = fmaf(ef, ln2_lo, c) - t;
    return fmaf(ef, ln2_hi, f + lo);
}

/* softplus(x) = max(x, 0) + log1p(exp(-|x|)), with no threshold. */
float kdaref_softplus_f32(float x)
{
    float pos = (x > 0.0f) ? x : 0.0f;
    float ax = fabsf(x);
    return pos + kdaref_log1p_f32(kdaref_exp_f32(-ax));
}

/* sigmoid(b) = 1 / (1 + exp(-b)), one IEEE division. */
float kdaref_sigmoid_f32(float b)
{
    return 1.0f / (1.0f + kdaref_exp_f32(-b));
}

/*
 * The gate, element by element:
 *   g[n,h,c] = -(exp(A_log[idx]) * softplus(f[n,h,c] + dt_bias[h,c]))
 *   beta[n,h] = sigmoid(b[n,h])
 * alog_mode selects the shape of A_log: 0 -> [H] (per head, the shape the
 * public configuration, HF code and FlashKDA check expect), 1 -> [K] (per
 * channel, the [128] shape found in the checkpoint header), 2 -> [H,K].
 * K3_ARTIFACT_AUDIT.md section 5.2 records this A_log shape disagreement.
 * f and b arrive as binary32 (a bf16 input is widened exactly beforehand).
 */
void kdaref_gate_f32(const float *f, const float *b, const float *A_log, int alog_mode,
                     const float *dt_bias, float *g, float *beta,
                     int64_t N, int H, int K)
{
    for (int64_t n = 0; n < N; n++) {
        for (int h = 0; h < H; h++) {
            for (int c = 0; c < K; c++) {
                int64_t i = (n * H + h) * (int64_t)K + c;
                float a_log;
                if (alog_mode == 0) a_log = A_log[h];
                else if (alog_mode == 1) a_log = A_log[c];
                else a_log = A_log[(int64_t)h * K + c];
                float x = f[i] + dt_bias[(int64_t)h * K + c];
                float sp = kdaref_softplus_f32(x);
                float a = kdaref_exp_f32(a_log);
                g[i] = -(a * sp);
            }
            if (b != NULL && beta != NULL)
                beta[n * H + h] = kdaref_sigmoid_f32(b[n * H + h]);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* fp64 recurrence and chunked form                                           */
/* ------------------------------------------------------------------------- */

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int32_t *cu_seqlens;
    int B, H, K, V;
    int64_t N;
    double scale;
    const double *S0;
    double *o, *S_final;
    int chunk, frame;      /* chunked form only */
    int nthreads;
    int thread_id;
    int status;
} job_t;

static void seq_range(const job_t *j, int seq, int64_t *t0, int64_t *t1)
{
    if (j->cu_seqlens) { *t0 = j->cu_seqlens[seq]; *t1 = j->cu_seqlens[seq + 1]; }
    else { *t0 = 0; *t1 = j->N; }
}

static void load_state(const job_t *j, int seq, int h, double *S)
{
    size_t n = (size_t)j->K * j->V;
    if (j->S0) memcpy(S, j->S0 + ((size_t)seq * j->H + h) * n, n * sizeof(double));
    else memset(S, 0, n * sizeof(double));
}

static void store_state(const job_t *j, int seq, int h, const double *S)
{
    size_t n = (size_t)j->K * j->V;
    if (j->S_final) memcpy(j->S_final + ((size_t)seq * j->H + h) * n, S, n * sizeof(double));
}

/* One (sequence, head): the recurrence, token by token, in fp64. */
static int recurrent_unit(const job_t *j, int seq, int h)
{
    const int K = j->K, V = j->V, H = j->H;
    double *S = malloc(sizeof(double) * (size_t)K * V);
    double *w = malloc(sizeof(double) * V);
    double *qs = malloc(sizeof(double) * K);
    if (!S || !w || !qs) { free(S); free(w); free(qs); return 1; }
    load_state(j, seq, h, S);
    int64_t t0, t1;
    seq_range(j, seq, &t0, &t1);
    for (int64_t t = t0; t < t1; t++) {
        const double *qt = j->q + (t * H + h) * K;
        const double *kt = j->k + (t * H + h) * K;
        const double *vt = j->v + (t * H + h) * V;
        const double *gt = j->g + (t * H + h) * K;
        const double bt = j->beta[t * H + h];
        double *ot = j->o + (t * H + h) * V;
        /* S' = Diag(exp(g_t)) S */
        for (int a = 0; a < K; a++) {
            double d = exp(gt[a]);
            for (int c = 0; c < V; c++) S[a * V + c] *= d;
        }
        /* w = S'^T k_t */
        for (int c = 0; c < V; c++) w[c] = 0.0;
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) w[c] += S[a * V + c] * kt[a];
        /* u_t = beta_t (v_t - w), kept in w */
        for (int c = 0; c < V; c++) w[c] = bt * (vt[c] - w[c]);
        /* S_t = S' + k_t u_t^T */
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) S[a * V + c] += kt[a] * w[c];
        /* o_t = S_t^T (scale q_t) */
        for (int a = 0; a < K; a++) qs[a] = j->scale * qt[a];
        for (int c = 0; c < V; c++) ot[c] = 0.0;
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) ot[c] += S[a * V + c] * qs[a];
    }
    store_state(j, seq, h, S);
    free(S); free(w); free(qs);
    return 0;
}

/*
 * One (sequence, head) in the chunked form, fp64.  Within a chunk of L
 * tokens starting from state S (rows r, s index tokens of the chunk):
 *   Gam_r      = sum_{i<=r} g_i                       (per channel)
 *   A_kk[r,s]  = beta_r <k_r * exp(Gam_r - Gam_s), k_s>      (s < r)
 *   A_qk[r,s]  = scale <q_r * exp(Gam_r - Gam_s), k_s>       (s <= r)
 *   T          = (I + A_kk)^{-1}                       (unit lower triangular)
 *   W          = T Diag(beta) Kbar,  Kbar_r = k_r * exp(Gam_r)
 *   Ut         = T Diag(beta) V
 *   U          = Ut - W S
 *   O          = Qbar S + A_qk U,    Qbar_r = scale q_r * exp(Gam_r)
 *   S         <- Diag(exp(Gam_L)) S + Khat^T U,  Khat_r = k_r * exp(Gam_L - Gam_r)
 * When frame < chunk the factor exp(Gam_r - Gam_s) of A_kk/A_qk is evaluated
 * as exp(Gam_r - ref) * exp(ref - Gam_s) with ref the Gam of the first row of
 * r's frame (rows grouped frame at a time), the factorisation a tensor-core
 * implementation needs; frame >= chunk evaluates the difference directly.
 */
static int chunked_unit(const job_t *j, int seq, int h)
{
    const int K = j->K, V = j->V, H = j->H, C = j->chunk;
    const int F = (j->frame > 0 && j->frame < C) ? j->frame : C;
    size_t CK = (size_t)C * K, CV = (size_t)C * V, CC = (size_t)C * C;
    double *S = malloc(sizeof(double) * (size_t)K * V);
    double *Gam = malloc(sizeof(double) * CK);
    double *Akk = malloc(sizeof(double) * CC), *Aqk = malloc(sizeof(double) * CC);
    double *T = malloc(sizeof(double) * CC);
    double *W = malloc(sizeof(double) * CK), *Ut = malloc(sizeof(double) * CV);
    double *U = malloc(sizeof(double) * CV);
    double *Kbar = malloc(sizeof(double) * CK), *Qbar = malloc(sizeof(double) * CK);
    double *Khat = malloc(sizeof(double) * CK);
    int ok = S && Gam && Akk && Aqk && T && W && Ut && U && Kbar && Qbar && Khat;
    if (!ok) goto done;
    load_state(j, seq, h, S);
    int64_t t0, t1;
    seq_range(j, seq, &t0, &t1);
    for (int64_t c0 = t0; c0 < t1; c0 += C) {
        int L = (int)((t1 - c0 < C) ? (t1 - c0) : C);
#define Q_(r, a) (j->q[((c0 + (r)) * H + h) * K + (a)])
#define K_(r, a) (j->k[((c0 + (r)) * H + h) * K + (a)])
#define V_(r, c) (j->v[((c0 + (r)) * H + h) * V + (c)])
#define G_(r, a) (j->g[((c0 + (r)) * H + h) * K + (a)])
#define B_(r) (j->beta[(c0 + (r)) * H + h])
        for (int a = 0; a < K; a++) {
            double acc = 0.0;
            for (int r = 0; r < L; r++) { acc += G_(r, a); Gam[(size_t)r * K + a] = acc; }
        }
        for (int r = 0; r < L; r++) {
            int ref = (r / F) * F;
            for (int s = 0; s < L; s++) {
                double akk = 0.0, aqk = 0.0;
                if (s <= r) {
                    for (int a = 0; a < K; a++) {
                        double Gr = Gam[(size_t)r * K + a], Gs = Gam[(size_t)s * K + a];
                        double e;
                        if (F < C) {
                            double Gref = Gam[(size_t)ref * K + a];
                            e = exp(Gr - Gref) * exp(Gref - Gs);
                        } else {
                            e = exp(Gr - Gs);
                        }
                        akk += K_(r, a) * e * K_(s, a);
                        aqk += Q_(r, a) * e * K_(s, a);
                    }
                }
                Akk[(size_t)r * C + s] = (s < r) ? B_(r) * akk : 0.0;
                Aqk[(size_t)r * C + s] = (s <= r) ? j->scale * aqk : 0.0;
            }
        }
        /* T = (I + A_kk)^{-1} by forward substitution, column by column. */
        for (int col = 0; col < L; col++) {
            for (int r = 0; r < L; r++) {
                double acc = (r == col) ? 1.0 : 0.0;
                for (int s = 0; s < r; s++) acc -= Akk[(size_t)r * C + s] * T[(size_t)s * C + col];
                T[(size_t)r * C + col] = acc;
            }
        }
        for (int r = 0; r < L; r++) {
            for (int a = 0; a < K; a++) {
                double Gr = Gam[(size_t)r * K + a], GL = Gam[(size_t)(L - 1) * K + a];
                Kbar[(size_t)r * K + a] = K_(r, a) * exp(Gr);
                Qbar[(size_t)r * K + a] = j->scale * Q_(r, a) * exp(Gr);
                Khat[(size_t)r * K + a] = K_(r, a) * exp(GL - Gr);
            }
        }
        for (int r = 0; r < L; r++) {
            for (int a = 0; a < K; a++) {
                double acc = 0.0;
                for (int s = 0; s < L; s++) acc += T[(size_t)r * C + s] * B_(s) * Kbar[(size_t)s * K + a];
                W[(size_t)r * K + a] = acc;
            }
            for (int c = 0; c < V; c++) {
                double acc = 0.0;
                for (int s = 0; s < L; s++) acc += T[(size_t)r * C + s] * B_(s) * V_(s, c);
                Ut[(size_t)r * V + c] = acc;
            }
        }
        for (int r = 0; r < L; r++) {
            for (int c = 0; c < V; c++) {
                double acc = Ut[(size_t)r * V + c];
                for (int a = 0; a < K; a++) acc -= W[(size_t)r * K + a] * S[(size_t)a * V + c];
                U[(size_t)r * V + c] = acc;
            }
        }
        for (int r = 0; r < L; r++) {
            double *orow = j->o + ((c0 + r) * H + h) * V;
            for (int c = 0; c < V; c++) {
                double acc = 0.0;
                for (int a = 0; a < K; a++) acc += Qbar[(size_t)r * K + a] * S[(size_t)a * V + c];
                for (int s = 0; s <= r; s++) acc += Aqk[(size_t)r * C + s] * U[(size_t)s * V + c];
                orow[c] = acc;
            }
        }
        for (int a = 0; a < K; a++) {
            double d = exp(Gam[(size_t)(L - 1) * K + a]);
            for (int c = 0; c < V; c++) {
                double acc = d * S[(size_t)a * V + c];
                for (int r = 0; r < L; r++) acc += Khat[(size_t)r * K + a] * U[(size_t)r * V + c];
                S[(size_t)a * V + c] = acc;
            }
        }
#undef Q_
#undef K_
#undef V_
#undef G_
#undef B_
    }
    store_state(j, seq, h, S);
done:
    free(S); free(Gam); free(Akk); free(Aqk); free(T); free(W); free(Ut); free(U);
    free(Kbar); free(Qbar); free(Khat);
    return ok ? 0 : 1;
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    int units = j->B * j->H;
    for (int u = j->thread_id; u < units; u += j->nthreads) {
        int seq = u / j->H, h = u % j->H;
        int rc = (j->chunk > 0) ? chunked_unit(j, seq, h) : recurrent_unit(j, seq, h);
        if (rc) j->status = rc;
    }
    return NULL;
}

static int run_jobs(job_t *tmpl)
{
    int nt = tmpl->nthreads < 1 ? 1 : tmpl->nthreads;
    int units = tmpl->B * tmpl->H;
    if (nt > units) nt = units > 0 ? units : 1;
    job_t *jobs = malloc(sizeof(job_t) * nt);
    pthread_t *th = malloc(sizeof(pthread_t) * nt);
    if (!jobs || !th) { free(jobs); free(th); return 1; }
    int status = 0;
    for (int i = 0; i < nt; i++) {
        jobs[i] = *tmpl;
        jobs[i].nthreads = nt;
        jobs[i].thread_id = i;
        jobs[i].status = 0;
    }
    for (int i = 1; i < nt; i++)
        if (pthread_create(&th[i], NULL, worker, &jobs[i])) { jobs[i].status = 2; th[i] = 0; }
    worker(&jobs[0]);
    for (int i = 1; i < nt; i++)
        if (jobs[i].status != 2) pthread_join(th[i], NULL);
    for (int i = 0; i < nt; i++) if (jobs[i].status) status = jobs[i].status;
    free(jobs); free(th);
    return status;
}

static int check_args(const double *q, const double *k, const double *v, const double *g,
                      const double *beta, const int32_t *cu, int B, int64_t N, int H, int K,
                      int V, double *o)
{
    if (!q || !k || !v || !g || !beta || !o) return 3;
    if (B < 1 || N < 0 || H < 1 || K < 1 || V < 1) return 3;
    if (!cu && B != 1) return 3;
    if (cu) {
        if (cu[0] != 0 || cu[B] != N) return 3;
        for (int i = 0; i < B; i++) if (cu[i + 1] < cu[i]) return 3;
    }
    return 0;
}

/*
 * The oracle: the fp64 recurrence over each (sequence, head), sequences given
 * by cu_seqlens[B+1] token offsets into the packed [N, H, *] arrays (NULL:
 * one sequence of N tokens).  initial_state [B,H,K,V] may be NULL (zero);
 * final_state [B,H,K,V] may be NULL.  Returns 0 on success.
 */
int kdaref_recurrent(const double *q, const double *k, const double *v, const double *g,
                     const double *beta, const int32_t *cu_seqlens, int B, int64_t N, int H,
                     int K, int V, double scale, const double *initial_state, double *o,
                     double *final_state, int nthreads)
{
    int rc = check_args(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, o);
    if (rc) return rc;
    job_t j = {q, k, v, g, beta, cu_seqlens, B, H, K, V, N, scale, initial_state, o,
               final_state, 0, 0, nthreads, 0, 0};
    return run_jobs(&j);
}

/* The fp64 chunked form with chunk size `chunk` and frame size `frame`. */
int kdaref_chunked(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const int32_t *cu_seqlens, int B, int64_t N, int H,
                   int K, int V, double scale, const double *initial_state, double *o,
                   double *final_state, int chunk, int frame, int nthreads)
{
    int rc = check_args(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, o);
    if (rc) return rc;
    if (chunk < 1) return 3;
    job_t j = {q, k, v, g, beta, cu_seqlens, B, H, K, V, N, scale, initial_state, o,
               final_state, chunk, frame, nthreads, 0, 0};
    return run_jobs(&j);
}

/* ------------------------------------------------------------------------- */
/* Reverse mode of the recurrence (the training regime's gradients), fp64      */
/* ------------------------------------------------------------------------- */

typedef struct {
    job_t f;                        /* the forward problem */
    const double *dO, *dSf;         /* [N,H,V]; [B,H,K,V] or NULL (zero) */
    double *dq, *dk, *dv, *dg, *dbeta, *dS0;
} bjob_t;

/*
 * One (sequence, head).  The forward recurrence is rerun keeping every state
 * S_t; then, from G = dL/dS_T, for t = T..1 with S' = Diag(exp g_t) S_{t-1},
 * w = S'^T k_t, u = beta_t (v_t - w), S_t = S' + k_t u^T, o_t = S_t^T (scale q_t):
 *   G   += (scale q_t) do_t^T           (o_t reads S_t)
 *   dq_t = scale S_t do_t
 *   du   = G^T k_t;   dk_t = G u;   dv_t = beta_t du;   dbeta_t = du . (v_t - w)
 *   dw   = -beta_t du;   dS' = G + k_t dw^T;   dk_t += S' dw
 *   dg_t = rowsum(dS' (.) S')           (S' = Diag(exp g_t) S_{t-1})
 *   G    = Diag(exp g_t) dS'            (= dL/dS_{t-1})
 * and dL/dS_0 = G.  Each line is the derivative of one forward line.
 */
static int backward_unit(const bjob_t *bj, int seq, int h)
{
    const job_t *j = &bj->f;
    const int K = j->K, V = j->V, H = j->H;
    const size_t KV = (size_t)K * V;
    int64_t t0, t1;
    seq_range(j, seq, &t0, &t1);
    const int64_t L = t1 - t0;
    double *Sall = malloc(sizeof(double) * KV * (size_t)(L + 1));
    double *Sp = malloc(sizeof(double) * KV);
    double *G = malloc(sizeof(double) * KV);
    double *w = malloc(sizeof(double) * V);
    double *u = malloc(sizeof(double) * V);
    double *du = malloc(sizeof(double) * V);
    double *dw = malloc(sizeof(double) * V);
    double *d = malloc(sizeof(double) * K);
    int ok = Sall && Sp && G && w && u && du && dw && d;
    if (!ok) goto done;
    load_state(j, seq, h, Sall);
    for (int64_t i = 0; i < L; i++) {            /* forward, keeping S_t at Sall[i + 1] */
        const int64_t t = t0 + i;
        const double *kt = j->k + (t * H + h) * K, *vt = j->v + (t * H + h) * V;
        const double *gt = j->g + (t * H + h) * K;
        const double bt = j->beta[t * H + h];
        const double *Sprev = Sall + (size_t)i * KV;
        double *S = Sall + (size_t)(i + 1) * KV;
        for (int a = 0; a < K; a++) {
            const double e = exp(gt[a]);
            for (int c = 0; c < V; c++) S[a * V + c] = e * Sprev[a * V + c];
        }
        for (int c = 0; c < V; c++) w[c] = 0.0;
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) w[c] += S[a * V + c] * kt[a];
        for (int c = 0; c < V; c++) u[c] = bt * (vt[c] - w[c]);
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) S[a * V + c] += kt[a] * u[c];
    }
    if (bj->dSf) memcpy(G, bj->dSf + ((size_t)seq * H + h) * KV, KV * sizeof(double));
    else memset(G, 0, KV * sizeof(double));
    for (int64_t i = L - 1; i >= 0; i--) {
        const int64_t t = t0 + i;
        const double *qt = j->q + (t * H + h) * K, *kt = j->k + (t * H + h) * K;
        const double *vt = j->v + (t * H + h) * V, *gt = j->g + (t * H + h) * K;
        const double *dot = bj->dO + (t * H + h) * V;
        const double bt = j->beta[t * H + h];
        const double *Sprev = Sall + (size_t)i * KV, *St = Sall + (size_t)(i + 1) * KV;
        double *dqt = bj->dq + (t * H + h) * K, *dkt = bj->dk + (t * H + h) * K;
        double *dvt = bj->dv + (t * H + h) * V, *dgt = bj->dg + (t * H + h) * K;
        for (int a = 0; a < K; a++) {                      /* S' and the step's u */
            d[a] = exp(gt[a]);
            for (int c = 0; c < V; c++) Sp[a * V + c] = d[a] * Sprev[a * V + c];
        }
        for (int c = 0; c < V; c++) w[c] = 0.0;
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) w[c] += Sp[a * V + c] * kt[a];
        for (int c = 0; c < V; c++) u[c] = bt * (vt[c] - w[c]);
        for (int a = 0; a < K; a++)                        /* G += (scale q) do^T */
            for (int c = 0; c < V; c++) G[a * V + c] += j->scale * qt[a] * dot[c];
        for (int a = 0; a < K; a++) {                      /* dq = scale S_t do */
            double acc = 0.0;
            for (int c = 0; c < V; c++) acc += St[a * V + c] * dot[c];
            dqt[a] = j->scale * acc;
        }
        for (int c = 0; c < V; c++) du[c] = 0.0;           /* du = G^T k */
        for (int a = 0; a < K; a++)
            for (int c = 0; c < V; c++) du[c] += G[a * V + c] * kt[a];
        double db = 0.0;
        for (int c = 0; c < V; c++) {
            dvt[c] = bt * du[c];
            db += du[c] * (vt[c] - w[c]);
            dw[c] = -bt * du[c];
        }
        bj->dbeta[t * H + h] = db;
        for (int a = 0; a < K; a++) {
            double gu = 0.0, sdw = 0.0, dgs = 0.0;
            for (int c = 0; c < V; c++) {
                const double dsp = G[a * V + c] + kt[a] * dw[c];    /* dS' */
                gu += G[a * V + c] * u[c];
                sdw += Sp[a * V + c] * dw[c];
                dgs += dsp * Sp[a * V + c];
                G[a * V + c] = d[a] * dsp;                         /* dL/dS_{t-1} */
            }
            dkt[a] = gu + sdw;
            dgt[a] = dgs;
        }
    }
    if (bj->dS0) memcpy(bj->dS0 + ((size_t)seq * H + h) * KV, G, KV * sizeof(double));
done:
    free(Sall); free(Sp); free(G); free(w); free(u); free(du); free(dw); free(d);
    return ok ? 0 : 1;
}

typedef struct {
    bjob_t *bj;
    int nthreads, thread_id, status;
} bworker_t;

static void *bworker(void *arg)
{
    bworker_t *w = (bworker_t *)arg;
    const int units = w->bj->f.B * w->bj->f.H;
    for (int u = w->thread_id; u < units; u += w->nthreads) {
        int rc = backward_unit(w->bj, u / w->bj->f.H, u % w->bj->f.H);
        if (rc) w->status = rc;
    }
    return NULL;
}

/*
 * Gradients of the recurrence (kdaref_recurrent) with respect to q, k, v, g,
 * beta and the initial state, given dO [N,H,V] and dS_final [B,H,K,V] (NULL:
 * zero).  dS0 may be NULL.  Every output is written in full.  Returns 0 on
 * success.
 */
int kdaref_recurrent_backward(const double *q, const double *k, const double *v,
                              const double *g, const double *beta, const int32_t *cu_seqlens,
                              int B, int64_t N, int H, int K, int V, double scale,
                              const double *initial_state, const double *dO,
                              const double *dS_final, double *dq, double *dk, double *dv,
                              double *dg, double *dbeta, double *dS0, int nthreads)
{
    int rc = check_args(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, dq);
    if (rc) return rc;
    if (!dO || !dk || !dv || !dg || !dbeta) return 3;
    bjob_t bj;
    memset(&bj, 0, sizeof bj);
    bj.f = (job_t){q, k, v, g, beta, cu_seqlens, B, H, K, V, N, scale, initial_state, NULL,
                   NULL, 0, 0, 1, 0, 0};
    bj.dO = dO; bj.dSf = dS_final;
    bj.dq = dq; bj.dk = dk; bj.dv = dv; bj.dg = dg; bj.dbeta = dbeta; bj.dS0 = dS0;
    int nt = nthreads < 1 ? 1 : nthreads;
    if (nt > B * H) nt = B * H;
    bworker_t *ws = malloc(sizeof(bworker_t) * nt);
    pthread_t *th = malloc(sizeof(pthread_t) * nt);
    if (!ws || !th) { free(ws); free(th); return 1; }
    for (int i = 0; i < nt; i++) ws[i] = (bworker_t){&bj, nt, i, 0};
    for (int i = 1; i < nt; i++)
        if (pthread_create(&th[i], NULL, bworker, &ws[i])) { ws[i].status = 2; th[i] = 0; }
    bworker(&ws[0]);
    int status = 0;
    for (int i = 1; i < nt; i++)
        if (ws[i].status != 2) pthread_join(th[i], NULL);
    for (int i = 0; i < nt; i++) if (ws[i].status) status = ws[i].status;
    free(ws); free(th);
    return status;
}

/* Element-wise array forms of the scalar functions (used by the ulp sweeps). */
void kdaref_exp_f32_array(const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++) y[i] = kdaref_exp_f32(x[i]);
}

void kdaref_log1p_f32_array(const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; i++) y[i] = kdaref_log1p_f32(x[i]);
}
