/*
 * gdn_oracle.c -- plain, slow, sequential fp64 oracle of the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * measured against.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call it; the library never does, and it
 * shares no code, header or table with the CUDA path.
 *
 * Everything is double precision, loops are written out, and nothing is
 * blocked, fused or reordered beyond what the cited passage states, so that a
 * reader can hold each function against the page it follows.
 *
 * Sources (titles of the web pages the method is taken from):
 *   [GDN-book]  "6.6 Gated DeltaNet (线性注意力)", sections 6.6.2-6.6.4 and 6.6.8
 *   [LinAttn]   "5. 线性注意力", sub-sections "门控 RMSNorm" and
 *               "Delta Rule 的 Chunk 实现" (the chunked algorithm)
 *   [LLM-Alg-2] "[LLM Algorithms-2] Gated DeltaNet", sections 2.1, 2.2, 4, 4.3, 5, 7
 *   [GDN-detail]"Gated DeltaNet详解" (recurrent forward with state d_v x d_k)
 *   [LinAttn-conv] "5. 线性注意力", sub-section "因果卷积(Causal Conv1d)" and the
 *               forward code after it (depthwise conv, kernel 4, then SiLU; the
 *               repeat_interleave of the q/k heads when num_v_heads > num_k_heads)
 *   [GDN-book-mix] "6.6 Gated DeltaNet", 6.6.7 (Kimi Linear: alpha_t a vector
 *               over the feature channels instead of one scalar per head)
 *
 * Conventions shared by every entry point (all arrays row-major, contiguous):
 *   q, k      [total_T][Hk][dk]     v, y      [total_T][H][dv]
 *             value head h reads query/key head h / (H / Hk)   ([LinAttn-conv]
 *             repeat_interleave; Hk == H is the plain case)
 *   g, beta   [total_T][H]          g is the log-decay, alpha_t = exp(g_t)
 *   g         [total_T][H][dk]      instead, when the decay is per key channel
 *             ([GDN-book-mix]; the reading taken: alpha scales the key columns
 *             of S, S <- S diag(alpha_t), the vector form of alpha_t S)
 *   state     [num_seqs][H][dv][dk] (the [LLM-Alg-2] section 1 orientation:
 *                                    S maps a key to a value, y = S q)
 *   cu_seqlens[num_seqs + 1]        prefix sums of the sequence lengths
 * Of the points the pages leave open, two change the numbers of every call:
 * (a) the delta is read from the decayed state ([LLM-Alg-2] 4.3) and (b)
 * l2(x) = x / sqrt(sum x^2 + 1e-6) ([GDN-book] 6.6.4 l2norm).  The readings
 * behind the options (decay per key channel, grouped heads, convolution
 * history) are stated beside the entry points that use them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define L2_EPS 1e-6

/* ------------------------------------------------------------------------ */
/* small helpers                                                            */
/* ------------------------------------------------------------------------ */

/* q/k normalisation of [GDN-book] 6.6.4: x * rsqrt(sum(x*x) + eps). */
static void l2_normalise(const double* x, double* out, int n, int enabled)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double f = enabled ? 1.0 / sqrt(ss + L2_EPS) : 1.0;
    for (int i = 0; i < n; ++i) out[i] = x[i] * f;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus(x) = log(1 + e^x), written so that large x does not overflow. */
static double softplus(double x)
{
    if (x > 30.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* Describes one slab: one sequence of one head, with row strides. */
typedef struct {
    int T, dk, dv;
    const double *q, *k, *v, *g, *beta; /* pointers at the slab's first token */
    long qk_stride, v_stride, gate_stride; /* elements between consecutive tokens */
    long g_stride;                      /* elements between consecutive tokens of g */
    int g_per_channel;                  /* g holds dk log-decays per token */
    double scale;
    int use_l2;
    const double* S0; /* dv*dk or NULL */
    double* y;        /* y rows, stride v_stride */
    double* S_out;    /* dv*dk or NULL */
} slab_t;

/* ------------------------------------------------------------------------ */
/* 1. token-by-token recurrence                                             */
/* ------------------------------------------------------------------------ */
/*
 * [LLM-Alg-2] section 4 (boxed update) and 4.3; the same order as the loop of
 * [GDN-book] 6.6.4 and [GDN-detail]'s recurrent forward:
 *     S      <- alpha_t * S                      decay first
 *     e      <- v_t - S k_t                      prediction from the decayed state
 *     S      <- S + beta_t * e k_t^T             rank-one write
 *     y_t    <- S q_t                            read after the write
 * with q_t = l2(q_t) * scale and k_t = l2(k_t) ([GDN-book] 6.6.4).
 */
static void recurrence_slab(const slab_t* s)
{
    const int dk = s->dk, dv = s->dv;
    double* S = (double*)calloc((size_t)dv * dk, sizeof(double));
    double* qn = (double*)malloc(sizeof(double) * dk);
    double* kn = (double*)malloc(sizeof(double) * dk);
    double* e = (double*)malloc(sizeof(double) * dv);
    double* al = (double*)malloc(sizeof(double) * dk);
    if (s->S0) memcpy(S, s->S0, sizeof(double) * dv * dk);

    for (int t = 0; t < s->T; ++t) {
        const double* qt = s->q + (long)t * s->qk_stride;
        const double* kt = s->k + (long)t * s->qk_stride;
        const double* vt = s->v + (long)t * s->v_stride;
        const double* gt = s->g + (long)t * s->g_stride;
        double beta = s->beta[(long)t * s->gate_stride];
        l2_normalise(qt, qn, dk, s->use_l2);
        l2_normalise(kt, kn, dk, s->use_l2);
        for (int j = 0; j < dk; ++j) qn[j] *= s->scale;

        /* alpha_t S, or S diag(alpha_t) when the decay is per key channel */
        const double a0 = exp(gt[0]);
        for (int j = 0; j < dk; ++j) al[j] = s->g_per_channel ? exp(gt[j]) : a0;
        for (int r = 0; r < dv; ++r)
            for (int j = 0; j < dk; ++j) S[(long)r * dk + j] *= al[j];
        for (int r = 0; r < dv; ++r) {
            double pred = 0.0;
            for (int j = 0; j < dk; ++j) pred += S[(long)r * dk + j] * kn[j];
            e[r] = vt[r] - pred;
        }
        for (int r = 0; r < dv; ++r)
            for (int j = 0; j < dk; ++j) S[(long)r * dk + j] += beta * e[r] * kn[j];
        double* yt = s->y + (long)t * s->v_stride;
        for (int r = 0; r < dv; ++r) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(long)r * dk + j] * qn[j];
            yt[r] = acc;
        }
    }
    if (s->S_out) memcpy(s->S_out, S, sizeof(double) * dv * dk);
    free(S); free(qn); free(kn); free(e); free(al);
}

/* ------------------------------------------------------------------------ */
/* 2. chunked (UT / WY) form                                                */
/* ------------------------------------------------------------------------ */

/*
 * Decay matrix of one chunk, [LinAttn] "阶段 1": gcum = inclusive cumulative
 * sum of g; decay[i][j] = exp(gcum[i] - gcum[j]) for i >= j, 0 above the
 * diagonal (the causal mask is stated explicitly rather than relying on
 * tril() before exp()).  out is L*L.
 */
void gdn_oracle_chunk_decay(const double* g, int L, double* gcum, double* out)
{
    double acc = 0.0;
    for (int i = 0; i < L; ++i) { acc += g[i]; gcum[i] = acc; }
    for (int i = 0; i < L; ++i)
        for (int j = 0; j < L; ++j)
            out[(long)i * L + j] = (j <= i) ? exp(gcum[i] - gcum[j]) : 0.0;
}

/*
 * [LinAttn] "Delta Rule 的 Chunk 实现": the sequence is cut into chunks of C
 * tokens; a last, shorter chunk is handled at its own length L (identical to
 * the page's zero padding, because padded tokens carry k = v = beta = 0 and
 * g = 0 and therefore leave S and the real outputs unchanged).
 * Per chunk, with Kb = diag(beta) K, Vb = diag(beta) V:
 *   stage 1  gcum, decay                      (gdn_oracle_chunk_decay)
 *   stage 2  attn = -(Kb K^T) * decay, strictly lower;
 *            row substitution attn[i,:i] += sum_m attn[i,m] attn[m,:i], then + I,
 *            so attn = (I + A)^-1 with A = (Kb K^T) * decay strictly lower;
 *            value      = attn Vb                         ("U")
 *            k_cumdecay = attn (Kb * exp(gcum))           ("W")
 *   stage 3  v_new = value - k_cumdecay S^T               (S is dv x dk here)
 *            out   = (Q * exp(gcum)) S^T + (Q K^T * decay) v_new
 *            S     = S exp(gcum[L-1]) + v_new^T (K * exp(gcum[L-1] - gcum))
 * The page writes S as dk x dv; with the dv x dk orientation used here the
 * products S and S^T swap, nothing else changes.
 */
static void chunked_slab(const slab_t* s, int C)
{
    const int dk = s->dk, dv = s->dv;
    double* S = (double*)calloc((size_t)dv * dk, sizeof(double));
    double* Q = (double*)malloc(sizeof(double) * C * dk);
    double* K = (double*)malloc(sizeof(double) * C * dk);
    double* V = (double*)malloc(sizeof(double) * C * dv);
    double* bt = (double*)malloc(sizeof(double) * C);
    double* gg = (double*)malloc(sizeof(double) * C);
    double* gcum = (double*)malloc(sizeof(double) * C);
    double* decay = (double*)malloc(sizeof(double) * C * C);
    double* attn = (double*)malloc(sizeof(double) * C * C);
    double* rowbuf = (double*)malloc(sizeof(double) * C);
    double* value = (double*)malloc(sizeof(double) * C * dv);
    double* kcum = (double*)malloc(sizeof(double) * C * dk);
    double* vnew = (double*)malloc(sizeof(double) * C * dv);
    double* qk = (double*)malloc(sizeof(double) * C * C);
    double* Snext = (double*)malloc(sizeof(double) * dv * dk);
    if (s->S0) memcpy(S, s->S0, sizeof(double) * dv * dk);

    for (int c0 = 0; c0 < s->T; c0 += C) {
        const int L = (s->T - c0 < C) ? (s->T - c0) : C;
        for (int i = 0; i < L; ++i) {
            long t = c0 + i;
            l2_normalise(s->q + t * s->qk_stride, Q + (long)i * dk, dk, s->use_l2);
            l2_normalise(s->k + t * s->qk_stride, K + (long)i * dk, dk, s->use_l2);
            for (int j = 0; j < dk; ++j) Q[(long)i * dk + j] *= s->scale;
            for (int r = 0; r < dv; ++r) V[(long)i * dv + r] = s->v[t * s->v_stride + r];
            bt[i] = s->beta[t * s->gate_stride];
            gg[i] = s->g[t * s->g_stride];
        }
        /* stage 1 */
        gdn_oracle_chunk_decay(gg, L, gcum, decay);
        /* stage 2: attn = -(Kb K^T) * decay, zero on and above the diagonal */
        for (int i = 0; i < L; ++i)
            for (int j = 0; j < L; ++j) {
                double a = 0.0;
                if (j < i) {
                    double dot = 0.0;
                    for (int x = 0; x < dk; ++x) dot += K[(long)i * dk + x] * K[(long)j * dk + x];
                    a = -bt[i] * dot * decay[(long)i * L + j];
                }
                attn[(long)i * L + j] = a;
            }
        /* row substitution; rows above i already hold their final values */
        for (int i = 1; i < L; ++i) {
            for (int j = 0; j < i; ++j) rowbuf[j] = attn[(long)i * L + j];
            for (int j = 0; j < i; ++j) {
                double acc = 0.0;
                for (int m = 0; m < i; ++m) acc += rowbuf[m] * attn[(long)m * L + j];
                attn[(long)i * L + j] = rowbuf[j] + acc;
            }
        }
        for (int i = 0; i < L; ++i) attn[(long)i * L + i] += 1.0;
        /* value = attn Vb ; k_cumdecay = attn (Kb * exp(gcum)) */
        for (int i = 0; i < L; ++i) {
            for (int r = 0; r < dv; ++r) {
                double acc = 0.0;
                for (int j = 0; j < L; ++j) acc += attn[(long)i * L + j] * bt[j] * V[(long)j * dv + r];
                value[(long)i * dv + r] = acc;
            }
            for (int x = 0; x < dk; ++x) {
                double acc = 0.0;
                for (int j = 0; j < L; ++j)
                    acc += attn[(long)i * L + j] * bt[j] * exp(gcum[j]) * K[(long)j * dk + x];
                kcum[(long)i * dk + x] = acc;
            }
        }
        /* stage 3 */
        for (int i = 0; i < L; ++i)
            for (int r = 0; r < dv; ++r) {
                double acc = 0.0;
                for (int x = 0; x < dk; ++x) acc += kcum[(long)i * dk + x] * S[(long)r * dk + x];
                vnew[(long)i * dv + r] = value[(long)i * dv + r] - acc;
            }
        for (int i = 0; i < L; ++i)
            for (int j = 0; j < L; ++j) {
                double dot = 0.0;
                if (j <= i)
                    for (int x = 0; x < dk; ++x) dot += Q[(long)i * dk + x] * K[(long)j * dk + x];
                qk[(long)i * L + j] = dot * decay[(long)i * L + j];
            }
        for (int i = 0; i < L; ++i) {
            double* yt = s->y + (long)(c0 + i) * s->v_stride;
            for (int r = 0; r < dv; ++r) {
                double inter = 0.0, intra = 0.0;
                for (int x = 0; x < dk; ++x) inter += Q[(long)i * dk + x] * S[(long)r * dk + x];
                inter *= exp(gcum[i]);
                for (int j = 0; j < L; ++j) intra += qk[(long)i * L + j] * vnew[(long)j * dv + r];
                yt[r] = inter + intra;
            }
        }
        const double glast = gcum[L - 1];
        for (int r = 0; r < dv; ++r)
            for (int x = 0; x < dk; ++x) {
                double acc = 0.0;
                for (int j = 0; j < L; ++j)
                    acc += vnew[(long)j * dv + r] * K[(long)j * dk + x] * exp(glast - gcum[j]);
                Snext[(long)r * dk + x] = S[(long)r * dk + x] * exp(glast) + acc;
            }
        memcpy(S, Snext, sizeof(double) * dv * dk);
    }
    if (s->S_out) memcpy(s->S_out, S, sizeof(double) * dv * dk);
    free(S); free(Q); free(K); free(V); free(bt); free(gg); free(gcum); free(decay);
    free(attn); free(rowbuf); free(value); free(kcum); free(vnew); free(qk); free(Snext);
}

/* ------------------------------------------------------------------------ */
/* 3. transition-product (unrolled) form                                    */
/* ------------------------------------------------------------------------ */
/*
 * [LLM-Alg-2] section 7: S_t = S_{t-1} A_t + B_t with
 *     A_t = alpha_t (I - beta_t k_t k_t^T)   (dk x dk)
 *         = diag(alpha_t) (I - beta_t k_t k_t^T) when alpha_t is per key channel
 *     B_t = beta_t v_t k_t^T                 (dv x dk)
 * unrolled to S_t = S_0 A_1...A_t + sum_{i<=t} B_i A_{i+1}...A_t, y_t = S_t q_t.
 * Every product is formed explicitly with dense matrices, for every t; this is
 * O(T^3 d^3) and meant for T of a few tens at most.
 */
static void matmul_dd(const double* X, const double* Y, double* Z, int m, int n, int p)
{ /* Z[m x p] = X[m x n] Y[n x p] */
    for (int i = 0; i < m; ++i)
        for (int j = 0; j < p; ++j) {
            double acc = 0.0;
            for (int x = 0; x < n; ++x) acc += X[(long)i * n + x] * Y[(long)x * p + j];
            Z[(long)i * p + j] = acc;
        }
}

static void transition_product_slab(const slab_t* s)
{
    const int dk = s->dk, dv = s->dv, T = s->T;
    double* A = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * dk * dk);
    double* B = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * dv * dk);
    double* P = (double*)malloc(sizeof(double) * dk * dk);
    double* Ptmp = (double*)malloc(sizeof(double) * dk * dk);
    double* St = (double*)malloc(sizeof(double) * dv * dk);
    double* term = (double*)malloc(sizeof(double) * dv * dk);
    double* qn = (double*)malloc(sizeof(double) * dk);
    double* kn = (double*)malloc(sizeof(double) * dk);

    for (int t = 0; t < T; ++t) {
        l2_normalise(s->k + (long)t * s->qk_stride, kn, dk, s->use_l2);
        const double* gt = s->g + (long)t * s->g_stride;
        double beta = s->beta[(long)t * s->gate_stride];
        const double* vt = s->v + (long)t * s->v_stride;
        for (int i = 0; i < dk; ++i) {
            double alpha = exp(s->g_per_channel ? gt[i] : gt[0]);
            for (int j = 0; j < dk; ++j)
                A[(long)t * dk * dk + (long)i * dk + j] = alpha * ((i == j ? 1.0 : 0.0) - beta * kn[i] * kn[j]);
        }
        for (int r = 0; r < dv; ++r)
            for (int j = 0; j < dk; ++j) B[(long)t * dv * dk + (long)r * dk + j] = beta * vt[r] * kn[j];
    }
    for (int t = 0; t < T; ++t) {
        /* S_0 A_1 ... A_t */
        for (int i = 0; i < dk * dk; ++i) P[i] = (i / dk == i % dk) ? 1.0 : 0.0;
        for (int u = 0; u <= t; ++u) {
            matmul_dd(P, A + (long)u * dk * dk, Ptmp, dk, dk, dk);
            memcpy(P, Ptmp, sizeof(double) * dk * dk);
        }
        if (s->S0) matmul_dd(s->S0, P, St, dv, dk, dk);
        else memset(St, 0, sizeof(double) * dv * dk);
        /* + sum_i B_i A_{i+1} ... A_t */
        for (int i = 0; i <= t; ++i) {
            for (int x = 0; x < dk * dk; ++x) P[x] = (x / dk == x % dk) ? 1.0 : 0.0;
            for (int u = i + 1; u <= t; ++u) {
                matmul_dd(P, A + (long)u * dk * dk, Ptmp, dk, dk, dk);
                memcpy(P, Ptmp, sizeof(double) * dk * dk);
            }
            matmul_dd(B + (long)i * dv * dk, P, term, dv, dk, dk);
            for (int x = 0; x < dv * dk; ++x) St[x] += term[x];
        }
        l2_normalise(s->q + (long)t * s->qk_stride, qn, dk, s->use_l2);
        double* yt = s->y + (long)t * s->v_stride;
        for (int r = 0; r < dv; ++r) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += St[(long)r * dk + j] * qn[j] * s->scale;
            yt[r] = acc;
        }
        if (t == T - 1 && s->S_out) memcpy(s->S_out, St, sizeof(double) * dv * dk);
    }
    if (T == 0 && s->S_out) {
        if (s->S0) memcpy(s->S_out, s->S0, sizeof(double) * dv * dk);
        else memset(s->S_out, 0, sizeof(double) * dv * dk);
    }
    free(A); free(B); free(P); free(Ptmp); free(St); free(term); free(qn); free(kn);
}

/* ------------------------------------------------------------------------ */
/* varlen driver: one slab per (sequence, head), spread over threads        */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int32_t* cu;
    int num_seqs, H, Hk, dk, dv, g_per_channel, use_l2, form, C;
    double scale;
    const double* S0;
    double* y;
    double* S_final;
    long next_unit; /* shared work counter, guarded by mu */
    pthread_mutex_t mu;
} job_t;

static void run_unit(job_t* j, long unit)
{
    int n = (int)(unit / j->H), h = (int)(unit % j->H);
    long bos = j->cu[n], eos = j->cu[n + 1];
    slab_t s;
    s.T = (int)(eos - bos);
    s.dk = j->dk;
    s.dv = j->dv;
    const int hk = h / (j->H / j->Hk); /* repeat_interleave of the query/key heads */
    s.qk_stride = (long)j->Hk * j->dk;
    s.v_stride = (long)j->H * j->dv;
    s.gate_stride = j->H;
    s.g_per_channel = j->g_per_channel;
    s.g_stride = j->g_per_channel ? (long)j->H * j->dk : j->H;
    s.q = j->q + bos * s.qk_stride + (long)hk * j->dk;
    s.k = j->k + bos * s.qk_stride + (long)hk * j->dk;
    s.v = j->v + bos * s.v_stride + (long)h * j->dv;
    s.g = j->g + bos * s.g_stride + (long)h * (j->g_per_channel ? j->dk : 1);
    s.beta = j->beta + bos * j->H + h;
    s.scale = j->scale;
    s.use_l2 = j->use_l2;
    long slab = (long)j->dv * j->dk;
    s.S0 = j->S0 ? j->S0 + unit * slab : NULL;
    s.S_out = j->S_final ? j->S_final + unit * slab : NULL;
    s.y = j->y + bos * s.v_stride + (long)h * j->dv;
    if (j->form == 0) recurrence_slab(&s);
    else if (j->form == 1) chunked_slab(&s, j->C);
    else transition_product_slab(&s);
}

static void* worker(void* arg)
{
    job_t* j = (job_t*)arg;
    const long total = (long)j->num_seqs * j->H;
    for (;;) {
        pthread_mutex_lock(&j->mu);
        long u = j->next_unit++;
        pthread_mutex_unlock(&j->mu);
        if (u >= total) break;
        run_unit(j, u);
    }
    return NULL;
}

static int run_job(job_t* j, int n_threads)
{
    for (int n = 0; n < j->num_seqs; ++n)
        if (j->cu[n + 1] < j->cu[n]) return -1;
    if (j->form == 1 && (j->C <= 0 || j->g_per_channel)) return -1; /* the page's chunk algorithm is scalar */
    if (j->Hk <= 0 || j->H % j->Hk != 0) return -1;
    j->next_unit = 0;
    pthread_mutex_init(&j->mu, NULL);
    if (n_threads <= 1) {
        worker(j);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
        for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, worker, j);
        for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&j->mu);
    return 0;
}

/*
 * form: 0 = token-by-token recurrence, 1 = chunked form with chunk size C,
 *       2 = transition product.  Hk = number of query/key heads (H a multiple of
 *       it); g_per_channel = 1 when g is [total_T][H][dk] (not for form 1).
 *       Returns 0, or -1 on a malformed cu_seqlens or an unsupported request.
 */
int gdn_oracle_forward(int form, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, const int32_t* cu_seqlens,
                       int num_seqs, int H, int Hk, int dk, int dv, int g_per_channel,
                       double scale, int use_qk_l2norm,
                       const double* S0, double* y, double* S_final, int C, int n_threads)
{
    job_t j;
    j.q = q; j.k = k; j.v = v; j.g = g; j.beta = beta; j.cu = cu_seqlens;
    j.num_seqs = num_seqs; j.H = H; j.Hk = Hk; j.dk = dk; j.dv = dv; j.use_l2 = use_qk_l2norm;
    j.g_per_channel = g_per_channel;
    j.form = form; j.C = C; j.scale = scale; j.S0 = S0; j.y = y; j.S_final = S_final;
    return run_job(&j, n_threads);
}

/* ------------------------------------------------------------------------ */
/* gated output and gate preparation                                        */
/* ------------------------------------------------------------------------ */

/*
 * [LinAttn] "门控 RMSNorm" (RMSNormGated) and [GDN-book] 6.6.2 o_t:
 *     o = w * y / sqrt(mean(y^2) + eps) * z * sigmoid(z)     per row of dv
 * w == NULL means w = 1 (the page's one-initialised weight).  No intermediate
 * rounding (the page's cast back to the input dtype is not modelled).
 */
void gdn_oracle_gate_rmsnorm_silu(const double* y, const double* z, const double* w, double eps,
                                  double* out, long rows, int dv)
{
    for (long r = 0; r < rows; ++r) {
        const double* yr = y + r * dv;
        const double* zr = z + r * dv;
        double ms = 0.0;
        for (int c = 0; c < dv; ++c) ms += yr[c] * yr[c];
        ms /= dv;
        double inv = 1.0 / sqrt(ms + eps);
        for (int c = 0; c < dv; ++c) {
            double wc = w ? w[c] : 1.0;
            out[r * dv + c] = wc * yr[c] * inv * zr[c] * sigmoid(zr[c]);
        }
    }
}

/*
 * [GDN-book] 6.6.3 decay gate and update gate:
 *     g    = log(alpha) = -exp(A_log[h]) * softplus(a + dt_bias[h])
 *     beta = sigmoid(b)
 * a, b, g, beta are [total_T][H]; A_log, dt_bias are [H]; dt_bias and b may be
 * NULL (dt_bias = 0; beta not produced).
 */
void gdn_oracle_gates_from_logits(const double* a, const double* A_log, const double* dt_bias,
                                  const double* b, double* g, double* beta, long total_T, int H)
{
    for (long t = 0; t < total_T; ++t)
        for (int h = 0; h < H; ++h) {
            long i = t * H + h;
            double bias = dt_bias ? dt_bias[h] : 0.0;
            g[i] = -exp(A_log[h]) * softplus(a[i] + bias);
            if (b && beta) beta[i] = sigmoid(b[i]);
        }
}

/* ------------------------------------------------------------------------ */
/* causal depthwise short convolution                                       */
/* ------------------------------------------------------------------------ */

/*
 * [LinAttn-conv]: a depthwise Conv1d (one K-tap filter per channel, no bias)
 * with K-1 zeros of left padding, cut back to the sequence length, then SiLU:
 *     out[t][c] = silu( sum_{j<K} w[c][j] * xp[t + j][c] ),
 *     xp = [K-1 history rows ; x_0 ... x_{T-1}]
 * so tap K-1 multiplies the current token (the page's step-by-step picture).
 * The history rows are zeros (the page's padding) or, for a sequence continued
 * from an earlier call, its carried state, oldest first: state[c][j] =
 * xp[j][c].  After the sequence, state_out holds the last K-1 rows of xp.
 * x, out [total_T][channels]; w [channels][K]; state_in/out
 * [num_seqs][channels][K-1] (either may be NULL); silu = 0 skips the SiLU.
 * Returns -1 on a malformed cu_seqlens.
 */
int gdn_oracle_short_conv(const double* x, const double* w, const int32_t* cu_seqlens, int num_seqs,
                          int channels, int K, const double* state_in, double* out,
                          double* state_out, int silu)
{
    for (int n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    double* xp = NULL;
    for (int n = 0; n < num_seqs; ++n) {
        const long bos = cu_seqlens[n], T = cu_seqlens[n + 1] - cu_seqlens[n];
        xp = (double*)realloc(xp, sizeof(double) * (size_t)(T + K - 1 > 0 ? T + K - 1 : 1));
        for (int c = 0; c < channels; ++c) {
            for (int j = 0; j < K - 1; ++j)
                xp[j] = state_in ? state_in[((long)n * channels + c) * (K - 1) + j] : 0.0;
            for (long t = 0; t < T; ++t) xp[K - 1 + t] = x[(bos + t) * channels + c];
            for (long t = 0; t < T; ++t) {
                double acc = 0.0;
                for (int j = 0; j < K; ++j) acc += w[(long)c * K + j] * xp[t + j];
                out[(bos + t) * channels + c] = silu ? acc * sigmoid(acc) : acc;
            }
            if (state_out)
                for (int j = 0; j < K - 1; ++j)
                    state_out[((long)n * channels + c) * (K - 1) + j] = xp[T + j];
        }
    }
    free(xp);
    return 0;
}
