/*
 * dn_oracle.c -- fp64 CPU oracle for the chunkwise gated delta rule forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * Sources (web pages on the method; cited by title and section):
 *   [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现"
 *          (DeltaNet chunkwise parallelism: WY derivation and Triton kernels)
 *   [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么"
 *          (what the ChunkGatedDeltaRule operator computes)
 *
 * Two independent forms of the forward are implemented:
 *
 *   dn_oracle_recurrent  -- the definition: a token-by-token recurrence
 *                           ([WY] §1, [CGDR] §1), written out plainly.
 *   dn_oracle_chunked    -- the chunk algorithm in the pages' order: gate
 *                           prefix sum, WY matrix A, T = (I-A)^-1, W and U,
 *                           v_new, output, state ([CGDR] §3.1-§3.3,
 *                           [WY] §2.3-§2.4).  Used to pin the chunk algebra.
 *
 * and the gradient of the forward:
 *
 *   dn_oracle_recurrent_bwd -- reverse-mode differentiation of the token
 *                           recurrence, token by token in reverse order
 *                           ([WY] §3.4 names the gradients dq, dk, dv,
 *                           dbeta and dh0 of the backward, and [WY] §6 its
 *                           tests; dg is the gradient of the gated form).
 *                           The pages print no backward formula, so this is
 *                           the chain rule applied to each step of the
 *                           definition; the tests pin it by finite
 *                           differences of dn_oracle_recurrent.
 *
 * Readings taken where the pages are silent or garbled:
 *   - decay placement: the state is decayed *before* the delta read, i.e.
 *       S_t = e^{g_t} S_{t-1} + b_t k_t (v_t - k_t^T e^{g_t} S_{t-1})^T.
 *     [CGDR] §1 step 3 says "forget first, then write", and the chunk form of
 *     [CGDR] §3.1-§3.2 (A with e^{G_i-G_j}, G inclusive) equals this recurrence
 *     only.  read_mode = 1 selects the literal (undecayed) read
 *     v_t - k_t^T S_{t-1} of [CGDR] §1's formula; it exists only so the tests
 *     can show that the chunk form disagrees with it.
 *   - o_t reads the state after token t's update ([WY] §1 listing order), so
 *     the in-chunk output mask keeps j <= i (diagonal included).
 *   - G is an inclusive prefix sum that restarts at every chunk.
 *   - the cumulative decay in [CGDR] §3.2 (1) is e^{G_i}.
 *   - scale multiplies q only.
 *   - GQA: v-head h reads q/k head h / (Nv/Nk) ([CGDR] §1, last paragraph).
 *
 * Layouts (row-major, tokens flattened over the batch):
 *   q, k  [B*T, Nk, dk]     v, o  [B*T, Nv, dv]     beta, g  [B*T, Nv]
 *   h0, ht [N, Nv, dk, dv]
 * Sequence n covers tokens [cu[n], cu[n+1]) when cu_seqlens is given (B==1),
 * else [n*T, (n+1)*T) with N == B.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *beta, *g, *h0;
    const int64_t *cu;
    int n_seqs, B, T, Nk, Nv, dk, dv;
    double scale;
    double *o, *ht;
    int chunk;      /* chunked form only */
    int read_mode;  /* recurrent form only: 0 decayed read, 1 literal read */
    const int32_t *units; /* unit u = n * Nv + h */
    int n_units;
    int next;       /* work counter */
    int failed;
    pthread_mutex_t lock;
} job_t;

static void seq_bounds(const job_t *J, int n, int64_t *bos, int64_t *eos)
{
    if (J->cu) {
        *bos = J->cu[n];
        *eos = J->cu[n + 1];
    } else {
        *bos = (int64_t)n * J->T;
        *eos = (int64_t)(n + 1) * J->T;
    }
}

/* ---------------------------------------------------------------------- */
/* The definition: token recurrence ([WY] §1, [CGDR] §1).                  */
/* ---------------------------------------------------------------------- */
static void recurrent_unit(const job_t *J, int n, int h, double *S, double *delta)
{
    const int dk = J->dk, dv = J->dv, Nk = J->Nk, Nv = J->Nv;
    const int hk = h / (Nv / Nk);
    int64_t bos, eos;
    seq_bounds(J, n, &bos, &eos);

    if (J->h0)
        memcpy(S, J->h0 + ((size_t)n * Nv + h) * dk * dv, sizeof(double) * dk * dv);
    else
        memset(S, 0, sizeof(double) * dk * dv);

    for (int64_t t = bos; t < eos; ++t) {
        const double *qt = J->q + ((size_t)t * Nk + hk) * dk;
        const double *kt = J->k + ((size_t)t * Nk + hk) * dk;
        const double *vt = J->v + ((size_t)t * Nv + h) * dv;
        const double bt = J->beta[(size_t)t * Nv + h];
        const double alpha = J->g ? exp(J->g[(size_t)t * Nv + h]) : 1.0;

        if (J->read_mode == 0) {
            /* forget first: S <- alpha S */
            for (int i = 0; i < dk * dv; ++i) S[i] *= alpha;
            /* delta = beta (v - S^T k) */
            for (int c = 0; c < dv; ++c) {
                double r = 0.0;
                for (int d = 0; d < dk; ++d) r += kt[d] * S[d * dv + c];
                delta[c] = bt * (vt[c] - r);
            }
        } else {
            /* literal read of the old state, then forget */
            for (int c = 0; c < dv; ++c) {
                double r = 0.0;
                for (int d = 0; d < dk; ++d) r += kt[d] * S[d * dv + c];
                delta[c] = bt * (vt[c] - r);
            }
            for (int i = 0; i < dk * dv; ++i) S[i] *= alpha;
        }
        /* write: S <- S + k delta^T */
        for (int d = 0; d < dk; ++d)
            for (int c = 0; c < dv; ++c) S[d * dv + c] += kt[d] * delta[c];
        /* read: o_t = scale S^T q_t */
        double *ot = J->o + ((size_t)t * Nv + h) * dv;
        for (int c = 0; c < dv; ++c) {
            double r = 0.0;
            for (int d = 0; d < dk; ++d) r += qt[d] * S[d * dv + c];
            ot[c] = J->scale * r;
        }
    }
    if (J->ht)
        memcpy(J->ht + ((size_t)n * Nv + h) * dk * dv, S, sizeof(double) * dk * dv);
}

/* ---------------------------------------------------------------------- */
/* The chunk algorithm ([CGDR] §3, [WY] §2.3-§2.4), one chunk of L tokens. */
/* ---------------------------------------------------------------------- */

/*
 * Steps a1-a4 for one chunk: G, A, T = (I - A)^-1, W, U.
 *   K [L, ldk] (row stride ldk), V [L, ldv], beta[L] and g[L] with strides.
 *   Outputs (row-major, L rows): G[L], Tm[L*L], W[L*dk], U[L*dv].
 * g may be NULL (no gate).
 */
void dn_oracle_wy_chunk(int L, int dk, int dv,
                        const double *K, long ldk, const double *V, long ldv,
                        const double *beta, long ldb, const double *g, long ldg,
                        double *G, double *Tm, double *W, double *U)
{
    /* a1: inclusive in-chunk prefix sum of the log gate ([CGDR] §3, G_i). */
    double acc = 0.0;
    for (int i = 0; i < L; ++i) {
        acc += g ? g[(long)i * ldg] : 0.0;
        G[i] = acc;
    }
    /* a2: A_ij = -beta_i (k_i . k_j) e^{G_i - G_j}, j < i ([CGDR] §3.1 step 1). */
    double *A = (double *)calloc((size_t)L * L, sizeof(double));
    for (int i = 0; i < L; ++i)
        for (int j = 0; j < i; ++j) {
            double kk = 0.0;
            for (int d = 0; d < dk; ++d) kk += K[(long)i * ldk + d] * K[(long)j * ldk + d];
            A[i * L + j] = -beta[(long)i * ldb] * kk * exp(G[i] - G[j]);
        }
    /* a3: T = (I - A)^-1.  [CGDR] §3.1 step 2 builds it row by row: row i is
     * row i of A plus the A-weighted sum of the finished rows above it, and
     * the diagonal is set to 1 ([CGDR] §3.1 step 3). */
    for (int i = 0; i < L; ++i) {
        for (int j = 0; j < L; ++j) Tm[i * L + j] = 0.0;
        for (int j = 0; j < i; ++j) {
            double s = A[i * L + j];
            for (int m = j + 1; m < i; ++m) s += A[i * L + m] * Tm[m * L + j];
            Tm[i * L + j] = s;
        }
        Tm[i * L + i] = 1.0;
    }
    free(A);
    /* a4: W = T diag(beta e^G) K, U = T diag(beta) V ([CGDR] §3.2 (1)-(2),
     * [WY] §2.3 with diag(beta) moved onto K and V as in [WY] §3.3). */
    for (int i = 0; i < L; ++i) {
        for (int d = 0; d < dk; ++d) {
            double s = 0.0;
            for (int j = 0; j <= i; ++j)
                s += Tm[i * L + j] * beta[(long)j * ldb] * exp(G[j]) * K[(long)j * ldk + d];
            W[(long)i * dk + d] = s;
        }
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int j = 0; j <= i; ++j)
                s += Tm[i * L + j] * beta[(long)j * ldb] * V[(long)j * ldv + c];
            U[(long)i * dv + c] = s;
        }
    }
}

static void chunked_unit(const job_t *J, int n, int h, double *S)
{
    const int dk = J->dk, dv = J->dv, Nk = J->Nk, Nv = J->Nv, C = J->chunk;
    const int hk = h / (Nv / Nk);
    int64_t bos, eos;
    seq_bounds(J, n, &bos, &eos);

    double *G = (double *)malloc(sizeof(double) * C);
    double *Tm = (double *)malloc(sizeof(double) * C * C);
    double *W = (double *)malloc(sizeof(double) * C * dk);
    double *U = (double *)malloc(sizeof(double) * C * dv);
    double *Vn = (double *)malloc(sizeof(double) * C * dv);
    double *Snew = (double *)malloc(sizeof(double) * dk * dv);

    if (J->h0)
        memcpy(S, J->h0 + ((size_t)n * Nv + h) * dk * dv, sizeof(double) * dk * dv);
    else
        memset(S, 0, sizeof(double) * dk * dv);

    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        const double *K = J->k + ((size_t)t0 * Nk + hk) * dk;
        const double *Q = J->q + ((size_t)t0 * Nk + hk) * dk;
        const double *V = J->v + ((size_t)t0 * Nv + h) * dv;
        const long ldk = (long)Nk * dk, ldv = (long)Nv * dv;
        const double *bt = J->beta + (size_t)t0 * Nv + h;
        const double *gt = J->g ? J->g + (size_t)t0 * Nv + h : NULL;

        dn_oracle_wy_chunk(L, dk, dv, K, ldk, V, ldv, bt, Nv, gt, Nv, G, Tm, W, U);

        /* a5: v_new = U - W S_in ([CGDR] §3.2 (3), [WY] §2.4). */
        for (int i = 0; i < L; ++i)
            for (int c = 0; c < dv; ++c) {
                double s = 0.0;
                for (int d = 0; d < dk; ++d) s += W[(long)i * dk + d] * S[d * dv + c];
                Vn[i * dv + c] = U[(long)i * dv + c] - s;
            }
        /* a6: o_i = scale e^{G_i} q_i^T S_in
         *         + scale sum_{j<=i} (q_i . k_j) e^{G_i-G_j} v_new_j
         * ([CGDR] §3.2 (4)-(5), [WY] §2.4). */
        for (int i = 0; i < L; ++i) {
            double *oi = J->o + ((size_t)(t0 + i) * Nv + h) * dv;
            for (int c = 0; c < dv; ++c) {
                double inter = 0.0;
                for (int d = 0; d < dk; ++d) inter += Q[(long)i * ldk + d] * S[d * dv + c];
                oi[c] = J->scale * exp(G[i]) * inter;
            }
            for (int j = 0; j <= i; ++j) {
                double qk = 0.0;
                for (int d = 0; d < dk; ++d) qk += Q[(long)i * ldk + d] * K[(long)j * ldk + d];
                const double a = J->scale * qk * exp(G[i] - G[j]);
                for (int c = 0; c < dv; ++c) oi[c] += a * Vn[j * dv + c];
            }
        }
        /* a5 (state): S_out = e^{G_L} S_in + sum_i e^{G_L - G_i} k_i v_new_i^T
         * ([CGDR] §3.2 (6)); G_L is the prefix at the last real token. */
        const double GL = G[L - 1];
        for (int d = 0; d < dk; ++d)
            for (int c = 0; c < dv; ++c) {
                double s = exp(GL) * S[d * dv + c];
                for (int i = 0; i < L; ++i)
                    s += exp(GL - G[i]) * K[(long)i * ldk + d] * Vn[i * dv + c];
                Snew[d * dv + c] = s;
            }
        memcpy(S, Snew, sizeof(double) * dk * dv);
    }
    if (J->ht)
        memcpy(J->ht + ((size_t)n * Nv + h) * dk * dv, S, sizeof(double) * dk * dv);

    free(G); free(Tm); free(W); free(U); free(Vn); free(Snew);
}

/* ---------------------------------------------------------------------- */
/* Thread pool over (sequence, v-head) units.                              */
/* ---------------------------------------------------------------------- */
static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * J->dk * J->dv);
    double *delta = (double *)malloc(sizeof(double) * J->dv);
    if (!S || !delta) {
        pthread_mutex_lock(&J->lock);
        J->failed = 1;
        pthread_mutex_unlock(&J->lock);
        free(S); free(delta);
        return NULL;
    }
    const int total = J->units ? J->n_units : J->n_seqs * J->Nv;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int w = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (w >= total) break;
        const int u = J->units ? J->units[w] : w;
        const int n = u / J->Nv, h = u % J->Nv;
        if (J->chunk > 0)
            chunked_unit(J, n, h, S);
        else
            recurrent_unit(J, n, h, S, delta);
    }
    free(S);
    free(delta);
    return NULL;
}

static int run(job_t *J, int n_threads)
{
    if (J->Nk <= 0 || J->Nv <= 0 || J->Nv % J->Nk != 0 || J->dk <= 0 || J->dv <= 0) return 1;
    if (J->cu && J->B != 1) return 1;
    if (!J->cu && J->n_seqs != J->B) return 1;
    if (n_threads <= 0) {
        long nc = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = nc > 0 ? (int)nc : 1;
    }
    const int total = J->units ? J->n_units : J->n_seqs * J->Nv;
    if (n_threads > total) n_threads = total > 0 ? total : 1;
    pthread_mutex_init(&J->lock, NULL);
    J->next = 0;
    J->failed = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&th[i], NULL, worker, J) == 0) ++started;
    if (started == 0) worker(J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->lock);
    return J->failed ? 2 : 0;
}

/* Number of threads run() would use for n_threads <= 0. */
int dn_oracle_default_threads(void)
{
    long nc = sysconf(_SC_NPROCESSORS_ONLN);
    return nc > 0 ? (int)nc : 1;
}

int dn_oracle_recurrent(const double *q, const double *k, const double *v,
                        const double *beta, const double *g, const double *h0,
                        const int64_t *cu_seqlens, int n_seqs, int B, int T,
                        int Nk, int Nv, int dk, int dv, double scale,
                        double *o, double *ht, int read_mode,
                        const int32_t *units, int n_units, int n_threads)
{
    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.cu = cu_seqlens; J.n_seqs = n_seqs; J.B = B; J.T = T;
    J.Nk = Nk; J.Nv = Nv; J.dk = dk; J.dv = dv; J.scale = scale;
    J.o = o; J.ht = ht; J.chunk = 0; J.read_mode = read_mode;
    J.units = units; J.n_units = n_units;
    return run(&J, n_threads);
}

int dn_oracle_chunked(const double *q, const double *k, const double *v,
                      const double *beta, const double *g, const double *h0,
                      const int64_t *cu_seqlens, int n_seqs, int B, int T,
                      int Nk, int Nv, int dk, int dv, double scale, int chunk,
                      double *o, double *ht,
                      const int32_t *units, int n_units, int n_threads)
{
    if (chunk <= 0) return 1;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.cu = cu_seqlens; J.n_seqs = n_seqs; J.B = B; J.T = T;
    J.Nk = Nk; J.Nv = Nv; J.dk = dk; J.dv = dv; J.scale = scale;
    J.o = o; J.ht = ht; J.chunk = chunk; J.read_mode = 0;
    J.units = units; J.n_units = n_units;
    return run(&J, n_threads);
}

/* ---------------------------------------------------------------------- */
/* Gradient of the token recurrence (reverse mode).                        */
/* ---------------------------------------------------------------------- */
/*
 * For the loss l = sum(do . o) + sum(dht . ht) of one forward, given do and
 * dht (dht may be NULL: zero), the gradients of l with respect to q, k, v,
 * beta, g and h0.  Per token of the forward (decayed read, reading 1):
 *     a = e^{g_t};  S' = a S_{t-1};  p = S'^T k_t;  d = beta_t (v_t - p);
 *     S_t = S' + k_t d^T;  o_t = scale S_t^T q_t.
 * Walking the tokens backwards with dS = dl/dS_t (dht after the last one):
 *     dS     += scale q_t do_t^T          dq_t  += scale S_t do_t
 *     dd      = dS^T k_t                  dk_t  += dS d
 *     dbeta_t = dd . (v_t - p)            dv_t   = beta_t dd
 *     dp      = -beta_t dd                dS    += k_t dp^T     dk_t += S' dp
 *     dg_t    = <dS, S'>                  dS     = a dS         (= dl/dS_{t-1})
 * and dh0 = dS after the first token.  The states are recomputed from
 * checkpoints taken every CK tokens of a forward pass.
 *
 * Work is split over (sequence, key head) groups, so that one thread owns
 * every value head that reads a key head and sums their dq and dk.
 */
typedef struct {
    const double *q, *k, *v, *beta, *g, *h0, *dout, *dht;
    const int64_t *cu;
    int n_seqs, B, T, Nk, Nv, dk, dv;
    double scale;
    double *dq, *dk_, *dv_, *dbeta, *dg, *dh0;
    const int32_t *groups; /* group u = n * Nk + hk */
    int n_groups;
    int next, failed;
    pthread_mutex_t lock;
} bjob_t;

enum { CK = 64 };

static void bwd_unit(const bjob_t *J, int n, int h, double *ck, double *St, double *dS,
                     double *Sp, double *tmp)
{
    const int dk = J->dk, dv = J->dv, Nk = J->Nk, Nv = J->Nv;
    const int hk = h / (Nv / Nk);
    const size_t sz = (size_t)dk * dv;
    int64_t bos, eos;
    if (J->cu) {
        bos = J->cu[n];
        eos = J->cu[n + 1];
    } else {
        bos = (int64_t)n * J->T;
        eos = (int64_t)(n + 1) * J->T;
    }
    const int64_t len = eos - bos;
    const int64_t nck = (len + CK - 1) / CK;

    /* forward pass: the state before each block of CK tokens */
    double *S = St;  /* scratch for the running state */
    if (J->h0)
        memcpy(S, J->h0 + ((size_t)n * Nv + h) * sz, sizeof(double) * sz);
    else
        memset(S, 0, sizeof(double) * sz);
    for (int64_t c = 0; c < nck; ++c) {
        memcpy(ck + (size_t)c * sz, S, sizeof(double) * sz);
        const int64_t t1 = bos + (c + 1) * CK < eos ? bos + (c + 1) * CK : eos;
        for (int64_t t = bos + c * CK; t < t1; ++t) {
            const double *kt = J->k + ((size_t)t * Nk + hk) * dk;
            const double *vt = J->v + ((size_t)t * Nv + h) * dv;
            const double bt = J->beta[(size_t)t * Nv + h];
            const double a = J->g ? exp(J->g[(size_t)t * Nv + h]) : 1.0;
            for (size_t i = 0; i < sz; ++i) S[i] *= a;
            for (int c2 = 0; c2 < dv; ++c2) {
                double r = 0.0;
                for (int d = 0; d < dk; ++d) r += kt[d] * S[d * dv + c2];
                tmp[c2] = bt * (vt[c2] - r);
            }
            for (int d = 0; d < dk; ++d)
                for (int c2 = 0; c2 < dv; ++c2) S[d * dv + c2] += kt[d] * tmp[c2];
        }
    }

    /* backward pass */
    if (J->dht)
        memcpy(dS, J->dht + ((size_t)n * Nv + h) * sz, sizeof(double) * sz);
    else
        memset(dS, 0, sizeof(double) * sz);
    double *p = tmp, *dlt = tmp + dv, *ddl = tmp + 2 * dv, *dp = tmp + 3 * dv;
    for (int64_t c = nck - 1; c >= 0; --c) {
        const int64_t t0 = bos + c * CK;
        const int L = (int)((eos - t0) < CK ? (eos - t0) : CK);
        /* states S_{t0-1} .. S_{t0+L-1} of this block: St[j] = state before token t0 + j */
        memcpy(St, ck + (size_t)c * sz, sizeof(double) * sz);
        for (int j = 0; j < L; ++j) {
            const int64_t t = t0 + j;
            const double *kt = J->k + ((size_t)t * Nk + hk) * dk;
            const double *vt = J->v + ((size_t)t * Nv + h) * dv;
            const double bt = J->beta[(size_t)t * Nv + h];
            const double a = J->g ? exp(J->g[(size_t)t * Nv + h]) : 1.0;
            const double *Sa = St + (size_t)j * sz;
            double *Sb = St + (size_t)(j + 1) * sz;
            for (size_t i = 0; i < sz; ++i) Sb[i] = a * Sa[i];
            for (int c2 = 0; c2 < dv; ++c2) {
                double r = 0.0;
                for (int d = 0; d < dk; ++d) r += kt[d] * Sb[d * dv + c2];
                dlt[c2] = bt * (vt[c2] - r);
            }
            for (int d = 0; d < dk; ++d)
                for (int c2 = 0; c2 < dv; ++c2) Sb[d * dv + c2] += kt[d] * dlt[c2];
        }
        for (int j = L - 1; j >= 0; --j) {
            const int64_t t = t0 + j;
            const double *qt = J->q + ((size_t)t * Nk + hk) * dk;
            const double *kt = J->k + ((size_t)t * Nk + hk) * dk;
            const double *vt = J->v + ((size_t)t * Nv + h) * dv;
            const double *dot = J->dout + ((size_t)t * Nv + h) * dv;
            const double bt = J->beta[(size_t)t * Nv + h];
            const double a = J->g ? exp(J->g[(size_t)t * Nv + h]) : 1.0;
            const double *Sprev = St + (size_t)j * sz, *Snow = St + (size_t)(j + 1) * sz;
            double *dqt = J->dq + ((size_t)t * Nk + hk) * dk;
            double *dkt = J->dk_ + ((size_t)t * Nk + hk) * dk;
            double *dvt = J->dv_ + ((size_t)t * Nv + h) * dv;
            /* recompute S', p and d of this token */
            for (size_t i = 0; i < sz; ++i) Sp[i] = a * Sprev[i];
            for (int c2 = 0; c2 < dv; ++c2) {
                double r = 0.0;
                for (int d = 0; d < dk; ++d) r += kt[d] * Sp[d * dv + c2];
                p[c2] = r;
                dlt[c2] = bt * (vt[c2] - r);
            }
            /* o_t = scale S_t^T q_t */
            for (int d = 0; d < dk; ++d) {
                double r = 0.0;
                for (int c2 = 0; c2 < dv; ++c2) {
                    dS[d * dv + c2] += J->scale * qt[d] * dot[c2];
                    r += Snow[d * dv + c2] * dot[c2];
                }
                dqt[d] += J->scale * r;
            }
            /* S_t = S' + k d^T */
            for (int c2 = 0; c2 < dv; ++c2) {
                double r = 0.0;
                for (int d = 0; d < dk; ++d) r += dS[d * dv + c2] * kt[d];
                ddl[c2] = r;
            }
            for (int d = 0; d < dk; ++d) {
                double r = 0.0;
                for (int c2 = 0; c2 < dv; ++c2) r += dS[d * dv + c2] * dlt[c2];
                dkt[d] += r;
            }
            /* d = beta (v - p) */
            double db = 0.0;
            for (int c2 = 0; c2 < dv; ++c2) {
                db += ddl[c2] * (vt[c2] - p[c2]);
                dvt[c2] = bt * ddl[c2];
                dp[c2] = -bt * ddl[c2];
            }
            J->dbeta[(size_t)t * Nv + h] = db;
            /* p = S'^T k */
            for (int d = 0; d < dk; ++d) {
                double r = 0.0;
                for (int c2 = 0; c2 < dv; ++c2) {
                    dS[d * dv + c2] += kt[d] * dp[c2];
                    r += Sp[d * dv + c2] * dp[c2];
                }
                dkt[d] += r;
            }
            /* S' = a S_{t-1} */
            double dgt = 0.0;
            for (size_t i = 0; i < sz; ++i) dgt += dS[i] * Sp[i];
            if (J->dg) J->dg[(size_t)t * Nv + h] = dgt;
            for (size_t i = 0; i < sz; ++i) dS[i] *= a;
        }
    }
    if (J->dh0) memcpy(J->dh0 + ((size_t)n * Nv + h) * sz, dS, sizeof(double) * sz);
}

static void *bwd_worker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    const size_t sz = (size_t)J->dk * J->dv;
    int64_t maxlen = J->T;
    if (J->cu)
        for (int n = 0; n < J->n_seqs; ++n)
            if (J->cu[n + 1] - J->cu[n] > maxlen) maxlen = J->cu[n + 1] - J->cu[n];
    const int64_t nck = (maxlen + CK - 1) / CK + 1;
    double *ck = (double *)malloc(sizeof(double) * sz * nck);
    double *St = (double *)malloc(sizeof(double) * sz * (CK + 1));
    double *dS = (double *)malloc(sizeof(double) * sz);
    double *Sp = (double *)malloc(sizeof(double) * sz);
    double *tmp = (double *)malloc(sizeof(double) * 4 * J->dv);
    if (!ck || !St || !dS || !Sp || !tmp) {
        pthread_mutex_lock(&J->lock);
        J->failed = 1;
        pthread_mutex_unlock(&J->lock);
    } else {
        const int total = J->groups ? J->n_groups : J->n_seqs * J->Nk;
        const int r = J->Nv / J->Nk;
        for (;;) {
            pthread_mutex_lock(&J->lock);
            const int w = J->next++;
            pthread_mutex_unlock(&J->lock);
            if (w >= total) break;
            const int u = J->groups ? J->groups[w] : w;
            const int n = u / J->Nk, hk = u % J->Nk;
            /* zero this group's dq and dk rows, then add every value head's share */
            int64_t bos, eos;
            if (J->cu) {
                bos = J->cu[n];
                eos = J->cu[n + 1];
            } else {
                bos = (int64_t)n * J->T;
                eos = (int64_t)(n + 1) * J->T;
            }
            for (int64_t t = bos; t < eos; ++t) {
                memset(J->dq + ((size_t)t * J->Nk + hk) * J->dk, 0, sizeof(double) * J->dk);
                memset(J->dk_ + ((size_t)t * J->Nk + hk) * J->dk, 0, sizeof(double) * J->dk);
            }
            for (int h = hk * r; h < (hk + 1) * r; ++h) bwd_unit(J, n, h, ck, St, dS, Sp, tmp);
        }
    }
    free(ck); free(St); free(dS); free(Sp); free(tmp);
    return NULL;
}

int dn_oracle_recurrent_bwd(const double *q, const double *k, const double *v,
                            const double *beta, const double *g, const double *h0,
                            const int64_t *cu_seqlens, int n_seqs, int B, int T,
                            int Nk, int Nv, int dk, int dv, double scale,
                            const double *dout, const double *dht,
                            double *dq, double *dk_out, double *dv_out, double *dbeta,
                            double *dg, double *dh0,
                            const int32_t *groups, int n_groups, int n_threads)
{
    if (Nk <= 0 || Nv <= 0 || Nv % Nk != 0 || dk <= 0 || dv <= 0) return 1;
    if (cu_seqlens && B != 1) return 1;
    if (!cu_seqlens && n_seqs != B) return 1;
    bjob_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0; J.dout = dout; J.dht = dht;
    J.cu = cu_seqlens; J.n_seqs = n_seqs; J.B = B; J.T = T;
    J.Nk = Nk; J.Nv = Nv; J.dk = dk; J.dv = dv; J.scale = scale;
    J.dq = dq; J.dk_ = dk_out; J.dv_ = dv_out; J.dbeta = dbeta; J.dg = dg; J.dh0 = dh0;
    J.groups = groups; J.n_groups = n_groups;
    if (n_threads <= 0) n_threads = dn_oracle_default_threads();
    const int total = groups ? n_groups : n_seqs * Nk;
    if (n_threads > total) n_threads = total > 0 ? total : 1;
    pthread_mutex_init(&J.lock, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&th[i], NULL, bwd_worker, &J) == 0) ++started;
    if (started == 0) bwd_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? 2 : 0;
}
