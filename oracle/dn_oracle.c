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
 * Two independent forms are implemented:
 *
 *   dn_oracle_recurrent  -- the definition: a token-by-token recurrence
 *                           ([WY] §1, [CGDR] §1), written out plainly.
 *   dn_oracle_chunked    -- the chunk algorithm in the pages' order: gate
 *                           prefix sum, WY matrix A, T = (I-A)^-1, W and U,
 *                           v_new, output, state ([CGDR] §3.1-§3.3,
 *                           [WY] §2.3-§2.4).  Used to pin the chunk algebra.
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
