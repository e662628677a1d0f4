/*
 * KDA oracle: the plain FP64 token-by-token recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. The CUDA path
 * shares no code, header or constant with it.
 *
 * What it computes (Kimi Delta Attention, the gated delta rule with a
 * per-channel decay; "FlashInfer PR #4262: CAKE KDA Prefill Highlights",
 * section 2, gives only its chunked kernel form, so the recurrence below is
 * the token-level definition that chunked form reduces to):
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t = scale * S_t^T q_t
 *
 * with S in R^{dk x dv}.  It is evaluated in the equivalent rank-one order
 *
 *   S <- Diag(exp g) S ;  w = S^T k ;  S <- S + beta k (v - w)^T ;  o = scale S^T q
 *
 * since (I - b k k^T) D S + b k v^T = D S + k (b (v - (D S)^T k))^T.
 *
 * The gate g is a per-channel natural-log decay computed from the raw gate a:
 *   mode 0 (lower bound):  g = lower_bound * sigmoid(a)   (the "bounded lb" gate,
 *                          FlashInfer PR #5551, decode ABI "use_lower_bound")
 *   mode 1 (softplus):     g = -softplus(a) = -(max(a,0) + log1p(exp(-|a|)))
 *                          (the unbounded "Kimi-Linear softplus" gate, PR #5565)
 *   mode 2 (log decay):    g = a  (a <= 0 given directly; a test affordance)
 *
 * Every input is taken as an FP64 value (the Python wrapper widens the stored
 * BF16/FP32 inputs exactly), so input quantisation is not counted as error.
 * Dimensions dk, dv are run-time values so hand-checkable cases with d = 1, 2
 * use the same code as d = 128.
 *
 * Work is split over chains (sequence, head) with one POSIX thread per
 * core; chains are independent, so the split does not change any result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_NOMEM -2

static double oracle_gate(double a, int mode, double lower_bound)
{
    if (mode == 0)
        return lower_bound / (1.0 + exp(-a));
    if (mode == 1)
        return -(fmax(a, 0.0) + log1p(exp(-fabs(a))));
    return a;
}

/*
 * One token step on one chain.  S is dk x dv row-major (S[i*dv + j]).
 * q, k, a have dk entries, v has dv entries; o receives dv entries.
 * w is dv entries of scratch.
 */
static void oracle_token_step(double *S, const double *q, const double *k, const double *v,
                              const double *a, double beta, int dk, int dv, double scale,
                              double lower_bound, int gate_mode, double *o, double *w)
{
    int i, j;
    /* decay: S <- Diag(exp g) S */
    for (i = 0; i < dk; ++i) {
        double d = exp(oracle_gate(a[i], gate_mode, lower_bound));
        double *row = S + (size_t)i * dv;
        for (j = 0; j < dv; ++j)
            row[j] *= d;
    }
    /* w = S^T k */
    for (j = 0; j < dv; ++j)
        w[j] = 0.0;
    for (i = 0; i < dk; ++i) {
        const double *row = S + (size_t)i * dv;
        double ki = k[i];
        for (j = 0; j < dv; ++j)
            w[j] += row[j] * ki;
    }
    /* S <- S + beta k (v - w)^T */
    for (j = 0; j < dv; ++j)
        w[j] = beta * (v[j] - w[j]);
    for (i = 0; i < dk; ++i) {
        double *row = S + (size_t)i * dv;
        double ki = k[i];
        for (j = 0; j < dv; ++j)
            row[j] += ki * w[j];
    }
    /* o = scale S^T q */
    for (j = 0; j < dv; ++j)
        o[j] = 0.0;
    for (i = 0; i < dk; ++i) {
        const double *row = S + (size_t)i * dv;
        double qi = q[i];
        for (j = 0; j < dv; ++j)
            o[j] += row[j] * qi;
    }
    for (j = 0; j < dv; ++j)
        o[j] *= scale;
}

typedef struct {
    const double *q, *k, *v, *a, *beta;
    const int32_t *cu_seqlens;
    const double *init_state;
    double *out, *final_state;
    const int32_t *chains;
    int32_t num_chains, num_heads, dk, dv, gate_mode;
    double scale, lower_bound;
    int32_t next; /* next chain index to take */
    pthread_mutex_t lock;
    int failed;
} prefill_job;

static void *prefill_worker(void *arg)
{
    prefill_job *job = (prefill_job *)arg;
    const int H = job->num_heads, dk = job->dk, dv = job->dv;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *w = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !w) {
        pthread_mutex_lock(&job->lock);
        job->failed = 1;
        pthread_mutex_unlock(&job->lock);
        free(S);
        free(w);
        return NULL;
    }
    for (;;) {
        int32_t idx, chain, n, h, t;
        pthread_mutex_lock(&job->lock);
        idx = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (idx >= job->num_chains)
            break;
        chain = job->chains ? job->chains[idx] : idx;
        n = chain / H;
        h = chain % H;
        if (job->init_state)
            memcpy(S, job->init_state + (size_t)chain * dk * dv, sizeof(double) * (size_t)dk * dv);
        else
            memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (t = job->cu_seqlens[n]; t < job->cu_seqlens[n + 1]; ++t) {
            size_t th = (size_t)t * H + h;
            oracle_token_step(S, job->q + th * dk, job->k + th * dk, job->v + th * dv,
                              job->a + th * dk, job->beta[th], dk, dv, job->scale,
                              job->lower_bound, job->gate_mode, job->out + th * dv, w);
        }
        if (job->final_state)
            memcpy(job->final_state + (size_t)chain * dk * dv, S, sizeof(double) * (size_t)dk * dv);
    }
    free(S);
    free(w);
    return NULL;
}

static int resolve_threads(int threads, int work)
{
    if (threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        threads = n > 0 ? (int)n : 1;
    }
    if (threads > work)
        threads = work;
    return threads < 1 ? 1 : threads;
}

static int run_pool(void *(*fn)(void *), void *job, int threads)
{
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    int i, started = 0;
    if (!tid)
        return ORACLE_ERR_NOMEM;
    for (i = 0; i < threads; ++i) {
        if (pthread_create(&tid[i], NULL, fn, job) != 0)
            break;
        ++started;
    }
    if (started == 0)
        fn(job); /* no thread could start: run on the caller's thread */
    for (i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    return ORACLE_OK;
}

/*
 * Varlen prefill.  Layouts (row-major): q, k, a: [T_total, H, dk]; v: [T_total, H, dv];
 * beta: [T_total, H]; cu_seqlens: [num_seqs + 1]; init_state, final_state:
 * [num_seqs, H, dk, dv] (init NULL = zeros, final NULL = not written);
 * out: [T_total, H, dv].  chains (NULL = all num_seqs*H chains) lists chain ids
 * n*H + h to evaluate; out rows of other chains are left untouched.
 * Returns the number of threads used, or a negative error.
 */
int oracle_kda_prefill(const double *q, const double *k, const double *v, const double *a,
                       const double *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                       int32_t num_heads, int32_t dk, int32_t dv, const double *init_state,
                       double scale, double lower_bound, int32_t gate_mode,
                       const int32_t *chains, int32_t num_chains, double *out,
                       double *final_state, int32_t threads)
{
    prefill_job job;
    int32_t n, rc;
    if (num_seqs < 0 || num_heads < 1 || dk < 1 || dv < 1 || !cu_seqlens || gate_mode < 0 ||
        gate_mode > 2)
        return ORACLE_ERR_ARG;
    for (n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return ORACLE_ERR_ARG;
    if (cu_seqlens[num_seqs] > 0 && (!q || !k || !v || !a || !beta || !out))
        return ORACLE_ERR_ARG;
    if (!chains)
        num_chains = num_seqs * num_heads;
    if (num_chains <= 0)
        return 1;
    memset(&job, 0, sizeof(job));
    job.q = q;
    job.k = k;
    job.v = v;
    job.a = a;
    job.beta = beta;
    job.cu_seqlens = cu_seqlens;
    job.init_state = init_state;
    job.out = out;
    job.final_state = final_state;
    job.chains = chains;
    job.num_chains = num_chains;
    job.num_heads = num_heads;
    job.dk = dk;
    job.dv = dv;
    job.gate_mode = gate_mode;
    job.scale = scale;
    job.lower_bound = lower_bound;
    pthread_mutex_init(&job.lock, NULL);
    threads = resolve_threads(threads, num_chains);
    rc = run_pool(prefill_worker, &job, threads);
    pthread_mutex_destroy(&job.lock);
    if (rc != ORACLE_OK)
        return rc;
    return job.failed ? ORACLE_ERR_NOMEM : threads;
}

typedef struct {
    const double *q, *k, *v, *a, *beta;
    double *state, *out;
    int32_t items, dk, dv, gate_mode, beta_logits;
    double scale, lower_bound, norm_eps;
    int32_t next;
    pthread_mutex_t lock;
    int failed;
} decode_job;

/* x <- x / sqrt(sum x^2 + eps): the L2 normalisation a decode call may apply to q and k. */
static void oracle_l2norm(double *x, const double *src, int n, double eps)
{
    double ss = 0.0;
    int i;
    for (i = 0; i < n; ++i)
        ss += src[i] * src[i];
    ss = 1.0 / sqrt(ss + eps);
    for (i = 0; i < n; ++i)
        x[i] = src[i] * ss;
}

static void *decode_worker(void *arg)
{
    decode_job *job = (decode_job *)arg;
    const int dk = job->dk, dv = job->dv;
    double *w = (double *)malloc(sizeof(double) * (size_t)(dv + 2 * dk));
    if (!w) {
        pthread_mutex_lock(&job->lock);
        job->failed = 1;
        pthread_mutex_unlock(&job->lock);
        return NULL;
    }
    for (;;) {
        int32_t it;
        pthread_mutex_lock(&job->lock);
        it = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (it >= job->items)
            break;
        {
            const double *qi = job->q + (size_t)it * dk, *ki = job->k + (size_t)it * dk;
            double beta = job->beta[it];
            double *qn = w + dv, *kn = w + dv + dk;
            if (job->norm_eps >= 0.0) {
                oracle_l2norm(qn, qi, dk, job->norm_eps);
                oracle_l2norm(kn, ki, dk, job->norm_eps);
                qi = qn;
                ki = kn;
            }
            if (job->beta_logits)
                beta = 1.0 / (1.0 + exp(-beta));
            oracle_token_step(job->state + (size_t)it * dk * dv, qi, ki, job->v + (size_t)it * dv,
                              job->a + (size_t)it * dk, beta, dk, dv, job->scale, job->lower_bound,
                              job->gate_mode, job->out + (size_t)it * dv, w);
        }
    }
    free(w);
    return NULL;
}

/*
 * T = 1 decode on already-gathered states.  Items are (row, head) pairs in
 * row-major order: q, k, a: [items, dk]; v, out: [items, dv]; beta: [items];
 * state: [items, dk, dv], updated in place.  The slot indirection of a state
 * pool is the caller's gather/scatter.
 */
int oracle_kda_decode_ex(const double *q, const double *k, const double *v, const double *a,
                         const double *beta, int32_t items, int32_t dk, int32_t dv, double *state,
                         double scale, double lower_bound, int32_t gate_mode, double norm_eps,
                         int32_t beta_logits, double *out, int32_t threads);

int oracle_kda_decode(const double *q, const double *k, const double *v, const double *a,
                      const double *beta, int32_t items, int32_t dk, int32_t dv, double *state,
                      double scale, double lower_bound, int32_t gate_mode, double *out,
                      int32_t threads)
{
    return oracle_kda_decode_ex(q, k, v, a, beta, items, dk, dv, state, scale, lower_bound, gate_mode,
                                -1.0, 0, out, threads);
}

/*
 * The same step with the two input options of a decode call (FlashInfer PR #5551, decode ABI:
 * "norm_eps"; PR #5573 section 3: the kernel stages sigmoid(beta) itself):
 *   norm_eps >= 0  q and k are first replaced by x / sqrt(sum x^2 + norm_eps)
 *   beta_logits    beta holds logits b and the step uses sigmoid(b) = 1 / (1 + exp(-b))
 */
int oracle_kda_decode_ex(const double *q, const double *k, const double *v, const double *a,
                         const double *beta, int32_t items, int32_t dk, int32_t dv, double *state,
                         double scale, double lower_bound, int32_t gate_mode, double norm_eps,
                         int32_t beta_logits, double *out, int32_t threads)
{
    decode_job job;
    int rc;
    if (items < 0 || dk < 1 || dv < 1 || gate_mode < 0 || gate_mode > 2)
        return ORACLE_ERR_ARG;
    if (items == 0)
        return 1;
    if (!q || !k || !v || !a || !beta || !state || !out)
        return ORACLE_ERR_ARG;
    memset(&job, 0, sizeof(job));
    job.q = q;
    job.k = k;
    job.v = v;
    job.a = a;
    job.beta = beta;
    job.state = state;
    job.out = out;
    job.items = items;
    job.dk = dk;
    job.dv = dv;
    job.gate_mode = gate_mode;
    job.scale = scale;
    job.lower_bound = lower_bound;
    job.norm_eps = norm_eps;
    job.beta_logits = beta_logits;
    pthread_mutex_init(&job.lock, NULL);
    threads = resolve_threads(threads, items);
    rc = run_pool(decode_worker, &job, threads);
    pthread_mutex_destroy(&job.lock);
    if (rc != ORACLE_OK)
        return rc;
    return job.failed ? ORACLE_ERR_NOMEM : threads;
}

/* The gate as the oracle evaluates it, exposed so its special values can be pinned. */
double oracle_kda_gate(double a, int32_t gate_mode, double lower_bound)
{
    return oracle_gate(a, gate_mode, lower_bound);
}
