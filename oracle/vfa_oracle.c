/*
 * vfa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the variable-length attention
 * path computes.  Only the test-suite, the package's smoke check and the
 * bench's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (the pages this follows):
 *   - "Varlen Flash Attention Implementation Plan" (rustytorch), Task 1
 *     Step 1 (the CUDA kernel: packed [total, heads, head_dim] layout,
 *     cu_seqlens prefix sums, scaled scores, causal and boundary masks,
 *     epilogue out = acc / l and lse = log(l) + m) and Task 2 Step 1
 *     (varlen_attention_cpu: per-sequence masked softmax times V).
 *   - an FP8 variant of the forward (the plan names FP8 kernel configuration
 *     types without content): q and k given as FP8 E4M3 codes with one
 *     descale factor per tensor, read as descale * code exactly;
 *   - the backward is the derivative of that forward (the plan names a
 *     backward without giving one), written out per query row;
 *   - "attention_ref.rs" (spark_storage): AttnState::new, step_tile_ref,
 *     finalize_ref -- the paged GQA decode state (m, l, o), its update over
 *     the tokens of the blocks listed for one tile, and the final o / l.
 *
 * All arithmetic is in double.  bf16 inputs are widened exactly.  Nothing is
 * blocked, fused or reordered beyond the definition: each (sequence, head,
 * query row) is computed on its own from the full set of keys it may see.
 *
 * Readings taken where the pages are silent or disagree (each is also listed
 * in the design notes):
 *   - causal alignment is top-left: local key j is visible to local query i
 *     iff j <= i (the kernel compares local positions k_pos > q_pos); the
 *     bottom-right alignment (the last query sees every key: j <= i + Lk - Lq)
 *     is offered as a second causal mode, and either mode may be narrowed to
 *     a sliding window of the window_left keys before the diagonal;
 *   - masked keys carry weight exactly zero (the kernel's -FLT_MAX sentinel
 *     and the CPU reference's -inf sentinel both give that);
 *   - an empty key set gives out = 0 and lse = -FLT_MAX (the kernel's
 *     inv_l = 0 and lse epilogue);
 *   - lse is the natural log of sum_j exp(scale * q.k_j);
 *   - decode: every listed block contributes all block_size tokens and the
 *     decode scale is 1/sqrt(head_dim), as in step_tile_ref; two optional
 *     arguments extend it for callers whose contexts end inside a block or
 *     who use another scale: a per-sequence count of the tile's tokens to
 *     absorb (the first n of the listed blocks' tokens, in list order) and an
 *     explicit scale.
 *
 * Parity pins (independent checks of this file) live in tests/: a numpy
 * brute-force formulation, torch float64 scaled_dot_product_attention, the
 * worked examples the plan's tests print, closed-form invariants, and the
 * tile-fragmentation invariance that attention_ref.rs states as its purpose.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Exact widening of a bfloat16 bit pattern to double. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Exact value of an FP8 E4M3 code (the OCP 8-bit floating-point format's
 * E4M3 encoding: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 is subnormal, 2^-6 * m / 8; no infinities; S.1111.111 is NaN).
 */
static double fp8_e4m3_to_double(uint8_t b)
{
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Packed layout [tokens, heads, head_dim]: element (t, h, d). */
static size_t packed_index(int64_t t, int h, int d, int num_heads, int head_dim)
{
    return ((size_t)t * (size_t)num_heads + (size_t)h) * (size_t)head_dim + (size_t)d;
}

int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ------------------------------------------------------------------------ */
/* Varlen attention forward                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *cu_q, *cu_k;
    int batch, num_heads, num_kv_heads, head_dim;
    double scale;
    int causal;
    int window_left;                        /* < 0: none; else keys j >= i + off - window_left */
    const uint8_t *q8, *k8;                 /* FP8 E4M3 q and k (then q, k unused), or NULL */
    double descale_q, descale_k;            /* q = descale_q * code, k = descale_k * code */
} varlen_problem;

/* q and k elements as real numbers: bf16 widened, or FP8 code times its descale. */
static double q_elem(const varlen_problem *p, size_t i)
{
    return p->q8 ? p->descale_q * fp8_e4m3_to_double(p->q8[i]) : bf16_to_double(p->q[i]);
}

static double k_elem(const varlen_problem *p, size_t i)
{
    return p->k8 ? p->descale_k * fp8_e4m3_to_double(p->k8[i]) : bf16_to_double(p->k[i]);
}

/*
 * One query row: local row i of sequence b, head h; its keys and values are
 * those of kv head kh = h / (H / Hkv) (kh = h when Hkv = H).
 *
 *   K_set = { j : 0 <= j < Lk_b  and  (causal == 0 or j <= i + off)
 *               and  (window_left < 0 or j >= i + off - window_left) }
 *   off   = 0 for causal == 1 (top-left), Lk_b - Lq_b for causal == 2
 *           (bottom-right); a window needs a causal mode
 *   s_j   = scale * sum_d q[tq, h, d] * k[cu_k[b] + j, kh, d]
 *   empty K_set: out = 0, lse = -FLT_MAX
 *   else: M = max_j s_j, Z = sum_j exp(s_j - M),
 *         out[d] = sum_j exp(s_j - M) * v[cu_k[b] + j, h, d] / Z,
 *         lse = M + ln Z
 *
 * `s` and `w` are caller scratch of at least Lk_b doubles; `kidx` of Lk_b ints.
 */
static void varlen_row(const varlen_problem *p, int b, int i, int h,
                       double *out_row, double *lse_out,
                       double *s, double *w, int *kidx)
{
    const int D = p->head_dim, H = p->num_heads, Hkv = p->num_kv_heads;
    const int kh = h / (H / Hkv);
    const int64_t tq = (int64_t)p->cu_q[b] + i;
    const int64_t k0 = p->cu_k[b];
    const int Lk = p->cu_k[b + 1] - p->cu_k[b];
    const int Lq = p->cu_q[b + 1] - p->cu_q[b];
    const int off = p->causal == 2 ? Lk - Lq : 0;

    int n = 0;
    for (int j = 0; j < Lk; ++j) {
        if (p->causal && j > i + off)
            continue;                       /* masked: weight exactly zero */
        if (p->window_left >= 0 && j < i + off - p->window_left)
            continue;                       /* left of the sliding window */
        kidx[n++] = j;
    }
    if (n == 0) {
        for (int d = 0; d < D; ++d)
            out_row[d] = 0.0;
        *lse_out = -(double)FLT_MAX;
        return;
    }
    for (int a = 0; a < n; ++a) {
        const int64_t tk = k0 + kidx[a];
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q_elem(p, packed_index(tq, h, d, H, D)) *
                   k_elem(p, packed_index(tk, kh, d, Hkv, D));
        s[a] = p->scale * dot;
    }
    double M = s[0];
    for (int a = 1; a < n; ++a)
        if (s[a] > M)
            M = s[a];
    double Z = 0.0;
    for (int a = 0; a < n; ++a) {
        w[a] = exp(s[a] - M);
        Z += w[a];
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int a = 0; a < n; ++a)
            acc += w[a] * bf16_to_double(p->v[packed_index(k0 + kidx[a], kh, d, Hkv, D)]);
        out_row[d] = acc / Z;
    }
    *lse_out = M + log(Z);
}

/* Work distribution: independent units handed out by an atomic counter. */
typedef struct {
    const varlen_problem *p;
    /* full mode: unit = (b, h); rows mode: unit = one (token, head) row */
    const int64_t *rows;   /* NULL in full mode; else pairs (token, head) */
    int64_t n_units;
    int64_t next;          /* shared counter */
    int max_lk;
    double *out, *lse;     /* full mode: packed [Tq,H,D] and [Tq,H]; rows mode: [n,D], [n] */
    int status;
} varlen_job;

/* Sequence that owns packed query token t: cu_q[b] <= t < cu_q[b+1]. */
static int owner_sequence(const int32_t *cu, int batch, int64_t t)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {              /* first b with cu[b+1] > t */
        int mid = (lo + hi) / 2;
        if (cu[mid + 1] > t)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

static void *varlen_worker(void *arg)
{
    varlen_job *job = (varlen_job *)arg;
    const varlen_problem *p = job->p;
    const int D = p->head_dim, H = p->num_heads;
    size_t nscratch = (size_t)(job->max_lk > 0 ? job->max_lk : 1);
    double *s = (double *)malloc(nscratch * sizeof(double));
    double *w = (double *)malloc(nscratch * sizeof(double));
    int *kidx = (int *)malloc(nscratch * sizeof(int));
    if (!s || !w || !kidx) {
        __atomic_store_n(&job->status, -1, __ATOMIC_SEQ_CST);
        free(s); free(w); free(kidx);
        return NULL;
    }
    for (;;) {
        int64_t u = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (u >= job->n_units)
            break;
        if (job->rows == NULL) {
            const int b = (int)(u / H), h = (int)(u % H);
            const int Lq = p->cu_q[b + 1] - p->cu_q[b];
            for (int i = 0; i < Lq; ++i) {
                const int64_t tq = (int64_t)p->cu_q[b] + i;
                varlen_row(p, b, i, h, job->out + packed_index(tq, h, 0, H, D),
                           job->lse + (size_t)tq * H + h, s, w, kidx);
            }
        } else {
            const int64_t tq = job->rows[2 * u];
            const int h = (int)job->rows[2 * u + 1];
            const int b = owner_sequence(p->cu_q, p->batch, tq);
            varlen_row(p, b, (int)(tq - p->cu_q[b]), h, job->out + (size_t)u * D,
                       job->lse + u, s, w, kidx);
        }
    }
    free(s); free(w); free(kidx);
    return NULL;
}

static int run_varlen_job(varlen_job *job, int nthreads)
{
    if (nthreads <= 0)
        nthreads = oracle_default_threads();
    if ((int64_t)nthreads > job->n_units)
        nthreads = job->n_units > 0 ? (int)job->n_units : 1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid)
        return -1;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, varlen_worker, job) != 0)
            break;
        ++started;
    }
    if (started == 0)
        varlen_worker(job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    if (job->status != 0)
        return -1;
    return started > 0 ? started : 1;
}

static int check_cu(const int32_t *cu, int batch)
{
    if (cu[0] != 0)
        return -2;
    for (int b = 0; b < batch; ++b)
        if (cu[b + 1] < cu[b])
            return -2;
    return 0;
}

static int max_len(const int32_t *cu, int batch)
{
    int m = 0;
    for (int b = 0; b < batch; ++b)
        if (cu[b + 1] - cu[b] > m)
            m = cu[b + 1] - cu[b];
    return m;
}

/*
 * Full varlen forward.  q: [cu_q[B], H, D], k/v: [cu_k[B], Hkv, D] (bf16 bits),
 * H a multiple of Hkv (query head h reads kv head h / (H / Hkv)).
 * out: double [cu_q[B], H, D]; lse: double [cu_q[B], H].
 * Returns the number of threads used (> 0), or < 0 on bad arguments.
 */
int oracle_varlen_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const int32_t *cu_q, const int32_t *cu_k, int batch,
                      int num_heads, int num_kv_heads, int head_dim, double scale, int causal,
                      int window_left, double *out, double *lse, int nthreads)
{
    if (batch < 1 || num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads != 0 ||
        head_dim < 1 || causal < 0 || causal > 2 || (window_left >= 0 && causal == 0))
        return -1;
    if (check_cu(cu_q, batch) || check_cu(cu_k, batch))
        return -2;
    varlen_problem p = {q, k, v, cu_q, cu_k, batch, num_heads, num_kv_heads, head_dim, scale,
                        causal, window_left};
    varlen_job job;
    memset(&job, 0, sizeof job);
    job.p = &p;
    job.rows = NULL;
    job.n_units = (int64_t)batch * num_heads;
    job.max_lk = max_len(cu_k, batch);
    job.out = out;
    job.lse = lse;
    return run_varlen_job(&job, nthreads);
}

/*
 * The forward with FP8 E4M3 q and k: q8 [cu_q[B], H, D] and k8 [cu_k[B], Hkv, D]
 * codes standing for descale_q * code and descale_k * code; v bf16.  Same
 * definition, outputs and return value as oracle_varlen_fwd.
 */
int oracle_varlen_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint16_t *v,
                          const int32_t *cu_q, const int32_t *cu_k, int batch, int num_heads,
                          int num_kv_heads, int head_dim, double scale, double descale_q,
                          double descale_k, int causal, int window_left, double *out,
                          double *lse, int nthreads)
{
    if (batch < 1 || num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads != 0 ||
        head_dim < 1 || causal < 0 || causal > 2 || (window_left >= 0 && causal == 0) ||
        !q8 || !k8)
        return -1;
    if (check_cu(cu_q, batch) || check_cu(cu_k, batch))
        return -2;
    varlen_problem p = {NULL, NULL, v, cu_q, cu_k, batch, num_heads, num_kv_heads, head_dim,
                        scale, causal, window_left, q8, k8, descale_q, descale_k};
    varlen_job job;
    memset(&job, 0, sizeof job);
    job.p = &p;
    job.rows = NULL;
    job.n_units = (int64_t)batch * num_heads;
    job.max_lk = max_len(cu_k, batch);
    job.out = out;
    job.lse = lse;
    return run_varlen_job(&job, nthreads);
}

/* Exact values of n FP8 E4M3 codes (for the decoder's own pins). */
void oracle_fp8_e4m3_decode(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fp8_e4m3_to_double(codes[i]);
}

/*
 * Sampled rows of the same forward.  rows: int64 pairs (packed token, head),
 * n_rows of them.  out_rows: double [n_rows, D]; lse_rows: double [n_rows].
 */
int oracle_varlen_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const int32_t *cu_q, const int32_t *cu_k, int batch,
                           int num_heads, int num_kv_heads, int head_dim, double scale,
                           int causal, int window_left, const int64_t *rows, int64_t n_rows,
                           double *out_rows, double *lse_rows, int nthreads)
{
    if (batch < 1 || num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads != 0 ||
        head_dim < 1 || n_rows < 0 || causal < 0 || causal > 2 ||
        (window_left >= 0 && causal == 0))
        return -1;
    if (check_cu(cu_q, batch) || check_cu(cu_k, batch))
        return -2;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= cu_q[batch] ||
            rows[2 * r + 1] < 0 || rows[2 * r + 1] >= num_heads)
            return -3;
    varlen_problem p = {q, k, v, cu_q, cu_k, batch, num_heads, num_kv_heads, head_dim, scale,
                        causal, window_left};
    varlen_job job;
    memset(&job, 0, sizeof job);
    job.p = &p;
    job.rows = rows;
    job.n_units = n_rows;
    job.max_lk = max_len(cu_k, batch);
    job.out = out_rows;
    job.lse = lse_rows;
    return run_varlen_job(&job, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Varlen attention backward                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Gradients of the forward above for an upstream gradient dout = dL/dout
 * (the pages only name a backward; this is the derivative of the forward's
 * definition, written out).  For one query row (b, i, h) with visible key
 * set K_set, weights P_j = exp(s_j - M) / Z (j in K_set) and
 *
 *   dP_j    = sum_d dout[tq, h, d] * v[k0 + j, kh, d]
 *   Delta   = sum_{j in K_set} P_j * dP_j
 *   dS_j    = P_j * (dP_j - Delta)                 (softmax Jacobian)
 *   dq[tq, h, :]     = scale * sum_j dS_j * k[k0 + j, kh, :]
 *   dk[k0 + j, kh, :] += scale * dS_j * q[tq, h, :]
 *   dv[k0 + j, kh, :] += P_j * dout[tq, h, :]
 *
 * dk and dv of kv head kh sum over the query heads h with h / (H / Hkv) = kh
 * and over every row that sees the key.  A row with an empty K_set adds
 * nothing and gets dq = 0.
 */
typedef struct {
    const varlen_problem *p;
    const uint16_t *dout;
    double *dq, *dk, *dv;
    int64_t n_units;       /* (b, kh) pairs */
    int64_t next;
    int max_lk;
    int status;
} bwd_job;

static void bwd_unit(bwd_job *job, int b, int kh, double *s, double *w, int *kidx)
{
    const varlen_problem *p = job->p;
    const int D = p->head_dim, H = p->num_heads, Hkv = p->num_kv_heads;
    const int group = H / Hkv;
    const int64_t q0 = p->cu_q[b], k0 = p->cu_k[b];
    const int Lq = p->cu_q[b + 1] - p->cu_q[b];
    const int Lk = p->cu_k[b + 1] - p->cu_k[b];
    const int off = p->causal == 2 ? Lk - Lq : 0;
    double *dp = (double *)malloc((size_t)(Lk > 0 ? Lk : 1) * sizeof(double));
    if (!dp) {
        __atomic_store_n(&job->status, -1, __ATOMIC_SEQ_CST);
        return;
    }
    for (int h = kh * group; h < (kh + 1) * group; ++h) {
        for (int i = 0; i < Lq; ++i) {
            const int64_t tq = q0 + i;
            int n = 0;
            for (int j = 0; j < Lk; ++j) {
                if (p->causal && j > i + off)
                    continue;
                if (p->window_left >= 0 && j < i + off - p->window_left)
                    continue;
                kidx[n++] = j;
            }
            double *dq_row = job->dq + packed_index(tq, h, 0, H, D);
            for (int d = 0; d < D; ++d)
                dq_row[d] = 0.0;
            if (n == 0)
                continue;
            /* softmax weights of the row */
            for (int a = 0; a < n; ++a) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_to_double(p->q[packed_index(tq, h, d, H, D)]) *
                           bf16_to_double(p->k[packed_index(k0 + kidx[a], kh, d, Hkv, D)]);
                s[a] = p->scale * dot;
            }
            double M = s[0];
            for (int a = 1; a < n; ++a)
                if (s[a] > M)
                    M = s[a];
            double Z = 0.0;
            for (int a = 0; a < n; ++a) {
                w[a] = exp(s[a] - M);
                Z += w[a];
            }
            for (int a = 0; a < n; ++a)
                w[a] /= Z;                              /* P_j */
            /* dP_j and Delta */
            double delta = 0.0;
            for (int a = 0; a < n; ++a) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_to_double(job->dout[packed_index(tq, h, d, H, D)]) *
                           bf16_to_double(p->v[packed_index(k0 + kidx[a], kh, d, Hkv, D)]);
                dp[a] = dot;
                delta += w[a] * dot;
            }
            for (int a = 0; a < n; ++a) {
                const double ds = w[a] * (dp[a] - delta);
                const int64_t tk = k0 + kidx[a];
                double *dk_row = job->dk + packed_index(tk, kh, 0, Hkv, D);
                double *dv_row = job->dv + packed_index(tk, kh, 0, Hkv, D);
                for (int d = 0; d < D; ++d) {
                    dq_row[d] += p->scale * ds *
                                 bf16_to_double(p->k[packed_index(tk, kh, d, Hkv, D)]);
                    dk_row[d] += p->scale * ds *
                                 bf16_to_double(p->q[packed_index(tq, h, d, H, D)]);
                    dv_row[d] += w[a] * bf16_to_double(job->dout[packed_index(tq, h, d, H, D)]);
                }
            }
        }
    }
    free(dp);
}

static void *bwd_worker(void *arg)
{
    bwd_job *job = (bwd_job *)arg;
    const int Hkv = job->p->num_kv_heads;
    size_t nscratch = (size_t)(job->max_lk > 0 ? job->max_lk : 1);
    double *s = (double *)malloc(nscratch * sizeof(double));
    double *w = (double *)malloc(nscratch * sizeof(double));
    int *kidx = (int *)malloc(nscratch * sizeof(int));
    if (!s || !w || !kidx) {
        __atomic_store_n(&job->status, -1, __ATOMIC_SEQ_CST);
        free(s); free(w); free(kidx);
        return NULL;
    }
    for (;;) {
        int64_t u = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (u >= job->n_units)
            break;
        bwd_unit(job, (int)(u / Hkv), (int)(u % Hkv), s, w, kidx);
    }
    free(s); free(w); free(kidx);
    return NULL;
}

/*
 * Full varlen backward.  q, dout: [cu_q[B], H, D]; k, v: [cu_k[B], Hkv, D]
 * (bf16 bits).  dq: double [cu_q[B], H, D]; dk, dv: double [cu_k[B], Hkv, D]
 * (overwritten).  Same masks and argument rules as oracle_varlen_fwd.
 * Returns the number of threads used (> 0), or < 0 on bad arguments.
 */
int oracle_varlen_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const uint16_t *dout, const int32_t *cu_q, const int32_t *cu_k,
                      int batch, int num_heads, int num_kv_heads, int head_dim, double scale,
                      int causal, int window_left, double *dq, double *dk, double *dv,
                      int nthreads)
{
    if (batch < 1 || num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads != 0 ||
        head_dim < 1 || causal < 0 || causal > 2 || (window_left >= 0 && causal == 0))
        return -1;
    if (check_cu(cu_q, batch) || check_cu(cu_k, batch))
        return -2;
    varlen_problem p = {q, k, v, cu_q, cu_k, batch, num_heads, num_kv_heads, head_dim, scale,
                        causal, window_left};
    memset(dk, 0, (size_t)cu_k[batch] * (size_t)num_kv_heads * (size_t)head_dim * sizeof(double));
    memset(dv, 0, (size_t)cu_k[batch] * (size_t)num_kv_heads * (size_t)head_dim * sizeof(double));
    bwd_job job;
    memset(&job, 0, sizeof job);
    job.p = &p;
    job.dout = dout;
    job.dq = dq;
    job.dk = dk;
    job.dv = dv;
    job.n_units = (int64_t)batch * num_kv_heads;
    job.max_lk = max_len(cu_k, batch);
    if (nthreads <= 0)
        nthreads = oracle_default_threads();
    if ((int64_t)nthreads > job.n_units)
        nthreads = (int)job.n_units;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid)
        return -1;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, bwd_worker, &job) != 0)
            break;
        ++started;
    }
    if (started == 0)
        bwd_worker(&job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    if (job.status != 0)
        return -1;
    return started > 0 ? started : 1;
}

/* ------------------------------------------------------------------------ */
/* Paged GQA decode (state m, l, o)                                          */
/* ------------------------------------------------------------------------ */

/* AttnState::new: m = -inf, l = 0, o = 0. */
void oracle_decode_init(double *m, double *l, double *o, int num_seqs,
                        int num_q_heads, int head_dim)
{
    const size_t n = (size_t)num_seqs * (size_t)num_q_heads;
    for (size_t i = 0; i < n; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0;
    }
    memset(o, 0, n * (size_t)head_dim * sizeof(double));
}

typedef struct {
    const uint16_t *q, *k_pool, *v_pool;
    const int32_t *tile_blocks, *tile_block_counts;
    const int32_t *tile_token_counts;      /* NULL: every token of every listed block */
    double scale;
    int tile_capacity, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
    int64_t num_blocks;
    double *m, *l, *o;
    int64_t next;
    int status;
} decode_job;

/*
 * One (sequence, q head) of one tile step.  The tokens of this step are all
 * block_size tokens of every block id tile_blocks[seq, 0:count] (or the first
 * tile_token_counts[seq] of them, taken in list order).  With x their logits
 * scale * (q . k), the state that describes every token seen
 * so far is m = max x, l = sum exp(x - m), o = sum exp(x - m) v; merging the
 * old state with this step's set re-expresses both sums at the new max.
 */
static void decode_unit(decode_job *job, int seq, int qh, double *x, int64_t *tok)
{
    const int D = job->head_dim, Hq = job->num_q_heads, Hkv = job->num_kv_heads;
    const int group = Hq / Hkv;
    const int kh = qh / group;
    const int count = job->tile_block_counts[seq];
    const int64_t take = job->tile_token_counts ? job->tile_token_counts[seq]
                                                : (int64_t)count * job->block_size;
    const size_t sidx = (size_t)seq * Hq + qh;
    const uint16_t *qrow = job->q + sidx * D;

    int64_t n = 0;
    for (int b = 0; b < count; ++b) {
        const int64_t blk = job->tile_blocks[(size_t)seq * job->tile_capacity + b];
        for (int t = 0; t < job->block_size && n < take; ++t) {
            /* pool layout [num_blocks, block_size, num_kv_heads, head_dim] */
            const int64_t base = ((blk * job->block_size + t) * Hkv + kh) * (int64_t)D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += bf16_to_double(qrow[d]) * bf16_to_double(job->k_pool[base + d]);
            x[n] = dot * job->scale;
            tok[n] = base;
            ++n;
        }
    }
    if (n == 0)
        return;                                   /* an empty tile leaves the state as it was */

    const double m_old = job->m[sidx];
    double m_new = m_old;
    for (int64_t a = 0; a < n; ++a)
        if (x[a] > m_new)
            m_new = x[a];
    const double carry = exp(m_old - m_new);      /* 0 when m_old = -inf */
    double l_new = job->l[sidx] * carry;
    double *orow = job->o + sidx * D;
    for (int d = 0; d < D; ++d)
        orow[d] *= carry;
    for (int64_t a = 0; a < n; ++a) {
        const double e = exp(x[a] - m_new);
        l_new += e;
        for (int d = 0; d < D; ++d)
            orow[d] += e * bf16_to_double(job->v_pool[tok[a] + d]);
    }
    job->m[sidx] = m_new;
    job->l[sidx] = l_new;
}

static void *decode_worker(void *arg)
{
    decode_job *job = (decode_job *)arg;
    const size_t cap_tokens = (size_t)(job->tile_capacity > 0 ? job->tile_capacity : 1) *
                              (size_t)job->block_size;
    double *x = (double *)malloc(cap_tokens * sizeof(double));
    int64_t *tok = (int64_t *)malloc(cap_tokens * sizeof(int64_t));
    if (!x || !tok) {
        __atomic_store_n(&job->status, -1, __ATOMIC_SEQ_CST);
        free(x); free(tok);
        return NULL;
    }
    const int64_t n_units = (int64_t)job->num_seqs * job->num_q_heads;
    for (;;) {
        int64_t u = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (u >= n_units)
            break;
        decode_unit(job, (int)(u / job->num_q_heads), (int)(u % job->num_q_heads), x, tok);
    }
    free(x); free(tok);
    return NULL;
}

/*
 * One tile step over every sequence.  q: [S, Hq, D]; pools: [num_blocks,
 * block_size, Hkv, D] (bf16 bits); tile_blocks: [S, tile_capacity];
 * tile_block_counts: [S]; tile_token_counts: [S] or NULL; scale <= 0 means
 * 1/sqrt(D).  m, l: double [S, Hq]; o: double [S, Hq, D] (in/out).
 * Returns threads used (> 0) or < 0 on bad arguments (nothing is changed).
 */
int oracle_decode_step(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                       int64_t num_blocks, const int32_t *tile_blocks,
                       const int32_t *tile_block_counts, const int32_t *tile_token_counts,
                       int tile_capacity, int num_seqs, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, double scale, double *m, double *l,
                       double *o, int nthreads)
{
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 ||
        block_size < 1 || tile_capacity < 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s) {
        const int c = tile_block_counts[s];
        if (c < 0 || c > tile_capacity)
            return -2;
        for (int b = 0; b < c; ++b) {
            const int32_t blk = tile_blocks[(size_t)s * tile_capacity + b];
            if (blk < 0 || blk >= num_blocks)
                return -3;
        }
        if (tile_token_counts &&
            (tile_token_counts[s] < 0 || (int64_t)tile_token_counts[s] > (int64_t)c * block_size))
            return -4;
    }
    decode_job job;
    memset(&job, 0, sizeof job);
    job.q = q; job.k_pool = k_pool; job.v_pool = v_pool;
    job.tile_blocks = tile_blocks; job.tile_block_counts = tile_block_counts;
    job.tile_token_counts = tile_token_counts;
    job.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)head_dim);
    job.tile_capacity = tile_capacity; job.num_seqs = num_seqs;
    job.num_q_heads = num_q_heads; job.num_kv_heads = num_kv_heads;
    job.head_dim = head_dim; job.block_size = block_size; job.num_blocks = num_blocks;
    job.m = m; job.l = l; job.o = o;

    const int64_t n_units = (int64_t)num_seqs * num_q_heads;
    if (nthreads <= 0)
        nthreads = oracle_default_threads();
    if ((int64_t)nthreads > n_units)
        nthreads = (int)n_units;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid)
        return -1;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, decode_worker, &job) != 0)
            break;
        ++started;
    }
    if (started == 0)
        decode_worker(&job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    if (job.status != 0)
        return -1;
    return started > 0 ? started : 1;
}

/* finalize_ref: out = o * (l > 0 ? 1 / l : 0), kept in double here. */
void oracle_decode_finalize(const double *l, const double *o, int num_seqs,
                            int num_q_heads, int head_dim, double *out)
{
    const size_t n = (size_t)num_seqs * (size_t)num_q_heads;
    for (size_t i = 0; i < n; ++i) {
        const double inv_l = l[i] > 0.0 ? 1.0 / l[i] : 0.0;
        for (int d = 0; d < head_dim; ++d)
            out[i * head_dim + d] = o[i * head_dim + d] * inv_l;
    }
}
