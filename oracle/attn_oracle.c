/*
 * attn_oracle.c -- fp64 CPU oracle for multi-head scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests, the smoke check and the bench's CPU
 * baseline leg may load this code; the product library never calls it and
 * shares no code, header or table with it.
 *
 * What it computes is the plain three-stage definition, row by row, in the
 * order the source pages give it:
 *
 *   stage 1  scores   s_j = scale * <q_i, k_j>        for every allowed key j
 *            (realizar cached/attention.rs, parallel_multihead_attention_gpu_cached:
 *             per-head Q.K^T product, then multiplication by scale = 1/sqrt(head_dim);
 *             ripvec-core Driver::fused_scale_mask_softmax: softmax(scores*scale + mask))
 *   stage 2  weights  w_j = exp(s_j - max) / sum exp(s_k - max) over allowed keys,
 *            disallowed keys weight 0, a row with no allowed key is all zeros
 *            (realizar cached/attention.rs, batched_causal_softmax: max over the
 *             visible range, exp and sum, normalise only when the sum is positive,
 *             hidden positions stay at their zero initialisation)
 *   stage 3  output   o_i = sum_j w_j v_j
 *            (realizar cached/attention.rs, parallel_multihead_attention_gpu_cached:
 *             weights times V per head)
 *
 * Which keys are allowed (readings of the pages, all integer arithmetic):
 *   - key padding: j < key_lens[b] when key_lens is given
 *     (ripvec-core Driver::build_attn_mask, 0/1 key mask; the additive -10000
 *      is read as exclusion, i.e. weight exactly 0)
 *   - mode 0, none:         every key (bidirectional encoder attention)
 *   - mode 1, causal:       j <= pos_offset + i
 *     (batched_causal_softmax: row i sees 0..=i; ferrum-kernels Backend::qk_norm_rope:
 *      token i sits at position pos_offset + i)
 *   - mode 2, window:       |pos_offset + i - j| <= window/2 (floor), window 0 = no window
 *     (ripvec-core Driver::fused_scale_mask_softmax_windowed)
 *   - mode 3, causal window: pos_offset + i - window < j <= pos_offset + i, window 0 = causal
 *     (ferrum-kernels Backend::flash_attention_batched_per_cache, sliding_window:
 *      the last w valid positions, 0 = full causal)
 *   - grouped-query heads: query head h reads key/value head h / (q_heads/kv_heads)
 *     (ferrum-kernels Backend::split_qkv, q_dim differs from kv_dim)
 *
 * Inputs are float arrays (every bf16 and fp32 value is exactly a float);
 * each element is widened to double before use and all arithmetic is fp64.
 * Layout: q [B, Hq, Lq, D], k and v [B, Hkv, Lk, D], row-major, contiguous.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const float *q, *k, *v;
    int B, Hq, Hkv, Lq, Lk, D, P, mode, window;
    const int *key_lens;
    double scale;
    const long long *rows;
    long long nrows;
    double *out;     /* [nrows, D] */
    double *weights; /* NULL or [nrows, Lk] */
    long long next;  /* shared work counter */
    pthread_mutex_t lock;
} job_t;

/* Allowed-key rule for one (query position, key index) pair. */
static int key_allowed(int mode, long long qpos, long long j, int window)
{
    switch (mode) {
    case 0:
        return 1;
    case 1:
        return j <= qpos;
    case 2: {
        if (window == 0) return 1;
        long long d = qpos - j;
        if (d < 0) d = -d;
        return d <= (long long)(window / 2);
    }
    case 3:
        if (j > qpos) return 0;
        if (window == 0) return 1;
        return j > qpos - (long long)window;
    default:
        return 0;
    }
}

/* One output row: the three stages, in fp64, with per-row scratch. */
static void one_row(const job_t *jb, long long row, double *out_row,
                    double *w_row, double *s, unsigned char *allowed)
{
    const int D = jb->D, Lk = jb->Lk;
    const long long i = row % jb->Lq;
    const long long bh = row / jb->Lq;
    const int hq = (int)(bh % jb->Hq);
    const int b = (int)(bh / jb->Hq);
    const int group = jb->Hq / jb->Hkv;
    const int hk = hq / group;
    const long long qpos = (long long)jb->P + i;
    const int klen = jb->key_lens ? jb->key_lens[b] : Lk;

    const float *qrow = jb->q + row * (long long)D;
    const float *kh = jb->k + ((long long)b * jb->Hkv + hk) * (long long)Lk * D;
    const float *vh = jb->v + ((long long)b * jb->Hkv + hk) * (long long)Lk * D;

    /* stage 1: scaled dot products of the allowed keys */
    int any = 0;
    for (long long j = 0; j < Lk; ++j) {
        allowed[j] = (unsigned char)(j < klen && key_allowed(jb->mode, qpos, j, jb->window));
        if (!allowed[j]) { s[j] = 0.0; continue; }
        double acc = 0.0;
        const float *krow = kh + j * D;
        for (int d = 0; d < D; ++d) acc += (double)qrow[d] * (double)krow[d];
        s[j] = jb->scale * acc;
        any = 1;
    }

    /* stage 2: softmax over the allowed keys; masked keys weight 0 */
    if (any) {
        double m = -INFINITY;
        for (long long j = 0; j < Lk; ++j)
            if (allowed[j] && s[j] > m) m = s[j];
        double sum = 0.0;
        for (long long j = 0; j < Lk; ++j) {
            s[j] = allowed[j] ? exp(s[j] - m) : 0.0;
            sum += s[j];
        }
        if (sum > 0.0)
            for (long long j = 0; j < Lk; ++j) s[j] /= sum;
    } else {
        for (long long j = 0; j < Lk; ++j) s[j] = 0.0;
    }

    /* stage 3: weighted sum of value rows */
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    for (long long j = 0; j < Lk; ++j) {
        if (s[j] == 0.0) continue;
        const float *vrow = vh + j * D;
        for (int d = 0; d < D; ++d) out_row[d] += s[j] * (double)vrow[d];
    }
    if (w_row) memcpy(w_row, s, sizeof(double) * (size_t)Lk);
}

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)jb->Lk + 8);
    unsigned char *allowed = (unsigned char *)malloc((size_t)jb->Lk + 8);
    if (!s || !allowed) { free(s); free(allowed); return (void *)1; }
    for (;;) {
        long long t;
        pthread_mutex_lock(&jb->lock);
        t = jb->next;
        jb->next += 1;
        pthread_mutex_unlock(&jb->lock);
        if (t >= jb->nrows) break;
        long long row = jb->rows ? jb->rows[t] : t;
        one_row(jb, row, jb->out + t * (long long)jb->D,
                jb->weights ? jb->weights + t * (long long)jb->Lk : NULL, s, allowed);
    }
    free(s);
    free(allowed);
    return NULL;
}

/*
 * Compute output rows of attention in fp64.
 * rows: flat row indices (b*Hq + hq)*Lq + i, or NULL for every row in order
 *       (then nrows must equal B*Hq*Lq).
 * out: [nrows, D] doubles. weights: NULL or [nrows, Lk] doubles (stage-2 weights).
 * nthreads <= 0 uses every online core. Returns 0, or -1 on invalid arguments,
 * -2 on allocation failure.
 */
int oracle_attention_rows(const float *q, const float *k, const float *v,
                          int B, int Hq, int Hkv, int Lq, int Lk, int D,
                          int pos_offset, int mode, int window, const int *key_lens,
                          double scale, const long long *rows, long long nrows,
                          double *out, double *weights, int nthreads)
{
    if (!q || !k || !v || !out) return -1;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Lq < 0 || Lk < 0 || D <= 0) return -1;
    if (Hq % Hkv != 0 || mode < 0 || mode > 3 || window < 0 || pos_offset < 0) return -1;
    if (!rows && nrows != (long long)B * Hq * Lq) return -1;
    if (rows)
        for (long long t = 0; t < nrows; ++t)
            if (rows[t] < 0 || rows[t] >= (long long)B * Hq * Lq) return -1;
    if (nrows == 0) return 0;

    job_t jb;
    jb.q = q; jb.k = k; jb.v = v;
    jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.Lq = Lq; jb.Lk = Lk; jb.D = D;
    jb.P = pos_offset; jb.mode = mode; jb.window = window; jb.key_lens = key_lens;
    jb.scale = scale; jb.rows = rows; jb.nrows = nrows; jb.out = out; jb.weights = weights;
    jb.next = 0;
    pthread_mutex_init(&jb.lock, NULL);

    long ncpu = sysconf(_SC_NPROCESSORS_ONLN);
    int nt = nthreads > 0 ? nthreads : (int)(ncpu > 0 ? ncpu : 1);
    if ((long long)nt > nrows) nt = (int)nrows;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) { pthread_mutex_destroy(&jb.lock); return -2; }
    int started = 0, rc = 0;
    for (int t = 0; t < nt; ++t) {
        if (pthread_create(&th[t], NULL, worker, &jb) != 0) break;
        ++started;
    }
    if (started == 0) rc = (worker(&jb) == NULL) ? 0 : -2;
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret) rc = -2;
    }
    free(th);
    pthread_mutex_destroy(&jb.lock);
    return rc;
}
