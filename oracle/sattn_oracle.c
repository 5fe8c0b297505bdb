/*
 * sattn oracle: plain, slow, fp64 reference for index-gathered attention with
 * sinks.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path links, loads or calls
 * this file; only the test suite, the package's smoke check and the CPU
 * baseline leg of the benchmark do. It shares no code, header or constant
 * table with the CUDA implementation.
 *
 * Every row r = (query, head) is computed as a literal masked softmax over an
 * explicit multiset S(r) of key rows, with no tiling, no online update and no
 * log2 tricks:
 *
 *   l_j  = scale * <q_r, k_j>            (+ sink_h on "key 0" in key-0 mode)
 *   Z    = sum_{j in S} exp(l_j)         (+ exp(sink_h) in null-logit mode)
 *   o_r  = sum_{j in S} exp(l_j) v_j / Z
 *   lse_r = ln Z
 *
 * evaluated with the maximum of {l_j} (and the null sink) subtracted first.
 * A row with nothing to attend gives o = 0 and lse = -inf (or lse = sink in
 * null-logit mode, where Z = exp(sink)).
 *
 * Sources (pages, by title and section):
 *  - "PR #49815 report" (vLLM, apply vision attention sinks in the window
 *    attention path): window visibility |i-j| <= w inside one sequence,
 *    non-causal; GQA head map h // (H/Hkv); key-0 bias semantics (the sink is
 *    added to the logit of each sequence's first key where it is visible);
 *    null-logit semantics (the sink is a denominator-only term) -- sections
 *    "Implementation" items 2-4 and the `_fwd_kernel` / `_reference` listings.
 *  - "DeepSeek-V4 CSA/HCA sparse attention walkthrough": gathered attention
 *    over topk_idxs into a single shared KV head (the same row is key and
 *    value), -1 entries contribute nothing (section 4.2), sink added to the
 *    softmax denominator (section 4.4).
 *  - "XAttention Offload Stream Synchronization Fix" (nano-vllm): per-chunk
 *    partial softmax statistics merged into global ones (technical details,
 *    three-stage KV chunking).
 *
 * Inputs are float32 arrays holding the exact values the GPU receives
 * (bf16 inputs widened exactly); all arithmetic is in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_SINK_NONE 0
#define ORACLE_SINK_KEY0_BIAS 1
#define ORACLE_SINK_NULL_LOGIT 2

/* ------------------------------------------------------------------------ */
/* Softmax over one row's explicit key multiset.                            */
/* ------------------------------------------------------------------------ */

/* n logits with their value rows (float32, length d). If null_sink, exp(sink)
 * joins the denominator only. Writes o[d] and *lse. */
static void softmax_row(int n, const double *logit, const float *const *vrow, int d,
                        int null_sink, double sink, double *o, double *lse)
{
    double m = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (logit[j] > m) m = logit[j];
    if (null_sink && sink > m) m = sink;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (m == -INFINITY) { /* nothing to attend to */
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
        double w = exp(logit[j] - m);
        z += w;
        for (int c = 0; c < d; ++c) o[c] += w * (double)vrow[j][c];
    }
    if (null_sink) z += exp(sink - m);
    for (int c = 0; c < d; ++c) o[c] /= z;
    *lse = m + log(z);
}

static double dot_qk(const float *q, const float *k, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += (double)q[c] * (double)k[c];
    return s;
}

/* ------------------------------------------------------------------------ */
/* A tiny parallel-for over rows (rows are independent).                    */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(const void *ctx, int64_t first, int64_t last, double *scratch);

struct pf_job {
    row_fn fn;
    const void *ctx;
    int64_t first, last;
    size_t scratch_doubles;
};

static void *pf_thread(void *arg)
{
    struct pf_job *job = (struct pf_job *)arg;
    double *scratch = (double *)malloc(job->scratch_doubles * sizeof(double) + 64);
    if (scratch) {
        job->fn(job->ctx, job->first, job->last, scratch);
        free(scratch);
    }
    return NULL;
}

static int g_threads = 0; /* 0 or less: every online core */

static int oracle_threads(void)
{
    if (g_threads > 0) return g_threads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int parallel_rows(row_fn fn, const void *ctx, int64_t nrows, size_t scratch_doubles)
{
    int nt = oracle_threads();
    if (nt > nrows) nt = (int)(nrows > 0 ? nrows : 1);
    if (nt <= 1) {
        double *scratch = (double *)malloc(scratch_doubles * sizeof(double) + 64);
        if (!scratch) return -1;
        fn(ctx, 0, nrows, scratch);
        free(scratch);
        return 0;
    }
    pthread_t *tid = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    struct pf_job *jobs = (struct pf_job *)calloc((size_t)nt, sizeof(struct pf_job));
    if (!tid || !jobs) { free(tid); free(jobs); return -1; }
    for (int t = 0; t < nt; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].first = nrows * t / nt;
        jobs[t].last = nrows * (t + 1) / nt;
        jobs[t].scratch_doubles = scratch_doubles;
        pthread_create(&tid[t], NULL, pf_thread, &jobs[t]);
    }
    for (int t = 0; t < nt; ++t) pthread_join(tid[t], NULL);
    free(tid);
    free(jobs);
    return 0;
}

/* Number of worker threads for every following call (0 or less: every online core). */
void oracle_set_threads(int n) { g_threads = n; }
int oracle_get_threads(void) { return oracle_threads(); }

/* ------------------------------------------------------------------------ */
/* Window attention over packed varlen sequences ("PR #49815 report").      */
/* ------------------------------------------------------------------------ */

struct window_ctx {
    const float *q, *k, *v, *sinks;
    const int32_t *cu_seqlens;
    int num_seqs, H, Hkv, d, wl, wr, causal, sink_mode;
    double scale;
    const int64_t *rows; /* optional subset of rows r = token * H + head */
    double *o, *lse;
};

/* Key j (local) is visible to query i (local) of the same sequence iff
 * -wl <= j - i <= wr (a negative bound means unbounded on that side) and, for
 * causal attention, j <= i. The pages' window w is wl = wr = w. */
static int window_visible(int i, int j, int wl, int wr, int causal)
{
    if (wl >= 0 && j < i - wl) return 0;
    if (wr >= 0 && j > i + wr) return 0;
    if (causal && j > i) return 0;
    return 1;
}

static void window_rows(const void *vctx, int64_t first, int64_t last, double *scratch)
{
    const struct window_ctx *c = (const struct window_ctx *)vctx;
    int64_t T = c->cu_seqlens[c->num_seqs];
    /* scratch layout: logits[T] | value-row pointers[T] */
    double *logit = scratch;
    const float **vrow = (const float **)(scratch + T);
    int groups = c->H / c->Hkv;
    for (int64_t n = first; n < last; ++n) {
        int64_t r = c->rows ? c->rows[n] : n;
        int64_t tok = r / c->H;
        int h = (int)(r % c->H);
        int g = h / groups; /* GQA: repeat_interleave of KV heads */
        int s = 0;
        while (s + 1 < c->num_seqs + 1 && c->cu_seqlens[s + 1] <= tok) ++s;
        int64_t start = c->cu_seqlens[s];
        int L = (int)(c->cu_seqlens[s + 1] - start);
        int i = (int)(tok - start);
        const float *qr = c->q + (tok * c->H + h) * (int64_t)c->d;
        double sink = c->sinks ? (double)c->sinks[h] : 0.0;
        int cnt = 0;
        for (int j = 0; j < L; ++j) {
            if (!window_visible(i, j, c->wl, c->wr, c->causal)) continue;
            int64_t kt = start + j;
            const float *kr = c->k + (kt * c->Hkv + g) * (int64_t)c->d;
            double l = c->scale * dot_qk(qr, kr, c->d);
            if (c->sink_mode == ORACLE_SINK_KEY0_BIAS && j == 0) l += sink;
            logit[cnt] = l;
            vrow[cnt] = c->v + (kt * c->Hkv + g) * (int64_t)c->d;
            ++cnt;
        }
        softmax_row(cnt, logit, vrow, c->d, c->sink_mode == ORACLE_SINK_NULL_LOGIT, sink,
                    c->o + n * (int64_t)c->d, c->lse + n);
    }
}

/* q[T,H,d], k/v[T,Hkv,d], cu_seqlens[num_seqs+1]; o[nrows,d], lse[nrows]
 * where nrows = T*H (rows == NULL) or nrows (the listed rows). */
int oracle_window(const float *q, const float *k, const float *v, const int32_t *cu_seqlens,
                  int num_seqs, int H, int Hkv, int d, int window_left, int window_right,
                  int causal, const float *sinks, int sink_mode, double scale,
                  const int64_t *rows, int64_t nrows, double *o, double *lse)
{
    if (H <= 0 || Hkv <= 0 || H % Hkv) return -1;
    if (sink_mode != ORACLE_SINK_NONE && !sinks) return -1;
    struct window_ctx c = {q, k, v, sinks, cu_seqlens, num_seqs, H, Hkv, d,
                           window_left, window_right, causal, sink_mode, scale, rows, o, lse};
    int64_t T = cu_seqlens[num_seqs];
    if (!rows) nrows = T * H;
    /* scratch: T logits + T pointers */
    return parallel_rows(window_rows, &c, nrows, (size_t)(2 * T + 2));
}

/* ------------------------------------------------------------------------ */
/* Index-gathered attention over one shared KV head (DeepSeek-V4 walkthrough) */
/* ------------------------------------------------------------------------ */

struct sparse_ctx {
    const float *q, *kv, *sinks;
    const int32_t *idx;
    int B, M, H, d, N, K, sink_mode;
    double scale;
    const int64_t *rows; /* optional subset of rows r = (b*M + m)*H + h */
    double *o, *lse;
};

static void sparse_rows(const void *vctx, int64_t first, int64_t last, double *scratch)
{
    const struct sparse_ctx *c = (const struct sparse_ctx *)vctx;
    double *logit = scratch;
    const float **vrow = (const float **)(scratch + c->K);
    for (int64_t n = first; n < last; ++n) {
        int64_t r = c->rows ? c->rows[n] : n;
        int64_t bm = r / c->H;
        int h = (int)(r % c->H);
        int64_t b = bm / c->M;
        const float *qr = c->q + r * (int64_t)c->d;
        const int32_t *list = c->idx + bm * (int64_t)c->K;
        double sink = c->sinks ? (double)c->sinks[h] : 0.0;
        int cnt = 0;
        for (int t = 0; t < c->K; ++t) {
            int32_t e = list[t];
            if (e < 0) continue; /* -1: invalid entry, contributes nothing */
            /* key row == value row: one shared KV head */
            const float *row = c->kv + (b * c->N + e) * (int64_t)c->d;
            double l = c->scale * dot_qk(qr, row, c->d);
            if (c->sink_mode == ORACLE_SINK_KEY0_BIAS && e == 0) l += sink;
            logit[cnt] = l;
            vrow[cnt] = row;
            ++cnt;
        }
        softmax_row(cnt, logit, vrow, c->d, c->sink_mode == ORACLE_SINK_NULL_LOGIT, sink,
                    c->o + n * (int64_t)c->d, c->lse + n);
    }
}

/* q[B,M,H,d], kv[B,N,d], idx[B,M,K] (entries -1 or in [0,N)); o[nrows,d], lse[nrows]. */
int oracle_sparse(const float *q, const float *kv, const int32_t *idx, int B, int M, int H,
                  int d, int N, int K, const float *sinks, int sink_mode, double scale,
                  const int64_t *rows, int64_t nrows, double *o, double *lse)
{
    if (sink_mode != ORACLE_SINK_NONE && !sinks) return -1;
    for (int64_t t = 0; t < (int64_t)B * M * K; ++t)
        if (idx[t] < -1 || idx[t] >= N) return -2;
    struct sparse_ctx c = {q, kv, sinks, idx, B, M, H, d, N, K, sink_mode, scale, rows, o, lse};
    if (!rows) nrows = (int64_t)B * M * H;
    return parallel_rows(sparse_rows, &c, nrows, (size_t)(2 * K + 2));
}

/* ------------------------------------------------------------------------ */
/* One KV chunk of block-sparse causal attention (nano-vllm XAttention).    */
/* ------------------------------------------------------------------------ */

struct block_ctx {
    const float *q, *k, *v;
    const uint8_t *mask;
    int M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end, causal, blk;
    double scale;
    const int64_t *rows; /* optional subset of rows r = i*H + h */
    double *o, *lse;
};

static void block_rows(const void *vctx, int64_t first, int64_t last, double *scratch)
{
    const struct block_ctx *c = (const struct block_ctx *)vctx;
    int QB = (c->M + c->blk - 1) / c->blk;
    int KB = (c->Nctx + c->blk - 1) / c->blk;
    int groups = c->H / c->Hkv;
    double *logit = scratch;
    const float **vrow = (const float **)(scratch + c->Nctx);
    for (int64_t n = first; n < last; ++n) {
        int64_t r = c->rows ? c->rows[n] : n;
        int i = (int)(r / c->H);
        int h = (int)(r % c->H);
        int g = h / groups;
        int64_t pos = (int64_t)c->q_pos0 + i;
        const float *qr = c->q + r * (int64_t)c->d;
        const uint8_t *mrow = c->mask + ((int64_t)h * QB + i / c->blk) * KB;
        int cnt = 0;
        for (int j = c->kv_begin; j < c->kv_end; ++j) {
            if (!mrow[j / c->blk]) continue;
            if (c->causal && j > pos) continue;
            const float *kr = c->k + ((int64_t)j * c->Hkv + g) * c->d;
            logit[cnt] = c->scale * dot_qk(qr, kr, c->d);
            vrow[cnt] = c->v + ((int64_t)j * c->Hkv + g) * c->d;
            ++cnt;
        }
        softmax_row(cnt, logit, vrow, c->d, 0, 0.0, c->o + n * (int64_t)c->d, c->lse + n);
    }
}

/* q[M,H,d] at positions q_pos0.., k/v[Nctx,Hkv,d], mask uint8[H, ceil(M/blk),
 * ceil(Nctx/blk)] (query block local, key block global); only keys in
 * [kv_begin, kv_end) are used. Writes the chunk's normalised partial output
 * and its lse (-inf where the row sees nothing in the chunk). */
int oracle_block_sparse(const float *q, const float *k, const float *v, const uint8_t *mask,
                        int M, int Nctx, int H, int Hkv, int d, int q_pos0, int kv_begin,
                        int kv_end, int causal, int blk, double scale, const int64_t *rows,
                        int64_t nrows, double *o, double *lse)
{
    if (H <= 0 || Hkv <= 0 || H % Hkv || blk <= 0) return -1;
    if (kv_begin < 0 || kv_end > Nctx || kv_begin > kv_end) return -1;
    struct block_ctx c = {q, k, v, mask, M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end,
                          causal, blk, scale, rows, o, lse};
    if (!rows) nrows = (int64_t)M * H;
    return parallel_rows(block_rows, &c, nrows, (size_t)(2 * (int64_t)Nctx + 2));
}

/* ------------------------------------------------------------------------ */
/* Merge of chunk partials through their log-sum-exp (nano-vllm XAttention) */
/* ------------------------------------------------------------------------ */

/* o_parts[C,R,d] (each normalised within its chunk), lse_parts[C,R];
 * sinks[H] or NULL (a null-logit term added once, head = r % H).
 *   lse = ln( sum_c exp(lse_c) [+ exp(sink)] ),  o = sum_c exp(lse_c - lse) o_c
 * which is the (m, l) merge m = max_c m_c, l = sum_c l_c exp(m_c - m). */
int oracle_merge(const double *o_parts, const double *lse_parts, int C, int64_t R, int d,
                 int H, const float *sinks, double *o, double *lse)
{
    for (int64_t r = 0; r < R; ++r) {
        double m = -INFINITY;
        for (int c = 0; c < C; ++c)
            if (lse_parts[(int64_t)c * R + r] > m) m = lse_parts[(int64_t)c * R + r];
        double sink = sinks ? (double)sinks[r % H] : -INFINITY;
        if (sinks && sink > m) m = sink;
        for (int x = 0; x < d; ++x) o[r * d + x] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int c = 0; c < C; ++c) z += exp(lse_parts[(int64_t)c * R + r] - m);
        if (sinks) z += exp(sink - m);
        double L = m + log(z);
        for (int c = 0; c < C; ++c) {
            double lc = lse_parts[(int64_t)c * R + r];
            if (lc == -INFINITY) continue;
            double w = exp(lc - L);
            const double *oc = o_parts + ((int64_t)c * R + r) * d;
            for (int x = 0; x < d; ++x) o[r * d + x] += w * oc[x];
        }
        lse[r] = L;
    }
    return 0;
}
