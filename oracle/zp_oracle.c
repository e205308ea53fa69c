/*
 * zp_oracle.c -- plain fp64 CPU oracle for the Compressed PagedAttention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Tests, the smoke check and the benchmark's CPU
 * baseline leg are the only callers.  The product path (the CUDA library) never
 * links, loads or calls this file, and this file includes nothing from it.
 *
 * Sources (page title, then section):
 *   [ZP-nl]  "Zipage: Maintain High Request Concurrency for LLM Reasoning through
 *            Compressed PagedAttention", gist.science Dutch summary,
 *            "Technische samenvatting / Methodologie".
 *   [ZP-ko]  the same paper, gist.science Korean summary, "기술 요약 / 2. 방법론".
 *   [PKV]    "Paged KV cache and continuous batching for LLMs" (upskillscore),
 *            "How it works".
 *
 * What is computed, step by step (one "unit" = one request x layer x kv head):
 *   plan       [ZP-nl Methodologie §1, §3; ZP-ko 방법론 C]: destination blocks.
 *   importance [ZP-ko 방법론 A, observation window]: softmax(q.k/sqrt(d)) of the
 *              last w queries over all cached keys (causal inside the window),
 *              averaged over the w queries and the G query heads of the group.
 *   redundancy [ZP-nl Methodologie §5; ZP-ko 방법론 E, Lightning Redundancy
 *              Score]: mean cosine similarity of a key to the other b-1 keys of
 *              its own block.
 *   score      importance - lambda * redundancy, for the C = T - w candidates.
 *   select     [ZP-ko 방법론 A]: keep the (N-1)*b - w best candidates (score
 *              descending, lower index first at equal score), then the window.
 *   compact    [ZP-nl Methodologie §1]: kept rows, in original order, fill the
 *              first N-1 blocks; block N is reserved for future decoding.
 *   commit     [ZP-nl Methodologie §1, §3; PKV]: tables, lengths, refcounts,
 *              released blocks back to the free stack.
 *   decode     [PKV]: attention of one query per head over the block table.
 *   prefill    [ZP-nl Methodologie §1, §3]: the same scoring, selection and
 *              compaction for a request admitted with more than N*b tokens;
 *              its excess blocks are released.
 *   alloc /    [PKV]: blocks for a request's first tokens (taken from the free
 *   release    stack) and, when it finishes or is preempted, every block of
 *              its table back (one reference each, pushed when it reaches 0).
 *   fork       [PKV]: a new request sharing every block of another one (parallel
 *              sampling stores the shared prompt once; refcounts count holders).
 *   append     [PKV; ZP-nl Methodologie §1]: the slot of each decoding request's
 *              next token (a new block only when the last one is full,
 *              copy-on-write of a shared block), the new token's K/V written
 *              there, and the requests whose cache just reached N_max full
 *              blocks (the compression trigger).
 *
 * Every floating-point quantity is computed in double from the exact widening
 * of the bf16 inputs.  No blocking, fusion or reordering beyond the definitions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ZPO_OK 0
#define ZPO_ERR_INVALID_ARG (-1)
#define ZPO_ERR_OUT_OF_BLOCKS (-3)
#define ZPO_ERR_DEVICE_CHECK (-4)

/* ---------------------------------------------------------------- bf16 */

double zpo_bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double once, to nearest even, onto the bf16 grid (8 significant
 * bits, fp32 exponent range).  Values beyond the largest finite bf16 become
 * infinities; NaN stays NaN. */
uint16_t zpo_double_to_bf16(double x)
{
    if (isnan(x))
        return (uint16_t)0x7fc0;
    double ax = fabs(x);
    uint16_t sign = signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
    if (ax == 0.0)
        return sign;
    int e;
    frexp(ax, &e);                 /* ax = m * 2^e, m in [0.5, 1) */
    int exp_unbiased = e - 1;      /* ax in [2^(e-1), 2^e) */
    if (exp_unbiased < -126)
        exp_unbiased = -126;       /* subnormal range: fixed spacing */
    double spacing = ldexp(1.0, exp_unbiased - 7);
    double q = rint(ax / spacing); /* default rounding mode: to nearest even */
    double r = q * spacing;
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7f80);
    float f = (float)r; /* exact: r lies on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7fff));
}

/* Element-wise zpo_double_to_bf16 over an array. */
void zpo_double_to_bf16_array(const double *x, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = zpo_double_to_bf16(x[i]);
}

static double dot_bf16(const uint16_t *a, const uint16_t *b, int d)
{
    double s = 0.0;
    for (int k = 0; k < d; ++k)
        s += zpo_bf16_to_double(a[k]) * zpo_bf16_to_double(b[k]);
    return s;
}

/* ---------------------------------------------------------- importance */

/* Observation-window importance of the C = T - w candidates of one unit.
 *   K: T rows of d bf16, in token order.
 *   Q: G*w rows of d bf16; row g*w + i is query head g at window slot i, the
 *      query of token C + i.
 * Query i attends to keys 0 .. C+i (causal); its softmax uses exactly those.
 * imp[j] = (1/(w*G)) * sum_{g,i} softmax_row(g,i)[j]   for j < C.
 * [ZP-ko 방법론 A, observation window]; formula as adopted by this library. */
void zpo_importance(const uint16_t *K, const uint16_t *Q, int T, int d, int w, int G,
                    double *imp)
{
    int C = T - w;
    double scale = 1.0 / sqrt((double)d);
    double *logit = (double *)malloc(sizeof(double) * (size_t)T);
    for (int j = 0; j < C; ++j)
        imp[j] = 0.0;
    for (int g = 0; g < G; ++g) {
        for (int i = 0; i < w; ++i) {
            const uint16_t *q = Q + (size_t)(g * w + i) * d;
            int visible = C + i + 1;
            double m = -INFINITY;
            for (int j = 0; j < visible; ++j) {
                logit[j] = dot_bf16(q, K + (size_t)j * d, d) * scale;
                if (logit[j] > m)
                    m = logit[j];
            }
            double S = 0.0;
            for (int j = 0; j < visible; ++j)
                S += exp(logit[j] - m);
            for (int j = 0; j < C; ++j)
                imp[j] += exp(logit[j] - m) / S;
        }
    }
    for (int j = 0; j < C; ++j)
        imp[j] /= (double)(w * G);
    free(logit);
}

/* ---------------------------------------------------------- redundancy */

/* Lightning Redundancy Score [ZP-nl Methodologie §5; ZP-ko 방법론 E]: only the
 * keys of the same block are compared, O(N*b^2) per unit.
 * red[j] = (1/(f-1)) * sum_{k in block(j), k != j} cos(K_j, K_k), where f is
 * the number of filled slots of the block (b, except for a partial last block
 * when T is not a multiple of b; a block with one key gives 0) and a
 * zero-norm key has cosine 0 with every key.  All T keys get a value; window
 * keys count as "other keys" of their block. */
void zpo_redundancy(const uint16_t *K, int T, int d, int b, double *red)
{
    double *norm = (double *)malloc(sizeof(double) * (size_t)b);
    for (int base = 0; base < T; base += b) {
        int f = T - base < b ? T - base : b;
        for (int j = 0; j < f; ++j) {
            const uint16_t *kj = K + (size_t)(base + j) * d;
            norm[j] = sqrt(dot_bf16(kj, kj, d));
        }
        for (int j = 0; j < f; ++j) {
            double sum = 0.0;
            for (int k = 0; k < f; ++k) {
                if (k == j)
                    continue;
                double c = 0.0;
                if (norm[j] > 0.0 && norm[k] > 0.0)
                    c = dot_bf16(K + (size_t)(base + j) * d, K + (size_t)(base + k) * d, d) /
                        (norm[j] * norm[k]);
                sum += c;
            }
            red[base + j] = f > 1 ? sum / (double)(f - 1) : 0.0;
        }
    }
    free(norm);
}

/* Redundancy over ALL keys of a unit: the O(N^2*b^2) score that the
 * Lightning Redundancy Score replaces [ZP-nl Methodologie §5; ZP-ko 방법론 E],
 * read with this library's definition (mean cosine similarity to the other
 * keys), the comparison set being every other key of the unit instead of
 * its block: red[j] = (1/(T-1)) * sum_{k != j} cos(K_j, K_k), a zero-norm
 * key having cosine 0 with every key.  Written pair by pair, O(T^2 d). */
void zpo_redundancy_global(const uint16_t *K, int T, int d, double *red)
{
    double *norm = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    for (int j = 0; j < T; ++j)
        norm[j] = sqrt(dot_bf16(K + (size_t)j * d, K + (size_t)j * d, d));
    for (int j = 0; j < T; ++j) {
        double sum = 0.0;
        for (int k = 0; k < T; ++k) {
            if (k == j || norm[j] == 0.0 || norm[k] == 0.0)
                continue;
            sum += dot_bf16(K + (size_t)j * d, K + (size_t)k * d, d) / (norm[j] * norm[k]);
        }
        red[j] = T > 1 ? sum / (double)(T - 1) : 0.0;
    }
    free(norm);
}

/* score[j] = imp[j] - lambda * red[j] for the C candidates. */
void zpo_unit_scores(const uint16_t *K, const uint16_t *Q, int T, int d, int b, int w, int G,
                     double lambda, double *imp, double *red, double *score)
{
    int C = T - w;
    zpo_importance(K, Q, T, d, w, G, imp);
    zpo_redundancy(K, T, d, b, red);
    for (int j = 0; j < C; ++j)
        score[j] = imp[j] - lambda * red[j];
}

/* -------------------------------------------------------------- select */

/* Candidate order: higher score first; at equal score the lower index first. */
static int better(const double *score, int32_t a, int32_t b)
{
    if (score[a] > score[b])
        return 1;
    if (score[a] < score[b])
        return 0;
    return a < b;
}

static void merge_sort(int32_t *idx, int32_t *tmp, int n, const double *score)
{
    if (n < 2)
        return;
    int h = n / 2;
    merge_sort(idx, tmp, h, score);
    merge_sort(idx + h, tmp, n - h, score);
    int i = 0, j = h, o = 0;
    while (i < h && j < n)
        tmp[o++] = better(score, idx[j], idx[i]) ? idx[j++] : idx[i++];
    while (i < h)
        tmp[o++] = idx[i++];
    while (j < n)
        tmp[o++] = idx[j++];
    memcpy(idx, tmp, sizeof(int32_t) * (size_t)n);
}

/* Token-wise eviction for one unit [ZP-ko 방법론 A]: of the C candidates keep
 * the n_keep best in the candidate order, then append the window C..T-1.
 * kept[] receives n_keep + w indices in ascending (original) order.
 * Evicting the lowest-score token one at a time with fixed scores removes the
 * same set, so a sort is the whole selection. */
void zpo_select(const double *score, int C, int w, int n_keep, int32_t *kept)
{
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
    unsigned char *keep = (unsigned char *)calloc((size_t)(C > 0 ? C : 1), 1);
    for (int j = 0; j < C; ++j)
        idx[j] = j;
    merge_sort(idx, tmp, C, score);
    for (int r = 0; r < n_keep; ++r)
        keep[idx[r]] = 1;
    int o = 0;
    for (int j = 0; j < C; ++j)
        if (keep[j])
            kept[o++] = j;
    for (int i = 0; i < w; ++i)
        kept[o++] = C + i;
    free(idx);
    free(tmp);
    free(keep);
}

/* ---------------------------------------------------------------- plan */

/* Destination blocks for the compressing requests [ZP-nl Methodologie §1, §3;
 * ZP-ko 방법론 C].  Reading adopted: with the refcounts as they are at call
 * start, block p of a request is rewritten in place when its refcount is 1 and
 * compressed into a fresh target block from the free stack when it is > 1 (a
 * shared block is never rewritten).  The reserved last block is kept when its
 * refcount is 1, else replaced by a fresh block.  Targets are popped from the
 * top of the free stack in (request, block) order.
 *
 * tables: rows of `stride` int32; request r uses row req_idx[r] (or r when
 * req_idx is NULL); lengths indexed the same way.  dst_table[r*N + p] receives
 * the destination block of (r, p).  Nothing is modified; returns a status and
 * the number of popped blocks in *n_pops. */
int zpo_plan(const int32_t *tables, int stride, const int32_t *lengths, const int32_t *req_idx,
             int R, int num_rows, int N, int b, int num_blocks, const int32_t *refcount,
             const int32_t *free_ids, int free_count, int32_t *dst_table, int *n_pops)
{
    *n_pops = 0;
    if (R < 0 || N < 2 || b < 2 || stride < N)
        return ZPO_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        if (row < 0 || row >= num_rows)
            return ZPO_ERR_INVALID_ARG;
        for (int r2 = 0; r2 < r; ++r2)
            if ((req_idx ? req_idx[r2] : r2) == row)
                return ZPO_ERR_INVALID_ARG;
        if (lengths[row] != N * b)
            return ZPO_ERR_INVALID_ARG;
        for (int p = 0; p < N; ++p) {
            int32_t blk = tables[(size_t)row * stride + p];
            if (blk < 0 || blk >= num_blocks || refcount[blk] < 1)
                return ZPO_ERR_INVALID_ARG;
        }
    }
    int pops = 0;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        for (int p = 0; p < N; ++p) {
            int32_t blk = tables[(size_t)row * stride + p];
            if (refcount[blk] > 1) {
                if (pops >= free_count)
                    return ZPO_ERR_OUT_OF_BLOCKS;
                int32_t t = free_ids[free_count - 1 - pops];
                if (t < 0 || t >= num_blocks || refcount[t] != 0)
                    return ZPO_ERR_DEVICE_CHECK;
                dst_table[(size_t)r * N + p] = t;
                ++pops;
            } else {
                dst_table[(size_t)r * N + p] = blk;
            }
        }
    }
    *n_pops = pops;
    return ZPO_OK;
}

/* Applies a plan [ZP-nl Methodologie §1, §3; PKV]: every replaced block loses
 * one reference per holder, in (request, block) order; a block whose count
 * reaches zero is pushed onto the free stack at that moment (after the pops).
 * Targets get refcount 1, rows get the destination table, lengths become
 * (N-1)*b.  Returns the new free count. */
int zpo_commit(int32_t *tables, int stride, int32_t *lengths, const int32_t *req_idx, int R,
               int N, int b, int32_t *refcount, int32_t *free_ids, int free_count,
               const int32_t *dst_table, int n_pops)
{
    int top = free_count - n_pops;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        for (int p = 0; p < N; ++p) {
            int32_t src = tables[(size_t)row * stride + p];
            int32_t dst = dst_table[(size_t)r * N + p];
            if (dst != src) {
                refcount[src] -= 1;
                if (refcount[src] == 0)
                    free_ids[top++] = src;
                refcount[dst] = 1;
                tables[(size_t)row * stride + p] = dst;
            }
        }
        lengths[row] = (N - 1) * b;
    }
    return top;
}

/* ------------------------------------------------------------ compress */

typedef struct {
    int L, Hkv, Hq, d, b, num_blocks;
    const uint16_t *const *kpool; /* [L] -> [num_blocks][Hkv][b][d] */
    const uint16_t *const *vpool;
    uint16_t *const *kout; /* [L] pools written with the compacted rows */
    uint16_t *const *vout;
    const int32_t *tables;
    int stride;
    const int32_t *req_idx;
    int R, N, w;
    double lambda;
    const uint16_t *window_q; /* [L][R][Hq][w][d] */
    const int32_t *dst_table;
    double *scores_out; /* [L][R][Hkv][score_stride] or NULL */
    int32_t *kept_out;  /* [L][R][Hkv][(N-1)b] or NULL */
    const int32_t *unit_len; /* tokens of each request row (prefill) or NULL: T = N*b */
    int score_stride;
    int next_unit;
    pthread_mutex_t mu;
} compress_job;

static size_t slab_off(const compress_job *J, int32_t blk, int h)
{
    return ((size_t)blk * J->Hkv + h) * (size_t)J->b * J->d;
}

static void compress_unit(compress_job *J, int unit)
{
    int h = unit % J->Hkv;
    int l = (unit / J->Hkv) % J->L;
    int r = unit / (J->Hkv * J->L);
    int row = J->req_idx ? J->req_idx[r] : r;
    int b = J->b, d = J->d, N = J->N, w = J->w;
    int T = J->unit_len ? J->unit_len[row] : N * b;
    int C = T - w, G = J->Hq / J->Hkv;
    int n_keep = (N - 1) * b - w;
    const int32_t *src_row = J->tables + (size_t)row * J->stride;
    const int32_t *dst_row = J->dst_table + (size_t)r * N;

    /* gather the unit's K and V rows in token order */
    uint16_t *K = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * d);
    uint16_t *V = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * d);
    for (int t = 0; t < T; ++t) {
        size_t off = slab_off(J, src_row[t / b], h) + (size_t)(t % b) * d;
        memcpy(K + (size_t)t * d, J->kpool[l] + off, sizeof(uint16_t) * d);
        memcpy(V + (size_t)t * d, J->vpool[l] + off, sizeof(uint16_t) * d);
    }
    const uint16_t *Q = J->window_q + (((size_t)l * J->R + r) * J->Hq + (size_t)h * G) * w * d;
    double *imp = (double *)malloc(sizeof(double) * (size_t)T);
    double *red = (double *)malloc(sizeof(double) * (size_t)T);
    double *score = (double *)malloc(sizeof(double) * (size_t)T);
    int32_t *kept = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N - 1) * b);
    zpo_unit_scores(K, Q, T, d, b, w, G, J->lambda, imp, red, score);
    zpo_select(score, C, w, n_keep, kept);

    /* compaction: destination token j <- source token kept[j] */
    for (int j = 0; j < (N - 1) * b; ++j) {
        size_t off = slab_off(J, dst_row[j / b], h) + (size_t)(j % b) * d;
        memcpy(J->kout[l] + off, K + (size_t)kept[j] * d, sizeof(uint16_t) * d);
        memcpy(J->vout[l] + off, V + (size_t)kept[j] * d, sizeof(uint16_t) * d);
    }
    size_t u = ((size_t)l * J->R + r) * J->Hkv + h;
    if (J->scores_out) {
        size_t so = u * (size_t)J->score_stride;
        for (int j = 0; j < C; ++j)
            J->scores_out[so + j] = score[j];
        for (int j = C; j < T; ++j)
            J->scores_out[so + j] = INFINITY;
    }
    if (J->kept_out)
        memcpy(J->kept_out + u * (size_t)(N - 1) * b, kept, sizeof(int32_t) * (size_t)(N - 1) * b);
    free(K);
    free(V);
    free(imp);
    free(red);
    free(score);
    free(kept);
}

static void *compress_worker(void *arg)
{
    compress_job *J = (compress_job *)arg;
    int units = J->R * J->L * J->Hkv;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->mu);
        if (u >= units)
            break;
        compress_unit(J, u);
    }
    return NULL;
}

/* Runs compress_unit on every unit of J over `nthreads` threads. */
static void run_units(compress_job *J, int nthreads)
{
    J->next_unit = 0;
    pthread_mutex_init(&J->mu, NULL);
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i)
        pthread_create(&th[i], NULL, compress_worker, J);
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->mu);
}

/* Whole compression of R requests over all L layers and Hkv heads.
 * kpool/vpool hold the input bytes and are only read; kout/vout receive the
 * compacted rows (they may be the same arrays as kpool/vpool only when no
 * unit reads a block another unit writes, which holds for valid caches since
 * shared blocks are never written; pass copies to be safe).  The integer state
 * (tables, lengths, refcount, free stack) is updated in place, or left as it
 * was when the status is not OK.  Units are spread over `nthreads` threads. */
int zpo_compress(int L, int Hkv, int Hq, int d, int b, int num_blocks,
                 const uint16_t *const *kpool, const uint16_t *const *vpool,
                 uint16_t *const *kout, uint16_t *const *vout,
                 int32_t *tables, int stride, int32_t *lengths, const int32_t *req_idx, int R,
                 int num_rows, const uint16_t *window_q, int N, int w, double lambda,
                 int32_t *free_ids, int32_t *free_count, int32_t *refcount,
                 double *scores_out, int32_t *kept_out, int nthreads)
{
    if (L < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv || d < 1 || w < 1 || w > b)
        return ZPO_ERR_INVALID_ARG;
    int32_t *dst = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1) * N);
    int pops = 0;
    int st = zpo_plan(tables, stride, lengths, req_idx, R, num_rows, N, b, num_blocks, refcount,
                      free_ids, *free_count, dst, &pops);
    if (st != ZPO_OK) {
        free(dst);
        return st;
    }
    compress_job J;
    J.L = L; J.Hkv = Hkv; J.Hq = Hq; J.d = d; J.b = b; J.num_blocks = num_blocks;
    J.kpool = kpool; J.vpool = vpool; J.kout = kout; J.vout = vout;
    J.tables = tables; J.stride = stride; J.req_idx = req_idx;
    J.R = R; J.N = N; J.w = w; J.lambda = lambda; J.window_q = window_q;
    J.dst_table = dst; J.scores_out = scores_out; J.kept_out = kept_out;
    J.unit_len = NULL; J.score_stride = N * b;
    run_units(&J, nthreads);
    *free_count = zpo_commit(tables, stride, lengths, req_idx, R, N, b, refcount, free_ids,
                             *free_count, dst, pops);
    free(dst);
    return ZPO_OK;
}

/* ------------------------------------------------------------- prefill */

/* Destination blocks of a compression at admission [ZP-nl Methodologie §1,
 * §3]: request r holds T_r = lengths[row] >= N*b tokens in blocks
 * 0 .. ceil(T_r/b)-1.  Blocks 0 .. N-1 get destinations by the rule of
 * zpo_plan (refcount 1 at call start: in place; > 1: a fresh target from the
 * top of the free stack, in (request, block) order); blocks N .. are excess
 * and will be released.  Checks: rows in range and distinct,
 * N*b <= T_r <= stride*b, every block of the request valid with refcount >= 1.
 * dst_table[r*N + p] receives the destination of (r, p < N). */
int zpo_plan_prefill(const int32_t *tables, int stride, const int32_t *lengths,
                     const int32_t *req_idx, int R, int num_rows, int N, int b, int num_blocks,
                     const int32_t *refcount, const int32_t *free_ids, int free_count,
                     int32_t *dst_table, int *n_pops)
{
    *n_pops = 0;
    if (R < 0 || N < 2 || b < 2 || stride < N)
        return ZPO_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        if (row < 0 || row >= num_rows)
            return ZPO_ERR_INVALID_ARG;
        for (int r2 = 0; r2 < r; ++r2)
            if ((req_idx ? req_idx[r2] : r2) == row)
                return ZPO_ERR_INVALID_ARG;
        int T = lengths[row];
        if (T < N * b || T > stride * b)
            return ZPO_ERR_INVALID_ARG;
        for (int p = 0; p < (T + b - 1) / b; ++p) {
            int32_t blk = tables[(size_t)row * stride + p];
            if (blk < 0 || blk >= num_blocks || refcount[blk] < 1)
                return ZPO_ERR_INVALID_ARG;
        }
    }
    int taken = 0;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        for (int p = 0; p < N; ++p) {
            int32_t src = tables[(size_t)row * stride + p];
            int32_t target = src;
            if (refcount[src] > 1) {
                if (taken >= free_count)
                    return ZPO_ERR_OUT_OF_BLOCKS;
                target = free_ids[free_count - 1 - taken];
                if (target < 0 || target >= num_blocks || refcount[target] != 0)
                    return ZPO_ERR_DEVICE_CHECK;
                ++taken;
            }
            dst_table[(size_t)r * N + p] = target;
        }
    }
    *n_pops = taken;
    return ZPO_OK;
}

/* Applies a prefill plan [ZP-nl Methodologie §1 "the excess blocks are
 * released", §3; PKV reference counts]: one request after the other, blocks
 * 0 .. N-1 as in zpo_commit, then every excess block N .. ceil(T_r/b)-1 loses
 * one reference, is pushed onto the free stack (after the pops) when that
 * empties it, and its table entry becomes -1.  Lengths become (N-1)*b.
 * Returns the new free count. */
int zpo_commit_prefill(int32_t *tables, int stride, int32_t *lengths, const int32_t *req_idx,
                       int R, int N, int b, int32_t *refcount, int32_t *free_ids, int free_count,
                       const int32_t *dst_table, int n_pops)
{
    int next_free = free_count - n_pops;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        int nblk = (lengths[row] + b - 1) / b;
        for (int p = 0; p < nblk; ++p) {
            int32_t *entry = tables + (size_t)row * stride + p;
            int32_t src = *entry;
            int32_t dst = p < N ? dst_table[(size_t)r * N + p] : -1;
            if (dst == src)
                continue;
            refcount[src] -= 1;
            if (refcount[src] == 0)
                free_ids[next_free++] = src;
            if (dst >= 0)
                refcount[dst] = 1;
            *entry = dst;
        }
        lengths[row] = (N - 1) * b;
    }
    return next_free;
}

/* Compression at admission of requests longer than the budget: per unit the
 * scores of zpo_unit_scores over its T_r tokens (window = the last w), the
 * (N-1)*b - w best candidates kept with the window (zpo_select), compacted
 * into the destinations of zpo_plan_prefill; then zpo_commit_prefill.
 * scores_out: [L][R][Hkv][stride*b] (+inf at window positions, entries at
 * T_r and beyond not written); other arguments as zpo_compress. */
int zpo_compress_prefill(int L, int Hkv, int Hq, int d, int b, int num_blocks,
                         const uint16_t *const *kpool, const uint16_t *const *vpool,
                         uint16_t *const *kout, uint16_t *const *vout, int32_t *tables,
                         int stride, int32_t *lengths, const int32_t *req_idx, int R,
                         int num_rows, const uint16_t *window_q, int N, int w, double lambda,
                         int32_t *free_ids, int32_t *free_count, int32_t *refcount,
                         double *scores_out, int32_t *kept_out, int nthreads)
{
    if (L < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv || d < 1 || w < 1 || w > b)
        return ZPO_ERR_INVALID_ARG;
    int32_t *dst = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1) * N);
    int pops = 0;
    int st = zpo_plan_prefill(tables, stride, lengths, req_idx, R, num_rows, N, b, num_blocks,
                              refcount, free_ids, *free_count, dst, &pops);
    if (st != ZPO_OK) {
        free(dst);
        return st;
    }
    compress_job J;
    J.L = L; J.Hkv = Hkv; J.Hq = Hq; J.d = d; J.b = b; J.num_blocks = num_blocks;
    J.kpool = kpool; J.vpool = vpool; J.kout = kout; J.vout = vout;
    J.tables = tables; J.stride = stride; J.req_idx = req_idx;
    J.R = R; J.N = N; J.w = w; J.lambda = lambda; J.window_q = window_q;
    J.dst_table = dst; J.scores_out = scores_out; J.kept_out = kept_out;
    J.unit_len = lengths; J.score_stride = stride * b;
    run_units(&J, nthreads);
    *free_count = zpo_commit_prefill(tables, stride, lengths, req_idx, R, N, b, refcount,
                                     free_ids, *free_count, dst, pops);
    free(dst);
    return ZPO_OK;
}

/* -------------------------------------------------------------- decode */

/* Paged decode attention [PKV]: for request r and query head hq (kv head
 * hq / (Hq/Hkv)), o = sum_t softmax_t(scale * q.k_t) v_t over the first
 * lengths[r] tokens, token t living in block tables[r*stride + t/b], slot t%b.
 * out64 (nullable) gets the exact double result, out_bf16 its single RNE
 * rounding.  A zero length gives a zero output. */
int zpo_decode_attn(const uint16_t *q, const uint16_t *kpool, const uint16_t *vpool,
                    const int32_t *tables, int stride, const int32_t *lengths, int R, int Hq,
                    int Hkv, int d, int b, int num_blocks, double scale, double *out64,
                    uint16_t *out_bf16)
{
    if (Hq % Hkv)
        return ZPO_ERR_INVALID_ARG;
    int G = Hq / Hkv;
    for (int r = 0; r < R; ++r) {
        int len = lengths[r];
        if (len < 0 || len > stride * b)
            return ZPO_ERR_INVALID_ARG;
        for (int p = 0; p < (len + b - 1) / b; ++p) {
            int32_t blk = tables[(size_t)r * stride + p];
            if (blk < 0 || blk >= num_blocks)
                return ZPO_ERR_INVALID_ARG;
        }
    }
    int maxlen = 1;
    for (int r = 0; r < R; ++r)
        if (lengths[r] > maxlen)
            maxlen = lengths[r];
    double *logit = (double *)malloc(sizeof(double) * (size_t)maxlen);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    for (int r = 0; r < R; ++r) {
        int len = lengths[r];
        for (int hq = 0; hq < Hq; ++hq) {
            int h = hq / G;
            const uint16_t *qv = q + ((size_t)r * Hq + hq) * d;
            double m = -INFINITY;
            for (int t = 0; t < len; ++t) {
                int32_t blk = tables[(size_t)r * stride + t / b];
                const uint16_t *k = kpool + (((size_t)blk * Hkv + h) * b + t % b) * d;
                logit[t] = scale * dot_bf16(qv, k, d);
                if (logit[t] > m)
                    m = logit[t];
            }
            double S = 0.0;
            for (int t = 0; t < len; ++t)
                S += exp(logit[t] - m);
            for (int k = 0; k < d; ++k)
                acc[k] = 0.0;
            for (int t = 0; t < len; ++t) {
                int32_t blk = tables[(size_t)r * stride + t / b];
                const uint16_t *v = vpool + (((size_t)blk * Hkv + h) * b + t % b) * d;
                double p = exp(logit[t] - m) / S;
                for (int k = 0; k < d; ++k)
                    acc[k] += p * zpo_bf16_to_double(v[k]);
            }
            for (int k = 0; k < d; ++k) {
                size_t o = ((size_t)r * Hq + hq) * d + k;
                if (out64)
                    out64[o] = acc[k];
                if (out_bf16)
                    out_bf16[o] = zpo_double_to_bf16(acc[k]);
            }
        }
    }
    free(logit);
    free(acc);
    return ZPO_OK;
}

/* -------------------------------------------------------------- append */

/* Reserves the slot of the next token of each listed request, one request
 * after the other in list order [PKV, "How it works": a new block is taken
 * only when the previous ones are full; a request about to write into a
 * shared block first copies it to a fresh block and drops one reference to
 * the original (copy-on-write); ZP-nl Methodologie §1: a request that holds
 * N_max full blocks is due for compression].
 *
 * For request r (row = req_idx[r], or r), p = lengths[row] is the position of
 * its new token, in block e = p / b, slot p % b:
 *   - table entry e < 0 (only allowed at slot 0): pop a fresh block;
 *   - else, if the block's CURRENT refcount is > 1: pop a fresh block, copy
 *     slots 0 .. p%b - 1 of every layer and kv head (K and V) into it, and
 *     take one reference off the original;
 *   - else the block is written in place.
 * A popped block comes from the top of the free stack and gets refcount 1.
 * Then lengths[row] = p + 1, and when n_max > 0 and p + 1 == n_max * b the
 * row is appended to trigger_rows.  Because refcounts are updated as the
 * loop goes, the last of several writers of one shared block in this call
 * finds it unshared and writes in place.
 *
 * Checked before anything changes (all or nothing): rows in range and
 * distinct, 0 <= p < stride*b, p < n_max*b when n_max > 0, the tail entry a
 * valid block (or negative at slot 0) with at least as many references as
 * rows of this call write into it -> INVALID_ARG; the
 * free stack long enough -> OUT_OF_BLOCKS; a popped id in range with
 * refcount 0, free_count within [0, capacity] -> DEVICE_CHECK.
 * kpool/vpool: L pools [num_blocks][Hkv][b][d], modified in place. */
int zpo_append_slots(int L, int Hkv, int d, int b, int num_blocks, uint16_t *const *kpool,
                     uint16_t *const *vpool, int32_t *tables, int stride, int num_rows,
                     int32_t *lengths, const int32_t *req_idx, int R, int n_max,
                     int32_t *refcount, int32_t *free_ids, int32_t *free_count, int capacity,
                     int32_t *trigger_rows, int32_t *trigger_count)
{
    if (R < 0 || b < 1 || stride < 1 || n_max < 0)
        return ZPO_ERR_INVALID_ARG;
    int fc = *free_count;
    if (fc < 0 || fc > capacity)
        return ZPO_ERR_DEVICE_CHECK;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        if (row < 0 || row >= num_rows)
            return ZPO_ERR_INVALID_ARG;
        for (int r2 = 0; r2 < r; ++r2)
            if ((req_idx ? req_idx[r2] : r2) == row)
                return ZPO_ERR_INVALID_ARG;
        int p = lengths[row];
        if (p < 0 || p >= stride * b || (n_max > 0 && p >= n_max * b))
            return ZPO_ERR_INVALID_ARG;
        int32_t blk = tables[(size_t)row * stride + p / b];
        if (blk >= num_blocks || (blk < 0 && p % b != 0) || (blk >= 0 && refcount[blk] < 1))
            return ZPO_ERR_INVALID_ARG;
        /* every writer of a block holds one of its references */
        int writers = 1;
        for (int r2 = 0; r2 < r && blk >= 0; ++r2) {
            int row2 = req_idx ? req_idx[r2] : r2;
            if (tables[(size_t)row2 * stride + lengths[row2] / b] == blk)
                ++writers;
        }
        if (blk >= 0 && writers > refcount[blk])
            return ZPO_ERR_INVALID_ARG;
    }

    /* dry run on a copy of the refcounts: the pops this call needs */
    int32_t *rc = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_blocks > 0 ? num_blocks : 1));
    memcpy(rc, refcount, sizeof(int32_t) * (size_t)num_blocks);
    int pops = 0;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        int p = lengths[row];
        int32_t blk = tables[(size_t)row * stride + p / b];
        if (blk < 0) {
            ++pops;
        } else if (rc[blk] > 1) {
            rc[blk] -= 1;
            ++pops;
        }
    }
    free(rc);
    if (pops > fc)
        return ZPO_ERR_OUT_OF_BLOCKS;
    for (int k = 0; k < pops; ++k) {
        int32_t t = free_ids[fc - 1 - k];
        if (t < 0 || t >= num_blocks || refcount[t] != 0)
            return ZPO_ERR_DEVICE_CHECK;
    }

    /* the real pass */
    int ntrig = 0;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        int p = lengths[row], e = p / b, slot = p % b;
        int32_t *entry = tables + (size_t)row * stride + e;
        int32_t blk = *entry;
        if (blk < 0 || refcount[blk] > 1) {
            int32_t fresh = free_ids[--fc];
            if (blk >= 0) {
                for (int l = 0; l < L; ++l)
                    for (int h = 0; h < Hkv; ++h) {
                        size_t from = ((size_t)blk * Hkv + h) * (size_t)b * d;
                        size_t to = ((size_t)fresh * Hkv + h) * (size_t)b * d;
                        memcpy(kpool[l] + to, kpool[l] + from, sizeof(uint16_t) * (size_t)slot * d);
                        memcpy(vpool[l] + to, vpool[l] + from, sizeof(uint16_t) * (size_t)slot * d);
                    }
                refcount[blk] -= 1;
            }
            refcount[fresh] = 1;
            *entry = fresh;
        }
        lengths[row] = p + 1;
        if (n_max > 0 && p + 1 == n_max * b) {
            if (trigger_rows)
                trigger_rows[ntrig] = row;
            ++ntrig;
        }
    }
    *free_count = fc;
    if (trigger_count)
        *trigger_count = ntrig;
    return ZPO_OK;
}

/* Writes the new token of each listed request into one layer's pools [PKV]:
 * the token at position p = lengths[row] - 1 (the slot zpo_append_slots
 * reserved) gets k_new[r][h] and v_new[r][h] for every kv head h.
 * k_new, v_new: [R][Hkv][d].  Checked first: rows in range, 1 <= lengths[row]
 * <= stride*b, the block at p / b in range -> INVALID_ARG, nothing written. */
int zpo_append_kv(int Hkv, int d, int b, int num_blocks, uint16_t *kpool, uint16_t *vpool,
                  const int32_t *tables, int stride, int num_rows, const int32_t *lengths,
                  const int32_t *req_idx, int R, const uint16_t *k_new, const uint16_t *v_new)
{
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        if (row < 0 || row >= num_rows)
            return ZPO_ERR_INVALID_ARG;
        int p = lengths[row] - 1;
        if (p < 0 || p >= stride * b)
            return ZPO_ERR_INVALID_ARG;
        int32_t blk = tables[(size_t)row * stride + p / b];
        if (blk < 0 || blk >= num_blocks)
            return ZPO_ERR_INVALID_ARG;
    }
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        int p = lengths[row] - 1;
        int32_t blk = tables[(size_t)row * stride + p / b];
        for (int h = 0; h < Hkv; ++h) {
            size_t to = (((size_t)blk * Hkv + h) * b + p % b) * d;
            size_t from = ((size_t)r * Hkv + h) * d;
            memcpy(kpool + to, k_new + from, sizeof(uint16_t) * (size_t)d);
            memcpy(vpool + to, v_new + from, sizeof(uint16_t) * (size_t)d);
        }
    }
    return ZPO_OK;
}

/* ------------------------------------------------------ alloc / release */

/* Blocks for the first tokens of empty requests [PKV, "How it works": blocks
 * are taken from the pool only as the tokens need them].  Request i (row =
 * req_idx[i], or i) gets counts[i] tokens: entries 0 .. ceil(counts[i]/b)-1
 * of its row become blocks popped from the top of the free stack, in
 * (request, block) order, each with refcount 1; lengths[row] = counts[i].
 * Checked first (all or nothing): rows in range and distinct, lengths[row]
 * == 0, 0 <= counts[i] <= stride*b, the entries to fill < 0 -> INVALID_ARG;
 * enough free blocks -> OUT_OF_BLOCKS; popped ids in range with refcount 0,
 * free_count within [0, capacity] -> DEVICE_CHECK. */
int zpo_alloc_rows(int32_t *tables, int stride, int num_rows, int32_t *lengths,
                   const int32_t *req_idx, int R, const int32_t *counts, int b, int num_blocks,
                   int32_t *refcount, int32_t *free_ids, int32_t *free_count, int capacity)
{
    int fc = *free_count;
    if (R < 0 || b < 1 || stride < 1)
        return ZPO_ERR_INVALID_ARG;
    if (fc < 0 || fc > capacity)
        return ZPO_ERR_DEVICE_CHECK;
    int need = 0;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        if (row < 0 || row >= num_rows)
            return ZPO_ERR_INVALID_ARG;
        for (int r2 = 0; r2 < r; ++r2)
            if ((req_idx ? req_idx[r2] : r2) == row)
                return ZPO_ERR_INVALID_ARG;
        if (lengths[row] != 0 || counts[r] < 0 || counts[r] > stride * b)
            return ZPO_ERR_INVALID_ARG;
        int nb = (counts[r] + b - 1) / b;
        for (int p = 0; p < nb; ++p)
            if (tables[(size_t)row * stride + p] >= 0)
                return ZPO_ERR_INVALID_ARG;
        need += nb;
    }
    if (need > fc)
        return ZPO_ERR_OUT_OF_BLOCKS;
    for (int k = 0; k < need; ++k) {
        int32_t t = free_ids[fc - 1 - k];
        if (t < 0 || t >= num_blocks || refcount[t] != 0)
            return ZPO_ERR_DEVICE_CHECK;
    }
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        int nb = (counts[r] + b - 1) / b;
        for (int p = 0; p < nb; ++p) {
            int32_t t = free_ids[--fc];
            refcount[t] = 1;
            tables[(size_t)row * stride + p] = t;
        }
        lengths[row] = counts[r];
    }
    *free_count = fc;
    return ZPO_OK;
}

/* Every block of finished or preempted requests back to the pool [PKV,
 * "How it works": a block's reference counter counts the tables that point
 * at it; finished requests leave the batch].  Request after request, entry
 * after entry, each entry >= 0 of the row loses one reference of its block,
 * which is pushed onto the free stack when that empties it; the entry becomes
 * -1 and lengths[row] becomes 0.  Checked first (all or nothing): rows in
 * range and distinct, entries < num_blocks, every block referenced by the
 * released rows at most refcount times -> INVALID_ARG; free_count within
 * [0, capacity] and room for the pushes -> DEVICE_CHECK. */
int zpo_release_rows(int32_t *tables, int stride, int num_rows, int32_t *lengths,
                     const int32_t *req_idx, int R, int num_blocks, int32_t *refcount,
                     int32_t *free_ids, int32_t *free_count, int capacity)
{
    int fc = *free_count;
    if (R < 0 || stride < 1)
        return ZPO_ERR_INVALID_ARG;
    if (fc < 0 || fc > capacity)
        return ZPO_ERR_DEVICE_CHECK;
    int32_t *rc = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_blocks > 0 ? num_blocks : 1));
    memcpy(rc, refcount, sizeof(int32_t) * (size_t)num_blocks);
    int pushes = 0, st = ZPO_OK;
    for (int r = 0; r < R && st == ZPO_OK; ++r) {
        int row = req_idx ? req_idx[r] : r;
        if (row < 0 || row >= num_rows) {
            st = ZPO_ERR_INVALID_ARG;
            break;
        }
        for (int r2 = 0; r2 < r; ++r2)
            if ((req_idx ? req_idx[r2] : r2) == row)
                st = ZPO_ERR_INVALID_ARG;
        for (int p = 0; p < stride && st == ZPO_OK; ++p) {
            int32_t blk = tables[(size_t)row * stride + p];
            if (blk < 0)
                continue;
            if (blk >= num_blocks || rc[blk] < 1) {
                st = ZPO_ERR_INVALID_ARG;
                break;
            }
            if (--rc[blk] == 0)
                ++pushes;
        }
    }
    free(rc);
    if (st != ZPO_OK)
        return st;
    if (fc + pushes > capacity)
        return ZPO_ERR_DEVICE_CHECK;
    for (int r = 0; r < R; ++r) {
        int row = req_idx ? req_idx[r] : r;
        for (int p = 0; p < stride; ++p) {
            int32_t *entry = tables + (size_t)row * stride + p;
            if (*entry < 0)
                continue;
            if (--refcount[*entry] == 0)
                free_ids[fc++] = *entry;
            *entry = -1;
        }
        lengths[row] = 0;
    }
    *free_count = fc;
    return ZPO_OK;
}

/* Forks requests [PKV, "How it works": parallel samples share the prompt's
 * blocks, each block's reference counter counts the tables pointing at it]:
 * pair i makes row dst[i] (empty: length 0, every entry < 0) a copy of row
 * src[i] -- the same table entries (a reserved empty block included) and the
 * same length -- and every block entry gains one reference.  Checked first
 * (all or nothing): rows in range, destinations distinct and none of them a
 * source of the same call, destinations empty, source entries < num_blocks
 * with refcount >= 1 -> INVALID_ARG. */
int zpo_fork_rows(int32_t *tables, int stride, int num_rows, int32_t *lengths,
                  const int32_t *src, const int32_t *dst, int n, int num_blocks,
                  int32_t *refcount)
{
    if (n < 0 || stride < 1)
        return ZPO_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        int s = src[i], d = dst[i];
        if (s < 0 || s >= num_rows || d < 0 || d >= num_rows || s == d)
            return ZPO_ERR_INVALID_ARG;
        for (int k = 0; k < n; ++k)
            if ((k != i && dst[k] == d) || src[k] == d)
                return ZPO_ERR_INVALID_ARG;
        if (lengths[d] != 0)
            return ZPO_ERR_INVALID_ARG;
        for (int p = 0; p < stride; ++p) {
            if (tables[(size_t)d * stride + p] >= 0)
                return ZPO_ERR_INVALID_ARG;
            int32_t blk = tables[(size_t)s * stride + p];
            if (blk >= num_blocks || (blk >= 0 && refcount[blk] < 1))
                return ZPO_ERR_INVALID_ARG;
        }
    }
    for (int i = 0; i < n; ++i) {
        int s = src[i], d = dst[i];
        for (int p = 0; p < stride; ++p) {
            int32_t blk = tables[(size_t)s * stride + p];
            tables[(size_t)d * stride + p] = blk;
            if (blk >= 0)
                refcount[blk] += 1;
        }
        lengths[d] = lengths[s];
    }
    return ZPO_OK;
}
