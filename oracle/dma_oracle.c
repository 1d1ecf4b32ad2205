/*
 * dma_oracle.c -- plain, slow, fp64 CPU oracle for dynamic-mask sparse attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
 * baseline call this code.  It shares nothing with the CUDA library: no header,
 * no helper, no table.  It is written to be checked by eye against the method:
 *
 *   Dynamic Mask Attention summary (lsdiaocha.cn, "HKUST-GZ / BAAI DMA"):
 *     §四  content-aware dynamic mask: every key gets an importance score from its
 *          value vector, through a learnable sampling weight and a per-head gate;
 *          each head gets its own mask; masked positions are skipped outright.
 *     §五  dynamic weight delta = exp(tau(v Delta) * A), tau non-negative;
 *          combine with the causal mask, keep the top-k historical positions at
 *          every time step, set the rest to -inf; skipped positions have weight
 *          exactly 0, so skipping equals the full masked computation.
 *
 * Readings taken where the page is silent (each is a line of the design notes):
 *   - tau = softplus, Delta = one weight vector w_h per KV head applied to that
 *     head's own value row, A = one scalar per KV head (default 1).
 *   - multiplying an attention weight by delta equals adding log(delta) =
 *     A * softplus(v . w_h) to its logit, so the score is added as a bias and
 *     ranking by it ranks by delta.
 *   - ranking uses the score rounded to fp32 (the kernel's precision); ties go
 *     to the lower key index; the bias added to the logit is the fp64 score.
 *   - row-wise mode: row i keeps the min(w, i+1) best keys among 0..i;
 *     global mode: row i keeps the keys j <= i among the w best of all keys.
 *   - the kept set of row i is that top set united with the window
 *     {i-window+1 .. i}.
 *   - block mode (block > 1): a block's score is the max of its keys' scores;
 *     row i ranks only complete blocks (last key <= i) and keeps the best
 *     floor(w/block) of them; a kept block brings all of its keys.
 *
 * Every key's top-set membership is an interval of rows: key j is in the top
 * set of rows lo_j <= i < expiry_j, lo_j = j for tokens and the block's last
 * key for blocks.  "Never kept" is written as expiry_j = min(lo_j, S).
 *
 * Layouts: Q [B][S][H][D]; K, V [B][S][Hkv][D]; W [Hkv][D]; scores and expiry
 * [B][Hkv][S].  Query head hq reads KV head hq / (H / Hkv).
 * Inputs arrive as fp32 (bf16 widens to fp32 exactly); all arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ROWWISE 0
#define ORACLE_GLOBAL 1

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- scoring -- */

/* tau: softplus(x) = log(1 + e^x), written in the overflow-safe form. */
static double softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* s[b,h,j] = A_h * softplus(<V[b,j,h,:], W[h,:]>) for keys key_begin <= j < key_end.
 * (DMA summary §五: the dynamic weight's exponent tau(v Delta) * A.) */
void oracle_score(const float* V, const float* W, const float* A, int B, int S, int Hkv, int D,
                  int key_begin, int key_end, double* scores)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h)
            for (int j = key_begin; j < key_end; ++j) {
                const float* v = V + (((int64_t)b * S + j) * Hkv + h) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += (double)v[d] * (double)W[h * D + d];
                double a = A ? (double)A[h] : 1.0;
                scores[((int64_t)b * Hkv + h) * S + j] = a * softplus(dot);
            }
}

/* -------------------------------------------------------------- selection -- */

/* The value a key is ranked by: its score rounded to fp32; NaN ranks lowest. */
static float rank_value(double s)
{
    float f = (float)s;
    return isnan(f) ? -INFINITY : f;
}

/* Total order: a beats b iff a's value is larger, or equal and a's index lower. */
static int beats(const float* val, int a, int b)
{
    return val[a] > val[b] || (val[a] == val[b] && a < b);
}

/* Binary min-heap whose root is the WORST member under the total order. */
typedef struct {
    const float* val;
    int* item;
    int n;
} worst_heap;

static void heap_swap(worst_heap* hp, int x, int y)
{
    int t = hp->item[x];
    hp->item[x] = hp->item[y];
    hp->item[y] = t;
}

static void heap_push(worst_heap* hp, int key)
{
    int c = hp->n++;
    hp->item[c] = key;
    while (c > 0) {
        int p = (c - 1) / 2;
        if (beats(hp->val, hp->item[p], hp->item[c])) {  /* parent better: child is worse, rises */
            heap_swap(hp, p, c);
            c = p;
        } else {
            break;
        }
    }
}

static int heap_pop_worst(worst_heap* hp)
{
    int top = hp->item[0];
    hp->item[0] = hp->item[--hp->n];
    int p = 0;
    for (;;) {
        int l = 2 * p + 1, r = l + 1, m = p;
        if (l < hp->n && beats(hp->val, hp->item[m], hp->item[l])) m = l;
        if (r < hp->n && beats(hp->val, hp->item[m], hp->item[r])) m = r;
        if (m == p) break;
        heap_swap(hp, p, m);
        p = m;
    }
    return top;
}

/* Row-wise top-k over a stream of n candidates (DMA summary §五: top-k at every
 * time step over the causal history).  Candidate c enters at step c; whenever
 * the kept set exceeds k, the worst member leaves and its leaving step is
 * recorded.  out_end[c] = step at which c left (c itself if it never entered),
 * or n if it was still kept after the last step. */
static void rowwise_topk_stream(const float* val, int n, int k, int* heap_buf, int* out_end)
{
    worst_heap hp = {val, heap_buf, 0};
    for (int c = 0; c < n; ++c) out_end[c] = n;
    for (int c = 0; c < n; ++c) {
        heap_push(&hp, c);
        if (hp.n > k) {
            int gone = heap_pop_worst(&hp);
            out_end[gone] = c;
        }
    }
}

static const float* sort_val;  /* comparator context for qsort (single-threaded use only) */
static int cmp_best_first(const void* pa, const void* pb)
{
    int a = *(const int*)pa, b = *(const int*)pb;
    if (beats(sort_val, a, b)) return -1;
    if (beats(sort_val, b, a)) return 1;
    return 0;
}

/* Global mode: winners are the k best of all n candidates.  out_win[c] = 1/0. */
static void global_topk(const float* val, int n, int k, int* order, int* out_win)
{
    for (int c = 0; c < n; ++c) order[c] = c;
#pragma omp critical(oracle_qsort)
    {
        sort_val = val;
        qsort(order, (size_t)n, sizeof(int), cmp_best_first);
    }
    for (int c = 0; c < n; ++c) out_win[c] = 0;
    for (int r = 0; r < n && r < k; ++r) out_win[order[r]] = 1;
}

/* Selection for one (batch, KV head) segment of S keys.
 * block == 1: token units.  block > 1: complete blocks of `block` keys.
 * Writes expiry[j] for every key j (see the header for its meaning). */
static void select_segment(const double* score, int S, int w, int block, int mode, int32_t* expiry)
{
    if (block <= 1) {
        float* val = (float*)calloc((size_t)(S > 0 ? S : 1), sizeof(float));
        int* buf = (int*)malloc(sizeof(int) * (size_t)(S + 1));
        int* res = (int*)malloc(sizeof(int) * (size_t)(S > 0 ? S : 1));
        for (int j = 0; j < S; ++j) val[j] = rank_value(score[j]);
        if (mode == ORACLE_ROWWISE) {
            rowwise_topk_stream(val, S, w, buf, res);
            for (int j = 0; j < S; ++j) expiry[j] = res[j];   /* left at row res[j]; == j if never */
        } else {
            global_topk(val, S, w, buf, res);
            for (int j = 0; j < S; ++j) expiry[j] = res[j] ? S : j;
        }
        free(val);
        free(buf);
        free(res);
        return;
    }
    /* Block units: block beta = keys [beta*block, beta*block + block).  It is
     * complete from row beta*block + block - 1 on.  Block-row r (r = 0, 1, ...)
     * is the set of rows that see exactly r + 1 complete blocks. */
    int nb = S / block;            /* complete blocks */
    int wb = w / block;            /* block budget */
    float* bval = (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
    int* buf = (int*)malloc(sizeof(int) * (size_t)(nb + 1));
    int* res = (int*)malloc(sizeof(int) * (size_t)(nb > 0 ? nb : 1));
    for (int bk = 0; bk < nb; ++bk) {
        float m = -INFINITY;
        for (int t = 0; t < block; ++t) {
            float v = rank_value(score[bk * block + t]);
            if (v > m) m = v;
        }
        bval[bk] = m;
    }
    if (mode == ORACLE_ROWWISE)
        rowwise_topk_stream(bval, nb, wb, buf, res);     /* res = block-row at which it left, nb if never */
    else
        global_topk(bval, nb, wb, buf, res);
    for (int j = 0; j < S; ++j) {
        int bk = j / block;
        int lo = bk * block + block - 1;
        int never = lo < S ? lo : S;
        if (bk >= nb) {
            expiry[j] = never;
            continue;
        }
        if (mode == ORACLE_ROWWISE) {
            if (res[bk] >= nb) {
                expiry[j] = S;                          /* still kept at the last row */
            } else {
                /* left at block-row E: kept for block-rows bk..E-1, i.e. rows
                 * up to (E+1)*block - 2, so the first row without it is E*block + block - 1. */
                int hi = res[bk] * block + block - 1;
                expiry[j] = hi > lo ? hi : never;
            }
        } else {
            expiry[j] = res[bk] ? S : never;
        }
    }
    free(bval);
    free(buf);
    free(res);
}

/* Selection for all B*Hkv segments.  scores, expiry: [B][Hkv][S]. */
void oracle_select(const double* scores, int B, int Hkv, int S, int w, int block, int mode, int32_t* expiry)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int seg = 0; seg < B * Hkv; ++seg)
        select_segment(scores + (int64_t)seg * S, S, w, block, mode, expiry + (int64_t)seg * S);
}

/* -------------------------------------------------------------- attention -- */

static int top_lo(int j, int block) { return block <= 1 ? j : (j / block) * block + block - 1; }

/* Is key j in the kept set of row i?  Top set by the expiry interval, united
 * with the local window {i-window+1 .. i}; never a key after the row. */
static int is_kept(int i, int j, int32_t expiry_j, int window, int block)
{
    if (j > i) return 0;
    if (j > i - window) return 1;
    return top_lo(j, block) <= i && i < expiry_j;
}

/* Dense masked softmax attention for one query row (DMA summary §五: masked
 * positions get -inf, hence weight exactly 0; the score is the logit's bias).
 * q [D]; K, V rows at stride kv_stride; x_buf holds i+1 logits. */
static void attend_row(const float* q, const float* K, const float* V, int64_t kv_stride, const double* score,
                       const int32_t* expiry, int i, int D, int window, int block, double scale, double* x_buf,
                       double* o, double* lse)
{
    double m = -INFINITY;
    for (int j = 0; j <= i; ++j) {
        if (!is_kept(i, j, expiry[j], window, block)) {
            x_buf[j] = -INFINITY;
            continue;
        }
        const float* k = K + (int64_t)j * kv_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)q[d] * (double)k[d];
        x_buf[j] = scale * dot + score[j];
        if (x_buf[j] > m) m = x_buf[j];
    }
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == -INFINITY) {  /* empty kept set: zero output, lse = -inf */
        *lse = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int j = 0; j <= i; ++j) {
        if (x_buf[j] == -INFINITY) continue;
        double p = exp(x_buf[j] - m);
        sum += p;
        const float* v = V + (int64_t)j * kv_stride;
        for (int d = 0; d < D; ++d) o[d] += p * (double)v[d];
    }
    for (int d = 0; d < D; ++d) o[d] /= sum;
    *lse = m + log(sum);
}

/* Prefill attention for the listed rows of every (batch, query head).
 * rows [n_rows]; O [B][n_rows][H][D]; lse [B][H][n_rows] (may be NULL). */
void oracle_attend_rows(const float* Q, const float* K, const float* V, const double* scores,
                        const int32_t* expiry, int B, int S, int H, int Hkv, int D, int window, int block,
                        double scale, int n_rows, const int32_t* rows, double* O, double* lse)
{
    int G = H / Hkv;
#pragma omp parallel
    {
        double* x_buf = (double*)malloc(sizeof(double) * (size_t)S);
#pragma omp for collapse(3) schedule(dynamic, 4)
        for (int b = 0; b < B; ++b)
            for (int hq = 0; hq < H; ++hq)
                for (int r = 0; r < n_rows; ++r) {
                    int i = rows[r];
                    int h = hq / G;
                    const float* q = Q + (((int64_t)b * S + i) * H + hq) * D;
                    const float* Kh = K + ((int64_t)b * S * Hkv + h) * D;
                    const float* Vh = V + ((int64_t)b * S * Hkv + h) * D;
                    const double* sc = scores + ((int64_t)b * Hkv + h) * S;
                    const int32_t* ex = expiry + ((int64_t)b * Hkv + h) * S;
                    double l;
                    attend_row(q, Kh, Vh, (int64_t)Hkv * D, sc, ex, i, D, window, block, scale, x_buf,
                               O + (((int64_t)b * n_rows + r) * H + hq) * D, &l);
                    if (lse) lse[((int64_t)b * H + hq) * n_rows + r] = l;
                }
        free(x_buf);
    }
}

/* Decode: one new query per sequence at position L-1 of a cache of length
 * L = cache_len[b].  Selection runs over that sequence's first L scores, and the
 * row is the last prefill row of a sequence of length L (same rule in training
 * and inference).  q [B][H][D]; Kc, Vc [B][Lmax][Hkv][D]; scores [B][Hkv][Lmax];
 * o [B][H][D]; lse [B][H] (may be NULL). */
void oracle_decode(const float* q, const float* Kc, const float* Vc, const int32_t* cache_len,
                   const double* scores, int B, int Lmax, int H, int Hkv, int D, int w, int window, int block,
                   int mode, double scale, double* o, double* lse)
{
    int G = H / Hkv;
#pragma omp parallel
    {
        double* x_buf = (double*)malloc(sizeof(double) * (size_t)Lmax);
        int32_t* ex = (int32_t*)malloc(sizeof(int32_t) * (size_t)Lmax);
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hkv; ++h) {
                int L = cache_len[b];
                const double* sc = scores + ((int64_t)b * Hkv + h) * Lmax;
                select_segment(sc, L, w, block, mode, ex);
                for (int g = 0; g < G; ++g) {
                    int hq = h * G + g;
                    double l;
                    attend_row(q + ((int64_t)b * H + hq) * D, Kc + ((int64_t)b * Lmax * Hkv + h) * D,
                               Vc + ((int64_t)b * Lmax * Hkv + h) * D, (int64_t)Hkv * D, sc, ex, L - 1, D, window,
                               block, scale, x_buf, o + ((int64_t)b * H + hq) * D, &l);
                    if (lse) lse[(int64_t)b * H + hq] = l;
                }
            }
        free(x_buf);
        free(ex);
    }
}

/* ------------------------------------------------------------- backward -- */
/*
 * Gradients of a loss L through the forward above, given dO = dL/dO (DMA
 * summary §四/§五/§七: the same mask in training and inference, and it is fully
 * differentiable in the kept positions; the top-k selection itself is piecewise
 * constant, so no gradient passes through the choice of keys, and a skipped
 * position -- weight exactly 0 -- receives exactly zero gradient).
 *
 * For row i (query head hq of KV head h) with kept set K_i:
 *   x_ij  = scale * <Q_i, K_j> + s_j          p_ij = exp(x_ij - lse_i) over K_i,
 *   lse_i = log sum_{j in K_i} exp(x_ij)      (the softmax of the forward)
 *   dP_ij = <dO_i, V_j>                       D_i  = sum_{j in K_i} p_ij dP_ij
 *   dx_ij = p_ij (dP_ij - D_i)                (softmax backward)
 *   dQ_i  = scale * sum_{j in K_i} dx_ij K_j
 *   dK_j  = scale * sum_{i : j in K_i} dx_ij Q_i
 *   dV_j  = sum_{i : j in K_i} p_ij dO_i
 *   ds_j  = sum_{i : j in K_i} dx_ij          (the score is the logit's bias)
 * where the key-side sums run over the rows of every query head of the group.
 * Computed in three phases, each a plain loop over independent outputs: the row
 * statistics (lse_i, D_i) of every row, then dQ row by row, then dK, dV and ds
 * key by key (each key's sum walks the rows i >= j and keeps those whose kept
 * set holds j).  Each output is written by one loop iteration, so the result
 * does not depend on the number of threads.
 *
 * Layouts as the forward; dQ [B][S][H][D], dK and dV [B][S][Hkv][D], ds
 * [B][Hkv][S], all fp64.  Segment seg = b * Hkv + h; seg_only < 0 means every
 * segment.  rows (n_rows entries, ascending) limits dQ to those rows and keys
 * (n_keys) limits dK, dV and ds to those keys; NULL means all.  Outputs not
 * computed are left as they were.
 */
static double kept_logit(const float* q, const float* k, double s, int D, double scale)
{
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += (double)q[d] * (double)k[d];
    return scale * dot + s;
}

static double dot_f(const float* a, const float* b, int D)
{
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += (double)a[d] * (double)b[d];
    return dot;
}

void oracle_attend_backward(const float* Q, const float* K, const float* V, const double* scores,
                            const int32_t* expiry, const float* dO, int B, int S, int H, int Hkv, int D, int window,
                            int block, double scale, int seg_only, const int32_t* rows, int n_rows,
                            const int32_t* keys, int n_keys, double* dQ, double* dK, double* dV, double* ds)
{
    const int G = H / Hkv;
    const int64_t kv_stride = (int64_t)Hkv * D;
    const int nseg = B * Hkv;
    const int nr = rows ? n_rows : S, nk = keys ? n_keys : S;
    /* row statistics of every row of the selected segments: lse_i and D_i */
    double* lse = (double*)malloc(sizeof(double) * (size_t)B * H * S);
    double* Dr = (double*)malloc(sizeof(double) * (size_t)B * H * S);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t t = 0; t < (int64_t)nseg * G * S; ++t) {
        const int i = (int)(t % S), g = (int)((t / S) % G), seg = (int)(t / ((int64_t)S * G));
        if (seg_only >= 0 && seg != seg_only) continue;
        const int b = seg / Hkv, h = seg % Hkv, hq = h * G + g;
        const int64_t qo = (((int64_t)b * S + i) * H + hq) * D, ro = ((int64_t)b * H + hq) * S + i;
        const float* Kh = K + ((int64_t)b * S * Hkv + h) * D;
        const float* Vh = V + ((int64_t)b * S * Hkv + h) * D;
        const double* sc = scores + (int64_t)seg * S;
        const int32_t* ex = expiry + (int64_t)seg * S;
        double m = -INFINITY;
        for (int j = 0; j <= i; ++j) {
            if (!is_kept(i, j, ex[j], window, block)) continue;
            const double x = kept_logit(Q + qo, Kh + (int64_t)j * kv_stride, sc[j], D, scale);
            if (x > m) m = x;
        }
        if (m == -INFINITY) { /* empty kept set: the output is the constant 0 */
            lse[ro] = -INFINITY;
            Dr[ro] = 0.0;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j <= i; ++j)
            if (is_kept(i, j, ex[j], window, block))
                sum += exp(kept_logit(Q + qo, Kh + (int64_t)j * kv_stride, sc[j], D, scale) - m);
        const double l = m + log(sum);
        double Di = 0.0;
        for (int j = 0; j <= i; ++j) {
            if (!is_kept(i, j, ex[j], window, block)) continue;
            const double p = exp(kept_logit(Q + qo, Kh + (int64_t)j * kv_stride, sc[j], D, scale) - l);
            Di += p * dot_f(dO + qo, Vh + (int64_t)j * kv_stride, D);
        }
        lse[ro] = l;
        Dr[ro] = Di;
    }
    /* dQ, row by row */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < (int64_t)nseg * G * nr; ++t) {
        const int ri = (int)(t % nr), g = (int)((t / nr) % G), seg = (int)(t / ((int64_t)nr * G));
        if (seg_only >= 0 && seg != seg_only) continue;
        const int i = rows ? rows[ri] : ri;
        const int b = seg / Hkv, h = seg % Hkv, hq = h * G + g;
        const int64_t qo = (((int64_t)b * S + i) * H + hq) * D, ro = ((int64_t)b * H + hq) * S + i;
        const float* Kh = K + ((int64_t)b * S * Hkv + h) * D;
        const float* Vh = V + ((int64_t)b * S * Hkv + h) * D;
        const double* sc = scores + (int64_t)seg * S;
        const int32_t* ex = expiry + (int64_t)seg * S;
        double* dq = dQ + qo;
        for (int d = 0; d < D; ++d) dq[d] = 0.0;
        if (lse[ro] == -INFINITY) continue;
        for (int j = 0; j <= i; ++j) {
            if (!is_kept(i, j, ex[j], window, block)) continue;
            const float* k = Kh + (int64_t)j * kv_stride;
            const double p = exp(kept_logit(Q + qo, k, sc[j], D, scale) - lse[ro]);
            const double dx = p * (dot_f(dO + qo, Vh + (int64_t)j * kv_stride, D) - Dr[ro]);
            for (int d = 0; d < D; ++d) dq[d] += scale * dx * (double)k[d];
        }
    }
    /* dK, dV and ds, key by key */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < (int64_t)nseg * nk; ++t) {
        const int kj = (int)(t % nk), seg = (int)(t / nk);
        if (seg_only >= 0 && seg != seg_only) continue;
        const int j = keys ? keys[kj] : kj;
        const int b = seg / Hkv, h = seg % Hkv;
        const int64_t ko = (((int64_t)b * S + j) * Hkv + h) * D;
        const double* sc = scores + (int64_t)seg * S;
        const int32_t* ex = expiry + (int64_t)seg * S;
        double* dk = dK + ko;
        double* dv = dV + ko;
        double dsj = 0.0;
        for (int d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
        for (int g = 0; g < G; ++g) {
            const int hq = h * G + g;
            for (int i = j; i < S; ++i) {
                if (!is_kept(i, j, ex[j], window, block)) continue;
                const int64_t qo = (((int64_t)b * S + i) * H + hq) * D, ro = ((int64_t)b * H + hq) * S + i;
                const double p = exp(kept_logit(Q + qo, K + ko, sc[j], D, scale) - lse[ro]);
                const double dx = p * (dot_f(dO + qo, V + ko, D) - Dr[ro]);
                for (int d = 0; d < D; ++d) {
                    dk[d] += scale * dx * (double)Q[qo + d];
                    dv[d] += p * (double)dO[qo + d];
                }
                dsj += dx;
            }
        }
        ds[(int64_t)seg * S + j] = dsj;
    }
    free(lse);
    free(Dr);
}

/* Through the score s_j = A_h * softplus(u_j), u_j = <V_j, W_h> (DMA summary
 * §五), given ds = dL/ds:
 *   dA_h  = sum_j ds_j softplus(u_j)
 *   du_j  = ds_j A_h sigmoid(u_j)             (softplus' = sigmoid)
 *   dW_h  = sum_j du_j V_j                    dV_j += du_j W_h
 * over every batch.  dV_add [B][S][Hkv][D] is added to (the value rows also
 * feed the attention); dW [Hkv][D] and dA [Hkv] are overwritten. */
static double sigmoid(double x) { return x >= 0 ? 1.0 / (1.0 + exp(-x)) : exp(x) / (1.0 + exp(x)); }

void oracle_score_backward(const float* V, const float* W, const float* A, const double* ds, int B, int S, int Hkv,
                           int D, double* dV_add, double* dW, double* dA)
{
#pragma omp parallel for schedule(static)
    for (int h = 0; h < Hkv; ++h) {
        double a = A ? (double)A[h] : 1.0;
        double da = 0.0;
        for (int d = 0; d < D; ++d) dW[h * D + d] = 0.0;
        for (int b = 0; b < B; ++b)
            for (int j = 0; j < S; ++j) {
                const float* v = V + (((int64_t)b * S + j) * Hkv + h) * D;
                double u = 0.0;
                for (int d = 0; d < D; ++d) u += (double)v[d] * (double)W[h * D + d];
                double g = ds[((int64_t)b * Hkv + h) * S + j];
                da += g * softplus(u);
                double du = g * a * sigmoid(u);
                for (int d = 0; d < D; ++d) {
                    dW[h * D + d] += du * (double)v[d];
                    dV_add[(((int64_t)b * S + j) * Hkv + h) * D + d] += du * (double)W[h * D + d];
                }
            }
        dA[h] = da;
    }
}
