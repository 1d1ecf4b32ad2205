/*
 * dma.h -- C ABI of the B300 (sm_103a) dynamic-mask sparse attention library.
 *
 * The method (Dynamic Mask Attention summary, lsdiaocha.cn, §四 and §五): every
 * key gets a content-derived importance score per KV head; at every time step
 * each head keeps the top-w historical keys (causal mask first, then top-k, the
 * rest set to -inf), optionally united with a local window; softmax attention
 * runs over the kept keys only, with the score added to the logit as a bias.
 * Skipped positions would have weight exactly 0, so skipping them computes the
 * same result as the full masked attention.
 *
 * Four calls make the forward hot path:
 *   dma_score_keys           s[b,h,j] = A_h * softplus(<V[b,j,h,:], W[h,:]>)
 *                            (dma_score_keys_bias: also the bias s or exp(s))
 *   dma_select_topk          per-key top-set intervals + per-query-tile key lists
 *                            (dma_select_topk_heads: a budget per KV head)
 *   dma_sparse_attn_prefill  masked softmax attention over the kept keys
 *   dma_sparse_attn_decode   the same for one new query row per sequence
 * plus page-granular decode over a paged KV cache (dma_score_keys_paged,
 * dma_select_pages, dma_sparse_attn_decode_paged),
 * the NSA-style three-branch fusion (dma_nsa_compress, dma_nsa_kept_pattern,
 * dma_nsa_combine),
 * and two for the backward pass (training through the same mask):
 *   dma_sparse_attn_prefill_backward  dQ, dK, dV and ds over the kept pairs
 *   dma_score_keys_backward           ds -> dW, dA and the score's share of dV
 *                                     (dma_score_keys_backward_bias: either bias form)
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates and frees every buffer; the library never
 *     allocates device memory.  Pointers named "device" must be device memory
 *     of the current CUDA device; nothing is read on the host except scalars.
 *   - Layout: dense, row-major, innermost dimension last, as written beside
 *     each argument.  Q [B][S][H][D]; K, V [B][S][Hkv][D]; query head hq uses
 *     KV head hq / (H / Hkv).  Every tensor base must be 16-byte aligned.
 *   - Supported shapes: D in {64, 128}; H % Hkv == 0; S >= 1; w >= 0;
 *     window >= 0.  dtype DMA_F32 or DMA_BF16 (round-to-nearest-even output).
 *   - Streams: every call only enqueues work on `stream` (NULL = the legacy
 *     default stream) and never synchronises, except dma_get_device_status.
 *   - Errors: argument errors return DMA_ERR_INVALID_ARG / DMA_ERR_UNSUPPORTED /
 *     DMA_ERR_WORKSPACE before anything is launched; a failed launch returns
 *     DMA_ERR_CUDA.  dma_last_error_message() gives a per-thread detail string.
 *     Conditions found on the device (a bounded wait that ran out, an internal
 *     capacity check) set a device status word read by dma_get_device_status.
 *   - Outputs alias no input, except where a call says so (dma_nsa_combine's O may
 *     be one of its branch outputs).
 */
#ifndef DMA_H_
#define DMA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dma_stream_t; /* a cudaStream_t */

typedef enum {
    DMA_OK = 0,
    DMA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned base, mismatched layout */
    DMA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (e.g. D = 96) */
    DMA_ERR_WORKSPACE = 3,    /* workspace pointer null or smaller than the size query says */
    DMA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    DMA_ERR_TIMEOUT = 5,      /* device status: a bounded wait inside a kernel ran out */
    DMA_ERR_DEVICE_CHECK = 6  /* device status: an internal capacity/bounds check failed */
} dma_status_t;

typedef enum { DMA_F32 = 0, DMA_BF16 = 1 } dma_dtype_t;

/* Row-wise: row i keeps the min(w, i+1) best keys among 0..i (top-k at every
 * time step, DMA summary §五).  Global: row i keeps the keys j <= i that are
 * among the w best of all S keys.  Both coincide on the last row. */
typedef enum { DMA_SEL_ROWWISE = 0, DMA_SEL_GLOBAL = 1 } dma_sel_mode_t;

/* FULL recomputes everything from the score array.  UPDATE (decode) merges the
 * newest key of each sequence into the top set of the previous row. */
typedef enum { DMA_SEL_FULL = 0, DMA_SEL_UPDATE = 1 } dma_sel_op_t;

/* What the logits get as their bias: LOG adds s = log delta (the default of
 * every call taking `scores`); EXP adds the dynamic weight delta = exp(s)
 * itself.  Either way the selection ranks s. */
typedef enum { DMA_BIAS_LOG = 0, DMA_BIAS_EXP = 1 } dma_bias_form_t;

/* Rows per query tile of the per-tile key lists. */
#define DMA_Q_TILE 128

/*
 * The kept-key representation.  Geometry fields are filled by dma_kept_layout;
 * the caller then allocates the arrays (device memory) and sets the pointers.
 *
 * Every key j has one top-set interval: j is in the top set of rows
 * lo_j <= i < expiry[j], where lo_j = j for token units (block == 1) and the
 * last key of j's block, (j / block) * block + block - 1, for block units.
 * expiry[j] <= lo_j means the key never enters the top set (it is then
 * min(lo_j, S)); expiry[j] == S means it is still kept at the last row.
 * The kept set of row i is that top set united with {i-window+1 .. i}.
 */
typedef struct {
    /* geometry (written by dma_kept_layout, checked by every consumer) */
    int32_t B, Hkv, S, w, window, block, mode;
    int32_t q_tile;       /* DMA_Q_TILE */
    int32_t n_qt;         /* ceil(S / q_tile) query tiles */
    int32_t cap;          /* entries of idx per (b, h) = S */
    int32_t top_cap;      /* entries of top_idx per (b, h): the top-set size bound */
    int32_t tile_stride;  /* entries of tile_idx per (b, h, tile) */
    int32_t bitmap_words; /* 32-bit words of bitmap per (b, h, tile) = ceil(S / 64 / 32) */
    /* caller-owned device arrays */
    int32_t* expiry;      /* [B][Hkv][S]                       required (FULL) */
    int32_t* idx;         /* [B][Hkv][cap]  keys ever kept by the top rule, ascending; required (FULL) */
    int32_t* count;       /* [B][Hkv]       entries used in idx; required (FULL) */
    int32_t* top_idx;     /* [B][Hkv][top_cap] top set of the last row, ascending; nullable (FULL),
                                            required (UPDATE and decode) */
    int32_t* top_count;   /* [B][Hkv]                           with top_idx */
    int32_t* tile_cnt;    /* [B][Hkv][n_qt]                     required by prefill */
    int32_t* tile_idx;    /* [B][Hkv][n_qt][tile_stride]: keys j <= q0 - window (all j <= q1 when
                                            window == 0) whose top interval meets the tile's rows
                                            [q0, q1]: first the keys in the top set of every row of
                                            the tile, then the others; each group in rank order
                                            (score descending, ties to the lower index; block
                                            units: block rank, then the block's keys ascending);
                                            the window band (q0-window, q1] is implicit */
    uint32_t* bitmap;     /* [B][Hkv][n_qt][bitmap_words]: bit (tile, 64-key block) set iff some key
                                            of the block is kept by some row of the tile; nullable */
} dma_kept_t;

/* ---------------------------------------------------------------- scoring --
 * DMA summary §五, dynamic weight delta = exp(tau(v Delta) * A): with tau =
 * softplus, Delta a per-KV-head vector W[h] and A a per-KV-head gate, the log
 * weight s = A_h * softplus(v . W[h]) is the additive logit bias and the
 * ranking key.
 *   V       device [B][S][Hkv][D] (dtype dt)   value rows
 *   W       device [Hkv][D] fp32               per-KV-head sampling weights
 *   A       device [Hkv] fp32 or NULL (= 1)    per-KV-head gate
 *   scores  device [B][Hkv][S] fp32            written for key_begin <= j < key_end only
 * 0 <= key_begin <= key_end <= S.  key_begin == key_end is a no-op.  Hkv <= 128
 * (DMA_ERR_UNSUPPORTED otherwise, before any launch).
 */
dma_status_t dma_score_keys(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin,
                            int key_end, const float* W, const float* A, float* scores, dma_stream_t stream);

/* dma_score_keys plus the bias array the attention calls take in place of the
 * scores (DMA summary §五 writes the weight as delta = exp(tau(v Delta) * A)):
 *   form    DMA_BIAS_LOG: bias = s (a copy of scores);
 *           DMA_BIAS_EXP: bias = exp(s) in fp32 (+inf where s > about 88.7)
 *   scores  device [B][Hkv][S] fp32   the ranking key, for dma_select_topk
 *   bias    device [B][Hkv][S] fp32   non-NULL, not scores; for the attention
 *           calls (prefill, decode, backward) as their `scores` argument
 * Both written for key_begin <= j < key_end only.  exp is increasing, so
 * ranking s keeps the sets that ranking delta would keep. */
dma_status_t dma_score_keys_bias(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin,
                                 int key_end, const float* W, const float* A, dma_bias_form_t form, float* scores,
                                 float* bias, dma_stream_t stream);

/* -------------------------------------------------------------- selection --
 * Fills the geometry of *kept for the given problem (pointers untouched) and
 * the workspace size dma_select_topk needs.  block is 1 (token units) or 64
 * (64-key blocks: block score = max of its keys' scores; row i ranks complete
 * blocks only, keeps floor(w / 64) of them).
 */
dma_status_t dma_kept_layout(int B, int Hkv, int S, int w, int window, int block, dma_sel_mode_t mode,
                             dma_kept_t* kept, size_t* select_ws_bytes);

/* DMA summary §五: combine the scores with the causal mask, keep the top-w at
 * every time step.  Ties go to the lower key index; scores are compared as
 * fp32 (-0 equals +0; NaN ranks below every number).
 *   scores   device [B][Hkv][S] fp32
 *   kept     geometry from dma_kept_layout with the same (B, Hkv, S, w, window,
 *            block, mode); arrays as documented in dma_kept_t
 *   op       FULL: writes expiry, idx/count, and (when non-NULL) top_idx/top_count,
 *            tile_cnt/tile_idx and bitmap.
 *            UPDATE: token units only; the newest key of sequence b sits at
 *            position seq_len[b] - 1 (seq_len NULL: S - 1); top_idx/top_count
 *            must hold the top set of the previous row; it becomes top-w of
 *            (previous set + newest key).  Nothing else is written.
 *   seq_len  device [B] int32 or NULL.  FULL requires NULL (all sequences have
 *            length S).
 *   ws       device workspace of at least *select_ws_bytes (FULL); UPDATE needs none.
 */
dma_status_t dma_select_topk(const float* scores, int B, int Hkv, int S, int w, int window, int block,
                             dma_sel_mode_t mode, dma_sel_op_t op, const int32_t* seq_len, dma_kept_t* kept,
                             void* ws, size_t ws_bytes, dma_stream_t stream);

/* Per-KV-head budgets (Sparse Frontier summary, budget allocation: uniform vs
 * adaptive across heads): dma_select_topk with KV head h of every sequence
 * keeping w_head[h] keys (block units: floor(w_head[h] / 64) blocks) at every
 * time step, selected exactly as a uniform budget of w_head[h] on that head.
 *   w        the largest budget: kept's layout (dma_kept_layout with this w) is
 *            sized for it, and the workspace is that of dma_select_topk
 *   w_head   device [Hkv] int32, 0 <= w_head[h] <= w; read on the device, so an
 *            entry outside the range is recorded as DMA_ERR_DEVICE_CHECK
 *            (dma_get_device_status) and clamped into [0, w]
 * Every other argument, and the result, as for dma_select_topk. */
dma_status_t dma_select_topk_heads(const float* scores, int B, int Hkv, int S, int w, const int32_t* w_head,
                                   int window, int block, dma_sel_mode_t mode, dma_sel_op_t op,
                                   const int32_t* seq_len, dma_kept_t* kept, void* ws, size_t ws_bytes,
                                   dma_stream_t stream);

/* -------------------------------------------------------------- attention --
 * DMA summary §四/§五: masked positions are skipped outright; the kept ones get
 * x_ij = scale * <Q_i, K_j> + s_j, softmax over the kept set, O_i = sum p_ij V_j.
 *   Q        device [B][S][H][D]      K, V  device [B][S][Hkv][D]   (dtype dt)
 *   scores   device [B][Hkv][S] fp32  (the bias; the same array the selection used)
 *   kept     after dma_select_topk(FULL) with tile_cnt/tile_idx set
 *   scale    > 0, or <= 0 for 1/sqrt(D)
 *   O        device [B][S][H][D] (dtype dt)
 *   lse      device [B][H][S] fp32 or NULL: log-sum-exp of the kept logits
 * A row with nothing kept gets O = 0 and lse = -inf.
 */
dma_status_t dma_sparse_attn_prefill(const void* Q, const void* K, const void* V, dma_dtype_t dt, int B, int S,
                                     int H, int Hkv, int D, const float* scores, const dma_kept_t* kept,
                                     float scale, void* O, float* lse, dma_stream_t stream);

/* Workspace bytes of dma_sparse_attn_decode. */
dma_status_t dma_decode_workspace_size(int B, int H, int Hkv, int D, int top_cap, int window, size_t* ws_bytes);

/* One new query row per sequence, at position L-1 of its cache of length
 * L = cache_len[b]; same kept-set rule as the last prefill row (DMA summary
 * §七: the same sparsity in training and inference; the full cache is kept and
 * only the selection changes).
 *   q          device [B][H][D]            Kc, Vc device [B][Lmax][Hkv][D]
 *   cache_len  device [B] int32 or NULL (= Lmax); 1 <= L <= Lmax
 *   scores     device [B][Hkv][Lmax] fp32
 *   kept       top_idx/top_count = the top set of row L-1 (FULL at S = L, or UPDATE)
 *   o          device [B][H][D] (dtype dt)    lse device [B][H] fp32 or NULL
 *   ws         device workspace of dma_decode_workspace_size bytes
 */
dma_status_t dma_sparse_attn_decode(const void* q, const void* Kc, const void* Vc, dma_dtype_t dt, int B, int Lmax,
                                    const int32_t* cache_len, int H, int Hkv, int D, const float* scores,
                                    const dma_kept_t* kept, float scale, void* o, float* lse, void* ws,
                                    size_t ws_bytes, dma_stream_t stream);

/* Decode for callers that cannot allocate device memory.  The method has no
 * counterpart for this call; it exists for callers that may not call cudaMalloc
 * at all -- a serving loop running on a fixed memory plan, a host library with
 * no access to the application's allocator, or code that must not risk the
 * device-wide synchronisation an allocation can cause.
 *
 * Same arguments and result as dma_sparse_attn_decode, without the workspace:
 * the split-K partials go to a 64 MiB array that the library holds in device
 * memory on every GPU that loads it, until the process exits.  The call itself
 * allocates nothing.
 *   - Limit: when the partials would need more than 64 MiB
 *     (4 * B * H * ceil((top_cap + window) / 64) * (D + 2) + 256 bytes), the call
 *     returns DMA_ERR_UNSUPPORTED before launching anything.
 *   - Set-up: the first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and keeps it for the process;
 *     make that first call before any stream capture.  A cudaDeviceReset of that
 *     device discards the array with the context: do not call this entry point on
 *     the device after such a reset.
 *   - Sharing: all calls on a device use the same array, which keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls that overlap
 *     on the GPU -- on different streams, or from different threads -- race on
 *     it and must be serialised by the caller.
 */
dma_status_t dma_sparse_attn_decode_noalloc(const void* q, const void* Kc, const void* Vc, dma_dtype_t dt, int B,
                                            int Lmax, const int32_t* cache_len, int H, int Hkv, int D,
                                            const float* scores, const dma_kept_t* kept, float scale, void* o,
                                            float* lse, dma_stream_t stream);

/* ----------------------------------------------------------- paged decode --
 * Page-granular decode over a paged KV cache.  Sparse Frontier summary, decode
 * findings: page-level (Quest) selection keeps the whole KV cache and picks pages
 * of it; DMA summary §五/§七: the same content-derived scores and top-k rule.  A
 * page's score is the maximum of its keys' scores (as for 64-key blocks); the
 * decode row L-1 keeps the floor(w / page_size) complete pages (last key <= L-1)
 * with the highest page scores, ties to the lower page index, united with the
 * window {L-window .. L-1}.
 *   K_pages, V_pages  device [n_pages][page_size][Hkv][D] (dtype dt)
 *   block_table       device [B][max_pages] int32: logical page p of sequence b
 *                     (keys p*page_size .. p*page_size+page_size-1) is physical
 *                     page block_table[b][p]; entries for pages past cache_len
 *                     are not read.  An entry outside [0, n_pages) is reported
 *                     as DMA_ERR_DEVICE_CHECK and its rows are not read.
 *   cache_len         device [B] int32 or NULL (= max_pages * page_size)
 *   page_size         16, 32, 64 or 128;  1 <= max_pages <= 8192
 * Scores are kept per logical position: scores [B][Hkv][max_pages * page_size],
 * page_scores [B][Hkv][max_pages], both fp32.
 */

/* Scores of keys key_begin <= j < min(key_end, cache_len[b]) of every sequence
 * (the dma_score_keys formula), read through the block table; when page_scores
 * is non-NULL, also the page score of every page holding a key of
 * [key_begin, key_end): the max over its keys below cache_len[b], whose scores
 * must all be in `scores` (scored now or earlier). */
dma_status_t dma_score_keys_paged(const void* V_pages, dma_dtype_t dt, int n_pages, const int32_t* block_table,
                                  int B, int max_pages, int page_size, const int32_t* cache_len, int Hkv, int D,
                                  int key_begin, int key_end, const float* W, const float* A, float* scores,
                                  float* page_scores, dma_stream_t stream);

/* dma_score_keys_paged plus the bias array the paged decode takes as its scores
 * (the exp form of dma_score_keys_bias for a paged cache): bias [B][Hkv][max_pages *
 * page_size] fp32, non-NULL and not scores, receives s (DMA_BIAS_LOG) or exp(s)
 * (DMA_BIAS_EXP) for the keys scored; the page scores stay the maxima of s, so
 * the page selection is unchanged. */
dma_status_t dma_score_keys_paged_bias(const void* V_pages, dma_dtype_t dt, int n_pages, const int32_t* block_table,
                                       int B, int max_pages, int page_size, const int32_t* cache_len, int Hkv, int D,
                                       int key_begin, int key_end, const float* W, const float* A,
                                       dma_bias_form_t form, float* scores, float* page_scores, float* bias,
                                       dma_stream_t stream);

/* The kept pages of every sequence's decode row, written as their keys:
 *   top_idx    device [B][Hkv][top_cap] int32: the keys of the kept pages, ascending
 *   top_count  device [B][Hkv] int32: their number
 *   top_cap    >= floor(w / page_size) * page_size
 * (the same top-set format as dma_kept_t.top_idx/top_count). */
dma_status_t dma_select_pages(const float* page_scores, int B, int Hkv, int max_pages, int page_size,
                              const int32_t* cache_len, int w, int32_t* top_idx, int32_t* top_count, int top_cap,
                              dma_stream_t stream);

/* dma_select_pages with a budget per KV head: head h keeps floor(w_head[h] /
 * page_size) pages.  w_head device [Hkv] int32 with 0 <= w_head[h] <= w (an entry
 * outside is recorded as DMA_ERR_DEVICE_CHECK and clamped); top_cap as for w. */
dma_status_t dma_select_pages_heads(const float* page_scores, int B, int Hkv, int max_pages, int page_size,
                                    const int32_t* cache_len, int w, const int32_t* w_head, int32_t* top_idx,
                                    int32_t* top_count, int top_cap, dma_stream_t stream);

/* Decode over the kept pages and the window (bf16 only; H / Hkv <= 16): the same
 * result as dma_sparse_attn_decode over a contiguous cache holding the same rows.
 *   q, o, lse, scale, ws  as for dma_sparse_attn_decode (ws of
 *                         dma_decode_workspace_size(B, H, Hkv, D, top_cap, window))
 *   scores                device [B][Hkv][max_pages * page_size] fp32
 *   top_idx, top_count, top_cap  from dma_select_pages */
dma_status_t dma_sparse_attn_decode_paged(const void* q, const void* K_pages, const void* V_pages, dma_dtype_t dt,
                                          int n_pages, const int32_t* block_table, int B, int max_pages,
                                          int page_size, const int32_t* cache_len, int H, int Hkv, int D,
                                          const float* scores, const int32_t* top_idx, const int32_t* top_count,
                                          int top_cap, int window, float scale, void* o, float* lse, void* ws,
                                          size_t ws_bytes, dma_stream_t stream);

/* --------------------------------------------------------------- backward --
 * DMA summary §四 (gradients flow through the top-k: kept positions get
 * gradients, masked ones exactly zero), §五 (skipping masked positions is exact
 * in the backward pass too) and §七 (the same sparsity in training and
 * inference).  With p_ij the forward's weights over row i's kept set:
 *   dP_ij = <dO_i, V_j>,  Delta_i = <dO_i, O_i>,  dx_ij = p_ij (dP_ij - Delta_i)
 *   dQ_i = scale sum_j dx_ij K_j      dK_j = scale sum_i dx_ij Q_i
 *   dV_j = sum_i p_ij dO_i            ds_j = sum_i dx_ij
 * (sums over i cover the rows of every query head of the KV head); pairs
 * outside the kept sets contribute nothing.  Through the score
 * s_j = A_h softplus(u_j), u_j = <V_j, W_h>:
 *   dA_h = sum ds_j softplus(u_j)     du_j = ds_j A_h sigmoid(u_j)
 *   dW_h = sum du_j V_j               dV_j += du_j W_h
 * The selection itself (top-w and the expiry intervals) is piecewise constant
 * in the scores and has no gradient of its own.
 */

/* Workspace bytes of dma_sparse_attn_prefill_backward and dma_score_keys_backward
 * (one size serves both). */
dma_status_t dma_backward_workspace_size(int B, int S, int H, int Hkv, int D, size_t* ws_bytes);

/* Gradients of dma_sparse_attn_prefill with respect to Q, K, V and the bias s.
 *   Q, K, V, dt, B, S, H, Hkv, D, scores, kept, scale
 *            exactly as given to the forward call (kept: the same selection,
 *            with expiry, tile_cnt and tile_idx)
 *   O        device [B][S][H][D] (dtype dt)  the forward's output
 *   lse      device [B][H][S] fp32           the forward's lse (required)
 *   dO       device [B][S][H][D] (dtype dt)  dL/dO
 *   dQ       device [B][S][H][D] fp32        written
 *   dK, dV   device [B][S][Hkv][D] fp32      written (not accumulated into)
 *   ds       device [B][Hkv][S] fp32         written: dL/ds
 *   ws       device workspace of dma_backward_workspace_size bytes, 16-byte aligned
 * Rows with nothing kept contribute nothing.  The bf16 path rounds p_ij and
 * dx_ij to bf16 as tensor-core operands and sums dK, dV, ds in fp32 in an order
 * that depends on scheduling; the fp32 path's sums have a fixed order.  Device
 * conditions (a bounded wait that ran out) are reported as for the forward. */
dma_status_t dma_sparse_attn_prefill_backward(const void* Q, const void* K, const void* V, dma_dtype_t dt, int B,
                                              int S, int H, int Hkv, int D, const float* scores,
                                              const dma_kept_t* kept, float scale, const void* O, const float* lse,
                                              const void* dO, float* dQ, float* dK, float* dV, float* ds, void* ws,
                                              size_t ws_bytes, dma_stream_t stream);

/* Gradients of dma_score_keys, given ds = dL/ds:
 *   V, dt, B, S, Hkv, D, W, A   as given to dma_score_keys (all S keys)
 *   ds       device [B][Hkv][S] fp32
 *   dV       device [B][S][Hkv][D] fp32   du_j W_h is ADDED to it (pass the
 *            attention backward's dV to get the total)
 *   dW       device [Hkv][D] fp32         written
 *   dA       device [Hkv] fp32 or NULL    written when non-NULL (with A NULL:
 *            the gradient with respect to a gate of 1)
 *   ws       device workspace of dma_backward_workspace_size bytes
 * dW and dA are summed in a fixed order (the same bits on every run). */
dma_status_t dma_score_keys_backward(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, const float* W,
                                     const float* A, const float* ds, float* dV, float* dW, float* dA, void* ws,
                                     size_t ws_bytes, dma_stream_t stream);

/* dma_score_keys_backward for a bias of the given form: with DMA_BIAS_EXP, ds is
 * the gradient of the added delta = exp(s), and the chain takes ds_j * delta_j
 * as the gradient of s_j (delta recomputed from V, W, A).  Arguments otherwise
 * as for dma_score_keys_backward. */
dma_status_t dma_score_keys_backward_bias(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D,
                                          const float* W, const float* A, dma_bias_form_t form, const float* ds,
                                          float* dV, float* dW, float* dA, void* ws, size_t ws_bytes,
                                          dma_stream_t stream);

/* ------------------------------------------------------- NSA-style fusion --
 * NSA post (news.news) §03: three branches side by side -- attention over
 * compressed blocks (a coarse view of everything), over selected blocks (the
 * important content) and over a sliding window (local context) -- mixed per
 * token by three gates from a small network.  The post gives no formulas; this
 * library reads them as:
 *   compressed  block beta is the mean of the K (V) rows of the complete 64-key
 *               block 64 beta .. 64 beta + 63, seen by rows i >= 64 beta + 63;
 *   selected    this library's 64-key block selection (dma_select_topk, block
 *               64) with no window;
 *   sliding     the keys i - window + 1 .. i;
 *   no branch adds a bias (pass an all-zero scores array to the attention calls);
 *   gates       g_b = sigmoid(<q_i, G[h][b]> + c[h][b]) for b = compressed,
 *               selected, sliding; O_i = sum_b g_b o_b,i.
 * Each branch runs through dma_sparse_attn_prefill (or _decode) with its own
 * kept structure; the compressed branch gathers from the arrays that
 * dma_nsa_compress writes.
 */

/* Block means in the layout the attention calls gather from:
 *   K, V    device [B][S][Hkv][D] (dtype dt)
 *   Kc, Vc  device [B][S][Hkv][D] (dtype dt), arrays of their own: row
 *           64 beta + 63 receives the mean of rows 64 beta .. 64 beta + 63 of
 *           block beta (summed in key order in fp32, rounded once to dt); no
 *           other row is written (nor read by the compressed pattern)
 *   blocks  block_begin <= beta < block_end, 0 <= block_begin <= block_end <=
 *           S / 64 (complete blocks only; decode compresses a block once, when
 *           its last key arrives) */
dma_status_t dma_nsa_compress(const void* K, const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D,
                              int block_begin, int block_end, void* Kc, void* Vc, dma_stream_t stream);

typedef enum { DMA_NSA_COMPRESSED = 0, DMA_NSA_WINDOW = 1 } dma_nsa_pattern_t;

/* Writes the kept structure of a fixed pattern (it depends on S and the window
 * only, so one structure serves every step and layer of that length):
 *   COMPRESSED  key 64 beta + 63 of every complete block is kept from its own row
 *               on, every other key never.  Layout: dma_kept_layout(B, Hkv, S,
 *               w = S / 64, window = 0, block = 1, DMA_SEL_GLOBAL) -- the arrays
 *               equal those of a global selection of the S / 64 best keys under
 *               scores that rank exactly those keys first.
 *   WINDOW      no key in any top set; the window alone.  Layout: dma_kept_layout(
 *               B, Hkv, S, w = 0, window, block = 1, either mode).
 *   seq_len     device [B] int32 or NULL (= S): top_idx/top_count become the
 *               set of the decode row seq_len[b] - 1.
 * Every array of *kept that is non-NULL is written (expiry is required). */
dma_status_t dma_nsa_kept_pattern(dma_nsa_pattern_t pattern, const int32_t* seq_len, dma_kept_t* kept,
                                  dma_stream_t stream);

/* The gated sum of the three branch outputs:
 *   Q                   device [B][S][H][D] (dtype dt)   the query rows (gate input)
 *   O_cmp, O_slc, O_win device [B][S][H][D] (dtype dt)   branch outputs
 *   G                   device [H][3][D] fp32            gate weights per query head
 *   c                   device [H][3] fp32               gate offsets
 *   O                   device [B][S][H][D] (dtype dt)   written (may alias a branch output)
 *   gates               device [B][S][H][3] fp32 or NULL written when non-NULL
 * Decode uses S = 1 (one row per sequence). */
dma_status_t dma_nsa_combine(const void* Q, const void* O_cmp, const void* O_slc, const void* O_win, dma_dtype_t dt,
                             int B, int S, int H, int D, const float* G, const float* c, void* O, float* gates,
                             dma_stream_t stream);

/* ------------------------------------------------------------------ misc -- */

/* Synchronises `stream`, returns the device status word (a dma_status_t value,
 * DMA_OK if nothing was recorded) in *device_status and clears it. */
dma_status_t dma_get_device_status(dma_stream_t stream, int* device_status);

const char* dma_status_string(dma_status_t s);

/* Detail of the last failing call on this host thread ("" if none). */
const char* dma_last_error_message(void);

/* Selects the prefill kernels, forward and backward: 0 = automatic (tensor-core
 * kernels for bf16 when available), 1 = SIMT kernels always.  Process-wide;
 * returns the old value. */
int dma_set_prefill_kernel(int which);

/* Fault detection (a test aid; no effect on results when left at the defaults).
 * Every wait inside the tensor-core prefill kernels (forward and backward) (on an mbarrier that a
 * copy, the tensor core or another warp completes) gives up after a time
 * limit: the kernel then records DMA_ERR_TIMEOUT in the device status word
 * (read by dma_get_device_status), every warp of the CTA leaves its loop, the
 * copies and tensor-core work already in flight land, and the kernel ends; the
 * CUDA context stays usable and O holds unspecified values for that launch.
 *
 * dma_set_wait_limit_ns: the limit in nanoseconds for launches made after the
 *   call (process-wide); 0 restores the default, which is DMA_TIMEOUT_NS from
 *   the environment when the library loads, else 2 s.  Returns the previous
 *   limit.
 * dma_set_fault_injection: DMA_FAULT_NONE, or DMA_FAULT_DROP_ARRIVE: in the
 *   prefill launches that follow, CTA 0 of the tensor-core kernel withholds the
 *   copy warps' completion signal for the K rows of its first key block, so the
 *   MMA warp's wait for them runs out (one bounded timeout, then the path
 *   above).  The default is DMA_FAULT_INJECT=drop_arrive in the environment
 *   when the library loads, else none.  Returns the previous mode, or -1 (and
 *   changes nothing) for an unknown mode. */
enum { DMA_FAULT_NONE = 0, DMA_FAULT_DROP_ARRIVE = 1 };
uint64_t dma_set_wait_limit_ns(uint64_t ns);
int dma_set_fault_injection(int mode);

int dma_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DMA_H_ */
