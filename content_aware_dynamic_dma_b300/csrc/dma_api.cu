// C ABI of libdma: argument validation, error reporting and kernel dispatch.
// Every entry point checks its arguments completely before it enqueues any
// work, so an argument error never leaves a partial launch behind.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dma_internal.cuh"

namespace dma {
namespace {

thread_local char g_msg[512] = "";

// Device status word: kernels record conditions they find (a bounded wait that
// ran out, an internal capacity check) here; dma_get_device_status reads and
// clears it.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

int g_prefill_kernel = 0;  // 0 automatic, 1 SIMT

// Wait limit of the kernels' bounded waits and the fault-injection mode, with their
// defaults from the environment (DMA_TIMEOUT_NS, DMA_FAULT_INJECT) read at load.
uint64_t env_wait_ns()
{
    const char* v = getenv("DMA_TIMEOUT_NS");
    if (!v || !*v) return kDefaultWaitNs;
    char* end = nullptr;
    const unsigned long long n = strtoull(v, &end, 10);
    return (end && *end == '\0' && n > 0) ? (uint64_t)n : kDefaultWaitNs;
}
int env_fault_mode()
{
    const char* v = getenv("DMA_FAULT_INJECT");
    return (v && (strcmp(v, "drop_arrive") == 0 || strcmp(v, "1") == 0)) ? DMA_FAULT_DROP_ARRIVE : DMA_FAULT_NONE;
}
std::atomic<uint64_t> g_wait_ns{env_wait_ns()};
std::atomic<int> g_fault_mode{env_fault_mode()};

dma_status_t fail(dma_status_t s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

dma_status_t ok()
{
    g_msg[0] = '\0';
    return DMA_OK;
}

dma_status_t cuda_fail(cudaError_t e, const char* where)
{
    return fail(DMA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Address of the status word on the current device (looked up once per device).
dma_status_t status_ptr(int** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(DMA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    *out = g_status_ptr[dev];
    return DMA_OK;
}

dma_status_t check_common(dma_dtype_t dt, int B, int S, int Hkv, int D)
{
    if (dt != DMA_F32 && dt != DMA_BF16) return fail(DMA_ERR_INVALID_ARG, "dtype %d is neither DMA_F32 nor DMA_BF16", (int)dt);
    if (B < 1 || S < 1 || Hkv < 1) return fail(DMA_ERR_INVALID_ARG, "B=%d S=%d Hkv=%d must be >= 1", B, S, Hkv);
    if (D != 64 && D != 128) return fail(DMA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
    if ((int64_t)B * S * Hkv * D > ((int64_t)1 << 40)) return fail(DMA_ERR_UNSUPPORTED, "tensor too large");
    return DMA_OK;
}

int64_t kept_top_budget(int w, int S, int block)
{
    int64_t k = block <= 1 ? w : (int64_t)(w / block) * block;
    return k < S ? k : S;
}

dma_status_t check_kept_geometry(const dma_kept_t* kept, int B, int Hkv, int S)
{
    if (!kept) return fail(DMA_ERR_INVALID_ARG, "kept is NULL");
    if (kept->B != B || kept->Hkv != Hkv || kept->S != S)
        return fail(DMA_ERR_INVALID_ARG, "kept layout (B=%d Hkv=%d S=%d) does not match the call (B=%d Hkv=%d S=%d)",
                    kept->B, kept->Hkv, kept->S, B, Hkv, S);
    dma_kept_t ref{};
    size_t ws = 0;
    dma_status_t s = dma_kept_layout(kept->B, kept->Hkv, kept->S, kept->w, kept->window, kept->block,
                                     (dma_sel_mode_t)kept->mode, &ref, &ws);
    if (s != DMA_OK) return s;
    if (ref.q_tile != kept->q_tile || ref.n_qt != kept->n_qt || ref.cap != kept->cap || ref.top_cap != kept->top_cap ||
        ref.tile_stride != kept->tile_stride || ref.bitmap_words != kept->bitmap_words)
        return fail(DMA_ERR_INVALID_ARG, "kept geometry was not produced by dma_kept_layout for these sizes");
    return DMA_OK;
}

}  // namespace

dma_status_t set_error(dma_status_t s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

}  // namespace dma

using namespace dma;

extern "C" {

int dma_version(void) { return 1; }

const char* dma_status_string(dma_status_t s)
{
    switch (s) {
    case DMA_OK: return "DMA_OK";
    case DMA_ERR_INVALID_ARG: return "DMA_ERR_INVALID_ARG";
    case DMA_ERR_UNSUPPORTED: return "DMA_ERR_UNSUPPORTED";
    case DMA_ERR_WORKSPACE: return "DMA_ERR_WORKSPACE";
    case DMA_ERR_CUDA: return "DMA_ERR_CUDA";
    case DMA_ERR_TIMEOUT: return "DMA_ERR_TIMEOUT";
    case DMA_ERR_DEVICE_CHECK: return "DMA_ERR_DEVICE_CHECK";
    }
    return "DMA_ERR_UNKNOWN";
}

const char* dma_last_error_message(void) { return g_msg; }

uint64_t dma_set_wait_limit_ns(uint64_t ns)
{
    return g_wait_ns.exchange(ns ? ns : env_wait_ns());
}

int dma_set_fault_injection(int mode)
{
    if (mode != DMA_FAULT_NONE && mode != DMA_FAULT_DROP_ARRIVE) return -1;
    return g_fault_mode.exchange(mode);
}

int dma_set_prefill_kernel(int which)
{
    int old = g_prefill_kernel;
    g_prefill_kernel = which;
    return old;
}

dma_status_t dma_get_device_status(dma_stream_t stream, int* device_status)
{
    if (!device_status) return fail(DMA_ERR_INVALID_ARG, "device_status is NULL");
    int* p = nullptr;
    dma_status_t s = status_ptr(&p);
    if (s != DMA_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    *device_status = v;
    return ok();
}

static dma_status_t score_impl(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin,
                               int key_end, const float* W, const float* A, dma_bias_form_t form, float* scores,
                               float* bias, dma_stream_t stream)
{
    dma_status_t s = check_common(dt, B, S, Hkv, D);
    if (s != DMA_OK) return s;
    if (!V || !W || !scores) return fail(DMA_ERR_INVALID_ARG, "V, W and scores must be non-NULL");
    if (!aligned16(V) || !aligned4(W) || !aligned4(scores) || (A && !aligned4(A)) || (bias && !aligned4(bias)))
        return fail(DMA_ERR_INVALID_ARG, "V must be 16-byte aligned; W, A, scores, bias 4-byte aligned");
    if (form != DMA_BIAS_LOG && form != DMA_BIAS_EXP) return fail(DMA_ERR_INVALID_ARG, "form=%d", (int)form);
    if (key_begin < 0 || key_end < key_begin || key_end > S)
        return fail(DMA_ERR_INVALID_ARG, "key range [%d, %d) outside [0, %d]", key_begin, key_end, S);
    if (Hkv > 128) return fail(DMA_ERR_UNSUPPORTED, "scoring takes up to 128 KV heads (Hkv=%d)", Hkv);
    cudaError_t e = launch_score(V, dt, B, S, Hkv, D, key_begin, key_end, W, A, scores, bias,
                                 form == DMA_BIAS_EXP ? 1 : 0, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "score kernel launch");
    return ok();
}

dma_status_t dma_score_keys(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin, int key_end,
                            const float* W, const float* A, float* scores, dma_stream_t stream)
{
    return score_impl(V, dt, B, S, Hkv, D, key_begin, key_end, W, A, DMA_BIAS_LOG, scores, nullptr, stream);
}

dma_status_t dma_score_keys_bias(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin,
                                 int key_end, const float* W, const float* A, dma_bias_form_t form, float* scores,
                                 float* bias, dma_stream_t stream)
{
    if (!bias) return fail(DMA_ERR_INVALID_ARG, "bias is NULL (dma_score_keys writes the scores alone)");
    if (bias == scores) return fail(DMA_ERR_INVALID_ARG, "bias and scores must be different arrays");
    return score_impl(V, dt, B, S, Hkv, D, key_begin, key_end, W, A, form, scores, bias, stream);
}

dma_status_t dma_kept_layout(int B, int Hkv, int S, int w, int window, int block, dma_sel_mode_t mode,
                             dma_kept_t* kept, size_t* select_ws_bytes)
{
    if (!kept || !select_ws_bytes) return fail(DMA_ERR_INVALID_ARG, "kept and select_ws_bytes must be non-NULL");
    if (B < 1 || Hkv < 1 || S < 1) return fail(DMA_ERR_INVALID_ARG, "B=%d Hkv=%d S=%d must be >= 1", B, Hkv, S);
    if (w < 0 || window < 0) return fail(DMA_ERR_INVALID_ARG, "w=%d and window=%d must be >= 0", w, window);
    if (block != 1 && block != 64) return fail(DMA_ERR_UNSUPPORTED, "block=%d (supported: 1, 64)", block);
    if (mode != DMA_SEL_ROWWISE && mode != DMA_SEL_GLOBAL) return fail(DMA_ERR_INVALID_ARG, "mode=%d", (int)mode);
    if (S > (1 << 28) || (int64_t)B * Hkv * S > ((int64_t)1 << 34))
        return fail(DMA_ERR_UNSUPPORTED, "selection over S=%d keys x %d segments is too large", S, B * Hkv);
    dma_kept_t k = *kept;
    k.B = B;
    k.Hkv = Hkv;
    k.S = S;
    k.w = w;
    k.window = window;
    k.block = block;
    k.mode = (int32_t)mode;
    k.q_tile = kQTile;
    k.n_qt = (S + kQTile - 1) / kQTile;
    k.cap = S;
    int64_t budget = kept_top_budget(w, S, block);
    k.top_cap = (int32_t)(budget > 0 ? budget : 1);
    int64_t stride = (int64_t)w + 3 * kQTile;
    int64_t s4 = ((int64_t)S + 3) / 4 * 4;
    if (stride > s4) stride = s4;
    k.tile_stride = (int32_t)((stride + 3) / 4 * 4);
    k.bitmap_words = ((S + kBitmapBlock - 1) / kBitmapBlock + 31) / 32;
    *kept = k;
    *select_ws_bytes = make_select_plan(B, Hkv, S, w, block).bytes;
    return ok();
}

static dma_status_t select_impl(const float* scores, int B, int Hkv, int S, int w, const int32_t* w_head, int window,
                                int block, dma_sel_mode_t mode, dma_sel_op_t op, const int32_t* seq_len,
                                dma_kept_t* kept, void* ws, size_t ws_bytes, dma_stream_t stream)
{
    if (!scores) return fail(DMA_ERR_INVALID_ARG, "scores is NULL");
    if (w_head && !aligned4(w_head)) return fail(DMA_ERR_INVALID_ARG, "w_head must be 4-byte aligned");
    if (!aligned4(scores)) return fail(DMA_ERR_INVALID_ARG, "scores must be 4-byte aligned");
    dma_status_t s = check_kept_geometry(kept, B, Hkv, S);
    if (s != DMA_OK) return s;
    if (kept->w != w || kept->window != window || kept->block != block || kept->mode != (int32_t)mode)
        return fail(DMA_ERR_INVALID_ARG, "kept layout (w=%d window=%d block=%d mode=%d) does not match the call",
                    kept->w, kept->window, kept->block, kept->mode);
    int* status = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (op == DMA_SEL_UPDATE) {
        if (block != 1) return fail(DMA_ERR_UNSUPPORTED, "UPDATE supports token units (block = 1) only");
        if (!kept->top_idx || !kept->top_count) return fail(DMA_ERR_INVALID_ARG, "UPDATE needs top_idx and top_count");
        if ((int64_t)kept->top_cap * 4 > 200 * 1024)
            return fail(DMA_ERR_UNSUPPORTED, "UPDATE supports budgets up to 51200 keys");
        if (seq_len && !aligned4(seq_len)) return fail(DMA_ERR_INVALID_ARG, "seq_len must be 4-byte aligned");
        if ((s = status_ptr(&status)) != DMA_OK) return s;
        cudaError_t e = launch_select_update(scores, kept, seq_len, w_head, status, st);
        if (e != cudaSuccess) return cuda_fail(e, "select update launch");
        return ok();
    }
    if (op != DMA_SEL_FULL) return fail(DMA_ERR_INVALID_ARG, "op=%d", (int)op);
    if (seq_len) return fail(DMA_ERR_UNSUPPORTED, "FULL selection takes seq_len = NULL (all sequences of length S)");
    if (!kept->expiry || !kept->idx || !kept->count)
        return fail(DMA_ERR_INVALID_ARG, "FULL needs expiry, idx and count");
    if ((kept->top_idx == nullptr) != (kept->top_count == nullptr))
        return fail(DMA_ERR_INVALID_ARG, "top_idx and top_count must both be set or both be NULL");
    if ((kept->tile_idx == nullptr) != (kept->tile_cnt == nullptr))
        return fail(DMA_ERR_INVALID_ARG, "tile_idx and tile_cnt must both be set or both be NULL");
    if (kept->bitmap && !kept->tile_idx) return fail(DMA_ERR_INVALID_ARG, "bitmap needs tile_idx/tile_cnt");
    SelectPlan plan = make_select_plan(B, Hkv, S, w, block);
    if (!ws || ws_bytes < plan.bytes)
        return fail(DMA_ERR_WORKSPACE, "select workspace of %zu bytes given, %zu needed", ws ? ws_bytes : (size_t)0,
                    plan.bytes);
    if (!aligned16(ws)) return fail(DMA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if ((s = status_ptr(&status)) != DMA_OK) return s;
    cudaError_t e = launch_select_full(scores, plan, kept, w_head, ws, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "select launch");
    return ok();
}

dma_status_t dma_select_topk(const float* scores, int B, int Hkv, int S, int w, int window, int block,
                             dma_sel_mode_t mode, dma_sel_op_t op, const int32_t* seq_len, dma_kept_t* kept, void* ws,
                             size_t ws_bytes, dma_stream_t stream)
{
    return select_impl(scores, B, Hkv, S, w, nullptr, window, block, mode, op, seq_len, kept, ws, ws_bytes, stream);
}

dma_status_t dma_select_topk_heads(const float* scores, int B, int Hkv, int S, int w, const int32_t* w_head,
                                   int window, int block, dma_sel_mode_t mode, dma_sel_op_t op,
                                   const int32_t* seq_len, dma_kept_t* kept, void* ws, size_t ws_bytes,
                                   dma_stream_t stream)
{
    if (!w_head) return fail(DMA_ERR_INVALID_ARG, "w_head is NULL (dma_select_topk takes one budget)");
    return select_impl(scores, B, Hkv, S, w, w_head, window, block, mode, op, seq_len, kept, ws, ws_bytes, stream);
}

dma_status_t dma_sparse_attn_prefill(const void* Q, const void* K, const void* V, dma_dtype_t dt, int B, int S, int H,
                                     int Hkv, int D, const float* scores, const dma_kept_t* kept, float scale,
                                     void* O, float* lse, dma_stream_t stream)
{
    dma_status_t s = check_common(dt, B, S, Hkv, D);
    if (s != DMA_OK) return s;
    if (H < 1 || H % Hkv != 0) return fail(DMA_ERR_INVALID_ARG, "H=%d must be a positive multiple of Hkv=%d", H, Hkv);
    if (!Q || !K || !V || !O || !scores) return fail(DMA_ERR_INVALID_ARG, "Q, K, V, O and scores must be non-NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned4(scores) || (lse && !aligned4(lse)))
        return fail(DMA_ERR_INVALID_ARG, "Q, K, V, O must be 16-byte aligned; scores, lse 4-byte aligned");
    if ((s = check_kept_geometry(kept, B, Hkv, S)) != DMA_OK) return s;
    if (!kept->expiry || !kept->tile_cnt || !kept->tile_idx)
        return fail(DMA_ERR_INVALID_ARG, "prefill needs kept->expiry, tile_cnt and tile_idx");
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)D);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (g_prefill_kernel == 0 && prefill_tc_supported(dt, B, S, H, Hkv, D)) {
        int* status = nullptr;
        if ((s = status_ptr(&status)) != DMA_OK) return s;
        e = launch_prefill_tc(Q, K, V, B, S, H, Hkv, D, scores, kept, scale, O, lse, status, g_wait_ns.load(),
                              g_fault_mode.load(), st);
    } else {
        e = launch_prefill_simt(Q, K, V, dt, B, S, H, Hkv, D, scores, kept, scale, O, lse, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

dma_status_t dma_decode_workspace_size(int B, int H, int Hkv, int D, int top_cap, int window, size_t* ws_bytes)
{
    if (!ws_bytes) return fail(DMA_ERR_INVALID_ARG, "ws_bytes is NULL");
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || top_cap < 0 || window < 0)
        return fail(DMA_ERR_INVALID_ARG, "bad sizes B=%d H=%d Hkv=%d top_cap=%d window=%d", B, H, Hkv, top_cap, window);
    if (D != 64 && D != 128) return fail(DMA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
    *ws_bytes = decode_ws_bytes(B, H, Hkv, D, top_cap, window);
    return ok();
}

dma_status_t dma_sparse_attn_decode(const void* q, const void* Kc, const void* Vc, dma_dtype_t dt, int B, int Lmax,
                                    const int32_t* cache_len, int H, int Hkv, int D, const float* scores,
                                    const dma_kept_t* kept, float scale, void* o, float* lse, void* ws,
                                    size_t ws_bytes, dma_stream_t stream)
{
    dma_status_t s = check_common(dt, B, Lmax, Hkv, D);
    if (s != DMA_OK) return s;
    if (H < 1 || H % Hkv != 0) return fail(DMA_ERR_INVALID_ARG, "H=%d must be a positive multiple of Hkv=%d", H, Hkv);
    if (H / Hkv > 16) return fail(DMA_ERR_UNSUPPORTED, "decode supports up to 16 query heads per KV head");
    if (!q || !Kc || !Vc || !o || !scores) return fail(DMA_ERR_INVALID_ARG, "q, Kc, Vc, o and scores must be non-NULL");
    if (!aligned16(q) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(o) || !aligned4(scores) ||
        (lse && !aligned4(lse)) || (cache_len && !aligned4(cache_len)))
        return fail(DMA_ERR_INVALID_ARG, "q, Kc, Vc, o must be 16-byte aligned; scores, lse, cache_len 4-byte aligned");
    if ((s = check_kept_geometry(kept, B, Hkv, Lmax)) != DMA_OK) return s;
    if (!kept->top_idx || !kept->top_count) return fail(DMA_ERR_INVALID_ARG, "decode needs kept->top_idx/top_count");
    size_t need = decode_ws_bytes(B, H, Hkv, D, kept->top_cap, kept->window);
    if (!ws || ws_bytes < need)
        return fail(DMA_ERR_WORKSPACE, "decode workspace of %zu bytes given, %zu needed", ws ? ws_bytes : (size_t)0, need);
    if (!aligned16(ws)) return fail(DMA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)D);
    cudaError_t e;
    if (decode_pipe_supported(dt, B, Lmax, H, Hkv, D)) {
        int* status = nullptr;
        if ((s = status_ptr(&status)) != DMA_OK) return s;
        e = launch_decode_pipe(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, D, scores, kept, scale, o, lse, ws, status,
                               reinterpret_cast<cudaStream_t>(stream));
    } else {
        e = launch_decode(q, Kc, Vc, dt, B, Lmax, cache_len, H, Hkv, D, scores, kept, scale, o, lse, ws,
                          reinterpret_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ok();
}

namespace {
// page_size a power of two in [16, 128]: its log2, else -1
int page_shift(int page_size)
{
    for (int s = 4; s <= 7; ++s)
        if (page_size == (1 << s)) return s;
    return -1;
}
}  // namespace

static dma_status_t score_paged_impl(const void* V_pages, dma_dtype_t dt, int n_pages, const int32_t* block_table,
                                     int B, int max_pages, int page_size, const int32_t* cache_len, int Hkv, int D,
                                     int key_begin, int key_end, const float* W, const float* A,
                                     dma_bias_form_t form, float* scores, float* page_scores, float* bias,
                                     dma_stream_t stream)
{
    if (form != DMA_BIAS_LOG && form != DMA_BIAS_EXP) return fail(DMA_ERR_INVALID_ARG, "form=%d", (int)form);
    if (bias && (bias == scores || !aligned4(bias)))
        return fail(DMA_ERR_INVALID_ARG, "bias must be a 4-byte aligned array of its own");
    const int ps = page_shift(page_size);
    if (ps < 0) return fail(DMA_ERR_UNSUPPORTED, "page_size=%d (supported: 16, 32, 64, 128)", page_size);
    if (max_pages < 1 || max_pages > 8192 || n_pages < 1)
        return fail(DMA_ERR_INVALID_ARG, "max_pages=%d (1..8192) and n_pages=%d (>= 1)", max_pages, n_pages);
    dma_status_t s = check_common(dt, B, max_pages * page_size, Hkv, D);
    if (s != DMA_OK) return s;
    if ((int64_t)n_pages * page_size * Hkv * D > ((int64_t)1 << 40)) return fail(DMA_ERR_UNSUPPORTED, "cache too large");
    if (!V_pages || !block_table || !W || !scores)
        return fail(DMA_ERR_INVALID_ARG, "V_pages, block_table, W and scores must be non-NULL");
    if (!aligned16(V_pages) || !aligned4(block_table) || !aligned4(W) || !aligned4(scores) || (A && !aligned4(A)) ||
        (page_scores && !aligned4(page_scores)) || (cache_len && !aligned4(cache_len)))
        return fail(DMA_ERR_INVALID_ARG, "V_pages must be 16-byte aligned; the other arrays 4-byte aligned");
    const int Lmax = max_pages * page_size;
    if (key_begin < 0 || key_end < key_begin || key_end > Lmax)
        return fail(DMA_ERR_INVALID_ARG, "key range [%d, %d) outside [0, %d]", key_begin, key_end, Lmax);
    int* status = nullptr;
    if ((s = status_ptr(&status)) != DMA_OK) return s;
    cudaError_t e = launch_score_paged(V_pages, dt, block_table, n_pages, B, max_pages, ps, Hkv, D, key_begin, key_end,
                                       cache_len, W, A, scores, page_scores, bias, form == DMA_BIAS_EXP ? 1 : 0,
                                       status, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged score launch");
    return ok();
}

dma_status_t dma_score_keys_paged(const void* V_pages, dma_dtype_t dt, int n_pages, const int32_t* block_table,
                                  int B, int max_pages, int page_size, const int32_t* cache_len, int Hkv, int D,
                                  int key_begin, int key_end, const float* W, const float* A, float* scores,
                                  float* page_scores, dma_stream_t stream)
{
    return score_paged_impl(V_pages, dt, n_pages, block_table, B, max_pages, page_size, cache_len, Hkv, D, key_begin,
                            key_end, W, A, DMA_BIAS_LOG, scores, page_scores, nullptr, stream);
}

dma_status_t dma_score_keys_paged_bias(const void* V_pages, dma_dtype_t dt, int n_pages, const int32_t* block_table,
                                       int B, int max_pages, int page_size, const int32_t* cache_len, int Hkv, int D,
                                       int key_begin, int key_end, const float* W, const float* A,
                                       dma_bias_form_t form, float* scores, float* page_scores, float* bias,
                                       dma_stream_t stream)
{
    if (!bias) return fail(DMA_ERR_INVALID_ARG, "bias is NULL (dma_score_keys_paged writes the scores alone)");
    return score_paged_impl(V_pages, dt, n_pages, block_table, B, max_pages, page_size, cache_len, Hkv, D, key_begin,
                            key_end, W, A, form, scores, page_scores, bias, stream);
}

static dma_status_t select_pages_impl(const float* page_scores, int B, int Hkv, int max_pages, int page_size,
                                      const int32_t* cache_len, int w, const int32_t* w_head, int32_t* top_idx,
                                      int32_t* top_count, int top_cap, dma_stream_t stream)
{
    const int ps = page_shift(page_size);
    if (ps < 0) return fail(DMA_ERR_UNSUPPORTED, "page_size=%d (supported: 16, 32, 64, 128)", page_size);
    if (B < 1 || Hkv < 1 || max_pages < 1 || max_pages > 8192 || w < 0)
        return fail(DMA_ERR_INVALID_ARG, "B=%d Hkv=%d max_pages=%d (1..8192) w=%d", B, Hkv, max_pages, w);
    if (!page_scores || !top_idx || !top_count)
        return fail(DMA_ERR_INVALID_ARG, "page_scores, top_idx and top_count must be non-NULL");
    if (!aligned4(page_scores) || !aligned4(top_idx) || !aligned4(top_count) || (cache_len && !aligned4(cache_len)) ||
        (w_head && !aligned4(w_head)))
        return fail(DMA_ERR_INVALID_ARG, "arrays must be 4-byte aligned");
    const int k_pages = w / page_size;
    if (top_cap < k_pages * page_size)
        return fail(DMA_ERR_INVALID_ARG, "top_cap=%d < floor(w / page_size) * page_size = %d", top_cap,
                    k_pages * page_size);
    int* status = nullptr;
    dma_status_t s;
    if (w_head && (s = status_ptr(&status)) != DMA_OK) return s;
    cudaError_t e = launch_select_pages(page_scores, B, Hkv, max_pages, ps, cache_len, w, w_head, top_idx, top_count,
                                        top_cap, status, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "page selection launch");
    return ok();
}

dma_status_t dma_select_pages(const float* page_scores, int B, int Hkv, int max_pages, int page_size,
                              const int32_t* cache_len, int w, int32_t* top_idx, int32_t* top_count, int top_cap,
                              dma_stream_t stream)
{
    return select_pages_impl(page_scores, B, Hkv, max_pages, page_size, cache_len, w, nullptr, top_idx, top_count,
                             top_cap, stream);
}

dma_status_t dma_select_pages_heads(const float* page_scores, int B, int Hkv, int max_pages, int page_size,
                                    const int32_t* cache_len, int w, const int32_t* w_head, int32_t* top_idx,
                                    int32_t* top_count, int top_cap, dma_stream_t stream)
{
    if (!w_head) return fail(DMA_ERR_INVALID_ARG, "w_head is NULL (dma_select_pages takes one budget)");
    return select_pages_impl(page_scores, B, Hkv, max_pages, page_size, cache_len, w, w_head, top_idx, top_count,
                             top_cap, stream);
}

dma_status_t dma_sparse_attn_decode_paged(const void* q, const void* K_pages, const void* V_pages, dma_dtype_t dt,
                                          int n_pages, const int32_t* block_table, int B, int max_pages,
                                          int page_size, const int32_t* cache_len, int H, int Hkv, int D,
                                          const float* scores, const int32_t* top_idx, const int32_t* top_count,
                                          int top_cap, int window, float scale, void* o, float* lse, void* ws,
                                          size_t ws_bytes, dma_stream_t stream)
{
    const int ps = page_shift(page_size);
    if (ps < 0) return fail(DMA_ERR_UNSUPPORTED, "page_size=%d (supported: 16, 32, 64, 128)", page_size);
    if (max_pages < 1 || max_pages > 8192 || n_pages < 1)
        return fail(DMA_ERR_INVALID_ARG, "max_pages=%d (1..8192) and n_pages=%d (>= 1)", max_pages, n_pages);
    dma_status_t s = check_common(dt, B, max_pages * page_size, Hkv, D);
    if (s != DMA_OK) return s;
    if (H < 1 || H % Hkv != 0) return fail(DMA_ERR_INVALID_ARG, "H=%d must be a positive multiple of Hkv=%d", H, Hkv);
    if (dt != DMA_BF16 || H / Hkv > 16)
        return fail(DMA_ERR_UNSUPPORTED, "paged decode supports bf16 with up to 16 query heads per KV head");
    if ((int64_t)n_pages * page_size * Hkv >= ((int64_t)1 << 31)) return fail(DMA_ERR_UNSUPPORTED, "cache too large");
    if (top_cap < 0 || window < 0) return fail(DMA_ERR_INVALID_ARG, "top_cap=%d window=%d", top_cap, window);
    if (!q || !K_pages || !V_pages || !block_table || !scores || !top_idx || !top_count || !o)
        return fail(DMA_ERR_INVALID_ARG, "q, K_pages, V_pages, block_table, scores, top_idx, top_count, o non-NULL");
    if (!aligned16(q) || !aligned16(K_pages) || !aligned16(V_pages) || !aligned16(o) || !aligned4(block_table) ||
        !aligned4(scores) || !aligned4(top_idx) || !aligned4(top_count) || (lse && !aligned4(lse)) ||
        (cache_len && !aligned4(cache_len)))
        return fail(DMA_ERR_INVALID_ARG, "q, K_pages, V_pages, o must be 16-byte aligned; the rest 4-byte aligned");
    const size_t need = decode_ws_bytes(B, H, Hkv, D, top_cap, window);
    if (!ws || ws_bytes < need)
        return fail(DMA_ERR_WORKSPACE, "decode workspace of %zu bytes given, %zu needed", ws ? ws_bytes : (size_t)0, need);
    if (!aligned16(ws)) return fail(DMA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)D);
    int* status = nullptr;
    if ((s = status_ptr(&status)) != DMA_OK) return s;
    cudaError_t e = launch_decode_paged(q, K_pages, V_pages, block_table, n_pages, B, max_pages, ps, cache_len, H, Hkv,
                                        D, scores, top_idx, top_count, top_cap, window, scale, o, lse, ws, status,
                                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
    return ok();
}

dma_status_t dma_backward_workspace_size(int B, int S, int H, int Hkv, int D, size_t* ws_bytes)
{
    if (!ws_bytes) return fail(DMA_ERR_INVALID_ARG, "ws_bytes is NULL");
    if (B < 1 || S < 1 || H < 1 || Hkv < 1 || H % Hkv != 0)
        return fail(DMA_ERR_INVALID_ARG, "bad sizes B=%d S=%d H=%d Hkv=%d", B, S, H, Hkv);
    if (D != 64 && D != 128) return fail(DMA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
    *ws_bytes = backward_ws_bytes(B, S, H, Hkv, D);
    return ok();
}

dma_status_t dma_sparse_attn_prefill_backward(const void* Q, const void* K, const void* V, dma_dtype_t dt, int B,
                                              int S, int H, int Hkv, int D, const float* scores,
                                              const dma_kept_t* kept, float scale, const void* O, const float* lse,
                                              const void* dO, float* dQ, float* dK, float* dV, float* ds, void* ws,
                                              size_t ws_bytes, dma_stream_t stream)
{
    dma_status_t s = check_common(dt, B, S, Hkv, D);
    if (s != DMA_OK) return s;
    if (H < 1 || H % Hkv != 0) return fail(DMA_ERR_INVALID_ARG, "H=%d must be a positive multiple of Hkv=%d", H, Hkv);
    if (!Q || !K || !V || !O || !dO || !scores || !lse || !dQ || !dK || !dV || !ds)
        return fail(DMA_ERR_INVALID_ARG, "Q, K, V, O, dO, scores, lse, dQ, dK, dV and ds must be non-NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
        !aligned16(dK) || !aligned16(dV) || !aligned4(scores) || !aligned4(lse) || !aligned4(ds))
        return fail(DMA_ERR_INVALID_ARG,
                    "Q, K, V, O, dO, dQ, dK, dV must be 16-byte aligned; scores, lse, ds 4-byte aligned");
    if ((s = check_kept_geometry(kept, B, Hkv, S)) != DMA_OK) return s;
    if (!kept->expiry || !kept->tile_cnt || !kept->tile_idx)
        return fail(DMA_ERR_INVALID_ARG, "the backward needs kept->expiry, tile_cnt and tile_idx");
    const size_t need = backward_ws_bytes(B, S, H, Hkv, D);
    if (!ws || ws_bytes < need)
        return fail(DMA_ERR_WORKSPACE, "backward workspace of %zu bytes given, %zu needed", ws ? ws_bytes : (size_t)0,
                    need);
    if (!aligned16(ws)) return fail(DMA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)D);
    int* status = nullptr;
    if ((s = status_ptr(&status)) != DMA_OK) return s;
    BwdArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.dO = dO;
    a.scores = scores;
    a.lse = lse;
    a.expiry = kept->expiry;
    a.tile_cnt = kept->tile_cnt;
    a.tile_idx = kept->tile_idx;
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    a.ds = ds;
    a.delta = static_cast<float*>(ws);
    a.delta_x = a.delta + (size_t)B * H * S;
    a.status = status;
    a.B = B;
    a.S = S;
    a.H = H;
    a.Hkv = Hkv;
    a.n_qt = kept->n_qt;
    a.tile_stride = kept->tile_stride;
    a.window = kept->window;
    a.block = kept->block;
    a.scale = scale;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool tc = g_prefill_kernel == 0 && bwd_tc_supported(dt, D);
    cudaError_t e = launch_bwd_prep(a, dt, D, tc, st);
    if (e == cudaSuccess) e = tc ? launch_bwd_tc(a, D, g_wait_ns.load(), st) : launch_bwd_simt(a, dt, D, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return ok();
}

static dma_status_t score_backward_impl(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, const float* W,
                                        const float* A, dma_bias_form_t form, const float* ds, float* dV, float* dW,
                                        float* dA, void* ws, size_t ws_bytes, dma_stream_t stream)
{
    if (form != DMA_BIAS_LOG && form != DMA_BIAS_EXP) return fail(DMA_ERR_INVALID_ARG, "form=%d", (int)form);
    dma_status_t s = check_common(dt, B, S, Hkv, D);
    if (s != DMA_OK) return s;
    if (!V || !W || !ds || !dV || !dW) return fail(DMA_ERR_INVALID_ARG, "V, W, ds, dV and dW must be non-NULL");
    if (!aligned16(V) || !aligned16(dV) || !aligned4(W) || !aligned4(ds) || !aligned4(dW) || (A && !aligned4(A)) ||
        (dA && !aligned4(dA)))
        return fail(DMA_ERR_INVALID_ARG, "V, dV must be 16-byte aligned; W, A, ds, dW, dA 4-byte aligned");
    const size_t need = backward_ws_bytes(B, S, Hkv, Hkv, D);
    if (!ws || ws_bytes < need)
        return fail(DMA_ERR_WORKSPACE, "score backward workspace of %zu bytes given, %zu needed",
                    ws ? ws_bytes : (size_t)0, need);
    if (!aligned16(ws)) return fail(DMA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    cudaError_t e = launch_score_bwd(V, dt, B, S, Hkv, D, W, A, form == DMA_BIAS_EXP ? 1 : 0, ds, dV, dW, dA, ws,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "score backward launch");
    return ok();
}

dma_status_t dma_score_keys_backward(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, const float* W,
                                     const float* A, const float* ds, float* dV, float* dW, float* dA, void* ws,
                                     size_t ws_bytes, dma_stream_t stream)
{
    return score_backward_impl(V, dt, B, S, Hkv, D, W, A, DMA_BIAS_LOG, ds, dV, dW, dA, ws, ws_bytes, stream);
}

dma_status_t dma_score_keys_backward_bias(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D,
                                          const float* W, const float* A, dma_bias_form_t form, const float* ds,
                                          float* dV, float* dW, float* dA, void* ws, size_t ws_bytes,
                                          dma_stream_t stream)
{
    return score_backward_impl(V, dt, B, S, Hkv, D, W, A, form, ds, dV, dW, dA, ws, ws_bytes, stream);
}

dma_status_t dma_nsa_compress(const void* K, const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D,
                              int block_begin, int block_end, void* Kc, void* Vc, dma_stream_t stream)
{
    dma_status_t s = check_common(dt, B, S, Hkv, D);
    if (s != DMA_OK) return s;
    if (!K || !V || !Kc || !Vc) return fail(DMA_ERR_INVALID_ARG, "K, V, Kc and Vc must be non-NULL");
    if (!aligned16(K) || !aligned16(V) || !aligned16(Kc) || !aligned16(Vc))
        return fail(DMA_ERR_INVALID_ARG, "K, V, Kc, Vc must be 16-byte aligned");
    if (Kc == K || Kc == V || Vc == K || Vc == V || Kc == Vc)
        return fail(DMA_ERR_INVALID_ARG, "Kc and Vc must be arrays of their own");
    if (block_begin < 0 || block_end < block_begin || block_end > S / 64)
        return fail(DMA_ERR_INVALID_ARG, "block range [%d, %d) outside the %d complete blocks", block_begin, block_end,
                    S / 64);
    cudaError_t e = launch_nsa_compress(K, V, dt, B, S, Hkv, D, block_begin, block_end, Kc, Vc,
                                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block compression launch");
    return ok();
}

dma_status_t dma_nsa_kept_pattern(dma_nsa_pattern_t pattern, const int32_t* seq_len, dma_kept_t* kept,
                                  dma_stream_t stream)
{
    if (!kept) return fail(DMA_ERR_INVALID_ARG, "kept is NULL");
    dma_status_t s = check_kept_geometry(kept, kept->B, kept->Hkv, kept->S);
    if (s != DMA_OK) return s;
    if (pattern == DMA_NSA_COMPRESSED) {
        if (kept->w != kept->S / 64 || kept->window != 0 || kept->block != 1 || kept->mode != DMA_SEL_GLOBAL)
            return fail(DMA_ERR_INVALID_ARG,
                        "the compressed pattern takes the layout (w = S / 64 = %d, window 0, block 1, GLOBAL); got "
                        "(w=%d window=%d block=%d mode=%d)", kept->S / 64, kept->w, kept->window, kept->block,
                        kept->mode);
    } else if (pattern == DMA_NSA_WINDOW) {
        if (kept->w != 0 || kept->block != 1)
            return fail(DMA_ERR_INVALID_ARG, "the window pattern takes the layout (w = 0, block 1); got (w=%d block=%d)",
                        kept->w, kept->block);
    } else {
        return fail(DMA_ERR_INVALID_ARG, "pattern=%d", (int)pattern);
    }
    if (!kept->expiry) return fail(DMA_ERR_INVALID_ARG, "kept->expiry is NULL");
    if ((kept->idx == nullptr) != (kept->count == nullptr))
        return fail(DMA_ERR_INVALID_ARG, "idx and count must both be set or both be NULL");
    if ((kept->top_idx == nullptr) != (kept->top_count == nullptr))
        return fail(DMA_ERR_INVALID_ARG, "top_idx and top_count must both be set or both be NULL");
    if ((kept->tile_idx == nullptr) != (kept->tile_cnt == nullptr))
        return fail(DMA_ERR_INVALID_ARG, "tile_idx and tile_cnt must both be set or both be NULL");
    if (kept->bitmap && !kept->tile_idx) return fail(DMA_ERR_INVALID_ARG, "bitmap needs tile_idx/tile_cnt");
    if (seq_len && !aligned4(seq_len)) return fail(DMA_ERR_INVALID_ARG, "seq_len must be 4-byte aligned");
    int* status = nullptr;
    if ((s = status_ptr(&status)) != DMA_OK) return s;
    cudaError_t e = launch_nsa_pattern(pattern == DMA_NSA_COMPRESSED ? 1 : 0, kept, seq_len, status,
                                       reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pattern launch");
    return ok();
}

dma_status_t dma_nsa_combine(const void* Q, const void* O_cmp, const void* O_slc, const void* O_win, dma_dtype_t dt,
                             int B, int S, int H, int D, const float* G, const float* c, void* O, float* gates,
                             dma_stream_t stream)
{
    dma_status_t s = check_common(dt, B, S, H, D);
    if (s != DMA_OK) return s;
    if (!Q || !O_cmp || !O_slc || !O_win || !G || !c || !O)
        return fail(DMA_ERR_INVALID_ARG, "Q, the three branch outputs, G, c and O must be non-NULL");
    if (!aligned16(Q) || !aligned16(O_cmp) || !aligned16(O_slc) || !aligned16(O_win) || !aligned16(O) ||
        !aligned4(G) || !aligned4(c) || (gates && !aligned4(gates)))
        return fail(DMA_ERR_INVALID_ARG, "Q, the branch outputs and O must be 16-byte aligned; G, c, gates 4-byte");
    cudaError_t e = launch_nsa_combine(Q, O_cmp, O_slc, O_win, dt, (int64_t)B * S * H, H, D, G, c, O, gates,
                                       reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fusion launch");
    return ok();
}

}  // extern "C"
