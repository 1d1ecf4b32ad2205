// Sparse attention decode: one new query row per sequence.
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §七: the full KV cache is kept
// and only the selection changes; training and inference share one sparsity
// rule.  Row L-1 of a cache of length L attends to the top set of that row
// (kept->top_idx, ascending) united with the window {L-window .. L-1}; window
// keys are taken from the band, so a top-set key inside the band is skipped in
// the list to avoid counting it twice.
//
// HBM-bound: the work is 2 * D * elem bytes of K and V per kept row per KV
// head.  Split-K: one CTA per (sequence, KV head, chunk of CH kept rows) issues
// all of its row gathers at once with 16-byte cp.async into shared memory (64 KB
// in flight per CTA), then computes the logits of all G = H / Hkv query heads of
// the group, a chunk-local softmax and the partial output.  A second kernel
// merges the chunks of each (sequence, query head) by their log-sum-exp.
#include <cmath>
#include <mutex>

#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxG = 16;

template <typename T>
constexpr int chunk_rows() { return sizeof(T) == 2 ? 128 : 64; }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Entry u of the (sequence, KV head) list: top-set keys outside the window,
// then the window band.  Returns -1 for an entry that contributes nothing.
__device__ __forceinline__ int list_key(int u, const int32_t* top, int n_top, int L, int window)
{
    if (u < n_top) {
        int j = top[u];
        return (j >= 0 && j < L - window && j <= L - 1) ? j : -1;
    }
    int j = L - window + (u - n_top);
    return (j >= 0 && j <= L - 1) ? j : -1;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_partial_kernel(
    const T* __restrict__ q, const T* __restrict__ Kc, const T* __restrict__ Vc, int Lmax,
    const int32_t* __restrict__ cache_len, int H, int Hkv, const float* __restrict__ scores,
    const int32_t* __restrict__ top_idx, const int32_t* __restrict__ top_count, int top_cap, int window, float scale,
    int nchunk, float* __restrict__ part_o, float* __restrict__ part_ml)
{
    constexpr int CH = chunk_rows<T>();
    constexpr int kElem = 16 / sizeof(T);
    constexpr int kCPR = D / kElem;  // 16-byte chunks per row
    constexpr int kDL = D / 32;      // elements per lane in the logit dot
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* k_s = reinterpret_cast<T*>(smem_raw);            // [CH][D]
    T* v_s = k_s + CH * D;                               // [CH][D]
    float* q_s = reinterpret_cast<float*>(v_s + CH * D); // [G][D]
    float* x_s = q_s + kMaxG * D;                        // [G][CH]
    int* j_s = reinterpret_cast<int*>(x_s + kMaxG * CH); // [CH]
    float* bias_s = reinterpret_cast<float*>(j_s + CH);  // [CH]

    const int seg = blockIdx.y, chunk = blockIdx.x;
    const int b = seg / Hkv, h = seg % Hkv;
    const int G = H / Hkv;
    // cache lengths outside [1, Lmax] are clamped so that no row outside the cache is read
    const int L = cache_len ? min(max(cache_len[b], 1), Lmax) : Lmax;
    const int n_top = min(max(top_count[seg], 0), top_cap);
    const int n_all = n_top + window;
    const int u0 = chunk * CH;
    if (u0 >= n_all) return;
    const int32_t* top = top_idx + (int64_t)seg * top_cap;
    const float* sc = scores + (int64_t)seg * Lmax;

    if (threadIdx.x < CH) {
        int u = u0 + threadIdx.x;
        int j = u < n_all ? list_key(u, top, n_top, L, window) : -1;
        j_s[threadIdx.x] = j;
        bias_s[threadIdx.x] = j >= 0 ? sc[j] : 0.f;
    }
    __syncthreads();
    // gather: all K and V rows of the chunk in flight at once
    const int64_t row_stride = (int64_t)Hkv * D;
    const T* Kh = Kc + ((int64_t)b * Lmax * Hkv + h) * D;
    const T* Vh = Vc + ((int64_t)b * Lmax * Hkv + h) * D;
    for (int c = threadIdx.x; c < CH * kCPR; c += kThreads) {
        const int r = c / kCPR, part = c % kCPR;
        const int j = j_s[r];
        if (j >= 0) {
            cp_async16(k_s + r * D + part * kElem, Kh + (int64_t)j * row_stride + part * kElem);
            cp_async16(v_s + r * D + part * kElem, Vh + (int64_t)j * row_stride + part * kElem);
        }
    }
    for (int t = threadIdx.x; t < G * D; t += kThreads) {
        const int g = t / D, d = t % D;
        q_s[t] = ld_f32<T>(q + ((int64_t)b * H + h * G + g) * D + d) * scale;
    }
    cp_async_wait_all();
    __syncthreads();

    // logits: one warp per row at a time, lanes split D
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < CH; r += kThreads / 32) {
        const int j = j_s[r];
        float kv[kDL];
#pragma unroll
        for (int e = 0; e < kDL; ++e) kv[e] = ld_f32<T>(k_s + r * D + lane * kDL + e);
        for (int g = 0; g < G; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < kDL; ++e) acc = fmaf(q_s[g * D + lane * kDL + e], kv[e], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) x_s[g * CH + r] = j >= 0 ? acc + bias_s[r] : -INFINITY;
        }
    }
    __syncthreads();
    // chunk-local softmax statistics per query head
    __shared__ float m_s[kMaxG], l_s[kMaxG];
    for (int g = warp; g < G; g += kThreads / 32) {
        float m = -INFINITY;
        for (int r = lane; r < CH; r += 32) m = fmaxf(m, x_s[g * CH + r]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int r = lane; r < CH; r += 32) {
            float x = x_s[g * CH + r];
            float p = x == -INFINITY ? 0.f : expf(x - m);
            x_s[g * CH + r] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            m_s[g] = m;
            l_s[g] = l;
        }
    }
    __syncthreads();
    // partial output: thread -> (query head, pair of d)
    for (int t = threadIdx.x; t < G * (D / 2); t += kThreads) {
        const int g = t / (D / 2), d = 2 * (t % (D / 2));
        float a0 = 0.f, a1 = 0.f;
        for (int r = 0; r < CH; ++r) {
            const float p = x_s[g * CH + r];
            if (p != 0.f) {
                a0 = fmaf(p, ld_f32<T>(v_s + r * D + d), a0);
                a1 = fmaf(p, ld_f32<T>(v_s + r * D + d + 1), a1);
            }
        }
        const int64_t pi = ((int64_t)b * H + h * G + g) * nchunk + chunk;
        part_o[pi * D + d] = a0;
        part_o[pi * D + d + 1] = a1;
    }
    if (threadIdx.x < G) {
        const int64_t pi = ((int64_t)b * H + h * G + threadIdx.x) * nchunk + chunk;
        part_ml[pi * 2] = m_s[threadIdx.x];
        part_ml[pi * 2 + 1] = l_s[threadIdx.x];
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(int H, int Hkv, const int32_t* __restrict__ top_count,
                                                         int top_cap, int window, int nchunk,
                                                         const float* __restrict__ part_o,
                                                         const float* __restrict__ part_ml, T* __restrict__ o,
                                                         float* __restrict__ lse)
{
    constexpr int CH = chunk_rows<T>();
    const int bh = blockIdx.x;  // b * H + hq
    const int b = bh / H, hq = bh % H;
    const int seg = b * Hkv + hq / (H / Hkv);
    const int used = min(nchunk, (min(max(top_count[seg], 0), top_cap) + window + CH - 1) / CH);
    const float* ml = part_ml + (int64_t)bh * nchunk * 2;
    float M = -INFINITY;
    for (int c = 0; c < used; ++c) M = fmaxf(M, ml[2 * c]);
    float Ls = 0.f, acc = 0.f;
    const int d = threadIdx.x;
    if (M != -INFINITY) {
        for (int c = 0; c < used; ++c) {
            const float mc = ml[2 * c];
            if (mc == -INFINITY) continue;
            const float wgt = expf(mc - M);
            Ls = fmaf(ml[2 * c + 1], wgt, Ls);
            acc = fmaf(part_o[((int64_t)bh * nchunk + c) * D + d], wgt, acc);
        }
    }
    o[(int64_t)bh * D + d] = to_out<T>(Ls > 0.f ? acc / Ls : 0.f);
    if (lse && d == 0) lse[bh] = Ls > 0.f ? M + logf(Ls) : -INFINITY;
}

int n_chunks(int top_cap, int window, int ch) { return (top_cap + window + ch - 1) / ch; }

template <typename T, int D>
cudaError_t launch_typed(const void* q, const void* Kc, const void* Vc, int B, int Lmax, const int32_t* cache_len,
                         int H, int Hkv, const float* scores, const dma_kept_t* kept, float scale, void* o, float* lse,
                         void* ws, cudaStream_t st)
{
    constexpr int CH = chunk_rows<T>();
    const int nchunk_ws = n_chunks(kept->top_cap, kept->window, 64);
    const int nchunk = n_chunks(kept->top_cap, kept->window, CH);
    float* part_o = static_cast<float*>(ws);
    float* part_ml = part_o + (size_t)B * H * nchunk_ws * D;
    size_t smem = 2 * sizeof(T) * CH * D + sizeof(float) * (kMaxG * D + kMaxG * CH) + 8 * CH;
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(nchunk, B * Hkv);
    decode_partial_kernel<T, D><<<grid, kThreads, smem, st>>>(
        static_cast<const T*>(q), static_cast<const T*>(Kc), static_cast<const T*>(Vc), Lmax, cache_len, H, Hkv,
        scores, kept->top_idx, kept->top_count, kept->top_cap, kept->window, scale, nchunk_ws, part_o, part_ml);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    decode_merge_kernel<T, D><<<B * H, D, 0, st>>>(H, Hkv, kept->top_count, kept->top_cap, kept->window, nchunk_ws,
                                                  part_o, part_ml,
                                                  static_cast<T*>(o), lse);
    return cudaGetLastError();
}

}  // namespace

size_t decode_ws_bytes(int B, int H, int Hkv, int D, int top_cap, int window)
{
    (void)Hkv;
    const size_t nchunk = (size_t)n_chunks(top_cap, window, 64);
    return sizeof(float) * (size_t)B * H * nchunk * (D + 2) + 256;
}

cudaError_t launch_decode(const void* q, const void* Kc, const void* Vc, dma_dtype_t dt, int B, int Lmax,
                          const int32_t* cache_len, int H, int Hkv, int D, const float* scores,
                          const dma_kept_t* kept, float scale, void* o, float* lse, void* ws, cudaStream_t st)
{
    if (H / Hkv > kMaxG) return cudaErrorInvalidValue;
    if (dt == DMA_BF16) {
        if (D == 128)
            return launch_typed<__nv_bfloat16, 128>(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, scores, kept, scale, o, lse,
                                                    ws, st);
        return launch_typed<__nv_bfloat16, 64>(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, scores, kept, scale, o, lse, ws,
                                               st);
    }
    if (D == 128)
        return launch_typed<float, 128>(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, scores, kept, scale, o, lse, ws, st);
    return launch_typed<float, 64>(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, scores, kept, scale, o, lse, ws, st);
}

}  // namespace dma

// ------------------------------------------------ decode without allocation --
//
// Some callers cannot call cudaMalloc at all: a serving loop that runs on a
// fixed memory plan, an embedding host library that has no access to the
// application's allocator, or code that may not trigger the device-wide
// synchronisation an allocation can imply.  For them the decode split-K
// partials live in this file-scope device array instead of a caller-provided
// workspace.  Every GPU that loads the library holds the array until the
// process exits.
namespace dma {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
void* g_scratch_addr[kNoAllocMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

}  // namespace dma

extern "C" dma_status_t dma_sparse_attn_decode_noalloc(const void* q, const void* Kc, const void* Vc, dma_dtype_t dt,
                                                       int B, int Lmax, const int32_t* cache_len, int H, int Hkv,
                                                       int D, const float* scores, const dma_kept_t* kept,
                                                       float scale, void* o, float* lse, dma_stream_t stream)
{
    using namespace dma;
    if (!kept) return set_error(DMA_ERR_INVALID_ARG, "kept is NULL");
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || kept->top_cap < 0 || kept->window < 0)
        return set_error(DMA_ERR_INVALID_ARG, "bad sizes B=%d H=%d Hkv=%d", B, H, Hkv);
    if (D != 64 && D != 128) return set_error(DMA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
    const size_t need = decode_ws_bytes(B, H, Hkv, D, kept->top_cap, kept->window);
    if (need > kNoAllocScratchBytes)
        return set_error(DMA_ERR_UNSUPPORTED,
                         "decode_noalloc needs %zu bytes of scratch, more than its fixed %zu; use "
                         "dma_sparse_attn_decode with a workspace", need, kNoAllocScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(DMA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kNoAllocMaxDevices) return set_error(DMA_ERR_UNSUPPORTED, "device ordinal %d", dev);
    void* scratch = nullptr;
    {
        // first call on this device: look up the array's device address with the
        // device current (the host-side name is only a stand-in for it)
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess)
                return set_error(DMA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    return dma_sparse_attn_decode(q, Kc, Vc, dt, B, Lmax, cache_len, H, Hkv, D, scores, kept, scale, o, lse,
                                  scratch, kNoAllocScratchBytes, stream);
}
