// Page-granular decode selection over a paged KV cache.
//
// Sparse Frontier summary (techwalker.com), decode findings: page-level (Quest)
// selection keeps the whole KV cache and chooses pages of it; DMA summary (lsdiaocha.cn)
// §五 and §七: the same content-derived key scores and top-k rule in every phase.  Here
// a page's score is the maximum of its keys' scores (as for the 64-key selection
// blocks), and the decode row L-1 keeps the floor(w / page_size) complete pages (last
// key <= L-1) with the highest page scores, ties to the lower page index; the window
// band is added by the decode kernel as for token units.
//
// Paged cache: K and V pages [n_pages][page_size][Hkv][D]; logical page p of sequence b
// (keys p * page_size .. p * page_size + page_size - 1) is physical page
// block_table[b][p].  Scores and page scores are kept per logical position.
#include <cmath>

#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kPagedThreads = 256;
constexpr int kPagedWarps = kPagedThreads / 32;
constexpr int kSelectThreads = 1024;

// Order-preserving key of the ranking (ascending = best first): the score as fp32, -0 as
// +0, NaN last.
__device__ __forceinline__ uint32_t rank_key(float s)
{
    if (s != s) return 0xffffffffu;
    if (s == 0.f) s = 0.f;
    uint32_t u = __float_as_uint(s);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~u;
}

// Physical row of logical key j of a sequence, or -1 when its page entry is out of range.
__device__ __forceinline__ int64_t paged_row(const int32_t* bt_b, int j, int pshift, int n_pages)
{
    const int phys = bt_b[j >> pshift];
    if (phys < 0 || phys >= n_pages) return -1;
    return ((int64_t)phys << pshift) + (j & ((1 << pshift) - 1));
}

// s[b][h][j] = A_h softplus(<V_j,h, W_h>) for keys key_begin <= j < min(key_end, L_b): one warp
// per (b, j); the Hkv value rows of a key are contiguous in its page.
template <typename T, int D>
__global__ void __launch_bounds__(kPagedThreads) score_paged_kernel(const T* __restrict__ Vp,
                                                                    const int32_t* __restrict__ bt, int n_pages,
                                                                    int max_pages, int pshift, int Hkv, int key_begin,
                                                                    int key_end, const int32_t* __restrict__ cache_len,
                                                                    const float* __restrict__ W,
                                                                    const float* __restrict__ A,
                                                                    float* __restrict__ scores,
                                                                    float* __restrict__ bias, int exp_form,
                                                                    int* status)
{
    constexpr int kElem = 16 / sizeof(T);
    constexpr int kCPR = D / kElem;  // lanes per row: 8, 16 or 32
    constexpr int kRowsPerWarp = 32 / kCPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int j = key_begin + blockIdx.x * kPagedWarps + warp;
    const int Lmax = max_pages << pshift;
    const int L = cache_len ? min(cache_len[b], Lmax) : Lmax;
    if (j >= key_end || j >= L) return;  // whole warp
    const int64_t row = paged_row(bt + (int64_t)b * max_pages, j, pshift, n_pages);
    if (row < 0) {
        if (lane == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
        return;
    }
    const T* base = Vp + row * Hkv * D;
    const int part = lane % kCPR;
    for (int h0 = 0; h0 < Hkv; h0 += kRowsPerWarp) {  // the same trip count for every lane
        const int h = h0 + lane / kCPR;
        const bool valid = h < Hkv;
        float acc = 0.f;
        if (valid) {
            const uint4 c = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)h * D) + part);
            const float* wr = W + h * D + part * kElem;
            if constexpr (sizeof(T) == 2) {
                const uint32_t u[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(bf16_lo(u[e]), wr[2 * e], acc);
                    acc = fmaf(bf16_hi(u[e]), wr[2 * e + 1], acc);
                }
            } else {
                acc = fmaf(__uint_as_float(c.x), wr[0], acc);
                acc = fmaf(__uint_as_float(c.y), wr[1], acc);
                acc = fmaf(__uint_as_float(c.z), wr[2], acc);
                acc = fmaf(__uint_as_float(c.w), wr[3], acc);
            }
        }
#pragma unroll
        for (int o = kCPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, kCPR);
        if (valid && part == 0) {
            // softplus(x) = max(x, 0) + log1p(exp(-|x|))
            const float sp = fmaxf(acc, 0.f) + log1pf(expf(-fabsf(acc)));
            const float sv = (A ? A[h] : 1.f) * sp;
            const int64_t o = ((int64_t)b * Hkv + h) * Lmax + j;
            scores[o] = sv;
            // the logits' bias, when asked for: s itself or (exp form) delta = exp(s)
            if (bias) bias[o] = exp_form ? expf(sv) : sv;
        }
    }
}

// ps[b][h][p] = max of scores[b][h][j] over the keys j < L_b of page p, for the pages that hold a
// key of [key_begin, key_end); one warp per (b, h, page).
__global__ void __launch_bounds__(kPagedThreads) page_max_kernel(const float* __restrict__ scores,
                                                                 const int32_t* __restrict__ cache_len, int Hkv,
                                                                 int max_pages, int pshift, int p_begin, int n_p,
                                                                 float* __restrict__ page_scores)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int t = blockIdx.x * kPagedWarps + warp;
    if (t >= n_p * Hkv) return;  // whole warp
    const int h = t / n_p, p = p_begin + t % n_p;
    const int Lmax = max_pages << pshift;
    const int L = cache_len ? min(cache_len[b], Lmax) : Lmax;
    const int P = 1 << pshift;
    const int j0 = p * P, j1 = min(L, j0 + P);
    const float* sc = scores + ((int64_t)b * Hkv + h) * Lmax;
    float m = -INFINITY;
    for (int j = j0 + lane; j < j1; j += 32) m = fmaxf(m, sc[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) page_scores[((int64_t)b * Hkv + h) * max_pages + p] = m;
}

// Ascending bitonic sort of n (a power of two) 64-bit keys in shared memory by the whole CTA.
__device__ void bitonic_sort(unsigned long long* keys, int n)
{
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
                const int idx = 2 * stride * (i / stride) + (i % stride);
                const int partner = idx + stride;
                const bool up = (idx & size) == 0;
                const unsigned long long x = keys[idx], y = keys[partner];
                if ((x > y) == up) {
                    keys[idx] = y;
                    keys[partner] = x;
                }
            }
            __syncthreads();
        }
    }
}

// The kept pages of the decode row of one (b, h) segment, written as their keys (ascending).
// The budget is w keys, or w_head[h] (clamped into [0, w], an entry outside recorded) when
// given: floor(budget / page size) pages.
__global__ void __launch_bounds__(kSelectThreads) select_pages_kernel(const float* __restrict__ page_scores,
                                                                      const int32_t* __restrict__ cache_len, int Hkv,
                                                                      int max_pages, int pshift, int w,
                                                                      const int32_t* __restrict__ w_head,
                                                                      int32_t* __restrict__ top_idx,
                                                                      int32_t* __restrict__ top_count, int top_cap,
                                                                      int* status)
{
    extern __shared__ unsigned long long keys[];  // [pow2 >= complete pages]
    const int seg = blockIdx.x, b = seg / Hkv;
    const int Lmax = max_pages << pshift;
    const int L = cache_len ? min(max(cache_len[b], 0), Lmax) : Lmax;
    const int n_c = min(L >> pshift, max_pages);  // complete pages
    int wb = w;
    if (w_head) {
        wb = w_head[seg % Hkv];
        if (wb < 0 || wb > w) {
            if (threadIdx.x == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
            wb = wb < 0 ? 0 : w;
        }
    }
    const int k = min(wb >> pshift, n_c);
    const float* ps = page_scores + (int64_t)seg * max_pages;
    const int P = 1 << pshift;
    if (k < n_c && n_c <= kSelectThreads) {
        // one thread per complete page: its rank is the number of pages that beat it (the same
        // (score rank, page index) order), and it is kept iff that is below k; the kept pages go
        // out in page order through a block-wide prefix of the kept flags
        __shared__ int warp_kept[kSelectThreads / 32];
        for (int i = threadIdx.x; i < n_c; i += blockDim.x)
            keys[i] = ((unsigned long long)rank_key(ps[i]) << 32) | (unsigned)i;
        __syncthreads();
        bool kept = false;
        if ((int)threadIdx.x < n_c) {
            const unsigned long long mine = keys[threadIdx.x];
            int rank = 0;
#pragma unroll 8
            for (int q = 0; q < n_c; ++q) rank += keys[q] < mine ? 1 : 0;
            kept = rank < k;
        }
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        const unsigned bal = __ballot_sync(0xffffffffu, kept);
        if (lane == 0) warp_kept[wid] = __popc(bal);
        __syncthreads();  // every rank is counted before keys[] is reused below
        int before = __popc(bal & ((1u << lane) - 1u));
        for (int w2 = 0; w2 < wid; ++w2) before += warp_kept[w2];
        if (kept) keys[before] = (unsigned)threadIdx.x;
        __syncthreads();
    } else if (k < n_c) {
        int n = 1;
        while (n < n_c) n <<= 1;
        // best first: (score rank, page index) ascending
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            keys[i] = i < n_c ? ((unsigned long long)rank_key(ps[i]) << 32) | (unsigned)i : ~0ull;
        __syncthreads();
        bitonic_sort(keys, n);
        // the k best, by page index
        int m = 1;
        while (m < k) m <<= 1;
        for (int i = threadIdx.x; i < m; i += blockDim.x) keys[i] = i < k ? (keys[i] & 0xffffffffull) : ~0ull;
        __syncthreads();
        bitonic_sort(keys, m);
    } else {
        for (int i = threadIdx.x; i < k; i += blockDim.x) keys[i] = (unsigned)i;
        __syncthreads();
    }
    int32_t* out = top_idx + (int64_t)seg * top_cap;
    for (int t = threadIdx.x; t < k * P; t += blockDim.x) out[t] = ((int)keys[t >> pshift] << pshift) + (t & (P - 1));
    if (threadIdx.x == 0) top_count[seg] = k * P;
}

// The same selection with one warp per (b, h) segment (two to a CTA: spread over more SMs than
// eight, 12% faster), for tables of up to 32 * kRounds pages:
// lane l holds the rank keys of pages l, l + 32, ... in registers.  A bitwise radix select,
// most significant bit first, finds the k-th smallest key: at each bit, the pages that agree
// with the bits chosen so far are counted by ballots, split by that bit; if enough of them
// have a 0 there, the bit is 0 and those with a 1 are out, otherwise it is 1 and those with a
// 0 are in.  The pages whose whole key equals the selected one then fill what is left, lowest
// page index first.  The kept pages go to shared memory in page order, then out as their keys.
constexpr int kWarpSelectWarps = 2;

template <int kRounds>
__global__ void __launch_bounds__(kWarpSelectWarps * 32) select_pages_warp_kernel(
    const float* __restrict__ page_scores, const int32_t* __restrict__ cache_len, int B, int Hkv, int max_pages,
    int pshift, int w, const int32_t* __restrict__ w_head, int32_t* __restrict__ top_idx,
    int32_t* __restrict__ top_count, int top_cap, int* status)
{
    __shared__ int32_t kept_pages[kWarpSelectWarps][32 * kRounds];
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x * kWarpSelectWarps + wid;
    if (seg >= B * Hkv) return;  // whole warp
    const int b = seg / Hkv;
    const int Lmax = max_pages << pshift;
    const int L = cache_len ? min(max(cache_len[b], 0), Lmax) : Lmax;
    const int n_c = min(L >> pshift, max_pages);  // complete pages
    int wb = w;
    if (w_head) {
        wb = w_head[seg % Hkv];
        if (wb < 0 || wb > w) {
            if (lane == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
            wb = wb < 0 ? 0 : w;
        }
    }
    const int k = min(wb >> pshift, n_c);
    const float* ps = page_scores + (int64_t)seg * max_pages;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t key[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int p = 32 * r + lane;
        key[r] = p < n_c ? rank_key(ps[p]) : 0xffffffffu;
    }
    uint32_t sel = 0;  // the bits of the k-th smallest key chosen so far
    int need = k;      // pages agreeing with those bits still to keep
    if (k > 0 && k < n_c) {
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t hi = bit == 31 ? 0u : ~0u << (bit + 1);  // the bits already chosen
            int zeros = 0;
#pragma unroll
            for (int r = 0; r < kRounds; ++r) {
                const bool zero = 32 * r + lane < n_c && ((key[r] ^ sel) & hi) == 0 && ((key[r] >> bit) & 1u) == 0;
                zeros += __popc(__ballot_sync(0xffffffffu, zero));
            }
            if (need > zeros) {
                need -= zeros;
                sel |= 1u << bit;
            }
        }
    }
    // kept: every page when k >= n_c; else a key below the selected one, or equal to it and
    // among the first `need` such pages
    int32_t* mine = kept_pages[wid];
    int n_kept = 0, n_tied = 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int p = 32 * r + lane;
        bool kept = p < n_c && k > 0;
        if (k < n_c) {
            const bool tied = p < n_c && key[r] == sel;
            const unsigned tb = __ballot_sync(0xffffffffu, tied);
            kept = k > 0 && ((p < n_c && key[r] < sel) || (tied && n_tied + __popc(tb & lt) < need));
            n_tied += __popc(tb);
        }
        const unsigned kb = __ballot_sync(0xffffffffu, kept);
        if (kept) mine[n_kept + __popc(kb & lt)] = p;
        n_kept += __popc(kb);
    }
    __syncwarp();
    const int P = 1 << pshift;
    int32_t* out = top_idx + (int64_t)seg * top_cap;
    for (int t = lane; t < k * P; t += 32) out[t] = (mine[t >> pshift] << pshift) + (t & (P - 1));
    if (lane == 0) top_count[seg] = k * P;
}

template <typename T, int D>
cudaError_t score_paged_typed(const void* Vp, const int32_t* bt, int n_pages, int B, int max_pages, int pshift,
                              int Hkv, int key_begin, int key_end, const int32_t* cache_len, const float* W,
                              const float* A, float* scores, float* page_scores, float* bias, int exp_form,
                              int* status, cudaStream_t st)
{
    const int nk = key_end - key_begin;
    dim3 grid((nk + kPagedWarps - 1) / kPagedWarps, B);
    score_paged_kernel<T, D><<<grid, kPagedThreads, 0, st>>>(static_cast<const T*>(Vp), bt, n_pages, max_pages,
                                                             pshift, Hkv, key_begin, key_end, cache_len, W, A, scores,
                                                             bias, exp_form, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !page_scores) return e;
    const int p_begin = key_begin >> pshift, n_p = ((key_end - 1) >> pshift) - p_begin + 1;
    dim3 g2((n_p * Hkv + kPagedWarps - 1) / kPagedWarps, B);
    page_max_kernel<<<g2, kPagedThreads, 0, st>>>(scores, cache_len, Hkv, max_pages, pshift, p_begin, n_p,
                                                 page_scores);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_paged(const void* Vp, dma_dtype_t dt, const int32_t* bt, int n_pages, int B, int max_pages,
                               int pshift, int Hkv, int D, int key_begin, int key_end, const int32_t* cache_len,
                               const float* W, const float* A, float* scores, float* page_scores, float* bias,
                               int exp_form, int* status, cudaStream_t st)
{
    if (key_end <= key_begin) return cudaSuccess;
    if (dt == DMA_BF16)
        return D == 128 ? score_paged_typed<__nv_bfloat16, 128>(Vp, bt, n_pages, B, max_pages, pshift, Hkv, key_begin,
                                                                key_end, cache_len, W, A, scores, page_scores, bias,
                                                                exp_form, status, st)
                        : score_paged_typed<__nv_bfloat16, 64>(Vp, bt, n_pages, B, max_pages, pshift, Hkv, key_begin,
                                                               key_end, cache_len, W, A, scores, page_scores, bias,
                                                               exp_form, status, st);
    return D == 128 ? score_paged_typed<float, 128>(Vp, bt, n_pages, B, max_pages, pshift, Hkv, key_begin, key_end,
                                                    cache_len, W, A, scores, page_scores, bias, exp_form, status, st)
                    : score_paged_typed<float, 64>(Vp, bt, n_pages, B, max_pages, pshift, Hkv, key_begin, key_end,
                                                   cache_len, W, A, scores, page_scores, bias, exp_form, status, st);
}

cudaError_t launch_select_pages(const float* page_scores, int B, int Hkv, int max_pages, int pshift,
                                const int32_t* cache_len, int w, const int32_t* w_head, int32_t* top_idx,
                                int32_t* top_count, int top_cap, int* status, cudaStream_t st)
{
    cudaError_t e = cudaSuccess;
    if (max_pages <= 1024) {
        const int grid = (B * Hkv + kWarpSelectWarps - 1) / kWarpSelectWarps;
        if (max_pages <= 512)
            select_pages_warp_kernel<16><<<grid, kWarpSelectWarps * 32, 0, st>>>(
                page_scores, cache_len, B, Hkv, max_pages, pshift, w, w_head, top_idx, top_count, top_cap, status);
        else
            select_pages_warp_kernel<32><<<grid, kWarpSelectWarps * 32, 0, st>>>(
                page_scores, cache_len, B, Hkv, max_pages, pshift, w, w_head, top_idx, top_count, top_cap, status);
        return cudaGetLastError();
    }
    int n = 1;
    while (n < max_pages) n <<= 1;
    const int smem = n * 8;
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(select_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
            cudaSuccess)
        return e;
    select_pages_kernel<<<B * Hkv, kSelectThreads, smem, st>>>(page_scores, cache_len, Hkv, max_pages, pshift, w,
                                                               w_head, top_idx, top_count, top_cap, status);
    return cudaGetLastError();
}

}  // namespace dma
