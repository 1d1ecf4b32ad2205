// Sparse attention prefill, SIMT kernel (fp32 inputs, and any dtype when the
// tensor-core kernel is not selected).
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §四/§五: positions whose mask
// is -inf are skipped outright -- no query-key product at all -- and since
// their weight would be exactly 0 the result equals the full masked softmax.
// For a query tile [q0, q1] the only keys touched are the tile's gathered list
// (keys outside the window band whose top-set interval meets the tile) and the
// window band (q0 - window, q1].  Per (row i, key j) the mask is
//     j <= i  and  (j > i - window  or  lo_j <= i < expiry_j)
// and the logit is scale * <Q_i, K_j> + s_j.
//
// Layout of the work: one CTA = 64 query rows of one query head; 4 threads per
// row, each holding D/4 of q and of the output accumulator.  Keys stream through
// shared memory 32 at a time (converted to fp32); each 32-key tile does one
// online-softmax rescale.
#include <cmath>

#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kRows = 64;
constexpr int kTPR = 4;  // threads per row
constexpr int kThreads = kRows * kTPR;
constexpr int kNK = 32;  // keys per shared-memory tile

template <typename T>
__device__ __forceinline__ void load_row_f32(const T* src, float* dst, int D, int part, int nparts)
{
    // copies one D-element row as fp32, 16 bytes of source per step
    constexpr int kElem = 16 / sizeof(T);
    for (int c = part; c < D / kElem; c += nparts) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + c);
        if constexpr (sizeof(T) == 2) {
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dst[c * 8 + 2 * e] = bf16_lo(u[e]);
                dst[c * 8 + 2 * e + 1] = bf16_hi(u[e]);
            }
        } else {
            reinterpret_cast<float4*>(dst)[c] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                                            __uint_as_float(v.z), __uint_as_float(v.w));
        }
    }
}

template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, int S, int H, int Hkv,
    const float* __restrict__ scores, const int32_t* __restrict__ expiry, const int32_t* __restrict__ tile_cnt,
    const int32_t* __restrict__ tile_idx, int n_qt, int tile_stride, int window, int block, float scale,
    T* __restrict__ O, float* __restrict__ lse)
{
    constexpr int kDP = D / kTPR;  // elements per thread
    constexpr int kC4 = kDP / 4;   // float4 chunks per thread
    __shared__ __align__(16) float k_s[kNK][D];
    __shared__ __align__(16) float v_s[kNK][D];
    __shared__ int j_s[kNK];
    __shared__ int lo_s[kNK];
    __shared__ int ex_s[kNK];
    __shared__ float b_s[kNK];

    const int b = blockIdx.z, hq = blockIdx.y;
    const int G = H / Hkv, h = hq / G;
    const int r0 = blockIdx.x * kRows;
    const int tile = r0 / kQTile;
    const int q0 = tile * kQTile, q1 = min(S, q0 + kQTile) - 1;
    const int seg = b * Hkv + h;
    const int row = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;
    const int i = r0 + row;

    // q slice: chunks sub, sub + 4, ... of 4 elements each
    float q[kDP];
    {
        const T* qp = Q + (((int64_t)b * S + min(i, S - 1)) * H + hq) * D;
#pragma unroll
        for (int c = 0; c < kC4; ++c) {
            int d0 = (c * kTPR + sub) * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) q[c * 4 + e] = (float)qp[d0 + e] * scale;
        }
    }
    float o[kDP];
#pragma unroll
    for (int t = 0; t < kDP; ++t) o[t] = 0.f;
    float m = -INFINITY, l = 0.f;

    const int n_g = tile_cnt[(int64_t)seg * n_qt + tile];
    const int32_t* gl = tile_idx + ((int64_t)seg * n_qt + tile) * tile_stride;
    const int band_lo = window > 0 ? max(0, q0 - window + 1) : q1 + 1;
    const int n_b = window > 0 ? q1 + 1 - band_lo : 0;
    const int n_all = n_g + n_b;
    const float* sc = scores + (int64_t)seg * S;
    const int32_t* ex = expiry + (int64_t)seg * S;
    const int64_t kv_row_stride = (int64_t)Hkv * D;
    const T* Kh = K + ((int64_t)b * S * Hkv + h) * D;
    const T* Vh = V + ((int64_t)b * S * Hkv + h) * D;

    for (int u0 = 0; u0 < n_all; u0 += kNK) {
        __syncthreads();
        if (threadIdx.x < kNK) {
            int u = u0 + threadIdx.x;
            int j = -1;
            if (u < n_all) j = u < n_g ? gl[u] : band_lo + (u - n_g);
            if (j >= S) j = -1;  // never produced by the selection; skipped rather than read
            j_s[threadIdx.x] = j;
            lo_s[threadIdx.x] = j >= 0 ? top_lo(j, block) : 0;
            ex_s[threadIdx.x] = j >= 0 ? ex[j] : 0;
            b_s[threadIdx.x] = j >= 0 ? sc[j] : 0.f;
        }
        __syncthreads();
        // 8 threads per key row: K and V rows to fp32 shared memory.  An empty slot (past the
        // end of the list) gets zeros: its weight is 0, and 0 times stale shared memory (NaN
        // bits left by an earlier kernel) would not be.
        {
            const int kr = threadIdx.x / 8, part = threadIdx.x % 8;
            const int j = j_s[kr];
            if (j >= 0) {
                load_row_f32<T>(Kh + (int64_t)j * kv_row_stride, k_s[kr], D, part, 8);
                load_row_f32<T>(Vh + (int64_t)j * kv_row_stride, v_s[kr], D, part, 8);
            } else {
                for (int d = part; d < D; d += 8) {
                    k_s[kr][d] = 0.f;
                    v_s[kr][d] = 0.f;
                }
            }
        }
        __syncthreads();
        float x[kNK];
        float mt = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < kNK; ++kk) {
            const float4* kr = reinterpret_cast<const float4*>(k_s[kk]);
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < kC4; ++c) {
                float4 kv = kr[c * kTPR + sub];
                acc = fmaf(q[c * 4 + 0], kv.x, acc);
                acc = fmaf(q[c * 4 + 1], kv.y, acc);
                acc = fmaf(q[c * 4 + 2], kv.z, acc);
                acc = fmaf(q[c * 4 + 3], kv.w, acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1, kTPR);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2, kTPR);
            const int j = j_s[kk];
            const bool kept = j >= 0 && j <= i && (j > i - window || (lo_s[kk] <= i && i < ex_s[kk]));
            x[kk] = kept ? acc + b_s[kk] : -INFINITY;
            mt = fmaxf(mt, x[kk]);
        }
        const float m_new = fmaxf(m, mt);
        if (m_new == -INFINITY) continue;
        const float alpha = expf(m - m_new);  // 0 when m = -inf
        l *= alpha;
#pragma unroll
        for (int t = 0; t < kDP; ++t) o[t] *= alpha;
#pragma unroll
        for (int kk = 0; kk < kNK; ++kk) {
            const float p = expf(x[kk] - m_new);
            l += p;
            const float4* vr = reinterpret_cast<const float4*>(v_s[kk]);
#pragma unroll
            for (int c = 0; c < kC4; ++c) {
                float4 vv = vr[c * kTPR + sub];
                o[c * 4 + 0] = fmaf(p, vv.x, o[c * 4 + 0]);
                o[c * 4 + 1] = fmaf(p, vv.y, o[c * 4 + 1]);
                o[c * 4 + 2] = fmaf(p, vv.z, o[c * 4 + 2]);
                o[c * 4 + 3] = fmaf(p, vv.w, o[c * 4 + 3]);
            }
        }
        m = m_new;
    }
    if (i >= S) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T* op = O + (((int64_t)b * S + i) * H + hq) * D;
#pragma unroll
    for (int c = 0; c < kC4; ++c) {
        int d0 = (c * kTPR + sub) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) op[d0 + e] = to_out<T>(o[c * 4 + e] * inv);
    }
    if (lse && sub == 0) lse[((int64_t)b * H + hq) * S + i] = l > 0.f ? m + logf(l) : -INFINITY;
}

template <typename T, int D>
cudaError_t launch_typed(const void* Q, const void* K, const void* V, int B, int S, int H, int Hkv,
                         const float* scores, const dma_kept_t* kept, float scale, void* O, float* lse,
                         cudaStream_t st)
{
    dim3 grid((S + kRows - 1) / kRows, H, B);
    prefill_simt_kernel<T, D><<<grid, kThreads, 0, st>>>(
        static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V), S, H, Hkv, scores,
        kept->expiry, kept->tile_cnt, kept->tile_idx, kept->n_qt, kept->tile_stride, kept->window, kept->block, scale,
        static_cast<T*>(O), lse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const void* Q, const void* K, const void* V, dma_dtype_t dt, int B, int S, int H,
                                int Hkv, int D, const float* scores, const dma_kept_t* kept, float scale, void* O,
                                float* lse, cudaStream_t st)
{
    if (dt == DMA_BF16) {
        if (D == 128) return launch_typed<__nv_bfloat16, 128>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, st);
        return launch_typed<__nv_bfloat16, 64>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, st);
    }
    if (D == 128) return launch_typed<float, 128>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, st);
    return launch_typed<float, 64>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, st);
}

}  // namespace dma
