// Key scoring: s[b,h,j] = A_h * softplus(<V[b,j,h,:], W[h,:]>).
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §五: the dynamic weight is
// delta = exp(tau(v Delta) * A) with tau non-negative; its logarithm, with tau =
// softplus, a per-KV-head vector Delta = W[h] and gate A_h, is the score.
//
// With a bias array, the kernel also writes the value the logits get: s itself,
// or (exp form) delta = exp(s), the dynamic weight as the summary writes it.  The
// selection ranks s either way: exp is increasing, so the kept sets are those of
// delta, without the ties that rounding large delta to fp32 would add.
//
// HBM-bound: every value row is read once (D * elem bytes) and 4 bytes are
// written per (key, head) and output array.  The rows of TJ consecutive keys and
// all Hkv heads are one contiguous span of V.  A CTA covers a fixed number of
// rows (TJ = that number / Hkv): each thread issues the 16-byte loads of all of
// its rows at once, every row is reduced by the lanes that hold it, each lane
// then takes the softplus of one row (no lane idles through another's), and the
// TJ scores of each head go out as one coalesced run.
#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreIters = 16;  // rows per thread: a CTA covers kScoreIters * (threads / lanes per row) rows

// Rows (j, h) of one CTA: floor(rows per CTA / Hkv) consecutive keys, all heads.
template <typename T, int D>
constexpr int score_rows_per_cta()
{
    return kScoreIters * (kScoreThreads / (D / (16 / (int)sizeof(T))));
}

template <typename T, int D>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const T* __restrict__ V, int S, int Hkv, int key_begin,
                                                              int key_end, int TJ, const float* __restrict__ W,
                                                              const float* __restrict__ A, float* __restrict__ out,
                                                              float* __restrict__ bias, int exp_form)
{
    constexpr int kElem = 16 / sizeof(T);    // elements per 16-byte chunk
    constexpr int kCPR = D / kElem;          // chunks (lanes) per row, 8..32
    constexpr int kGroups = kScoreThreads / kCPR;
    constexpr int kKeep = (kScoreIters + kCPR - 1) / kCPR;  // row sums each lane keeps for the softplus

    extern __shared__ float smem[];
    float* w_s = smem;                        // [Hkv][D]
    float* s_s = smem + Hkv * D;              // [Hkv][TJ]

    const int b = blockIdx.y;
    const int j0 = key_begin + blockIdx.x * TJ;
    const int nj = min(TJ, key_end - j0);
    const int lane_in_row = threadIdx.x % kCPR;
    const int group = threadIdx.x / kCPR;
    const int rows = nj * Hkv;  // rows (j, h) of this tile, contiguous in V
    const uint4* base = reinterpret_cast<const uint4*>(V + ((int64_t)b * S + j0) * Hkv * D);

    // every chunk of the thread's rows in flight at once, the weights staged meanwhile
    uint4 c[kScoreIters];
#pragma unroll
    for (int it = 0; it < kScoreIters; ++it) {
        const int r = it * kGroups + group;
        c[it] = r < rows ? __ldg(base + (int64_t)r * kCPR + lane_in_row) : make_uint4(0, 0, 0, 0);
    }
    for (int t = threadIdx.x; t < Hkv * D; t += kScoreThreads) w_s[t] = W[t];
    __syncthreads();

    // Row it of the group is reduced across its kCPR lanes (every lane ends with the sum);
    // lane it % kCPR keeps it for the softplus below.
    float keep[kKeep];
#pragma unroll
    for (int e = 0; e < kKeep; ++e) keep[e] = 0.f;
#pragma unroll
    for (int it = 0; it < kScoreIters; ++it) {
        const int r = it * kGroups + group;
        const float* wr = w_s + (r % Hkv) * D + lane_in_row * kElem;
        float acc = 0.f;
        if constexpr (sizeof(T) == 2) {
            const uint32_t u[4] = {c[it].x, c[it].y, c[it].z, c[it].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(bf16_lo(u[e]), wr[2 * e], acc);
                acc = fmaf(bf16_hi(u[e]), wr[2 * e + 1], acc);
            }
        } else {
            acc = fmaf(__uint_as_float(c[it].x), wr[0], acc);
            acc = fmaf(__uint_as_float(c[it].y), wr[1], acc);
            acc = fmaf(__uint_as_float(c[it].z), wr[2], acc);
            acc = fmaf(__uint_as_float(c[it].w), wr[3], acc);
        }
#pragma unroll
        for (int o = kCPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, kCPR);
        if (lane_in_row == it % kCPR) keep[it / kCPR] = acc;
    }
#pragma unroll
    for (int e = 0; e < kKeep; ++e) {
        const int it = e * kCPR + lane_in_row;
        const int r = it * kGroups + group;
        if (it < kScoreIters && r < rows) {
            const int h = r % Hkv;
            const float x = keep[e];
            // softplus(x) = max(x, 0) + log1p(exp(-|x|))
            const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
            s_s[h * TJ + r / Hkv] = (A ? A[h] : 1.f) * sp;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < Hkv * TJ; t += kScoreThreads) {
        const int h = t / TJ, jj = t % TJ;
        if (jj < nj) {
            const int64_t o = ((int64_t)b * Hkv + h) * S + j0 + jj;
            out[o] = s_s[t];
            if (bias) bias[o] = exp_form ? expf(s_s[t]) : s_s[t];
        }
    }
}

template <typename T, int D>
cudaError_t launch_typed(const void* V, int B, int S, int Hkv, int key_begin, int key_end, const float* W,
                         const float* A, float* scores, float* bias, int exp_form, cudaStream_t st)
{
    // keys per CTA: as many as fill its rows (the entry point accepts at most 128 KV heads, no
    // more than the rows of any instantiation, so every CTA covers at least one whole key)
    static_assert(score_rows_per_cta<T, D>() >= 128, "a CTA covers the rows of one key of 128 KV heads");
    const int TJ = std::max(1, score_rows_per_cta<T, D>() / Hkv);
    dim3 grid((key_end - key_begin + TJ - 1) / TJ, B);
    size_t smem = sizeof(float) * ((size_t)Hkv * D + (size_t)Hkv * TJ);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(score_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    score_kernel<T, D><<<grid, kScoreThreads, smem, st>>>(static_cast<const T*>(V), S, Hkv, key_begin, key_end, TJ,
                                                          W, A, scores, bias, exp_form);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin, int key_end,
                         const float* W, const float* A, float* scores, float* bias, int exp_form, cudaStream_t st)
{
    if (key_end <= key_begin) return cudaSuccess;
    if (dt == DMA_BF16) {
        if (D == 128)
            return launch_typed<__nv_bfloat16, 128>(V, B, S, Hkv, key_begin, key_end, W, A, scores, bias, exp_form, st);
        return launch_typed<__nv_bfloat16, 64>(V, B, S, Hkv, key_begin, key_end, W, A, scores, bias, exp_form, st);
    }
    if (D == 128) return launch_typed<float, 128>(V, B, S, Hkv, key_begin, key_end, W, A, scores, bias, exp_form, st);
    return launch_typed<float, 64>(V, B, S, Hkv, key_begin, key_end, W, A, scores, bias, exp_form, st);
}

}  // namespace dma
