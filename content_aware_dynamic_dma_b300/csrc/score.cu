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
// written per (key, head) and output array.  The rows of TJ consecutive keys and all Hkv heads are
// one contiguous span of V, so a CTA streams that span with 16-byte loads, each
// row reduced by the CPR lanes that hold it, and writes the TJ scores of each
// head as one coalesced run.
#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreTJ = 32;  // keys per CTA

template <typename T, int D>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const T* __restrict__ V, int S, int Hkv, int key_begin,
                                                              int key_end, const float* __restrict__ W,
                                                              const float* __restrict__ A, float* __restrict__ out,
                                                              float* __restrict__ bias, int exp_form)
{
    constexpr int kElem = 16 / sizeof(T);    // elements per 16-byte chunk
    constexpr int kCPR = D / kElem;          // chunks per row (8..32)
    constexpr int kGroups = kScoreThreads / kCPR;

    extern __shared__ float smem[];
    float* w_s = smem;                        // [Hkv][D]
    float* s_s = smem + Hkv * D;              // [Hkv][kScoreTJ]

    const int b = blockIdx.y;
    const int j0 = key_begin + blockIdx.x * kScoreTJ;
    const int nj = min(kScoreTJ, key_end - j0);
    for (int t = threadIdx.x; t < Hkv * D; t += kScoreThreads) w_s[t] = W[t];
    __syncthreads();

    const int lane_in_row = threadIdx.x % kCPR;
    const int group = threadIdx.x / kCPR;
    const int rows = nj * Hkv;  // rows (j, h) of this tile, contiguous in V
    const uint4* base = reinterpret_cast<const uint4*>(V + ((int64_t)b * S + j0) * Hkv * D);

    // The trip count is uniform over the CTA so that every lane reaches the shuffles.
#pragma unroll 4
    for (int r0 = 0; r0 < rows; r0 += kGroups) {
        const int r = r0 + group;
        const bool valid = r < rows;
        const int h = r % Hkv;
        uint4 c = valid ? __ldg(base + (int64_t)r * kCPR + lane_in_row) : make_uint4(0, 0, 0, 0);
        const float* wr = w_s + h * D + lane_in_row * kElem;
        float acc = 0.f;
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
#pragma unroll
        for (int o = kCPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, kCPR);
        if (valid && lane_in_row == 0) {
            // softplus(x) = max(x, 0) + log1p(exp(-|x|))
            float sp = fmaxf(acc, 0.f) + log1pf(expf(-fabsf(acc)));
            float a = A ? A[h] : 1.f;
            s_s[h * kScoreTJ + r / Hkv] = a * sp;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < Hkv * kScoreTJ; t += kScoreThreads) {
        int h = t / kScoreTJ, jj = t % kScoreTJ;
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
    dim3 grid((key_end - key_begin + kScoreTJ - 1) / kScoreTJ, B);
    size_t smem = sizeof(float) * (size_t)Hkv * (D + kScoreTJ);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(score_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    score_kernel<T, D><<<grid, kScoreThreads, smem, st>>>(static_cast<const T*>(V), S, Hkv, key_begin, key_end, W,
                                                          A, scores, bias, exp_form);
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
