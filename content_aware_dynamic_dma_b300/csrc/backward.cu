// Backward of the sparse attention and of the key scores: the preparation pass
// (Delta, and the zeroed accumulators of the tensor-core kernels), the SIMT
// kernels (fp32, and any dtype when the tensor-core kernels are not selected),
// and the score-path kernels.
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §四/§五/§七: the same mask is used
// in training and inference; gradients flow through the kept positions, and a
// skipped position -- weight exactly 0 in the forward -- gets exactly zero
// gradient.  So the backward, like the forward, touches kept (row, key) pairs
// only.  With p_ij the forward's softmax weights over row i's kept set and
// dO_i = dL/dO_i:
//   dP_ij = <dO_i, V_j>,    Delta_i = sum_j p_ij dP_ij = <dO_i, O_i>
//   dx_ij = p_ij (dP_ij - Delta_i)                       (softmax backward)
//   dQ_i = scale sum_j dx_ij K_j,   dK_j = scale sum_i dx_ij Q_i
//   dV_j = sum_i p_ij dO_i,         ds_j = sum_i dx_ij    (s_j is the logit bias)
// where the sums over i run over the rows of every query head of the KV head.
// Through the score s_j = A_h softplus(u_j), u_j = <V_j, W_h> (§五):
//   dA_h += ds_j softplus(u_j),     du_j = ds_j A_h sigmoid(u_j)
//   dW_h += du_j V_j,               dV_j += du_j W_h
// p_ij is recomputed as exp(scale <Q_i, K_j> + s_j - lse_i) from the forward's lse.
// Delta_i has two forms: <dO_i, O_i> from the forward's output (for bf16 that O is
// rounded, and its error, about 2^-9 |dO_i| |O_i|, is the same for every key of the
// row), and sum_j p_ij dP_ij summed over the kept pairs by the row-side kernel.  The
// key-side sums (dK, ds, and through ds dW and dA) add dx over thousands of rows, where a
// per-row error in Delta would not average out (sum_j ds_j = 0 holds only with the summed
// form); so the row-side kernel, which needs Delta before it has seen every key, uses
// the first form and writes the second for the key-side kernel.
//
// Key j is kept by row i iff  j <= i < j + window  or  lo_j <= i < expiry_j,
// and lo_j >= j, so the rows that keep j are [j, j + window) united with
// [lo_j, expiry_j): the SIMT key-side kernel walks exactly those rows, and the
// SIMT row-side kernel walks the query tile's key list (the same list the
// forward used).  Neither needs atomics: every output element has one writer.
#include <algorithm>
#include <cmath>

#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// <row, vec> over D elements: `row` in global memory (16-byte loads), `vec` fp32 in shared memory.
template <typename T, int D>
__device__ __forceinline__ float dot_row(const T* __restrict__ row, const float* vec)
{
    float acc = 0.f;
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = __ldg(r4 + c);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
            const float4 a = reinterpret_cast<const float4*>(vec)[2 * c];
            const float4 b = reinterpret_cast<const float4*>(vec)[2 * c + 1];
            acc = fmaf(bf16_lo(u[0]), a.x, acc);
            acc = fmaf(bf16_hi(u[0]), a.y, acc);
            acc = fmaf(bf16_lo(u[1]), a.z, acc);
            acc = fmaf(bf16_hi(u[1]), a.w, acc);
            acc = fmaf(bf16_lo(u[2]), b.x, acc);
            acc = fmaf(bf16_hi(u[2]), b.y, acc);
            acc = fmaf(bf16_lo(u[3]), b.z, acc);
            acc = fmaf(bf16_hi(u[3]), b.w, acc);
        }
    } else {
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
            const uint4 v = __ldg(r4 + c);
            const float4 a = reinterpret_cast<const float4*>(vec)[c];
            acc = fmaf(__uint_as_float(v.x), a.x, acc);
            acc = fmaf(__uint_as_float(v.y), a.y, acc);
            acc = fmaf(__uint_as_float(v.z), a.z, acc);
            acc = fmaf(__uint_as_float(v.w), a.w, acc);
        }
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ----------------------------------------------------------------- preparation
// Delta[b][hq][i] = <dO_i, O_i> (fp32), one group of kCPR lanes per (b, i, hq) row (16 bytes
// per lane); then, when dK is given, dK, dV, ds and delta_x are zeroed for the accumulating
// kernels.
template <typename T, int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_prep_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                                                               int B, int S, int H, float* __restrict__ delta,
                                                               float4* __restrict__ dK, float4* __restrict__ dV,
                                                               int64_t n_kv4, float* __restrict__ ds, int64_t n_ds,
                                                               float* __restrict__ delta_x)
{
    constexpr int kElem = 16 / sizeof(T);
    constexpr int kCPR = D / kElem;  // lanes per row: 8, 16 or 32
    constexpr int kRowsPerWarp = 32 / kCPR;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t rows = (int64_t)B * S * H;
    // warp-uniform trip count: every lane reaches the shuffles
    for (int64_t base = warp * kRowsPerWarp; base < rows; base += nwarps * kRowsPerWarp) {
        const int64_t r = base + lane / kCPR;
        const int part = lane % kCPR;
        float acc = 0.f;
        if (r < rows) {
            const uint4 o = __ldg(reinterpret_cast<const uint4*>(O + r * D) + part);
            const uint4 g = __ldg(reinterpret_cast<const uint4*>(dO + r * D) + part);
            if constexpr (sizeof(T) == 2) {
                const uint32_t uo[4] = {o.x, o.y, o.z, o.w}, ug[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(bf16_lo(uo[e]), bf16_lo(ug[e]), acc);
                    acc = fmaf(bf16_hi(uo[e]), bf16_hi(ug[e]), acc);
                }
            } else {
                acc = fmaf(__uint_as_float(o.x), __uint_as_float(g.x), acc);
                acc = fmaf(__uint_as_float(o.y), __uint_as_float(g.y), acc);
                acc = fmaf(__uint_as_float(o.z), __uint_as_float(g.z), acc);
                acc = fmaf(__uint_as_float(o.w), __uint_as_float(g.w), acc);
            }
        }
#pragma unroll
        for (int off = kCPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, kCPR);
        if (r < rows && part == 0) {
            const int hq = (int)(r % H);
            const int64_t bi = r / H;
            const int i = (int)(bi % S), b = (int)(bi / S);
            delta[((int64_t)b * H + hq) * S + i] = acc;
        }
    }
    if (dK) {
        const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        const int64_t nth = (int64_t)gridDim.x * blockDim.x;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t t = tid; t < n_kv4; t += nth) {
            dK[t] = z;
            dV[t] = z;
        }
        for (int64_t t = tid; t < n_ds; t += nth) ds[t] = 0.f;
        for (int64_t t = tid; t < rows; t += nth) delta_x[t] = 0.f;
    }
}

// ------------------------------------------------------------------ row side
// dQ_i: one warp per (b, query head, row i).  Each lane takes one key of the tile's list per
// step (gathered keys, then the window band) and tests whether row i keeps it.  A first sweep
// sums Delta_i = sum_j p_ij dP_ij (written for the key-side kernel); the second forms dx_ij and
// the warp accumulates dx_ij K_j, lanes splitting D.
template <typename T, int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_dq_simt_kernel(const BwdArgs a)
{
    constexpr int kDL = D / 32;
    __shared__ __align__(16) float q_s[kBwdWarps][D];
    __shared__ __align__(16) float g_s[kBwdWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, hq = blockIdx.y;
    const int i = blockIdx.x * kBwdWarps + warp;
    if (i >= a.S) return;  // whole warp
    const int G = a.H / a.Hkv, h = hq / G, seg = b * a.Hkv + h;
    const T* Qp = static_cast<const T*>(a.Q);
    const T* Kp = static_cast<const T*>(a.K);
    const T* Vp = static_cast<const T*>(a.V);
    const T* gp = static_cast<const T*>(a.dO);
    const int64_t qrow = (((int64_t)b * a.S + i) * a.H + hq) * D;
    for (int d = lane; d < D; d += 32) {
        q_s[warp][d] = to_f32<T>(Qp[qrow + d]);
        g_s[warp][d] = to_f32<T>(gp[qrow + d]);
    }
    __syncwarp();
    const float lse_i = a.lse[((int64_t)b * a.H + hq) * a.S + i];
    const int tile = i / kQTile;
    const int q0 = tile * kQTile, q1 = min(a.S, q0 + kQTile) - 1;
    const int n_g = min(max(a.tile_cnt[(int64_t)seg * a.n_qt + tile], 0), a.tile_stride);
    const int32_t* gl = a.tile_idx + ((int64_t)seg * a.n_qt + tile) * a.tile_stride;
    const int W = a.window;
    const int band_lo = W > 0 ? max(0, q0 - W + 1) : q1 + 1;
    const int n_all = n_g + (W > 0 ? q1 + 1 - band_lo : 0);
    const float* sc = a.scores + (int64_t)seg * a.S;
    const int32_t* ex = a.expiry + (int64_t)seg * a.S;
    const int64_t kv_stride = (int64_t)a.Hkv * D;
    const T* Kh = Kp + ((int64_t)b * a.S * a.Hkv + h) * D;
    const T* Vh = Vp + ((int64_t)b * a.S * a.Hkv + h) * D;
    // the key of list position u, or -1 when row i does not keep it
    auto kept_key = [&](int u) -> int {
        int j = -1;
        if (u < n_all) j = u < n_g ? gl[u] : band_lo + (u - n_g);
        if (j < 0 || j >= a.S || j > i) return -1;  // (out of range: never produced by the selection)
        const int lo = top_lo(j, a.block);
        return (i - j < W || (lo <= i && i < ex[j])) ? j : -1;
    };
    // pass 1: Delta_i = sum_j p_ij dP_ij over the kept keys
    float dsum = 0.f;
    for (int u0 = 0; u0 < n_all; u0 += 32) {
        const int j = kept_key(u0 + lane);
        if (j >= 0) {
            const float qk = dot_row<T, D>(Kh + (int64_t)j * kv_stride, q_s[warp]);
            const float gv = dot_row<T, D>(Vh + (int64_t)j * kv_stride, g_s[warp]);
            dsum = fmaf(expf(a.scale * qk + sc[j] - lse_i), gv, dsum);
        }
    }
    const float dl_i = warp_sum(dsum);
    if (lane == 0) a.delta_x[((int64_t)b * a.H + hq) * a.S + i] = dl_i;
    // pass 2: dQ_i
    float acc[kDL];
#pragma unroll
    for (int e = 0; e < kDL; ++e) acc[e] = 0.f;
    for (int u0 = 0; u0 < n_all; u0 += 32) {
        const int j = kept_key(u0 + lane);
        float dx = 0.f;
        if (j >= 0) {
            const float qk = dot_row<T, D>(Kh + (int64_t)j * kv_stride, q_s[warp]);
            const float gv = dot_row<T, D>(Vh + (int64_t)j * kv_stride, g_s[warp]);
            const float p = expf(a.scale * qk + sc[j] - lse_i);
            dx = p * (gv - dl_i);
        }
        for (int l = 0; l < 32; ++l) {
            const float dxl = __shfl_sync(0xffffffffu, dx, l);
            const int jl = __shfl_sync(0xffffffffu, j, l);
            if (dxl != 0.f) {  // the same for every lane
                const T* kr = Kh + (int64_t)jl * kv_stride;
#pragma unroll
                for (int e = 0; e < kDL; ++e) acc[e] = fmaf(dxl, to_f32<T>(kr[lane + 32 * e]), acc[e]);
            }
        }
    }
    float* dq = a.dQ + (((int64_t)b * a.S + i) * a.H + hq) * D;
#pragma unroll
    for (int e = 0; e < kDL; ++e) dq[lane + 32 * e] = a.scale * acc[e];
}

// ------------------------------------------------------------------ key side
// dK_j, dV_j, ds_j: one warp per (b, KV head, key j).  The rows that keep j are
// [j, min(S, j + window)) and then [max(lo_j, j + window), min(S, expiry_j)); each lane takes
// one row per step and forms p_ij and dx_ij for every query head of the KV head, then the
// warp accumulates dx_ij Q_i and p_ij dO_i, lanes splitting D.
template <typename T, int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_dkv_simt_kernel(const BwdArgs a)
{
    constexpr int kDL = D / 32;
    __shared__ __align__(16) float k_s[kBwdWarps][D];
    __shared__ __align__(16) float v_s[kBwdWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int j = blockIdx.x * kBwdWarps + warp;
    if (j >= a.S) return;  // whole warp
    const int G = a.H / a.Hkv, seg = b * a.Hkv + h;
    const T* Qp = static_cast<const T*>(a.Q);
    const T* Kp = static_cast<const T*>(a.K);
    const T* Vp = static_cast<const T*>(a.V);
    const T* gp = static_cast<const T*>(a.dO);
    const int64_t krow = (((int64_t)b * a.S + j) * a.Hkv + h) * D;
    for (int d = lane; d < D; d += 32) {
        k_s[warp][d] = to_f32<T>(Kp[krow + d]);
        v_s[warp][d] = to_f32<T>(Vp[krow + d]);
    }
    __syncwarp();
    const float s_j = a.scores[(int64_t)seg * a.S + j];
    const int lo = top_lo(j, a.block);
    const int e1 = (int)min((int64_t)a.S, (int64_t)j + a.window);
    const int e2 = min(a.S, a.expiry[(int64_t)seg * a.S + j]);
    const int r2 = max(lo, e1);
    const int n1 = e1 - j, n2 = max(0, e2 - r2);
    const int total = n1 + n2;
    float dk[kDL], dv[kDL];
#pragma unroll
    for (int e = 0; e < kDL; ++e) dk[e] = dv[e] = 0.f;
    float dsum = 0.f;
    for (int t0 = 0; t0 < total; t0 += 32) {
        const int t = t0 + lane;
        const int i = t < total ? (t < n1 ? j + t : r2 + (t - n1)) : -1;
        for (int gq = 0; gq < G; ++gq) {
            const int hq = h * G + gq;
            float p = 0.f, dx = 0.f;
            if (i >= 0) {
                const int64_t qrow = (((int64_t)b * a.S + i) * a.H + hq) * D;
                const float qk = dot_row<T, D>(Qp + qrow, k_s[warp]);
                const float gv = dot_row<T, D>(gp + qrow, v_s[warp]);
                const int64_t rs = ((int64_t)b * a.H + hq) * a.S + i;
                p = expf(a.scale * qk + s_j - a.lse[rs]);
                dx = p * (gv - a.delta_x[rs]);
            }
            dsum += dx;
            for (int l = 0; l < 32; ++l) {
                const int il = __shfl_sync(0xffffffffu, i, l);
                const float pl = __shfl_sync(0xffffffffu, p, l);
                const float dxl = __shfl_sync(0xffffffffu, dx, l);
                if (il >= 0) {  // the same for every lane
                    const int64_t qrow = (((int64_t)b * a.S + il) * a.H + hq) * D;
#pragma unroll
                    for (int e = 0; e < kDL; ++e) {
                        dk[e] = fmaf(dxl, to_f32<T>(Qp[qrow + lane + 32 * e]), dk[e]);
                        dv[e] = fmaf(pl, to_f32<T>(gp[qrow + lane + 32 * e]), dv[e]);
                    }
                }
            }
        }
    }
    dsum = warp_sum(dsum);
    const int64_t orow = (((int64_t)b * a.S + j) * a.Hkv + h) * D;
#pragma unroll
    for (int e = 0; e < kDL; ++e) {
        a.dK[orow + lane + 32 * e] = a.scale * dk[e];
        a.dV[orow + lane + 32 * e] = dv[e];
    }
    if (lane == 0) a.ds[(int64_t)seg * a.S + j] = dsum;
}

// --------------------------------------------------------------- score path
// One CTA per (chunk of kScoreBwdKeys keys, KV head, batch); a warp per key recomputes u_j,
// adds du_j W_h to dV_j (each (b, j, h) row has one writer) and accumulates du_j V_j and
// ds_j softplus(u_j); the CTA's sums go to its own slot of the partials array, which the
// finalize kernel adds up in a fixed order (no atomics: the result does not depend on
// scheduling).
constexpr int kScoreBwdKeys = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kBwdThreads) score_bwd_kernel(const T* __restrict__ V, int S, int Hkv,
                                                                const float* __restrict__ W,
                                                                const float* __restrict__ A, int exp_form,
                                                                const float* __restrict__ ds, float* __restrict__ dV,
                                                                float* __restrict__ part, int nchunk)
{
    constexpr int kDL = D / 32;
    __shared__ float red[kBwdWarps][D + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    float w[kDL], dw[kDL];
#pragma unroll
    for (int e = 0; e < kDL; ++e) {
        w[e] = W[h * D + lane + 32 * e];
        dw[e] = 0.f;
    }
    const float gate = A ? A[h] : 1.f;
    float da = 0.f;
    for (int jj = warp; jj < kScoreBwdKeys; jj += kBwdWarps) {
        const int j = c * kScoreBwdKeys + jj;
        if (j >= S) break;  // whole warp
        const int64_t row = (((int64_t)b * S + j) * Hkv + h) * D;
        float v[kDL];
        float u = 0.f;
#pragma unroll
        for (int e = 0; e < kDL; ++e) {
            v[e] = to_f32<T>(V[row + lane + 32 * e]);
            u = fmaf(v[e], w[e], u);
        }
        u = warp_sum(u);
        float g = ds[((int64_t)b * Hkv + h) * S + j];
        // softplus(u) = max(u, 0) + log1p(exp(-|u|)); sigmoid(u) = 1 / (1 + exp(-u))
        const float sp = fmaxf(u, 0.f) + log1pf(expf(-fabsf(u)));
        const float sg = 1.f / (1.f + expf(-u));
        // exp form: ds is dL/d delta with delta = exp(s), so dL/ds = ds * delta
        if (exp_form) g *= expf(gate * sp);
        const float du = g * gate * sg;
        da = fmaf(g, sp, da);
#pragma unroll
        for (int e = 0; e < kDL; ++e) {
            dV[row + lane + 32 * e] += du * w[e];
            dw[e] = fmaf(du, v[e], dw[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < kDL; ++e) red[warp][lane + 32 * e] = dw[e];
    if (lane == 0) red[warp][D] = da;
    __syncthreads();
    for (int d = threadIdx.x; d <= D; d += kBwdThreads) {
        float s = 0.f;
#pragma unroll
        for (int wv = 0; wv < kBwdWarps; ++wv) s += red[wv][d];
        part[(((int64_t)b * Hkv + h) * nchunk + c) * (D + 1) + d] = s;
    }
}

// dW[h][d] and dA[h]: the partials of every (batch, chunk) summed in index order.
__global__ void score_bwd_finalize_kernel(const float* __restrict__ part, int B, int Hkv, int nchunk, int D,
                                          float* __restrict__ dW, float* __restrict__ dA)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= Hkv * (D + 1)) return;
    const int h = t / (D + 1), d = t % (D + 1);
    float s = 0.f;
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < nchunk; ++c) s += part[(((int64_t)b * Hkv + h) * nchunk + c) * (D + 1) + d];
    if (d < D)
        dW[h * D + d] = s;
    else if (dA)
        dA[h] = s;
}

template <typename T, int D>
cudaError_t prep_typed(const BwdArgs& a, bool zero, cudaStream_t st)
{
    const int64_t rows = (int64_t)a.B * a.S * a.H;
    const int64_t n_kv4 = (int64_t)a.B * a.S * a.Hkv * D / 4;
    const int64_t work = rows * (D * (int64_t)sizeof(T) / 16) + (zero ? 2 * n_kv4 : 0);
    const int64_t blocks = std::min<int64_t>((work + kBwdThreads - 1) / kBwdThreads, 148 * 16);
    bwd_prep_kernel<T, D><<<(unsigned)std::max<int64_t>(blocks, 1), kBwdThreads, 0, st>>>(
        static_cast<const T*>(a.O), static_cast<const T*>(a.dO), a.B, a.S, a.H, a.delta,
        zero ? reinterpret_cast<float4*>(a.dK) : nullptr, reinterpret_cast<float4*>(a.dV), n_kv4, a.ds,
        (int64_t)a.B * a.Hkv * a.S, a.delta_x);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t simt_typed(const BwdArgs& a, cudaStream_t st)
{
    dim3 gq((a.S + kBwdWarps - 1) / kBwdWarps, a.H, a.B);
    bwd_dq_simt_kernel<T, D><<<gq, kBwdThreads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 gk((a.S + kBwdWarps - 1) / kBwdWarps, a.Hkv, a.B);
    bwd_dkv_simt_kernel<T, D><<<gk, kBwdThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t score_bwd_typed(const void* V, int B, int S, int Hkv, const float* W, const float* A, int exp_form,
                            const float* ds, float* dV, float* dW, float* dA, float* part, cudaStream_t st)
{
    const int nchunk = (S + kScoreBwdKeys - 1) / kScoreBwdKeys;
    dim3 grid(nchunk, Hkv, B);
    score_bwd_kernel<T, D><<<grid, kBwdThreads, 0, st>>>(static_cast<const T*>(V), S, Hkv, W, A, exp_form, ds, dV,
                                                         part, nchunk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n = Hkv * (D + 1);
    score_bwd_finalize_kernel<<<(n + 127) / 128, 128, 0, st>>>(part, B, Hkv, nchunk, D, dW, dA);
    return cudaGetLastError();
}

}  // namespace

size_t backward_ws_bytes(int B, int S, int H, int Hkv, int D)
{
    const size_t delta = 2 * (size_t)B * H * S * sizeof(float);  // delta and delta_x
    const size_t nchunk = ((size_t)S + kScoreBwdKeys - 1) / kScoreBwdKeys;
    const size_t part = (size_t)B * Hkv * nchunk * (D + 1) * sizeof(float);
    const size_t m = delta > part ? delta : part;
    return (m + 255) / 256 * 256;
}

cudaError_t launch_bwd_prep(const BwdArgs& a, dma_dtype_t dt, int D, bool zero, cudaStream_t st)
{
    if (dt == DMA_BF16) return D == 128 ? prep_typed<__nv_bfloat16, 128>(a, zero, st) : prep_typed<__nv_bfloat16, 64>(a, zero, st);
    return D == 128 ? prep_typed<float, 128>(a, zero, st) : prep_typed<float, 64>(a, zero, st);
}

cudaError_t launch_bwd_simt(const BwdArgs& a, dma_dtype_t dt, int D, cudaStream_t st)
{
    if (dt == DMA_BF16) return D == 128 ? simt_typed<__nv_bfloat16, 128>(a, st) : simt_typed<__nv_bfloat16, 64>(a, st);
    return D == 128 ? simt_typed<float, 128>(a, st) : simt_typed<float, 64>(a, st);
}

cudaError_t launch_score_bwd(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, const float* W,
                             const float* A, int exp_form, const float* ds, float* dV, float* dW, float* dA, void* ws,
                             cudaStream_t st)
{
    float* part = static_cast<float*>(ws);
    if (dt == DMA_BF16) {
        if (D == 128) return score_bwd_typed<__nv_bfloat16, 128>(V, B, S, Hkv, W, A, exp_form, ds, dV, dW, dA, part, st);
        return score_bwd_typed<__nv_bfloat16, 64>(V, B, S, Hkv, W, A, exp_form, ds, dV, dW, dA, part, st);
    }
    if (D == 128) return score_bwd_typed<float, 128>(V, B, S, Hkv, W, A, exp_form, ds, dV, dW, dA, part, st);
    return score_bwd_typed<float, 64>(V, B, S, Hkv, W, A, exp_form, ds, dV, dW, dA, part, st);
}

}  // namespace dma
