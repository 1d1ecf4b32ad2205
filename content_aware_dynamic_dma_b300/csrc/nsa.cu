// NSA-style three-branch attention (NSA post, news.news, §03): attention over
// compressed blocks, over selected blocks and over a sliding window, mixed per
// token by gates.  The selected branch is this library's 64-key block selection
// and sparse attention; this file adds what the other two branches and the
// fusion need:
//   - block compression: the mean of the K (V) rows of every complete 64-key
//     block, written at the row of the block's last key in arrays shaped like K
//     and V, so that the sparse attention kernels gather compressed rows by key
//     index like any other kept key;
//   - the kept-key structures of the two fixed patterns (compressed rows seen by
//     every row at or after them; the window alone), which depend only on the
//     sequence length and the window;
//   - the gated sum of the three branch outputs, gate = sigmoid(<q, G[h,b]> + c[h,b]).
#include "dma_internal.cuh"

namespace dma {
namespace {

constexpr int kNsaBlock = 64;
constexpr int kCompressThreads = 128;

// One CTA per (block beta, batch b, tensor K or V): the 64 rows of the block are one
// contiguous span of Hkv * D elements each; a thread owns 16-byte columns of it and sums
// them down the 64 rows in key order (fp32), then writes the mean in the input type.
template <typename T>
__global__ void __launch_bounds__(kCompressThreads) nsa_compress_kernel(const T* __restrict__ K,
                                                                       const T* __restrict__ V, int S, int row_elems,
                                                                       int block_begin, T* __restrict__ Kc,
                                                                       T* __restrict__ Vc)
{
    constexpr int kElem = 16 / sizeof(T);
    const int beta = block_begin + blockIdx.x, b = blockIdx.y;
    const T* src = blockIdx.z == 0 ? K : V;
    T* dst = blockIdx.z == 0 ? Kc : Vc;
    const int chunks = row_elems / kElem;
    const int64_t first = ((int64_t)b * S + (int64_t)beta * kNsaBlock) * row_elems;
    const uint4* in = reinterpret_cast<const uint4*>(src + first);
    uint4* out = reinterpret_cast<uint4*>(dst + first + (int64_t)(kNsaBlock - 1) * row_elems);
    for (int c = threadIdx.x; c < chunks; c += kCompressThreads) {
        float acc[kElem];
#pragma unroll
        for (int e = 0; e < kElem; ++e) acc[e] = 0.f;
#pragma unroll 8
        for (int r = 0; r < kNsaBlock; ++r) {
            const uint4 x = __ldg(in + (int64_t)r * chunks + c);
            if constexpr (sizeof(T) == 2) {
                const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e] += bf16_lo(u[e]);
                    acc[2 * e + 1] += bf16_hi(u[e]);
                }
            } else {
                acc[0] += __uint_as_float(x.x);
                acc[1] += __uint_as_float(x.y);
                acc[2] += __uint_as_float(x.z);
                acc[3] += __uint_as_float(x.w);
            }
        }
        constexpr float kInv = 1.0f / kNsaBlock;  // a power of two: exact
        uint4 y;
        if constexpr (sizeof(T) == 2) {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * e] * kInv, acc[2 * e + 1] * kInv);
                u[e] = *reinterpret_cast<const uint32_t*>(&p);
            }
            y = make_uint4(u[0], u[1], u[2], u[3]);
        } else {
            y = make_uint4(__float_as_uint(acc[0] * kInv), __float_as_uint(acc[1] * kInv),
                           __float_as_uint(acc[2] * kInv), __float_as_uint(acc[3] * kInv));
        }
        out[c] = y;
    }
}

// Per-key arrays of a pattern: expiry, the ever-kept list and the decode row's top set.
// Compressed: key 64 beta + 63 of a complete block is kept from its own row to the end;
// every other key never.  Window: no key is in a top set.
__global__ void nsa_pattern_keys_kernel(int compressed, int S, int cap, int top_cap, const int32_t* __restrict__ seq_len,
                                        int Hkv, int32_t* __restrict__ expiry, int32_t* __restrict__ idx,
                                        int32_t* __restrict__ count, int32_t* __restrict__ top_idx,
                                        int32_t* __restrict__ top_count, int* status)
{
    const int seg = blockIdx.y;
    const int nb = compressed ? S / kNsaBlock : 0;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < S) {
        const bool kept = j % kNsaBlock == kNsaBlock - 1 && j / kNsaBlock < nb;
        expiry[(int64_t)seg * S + j] = kept ? S : j;
        if (idx && j < nb) {
            if (j < cap)
                idx[(int64_t)seg * cap + j] = j * kNsaBlock + kNsaBlock - 1;
            else
                set_status(status, DMA_ERR_DEVICE_CHECK);
        }
    }
    // the decode row L - 1 (L = seq_len[b], or S) sees the complete blocks of its first L keys
    int L = S;
    if (seq_len) {
        L = seq_len[seg / Hkv];
        if (L < 1 || L > S) {
            if (j == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
            L = L < 1 ? 1 : S;
        }
    }
    const int n_top = compressed ? L / kNsaBlock : 0;
    if (top_idx && j < n_top) {
        if (j < top_cap)
            top_idx[(int64_t)seg * top_cap + j] = j * kNsaBlock + kNsaBlock - 1;
        else
            set_status(status, DMA_ERR_DEVICE_CHECK);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (count) count[seg] = nb;
        if (top_count) top_count[seg] = min(n_top, top_cap);
    }
}

// Per-tile lists and occupancy bitmap of a pattern: tile t of rows [q0, q1] lists the
// compressed keys 64 beta + 63 <= q1 in ascending order (those <= q0, kept by every row of
// the tile, come first by construction); the bitmap marks their blocks and the window band.
__global__ void nsa_pattern_tiles_kernel(int compressed, int S, int window, int n_qt, int tile_stride,
                                         int bitmap_words, int32_t* __restrict__ tile_cnt,
                                         int32_t* __restrict__ tile_idx, uint32_t* __restrict__ bitmap, int* status)
{
    const int seg = blockIdx.y, t = blockIdx.x;
    const int q0 = t * kQTile, q1 = min(S, q0 + kQTile) - 1;
    const int n_t = compressed ? (q1 + 1) / kNsaBlock : 0;
    int32_t* out = tile_idx + ((int64_t)seg * n_qt + t) * tile_stride;
    for (int e = threadIdx.x; e < n_t; e += blockDim.x) {
        if (e < tile_stride)
            out[e] = e * kNsaBlock + kNsaBlock - 1;
        else
            set_status(status, DMA_ERR_DEVICE_CHECK);
    }
    if (threadIdx.x == 0) tile_cnt[(int64_t)seg * n_qt + t] = min(n_t, tile_stride);
    if (!bitmap) return;
    const int band_lo = window > 0 ? max(0, q0 - window + 1) / kBitmapBlock : 1 << 30;
    const int band_hi = window > 0 ? q1 / kBitmapBlock : -1;
    uint32_t* bo = bitmap + ((int64_t)seg * n_qt + t) * bitmap_words;
    for (int wd = threadIdx.x; wd < bitmap_words; wd += blockDim.x) {
        uint32_t bits = 0;
        for (int l = 0; l < 32; ++l) {
            const int blk = 32 * wd + l;
            if (blk < n_t || (blk >= band_lo && blk <= band_hi)) bits |= 1u << l;
        }
        bo[wd] = bits;
    }
}

// kPer floats to consecutive elements, in one store of kPer * sizeof(T) bytes.
template <typename T, int kPer>
__device__ __forceinline__ void store_run(T* p, const float* v)
{
    if constexpr (sizeof(T) == 2) {
        uint32_t u[kPer / 2];
#pragma unroll
        for (int e = 0; e < kPer / 2; ++e) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            u[e] = *reinterpret_cast<const uint32_t*>(&b);
        }
        if constexpr (kPer == 4)
            *reinterpret_cast<uint2*>(p) = make_uint2(u[0], u[1]);
        else
            *reinterpret_cast<uint32_t*>(p) = u[0];
    } else {
        if constexpr (kPer == 4)
            *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        else
            *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    }
}

// The gated sum: per (b, i, h) a warp forms the three gates from the query row, then the
// weighted sum of the branch rows.  O may alias a branch output: each element is read
// before the same thread writes it.
constexpr int kCombineWarps = 8;

// kPer consecutive elements as floats, in one load of kPer * sizeof(T) bytes (4, 8 or 16).
template <typename T, int kPer>
__device__ __forceinline__ void load_run(const T* p, float* out)
{
    if constexpr (sizeof(T) == 2) {
        if constexpr (kPer == 4) {
            const uint2 x = *reinterpret_cast<const uint2*>(p);
            out[0] = bf16_lo(x.x), out[1] = bf16_hi(x.x), out[2] = bf16_lo(x.y), out[3] = bf16_hi(x.y);
        } else {
            const uint32_t x = *reinterpret_cast<const uint32_t*>(p);
            out[0] = bf16_lo(x), out[1] = bf16_hi(x);
        }
    } else {
        if constexpr (kPer == 4) {
            const float4 x = *reinterpret_cast<const float4*>(p);
            out[0] = x.x, out[1] = x.y, out[2] = x.z, out[3] = x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(p);
            out[0] = x.x, out[1] = x.y;
        }
    }
}

// One query head per warp: the warp keeps that head's gate weights in registers and walks
// rows (b, i) of it, n_warps / H rows apart.
template <typename T, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) nsa_combine_kernel(
    const T* __restrict__ Q, const T* Oc, const T* Os, const T* Ow, int64_t n_rows, int H, int n_warps,
    const float* __restrict__ G, const float* __restrict__ c, T* O, float* __restrict__ gates)
{
    constexpr int kPer = D / 32;  // consecutive elements per lane
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (gw >= n_warps) return;
    const int h = gw % H;
    float gw_r[3][kPer], cb[3];
#pragma unroll
    for (int br = 0; br < 3; ++br) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) gw_r[br][e] = __ldg(G + ((int64_t)h * 3 + br) * D + lane * kPer + e);
        cb[br] = __ldg(c + h * 3 + br);
    }
    const int64_t step = n_warps / H;
    // two rows per iteration: the loads of both are in flight before either's arithmetic
    auto finish = [&](int64_t r, const float* q, const float* oc, const float* os, const float* ow) {
        float g[3];
#pragma unroll
        for (int br = 0; br < 3; ++br) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < kPer; ++e) x = fmaf(q[e], gw_r[br][e], x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            g[br] = 1.f / (1.f + expf(-(x + cb[br])));
        }
        float v[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) v[e] = fmaf(g[0], oc[e], fmaf(g[1], os[e], g[2] * ow[e]));
        store_run<T, kPer>(O + r * D + lane * kPer, v);
        if (gates && lane < 3) gates[r * 3 + lane] = lane == 0 ? g[0] : (lane == 1 ? g[1] : g[2]);
    };
    for (int64_t bi = gw / H; bi < n_rows; bi += 2 * step) {
        const int64_t r0 = bi * H + h, r1 = (bi + step) * H + h;
        const bool two = bi + step < n_rows;  // warp-uniform
        float q0[kPer], oc0[kPer], os0[kPer], ow0[kPer], q1[kPer], oc1[kPer], os1[kPer], ow1[kPer];
        const int64_t b0 = r0 * D + lane * kPer, b1 = r1 * D + lane * kPer;
        load_run<T, kPer>(Q + b0, q0);
        load_run<T, kPer>(Oc + b0, oc0);
        load_run<T, kPer>(Os + b0, os0);
        load_run<T, kPer>(Ow + b0, ow0);
        if (two) {
            load_run<T, kPer>(Q + b1, q1);
            load_run<T, kPer>(Oc + b1, oc1);
            load_run<T, kPer>(Os + b1, os1);
            load_run<T, kPer>(Ow + b1, ow1);
        }
        finish(r0, q0, oc0, os0, ow0);
        if (two) finish(r1, q1, oc1, os1, ow1);
    }
}

template <typename T, int D>
cudaError_t combine_typed(const void* Q, const void* Oc, const void* Os, const void* Ow, int64_t rows, int H,
                          const float* G, const float* c, void* O, float* gates, cudaStream_t st)
{
    // as many warps as fit on the GPU at once, a multiple of H (at least H)
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, nsa_combine_kernel<T, D>, kCombineWarps * 32, 0);
    if (e != cudaSuccess) return e;
    const int64_t n_rows = rows / H;  // (b, i) pairs
    int64_t warps = (int64_t)sms * (per_sm > 0 ? per_sm : 1) * kCombineWarps;
    if (warps > n_rows * H) warps = n_rows * H;
    warps = warps / H * H;
    if (warps < H) warps = H;
    const int64_t grid = (warps + kCombineWarps - 1) / kCombineWarps;
    nsa_combine_kernel<T, D><<<(unsigned)grid, kCombineWarps * 32, 0, st>>>(
        static_cast<const T*>(Q), static_cast<const T*>(Oc), static_cast<const T*>(Os), static_cast<const T*>(Ow),
        n_rows, H, (int)warps, G, c, static_cast<T*>(O), gates);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_nsa_compress(const void* K, const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D,
                                int block_begin, int block_end, void* Kc, void* Vc, cudaStream_t st)
{
    if (block_end > S / kNsaBlock) block_end = S / kNsaBlock;
    if (block_end <= block_begin) return cudaSuccess;
    dim3 grid(block_end - block_begin, B, 2);
    if (dt == DMA_BF16)
        nsa_compress_kernel<__nv_bfloat16><<<grid, kCompressThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(K), static_cast<const __nv_bfloat16*>(V), S, Hkv * D, block_begin,
            static_cast<__nv_bfloat16*>(Kc), static_cast<__nv_bfloat16*>(Vc));
    else
        nsa_compress_kernel<float><<<grid, kCompressThreads, 0, st>>>(
            static_cast<const float*>(K), static_cast<const float*>(V), S, Hkv * D, block_begin,
            static_cast<float*>(Kc), static_cast<float*>(Vc));
    return cudaGetLastError();
}

cudaError_t launch_nsa_pattern(int compressed, const dma_kept_t* kept, const int32_t* seq_len, int* status,
                               cudaStream_t st)
{
    const int nseg = kept->B * kept->Hkv, S = kept->S;
    nsa_pattern_keys_kernel<<<dim3((S + 255) / 256, nseg), 256, 0, st>>>(
        compressed, S, kept->cap, kept->top_cap, seq_len, kept->Hkv, kept->expiry, kept->idx, kept->count,
        kept->top_idx, kept->top_count, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !kept->tile_idx) return e;
    nsa_pattern_tiles_kernel<<<dim3(kept->n_qt, nseg), 256, 0, st>>>(
        compressed, S, kept->window, kept->n_qt, kept->tile_stride, kept->bitmap_words, kept->tile_cnt,
        kept->tile_idx, kept->bitmap, status);
    return cudaGetLastError();
}

cudaError_t launch_nsa_combine(const void* Q, const void* Oc, const void* Os, const void* Ow, dma_dtype_t dt,
                               int64_t rows, int H, int D, const float* G, const float* c, void* O, float* gates,
                               cudaStream_t st)
{
    if (rows == 0) return cudaSuccess;
    if (dt == DMA_BF16)
        return D == 128 ? combine_typed<__nv_bfloat16, 128>(Q, Oc, Os, Ow, rows, H, G, c, O, gates, st)
                        : combine_typed<__nv_bfloat16, 64>(Q, Oc, Os, Ow, rows, H, G, c, O, gates, st);
    return D == 128 ? combine_typed<float, 128>(Q, Oc, Os, Ow, rows, H, G, c, O, gates, st)
                    : combine_typed<float, 64>(Q, Oc, Os, Ow, rows, H, G, c, O, gates, st);
}

}  // namespace dma
