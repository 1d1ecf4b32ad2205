// Internal declarations shared by the CUDA translation units of libdma.
// Nothing here is part of the C ABI (see include/dma.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dma.h"

namespace dma {

constexpr int kQTile = DMA_Q_TILE;
constexpr int kBitmapBlock = 64;  // keys per bit of the occupancy bitmap

// ---- small device helpers -------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// First row at which key j may enter the top set.
__host__ __device__ __forceinline__ int top_lo(int j, int block)
{
    return block <= 1 ? j : (j / block) * block + block - 1;
}

// Records a device-side condition (first one wins).
__device__ __forceinline__ void set_status(int* status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// ---- selection workspace --------------------------------------------------

struct SelectPlan {
    // problem
    int nseg;       // B * Hkv
    int S;          // keys per segment
    int n;          // ranked units per segment (S for tokens, S / block for blocks)
    int k;          // budget in units (w or w / block)
    int nchunk;     // radix-sort chunks per segment
    int T;          // rank chunk length of the expiry walk
    int nC;         // ceil(n / T)
    int X;          // position block length of the 2-D count table
    int nX;         // ceil(n / X)
    int nlc;        // list chunks per segment (of the key and rank-order compactions)
    int n_sg;       // super groups of query tiles per segment (1: the tile lists read the whole list)
    int sg_tiles;   // query tiles per super group
    int sg_cap;     // entries per super-group list
    // byte offsets into the workspace
    size_t off_key[2], off_val[2], off_hist, off_rank, off_tab, off_f0, off_bval, off_bexp, off_lcnt, off_krn;
    size_t off_sgu, off_sge, off_sgn;
    size_t bytes;
};

SelectPlan make_select_plan(int B, int Hkv, int S, int w, int block);

// Records the per-thread detail message returned by dma_last_error_message()
// and returns `s`.
dma_status_t set_error(dma_status_t s, const char* fmt, ...);

// ---- launchers (host) -----------------------------------------------------

cudaError_t launch_score(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, int key_begin, int key_end,
                         const float* W, const float* A, float* scores, float* bias, int exp_form, cudaStream_t st);

cudaError_t launch_nsa_compress(const void* K, const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D,
                                int block_begin, int block_end, void* Kc, void* Vc, cudaStream_t st);
cudaError_t launch_nsa_pattern(int compressed, const dma_kept_t* kept, const int32_t* seq_len, int* status,
                               cudaStream_t st);
cudaError_t launch_nsa_combine(const void* Q, const void* Oc, const void* Os, const void* Ow, dma_dtype_t dt,
                               int64_t rows, int H, int D, const float* G, const float* c, void* O, float* gates,
                               cudaStream_t st);

cudaError_t launch_select_full(const float* scores, const SelectPlan& plan, const dma_kept_t* kept,
                               const int32_t* w_head, void* ws, int* status, cudaStream_t st);
cudaError_t launch_select_update(const float* scores, const dma_kept_t* kept, const int32_t* seq_len,
                                 const int32_t* w_head, int* status, cudaStream_t st);

cudaError_t launch_prefill_simt(const void* Q, const void* K, const void* V, dma_dtype_t dt, int B, int S, int H,
                                int Hkv, int D, const float* scores, const dma_kept_t* kept, float scale, void* O,
                                float* lse, cudaStream_t st);

// Tensor-core prefill (bf16, D = 64 or 128).
bool prefill_tc_supported(dma_dtype_t dt, int B, int S, int H, int Hkv, int D);
// Default limit of the kernels' bounded waits.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// wait_ns: limit of every bounded wait in the kernel; fault_mode: DMA_FAULT_NONE or
// DMA_FAULT_DROP_ARRIVE (CTA 0 withholds one completion signal, for tests of the timeout path)
cudaError_t launch_prefill_tc(const void* Q, const void* K, const void* V, int B, int S, int H, int Hkv, int D,
                              const float* scores, const dma_kept_t* kept, float scale, void* O, float* lse,
                              int* status, uint64_t wait_ns, int fault_mode, cudaStream_t st);

// Pipelined bf16 decode (TMA row gathers, mma.sync, split-K).
bool decode_pipe_supported(dma_dtype_t dt, int B, int Lmax, int H, int Hkv, int D);
int decode_pipe_splits(int B, int Hkv, int top_cap, int window);
cudaError_t launch_decode_pipe(const void* q, const void* Kc, const void* Vc, int B, int Lmax,
                               const int32_t* cache_len, int H, int Hkv, int D, const float* scores,
                               const dma_kept_t* kept, float scale, void* o, float* lse, void* ws, int* status,
                               cudaStream_t st);

// ---- backward ---------------------------------------------------------------

// Arguments of the attention backward kernels (pointers as documented at
// dma_sparse_attn_prefill_backward).  Workspace: delta [B][H][S] = <dO_i, O_i> from the
// forward's (rounded) output; delta_x [B][H][S] = sum_j p_ij dP_ij summed by the row-side
// kernel over the kept pairs, for the key-side kernel.
struct BwdArgs {
    const void *Q, *K, *V, *O, *dO;
    const float* scores;
    const float* lse;
    const int32_t *expiry, *tile_cnt, *tile_idx;
    float *dQ, *dK, *dV, *ds, *delta, *delta_x;
    int* status;
    int B, S, H, Hkv, n_qt, tile_stride, window, block;
    float scale;
};

size_t backward_ws_bytes(int B, int S, int H, int Hkv, int D);
// Delta = <dO, O> per row; with `zero`, also dK = dV = ds = 0 (for the accumulating kernels).
cudaError_t launch_bwd_prep(const BwdArgs& a, dma_dtype_t dt, int D, bool zero, cudaStream_t st);
cudaError_t launch_bwd_simt(const BwdArgs& a, dma_dtype_t dt, int D, cudaStream_t st);
// Tensor-core backward (bf16, D = 64 or 128): dQ, then dK/dV/ds accumulated into zeroed arrays.
bool bwd_tc_supported(dma_dtype_t dt, int D);
cudaError_t launch_bwd_tc(const BwdArgs& a, int D, uint64_t wait_ns, cudaStream_t st);
cudaError_t launch_score_bwd(const void* V, dma_dtype_t dt, int B, int S, int Hkv, int D, const float* W,
                             const float* A, int exp_form, const float* ds, float* dV, float* dW, float* dA, void* ws,
                             cudaStream_t st);

// Paged decode cache (K/V pages [n_pages][1 << pshift][Hkv][D], block_table [B][max_pages]).
cudaError_t launch_score_paged(const void* Vp, dma_dtype_t dt, const int32_t* bt, int n_pages, int B, int max_pages,
                               int pshift, int Hkv, int D, int key_begin, int key_end, const int32_t* cache_len,
                               const float* W, const float* A, float* scores, float* page_scores, float* bias,
                               int exp_form, int* status, cudaStream_t st);
cudaError_t launch_select_pages(const float* page_scores, int B, int Hkv, int max_pages, int pshift,
                                const int32_t* cache_len, int w, const int32_t* w_head, int32_t* top_idx,
                                int32_t* top_count, int top_cap, int* status, cudaStream_t st);
cudaError_t launch_decode_paged(const void* q, const void* Kp, const void* Vp, const int32_t* block_table,
                                int n_pages, int B, int max_pages, int pshift, const int32_t* cache_len, int H,
                                int Hkv, int D, const float* scores, const int32_t* top_idx,
                                const int32_t* top_count, int top_cap, int window, float scale, void* o, float* lse,
                                void* ws, int* status, cudaStream_t st);

size_t decode_ws_bytes(int B, int H, int Hkv, int D, int top_cap, int window);
cudaError_t launch_decode(const void* q, const void* Kc, const void* Vc, dma_dtype_t dt, int B, int Lmax,
                          const int32_t* cache_len, int H, int Hkv, int D, const float* scores,
                          const dma_kept_t* kept, float scale, void* o, float* lse, void* ws, cudaStream_t st);

}  // namespace dma
