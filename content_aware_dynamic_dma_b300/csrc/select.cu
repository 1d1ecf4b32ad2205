// Causal top-w selection (Dynamic Mask Attention summary, lsdiaocha.cn, §五:
// combine the dynamic weights with the causal mask, keep the top-k historical
// positions at every time step, set the rest to -inf; §九: the keep budget is
// fixed in advance).
//
// Output representation: one interval per key.  Key j is in the top set of rows
// lo_j <= i < expiry[j].  For the row-wise rule this is exact because the top set
// of row i+1 is the top set of row i plus key i+1, minus at most one evicted key:
// once a key leaves it never returns.
//
// How expiry is computed (per (batch, KV head) segment of n ranked units):
//  1. Sort the units best-first by (fp32 score desc, position asc): a stable
//     4-pass LSD radix sort on an order-preserving 32-bit key, over chunks of
//     2048 units (histogram -> digit-major scan -> stable scatter).  This gives
//     p[t] (position of rank t) and rank[x].
//  2. The keys that beat unit u are exactly the ranks below rank[u].  u is in
//     the top set of row i iff fewer than k of them sit at positions <= i, so
//       expiry[u] = max(u, f(rank[u])),  f(t) = k-th smallest of {p[0..t-1]}
//     (f = infinity while t < k).  f is non-increasing in t.
//  3. f over a rank chunk [tc, tc+T) is a staircase walk: start from f(tc),
//     insert p[t] one at a time; an insertion below the current f moves f down
//     to the largest inserted position below it, found 128 positions per step
//     with warp ballots on rank[].  f(tc) itself comes from a 2-D count table
//     (ranks < tc per position block of X) and one ballot pass inside a block.
//  Global mode is rank[u] < k.  Block units run the same steps on block maxima
//  over complete blocks and expand the block interval to its keys.
//
// Then: the ever-kept key list (ascending), the last row's top set, per query
// tile of 128 rows the gathered key list (keys outside the window band whose
// interval meets the tile) and the 64-key block occupancy bitmap.
#include <cstdio>

#include "dma_internal.cuh"

namespace dma {

namespace {

constexpr int kRadixChunk = 2048;   // units per radix-sort chunk
constexpr int kRadixThreads = 256;  // 8 warps x 8 rounds x 32 lanes
constexpr int kRadixBins = 256;
constexpr int kRadixFuseChunks = 64;  // segments of up to 64 chunks: no separate scan launch

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int pow2_ceil(int x)
{
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Order-preserving key: ascending key = best first.  -0 is +0; NaN is last.
__device__ __forceinline__ uint32_t rank_key(float s)
{
    if (s != s) return 0xffffffffu;
    if (s == 0.f) s = 0.f;
    uint32_t u = __float_as_uint(s);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending in s
    return ~u;                                       // descending in s
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------- block max --

__global__ void block_max_kernel(const float* __restrict__ scores, int S, int nb, int block, float* __restrict__ bval)
{
    const int seg = blockIdx.y;
    const int bk = blockIdx.x * blockDim.x + threadIdx.x;
    if (bk >= nb) return;
    const float* s = scores + (int64_t)seg * S + (int64_t)bk * block;
    // The max is taken in key order, so the result is that of the keys' ranking
    // keys: NaN ranks lowest and is skipped by fmaxf.
    float m = -INFINITY;
    bool any = false;
    for (int t = 0; t < block; ++t) {
        float v = s[t];
        if (v == v) {
            m = any ? fmaxf(m, v) : v;
            any = true;
        }
    }
    bval[(int64_t)seg * nb + bk] = any ? m : __int_as_float(0x7fc00000);
}

// ---------------------------------------------------------------- radix sort --

// Pass input: either the raw values (first pass: key computed, value = position)
// or the previous pass's (key, value) buffers.
struct RadixIn {
    const float* values;  // first pass only
    const uint32_t* key;
    const int32_t* val;
};

__device__ __forceinline__ void radix_load(const RadixIn& in, int64_t seg_base, int e, int n, uint32_t& key,
                                           int32_t& val, bool& valid)
{
    valid = e < n;
    key = 0;
    val = 0;
    if (!valid) return;
    if (in.values) {
        key = rank_key(in.values[seg_base + e]);
        val = e;
    } else {
        key = in.key[seg_base + e];
        val = in.val[seg_base + e];
    }
}

__global__ void __launch_bounds__(kRadixThreads) radix_hist_kernel(RadixIn in, int n, int nchunk, int shift,
                                                                   uint32_t* __restrict__ hist)
{
    __shared__ uint32_t h[kRadixBins];
    const int seg = blockIdx.y, chunk = blockIdx.x;
    h[threadIdx.x] = 0;
    __syncthreads();
    const int64_t seg_base = (int64_t)seg * n;
    for (int r = 0; r < kRadixChunk / kRadixThreads; ++r) {
        int e = chunk * kRadixChunk + r * kRadixThreads + threadIdx.x;
        uint32_t key;
        int32_t val;
        bool valid;
        radix_load(in, seg_base, e, n, key, val, valid);
        if (valid) atomicAdd(&h[(key >> shift) & 0xff], 1u);
    }
    __syncthreads();
    hist[((int64_t)seg * kRadixBins + threadIdx.x) * nchunk + chunk] = h[threadIdx.x];
}

// Exclusive scan of a segment's [digit][chunk] counts, in place.
__global__ void __launch_bounds__(1024) radix_scan_kernel(uint32_t* __restrict__ hist, int nchunk)
{
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t carry;
    const int seg = blockIdx.x;
    uint32_t* h = hist + (int64_t)seg * kRadixBins * nchunk;
    const int total = kRadixBins * nchunk;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < total; base += 1024) {
        int e = base + threadIdx.x;
        uint32_t v = e < total ? h[e] : 0;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t t = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;  // inclusive over warps
        }
        __syncthreads();
        uint32_t before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
        if (e < total) h[e] = before;
        __syncthreads();
        if (threadIdx.x == 0) carry += warp_tot[31];
        __syncthreads();
    }
}

// Stable scatter of one chunk.  Warp w owns units [w*256, w*256+256) of the
// chunk and walks them in 8 rounds of 32, so (warp, round, lane) is the units'
// original order; __match_any_sync groups the lanes of one digit in a round.
// hist: with `counts`, the per-(digit, chunk) counts of radix_hist_kernel, from which each CTA
// computes its own offsets (digit d of chunk c starts after every key of a smaller digit and
// the digit-d keys of chunks before c); otherwise the offsets themselves (radix_scan_kernel
// ran: segments with many chunks).  rank: when non-null (the last pass), rank[value] = the
// key's place in the sorted order is written as well.
__global__ void __launch_bounds__(kRadixThreads) radix_scatter_kernel(RadixIn in, int n, int nchunk, int shift,
                                                                      const uint32_t* __restrict__ hist, bool counts,
                                                                      uint32_t* __restrict__ key_out,
                                                                      int32_t* __restrict__ val_out,
                                                                      int32_t* __restrict__ rank, int* status)
{
    constexpr int kWarps = kRadixThreads / 32;
    constexpr int kRounds = kRadixChunk / kRadixThreads;
    static_assert(kRadixThreads == kRadixBins, "one thread per digit");
    __shared__ uint32_t wc[kWarps][kRadixBins];
    __shared__ uint32_t gbase[kRadixBins];
    __shared__ uint32_t wtot[kWarps];
    const int seg = blockIdx.y, chunk = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = threadIdx.x; t < kWarps * kRadixBins; t += kRadixThreads) (&wc[0][0])[t] = 0;
    {
        const uint32_t* hd = hist + ((int64_t)seg * kRadixBins + threadIdx.x) * nchunk;
        if (counts) {
            uint32_t tot = 0, pre = 0;
            for (int c = 0; c < nchunk; ++c) {
                const uint32_t v = hd[c];
                tot += v;
                pre += c < chunk ? v : 0u;
            }
            // exclusive scan of the digit totals (thread = digit)
            uint32_t x = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) wtot[warp] = x;
            __syncthreads();
            uint32_t wb = 0;
            for (int w = 0; w < warp; ++w) wb += wtot[w];
            gbase[threadIdx.x] = wb + x - tot + pre;
        } else {
            gbase[threadIdx.x] = hd[chunk];
        }
    }
    __syncthreads();

    const int64_t seg_base = (int64_t)seg * n;
    const uint32_t lt = lanemask_lt();
    uint32_t key[kRounds];
    int32_t val[kRounds];
    uint32_t loc[kRounds];
    int dig[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        int e = chunk * kRadixChunk + warp * (kRounds * 32) + r * 32 + lane;
        bool valid;
        radix_load(in, seg_base, e, n, key[r], val[r], valid);
        int d = valid ? (int)((key[r] >> shift) & 0xff) : kRadixBins;
        dig[r] = d;
        uint32_t peers = __match_any_sync(0xffffffffu, d);
        uint32_t rk = __popc(peers & lt);
        loc[r] = valid ? wc[warp][d] + rk : 0;
        __syncwarp();
        if (valid && rk == 0) wc[warp][d] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {
        uint32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            uint32_t t = wc[w][threadIdx.x];
            wc[w][threadIdx.x] = run;
            run += t;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        int d = dig[r];
        if (d < kRadixBins) {
            uint32_t dl = gbase[d] + wc[warp][d] + loc[r];
            if (dl < (uint32_t)n) {
                key_out[seg_base + dl] = key[r];
                val_out[seg_base + dl] = val[r];
                if (rank) {
                    if (val[r] >= 0 && val[r] < n)
                        rank[seg_base + val[r]] = (int32_t)dl;
                    else
                        set_status(status, DMA_ERR_DEVICE_CHECK);
                }
            } else {
                set_status(status, DMA_ERR_DEVICE_CHECK);
            }
        }
    }
}

// ------------------------------------------------------------ unit budget --

// The budget in units of one segment (b, KV head h).  Uniform: k_max.  Per head
// (Sparse Frontier summary, budget allocation across heads): w_head[h] keys,
// floor(w_head[h] / block) units; an entry outside [0, w_max] -- the budget the
// kept layout was sized for -- is recorded and clamped into that range.
struct HeadBudget {
    const int32_t* w_head;  // device [Hkv] or nullptr
    int Hkv, block, w_max, k_max;
};

__device__ __forceinline__ int seg_budget(const HeadBudget& hb, int seg, int* status, bool report)
{
    if (!hb.w_head) return hb.k_max;
    int w = hb.w_head[seg % hb.Hkv];
    if (w < 0 || w > hb.w_max) {
        if (report) set_status(status, DMA_ERR_DEVICE_CHECK);
        w = w < 0 ? 0 : hb.w_max;
    }
    const int k = hb.block > 1 ? w / hb.block : w;
    return k < hb.k_max ? k : hb.k_max;
}

// ------------------------------------------------------------ expiry (global) --

__global__ void global_expiry_kernel(const int32_t* __restrict__ rank, int n, HeadBudget hb,
                                     int32_t* __restrict__ E, int* status)
{
    const int seg = blockIdx.y;
    const int k = seg_budget(hb, seg, status, blockIdx.x == 0 && threadIdx.x == 0);
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < n) E[(int64_t)seg * n + u] = rank[(int64_t)seg * n + u] < k ? n : u;
}

// ---------------------------------------------------------- expiry (row-wise) --

// tab[seg][c][xb] = number of ranks in chunk c whose position lies in block xb.
__global__ void count_table_kernel(const int32_t* __restrict__ p, int n, int T, int nC, int X, int nX,
                                   int32_t* __restrict__ tab)
{
    extern __shared__ int32_t cnt[];
    const int seg = blockIdx.y, c = blockIdx.x;
    for (int t = threadIdx.x; t < nX; t += blockDim.x) cnt[t] = 0;
    __syncthreads();
    const int t_end = min(n, (c + 1) * T);
    for (int t = c * T + threadIdx.x; t < t_end; t += blockDim.x) {
        const int x = p[(int64_t)seg * n + t];
        if (x >= 0 && x < n) atomicAdd(&cnt[x / X], 1);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < nX; t += blockDim.x) tab[((int64_t)seg * nC + c) * nX + t] = cnt[t];
}

// In place: tab[seg][c][xb] <- number of ranks < c*T in position block xb.  One
// thread per (segment, xb) column; the column's counts are read in batches so
// that the loads of a batch are in flight together.
constexpr int kPrefixBatch = 16;
__global__ void count_prefix_kernel(int32_t* __restrict__ tab, int nC, int nX)
{
    const int seg = blockIdx.y;
    const int xb = blockIdx.x * blockDim.x + threadIdx.x;
    if (xb >= nX) return;
    int32_t* col = tab + (int64_t)seg * nC * nX + xb;
    int32_t run = 0;
    for (int c0 = 0; c0 < nC; c0 += kPrefixBatch) {
        int32_t v[kPrefixBatch];
#pragma unroll
        for (int i = 0; i < kPrefixBatch; ++i) v[i] = c0 + i < nC ? col[(int64_t)(c0 + i) * nX] : 0;
#pragma unroll
        for (int i = 0; i < kPrefixBatch; ++i) {
            if (c0 + i < nC) col[(int64_t)(c0 + i) * nX] = run;
            run += v[i];
        }
    }
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, <= 1024).
__device__ int block_exclusive_scan(int v, int* warp_buf, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? warp_buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_buf[lane] = t;
    }
    __syncthreads();
    int before = (warp > 0 ? warp_buf[warp - 1] : 0) + x - v;
    *total = warp_buf[nw - 1];
    __syncthreads();
    return before;
}

// f0[seg][c] = f(t_start) with t_start = max(c*T, k): the k-th smallest position
// among ranks < t_start.  Only chunks that contain a rank >= k need it.
constexpr int kBoundaryThreads = 256;
__global__ void __launch_bounds__(kBoundaryThreads) boundary_kernel(const int32_t* __restrict__ p,
                                                                   const int32_t* __restrict__ rank,
                                                                   const int32_t* __restrict__ tab, int n,
                                                                   HeadBudget hb, int T, int nC, int X, int nX,
                                                                   int32_t* __restrict__ f0, int* status)
{
    extern __shared__ int32_t cnt[];  // [nX]
    __shared__ int warp_buf[32];
    __shared__ int sel_block, sel_need;
    const int seg = blockIdx.y, c = blockIdx.x;
    const int k = seg_budget(hb, seg, status, c == 0 && threadIdx.x == 0);
    const int t_begin = c * T, t_end = min(n, t_begin + T);
    const int t_start = max(t_begin, k);
    if (t_start >= t_end) return;
    if (k == 0) {
        if (threadIdx.x == 0) f0[(int64_t)seg * nC + c] = -1;
        return;
    }
    const int32_t* ps = p + (int64_t)seg * n;
    const int32_t* rs = rank + (int64_t)seg * n;
    for (int xb = threadIdx.x; xb < nX; xb += blockDim.x) cnt[xb] = tab[((int64_t)seg * nC + c) * nX + xb];
    __syncthreads();
    for (int t = t_begin + threadIdx.x; t < t_start; t += blockDim.x) {
        const int x = ps[t];
        if (x >= 0 && x < n) atomicAdd(&cnt[x / X], 1);
    }
    __syncthreads();
    // find the position block holding the k-th smallest inserted position
    if (threadIdx.x == 0) {
        int run = 0, xb = 0;
        for (; xb < nX; ++xb) {
            if (run + cnt[xb] >= k) break;
            run += cnt[xb];
        }
        sel_block = xb;
        sel_need = k - run;  // 1-based order inside the block
        // written first so that the walk never starts from an unset value
        f0[(int64_t)seg * nC + c] = -1;
        if (xb >= nX) set_status(status, DMA_ERR_DEVICE_CHECK);
    }
    __syncthreads();
    const int xb = sel_block, need = sel_need;
    if (xb >= nX) return;
    // positions of the block, in ascending order, flagged if inserted (rank < t_start)
    const int per = (X + blockDim.x - 1) / blockDim.x;
    const int x_lo = xb * X + threadIdx.x * per;
    int mine = 0;
    for (int q = 0; q < per; ++q) {
        int x = x_lo + q;
        if (x < min(n, (xb + 1) * X) && rs[x] < t_start) ++mine;
    }
    int total;
    int before = block_exclusive_scan(mine, warp_buf, &total);
    if (need > before && need <= before + mine) {
        int seen = before;
        for (int q = 0; q < per; ++q) {
            int x = x_lo + q;
            if (x < min(n, (xb + 1) * X) && rs[x] < t_start) {
                if (++seen == need) {
                    f0[(int64_t)seg * nC + c] = x;
                    break;
                }
            }
        }
    }
}

// One warp per (segment, rank chunk): E[p[t]] = max(p[t], f(t)).
// kSmem: the CTA first copies the segment's rank array into shared memory as
// 16-bit values (n <= 65536), so the downward scans for the staircase's next
// step read shared memory; every warp of the CTA walks one chunk of the same
// segment.  Otherwise the scans read rank[] from global memory.
constexpr int kWalkWarps = 4;
constexpr int kWalkSmemWarps = 32;
template <bool kSmem>
__global__ void walk_kernel(const int32_t* __restrict__ p, const int32_t* __restrict__ rank,
                            const int32_t* __restrict__ f0, int nseg, int n, HeadBudget hb, int T, int nC,
                            int32_t* __restrict__ E, int* status)
{
    extern __shared__ uint16_t rk16[];  // [n] (kSmem)
    const int lane = threadIdx.x & 31;
    int seg, c;
    if (kSmem) {
        seg = blockIdx.y;
        c = blockIdx.x * kWalkSmemWarps + (threadIdx.x >> 5);
        const int32_t* rsrc = rank + (int64_t)seg * n;
        for (int x = threadIdx.x; x < n; x += blockDim.x) rk16[x] = (uint16_t)rsrc[x];
        __syncthreads();
        if (c >= nC) return;
    } else {
        const int gw = blockIdx.x * kWalkWarps + (threadIdx.x >> 5);
        if (gw >= nseg * nC) return;
        seg = gw / nC;
        c = gw % nC;
    }
    const int k = seg_budget(hb, seg, status, false);  // reported by the boundary kernel
    const int32_t* ps = p + (int64_t)seg * n;
    const int32_t* rs = rank + (int64_t)seg * n;
    auto rank_at = [&](int pos) -> int { return kSmem ? (int)rk16[pos] : rs[pos]; };
    int32_t* Es = E + (int64_t)seg * n;
    const int t_begin = c * T, t_end = min(n, t_begin + T);
    const int t_start = min(t_end, max(t_begin, k));
    // ranks below k: fewer than k keys beat them, they are never evicted
    for (int t = t_begin + lane; t < t_start; t += 32) {
        const int x = ps[t];
        if (x >= 0 && x < n) Es[x] = n;
    }
    if (t_start >= t_end) return;
    int x = f0[(int64_t)seg * nC + c];
    if (x < -1 || x >= n) {
        if (lane == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
        return;
    }
    for (int t0 = t_start; t0 < t_end; t0 += 32) {
        const int my_t = t0 + lane;
        int my_p = my_t < t_end ? ps[my_t] : 0;
        if (my_p < 0 || my_p >= n) {
            set_status(status, DMA_ERR_DEVICE_CHECK);
            my_p = 0;
        }
        int my_x = 0;
        const int steps = min(32, t_end - t0);
        for (int q = 0; q < steps; ++q) {
            const int pt = __shfl_sync(0xffffffffu, my_p, q);
            if (lane == q) my_x = x;
            if (pt < x) {
                // f moves to the largest inserted position below x (p[t] itself qualifies)
                const int t = t0 + q;
                int base = x - 1;
                for (;;) {
                    int found = -1;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        int pos = base - s * 32 - lane;
                        bool flag = pos >= 0 && rank_at(pos) <= t;
                        uint32_t m = __ballot_sync(0xffffffffu, flag);
                        if (found < 0 && m) found = base - s * 32 - (__ffs(m) - 1);
                    }
                    if (found >= 0) {
                        x = found;
                        break;
                    }
                    base -= 128;
                    if (base < 0) {  // cannot happen for a valid permutation: p[t] itself qualifies
                        if (lane == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
                        x = -1;
                        break;
                    }
                }
            }
        }
        if (my_t < t_end) Es[my_p] = max(my_p, my_x);
    }
}

// ------------------------------------------------------- block units -> keys --

__global__ void expand_block_kernel(const int32_t* __restrict__ bexp, int S, int nb, int block,
                                    int32_t* __restrict__ expiry)
{
    const int seg = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= S) return;
    const int bk = j / block;
    const int lo = bk * block + block - 1;
    int e;
    if (bk >= nb) {
        e = min(lo, S);
    } else {
        const int E = bexp[(int64_t)seg * nb + bk];
        if (E >= nb) {
            e = S;
        } else {
            const int hi = E * block + block - 1;
            e = hi > lo ? hi : lo;
        }
    }
    expiry[(int64_t)seg * S + j] = e;
}

// ------------------------------------------------------------ compaction ------
//
// Three lists per segment, each written in two launches over chunks of kListChunk
// (counts, then writes at offsets summed from the counts of the chunks before):
//   idx      keys ever in the top set (lo_j < expiry_j), ascending
//   top_idx  keys in the top set of the last row (expiry_j >= S), ascending
//   kr       units ever in the top set, in rank order (best first), with their
//            expiry: the per-tile key lists are filtered from it
// A unit is one key (token units) or one block of `block` keys, whose keys share
// one interval.

constexpr int kListChunk = 4096;
constexpr int kListThreads = 512;
constexpr int kListPer = kListChunk / kListThreads;  // consecutive items per thread

// Block-wide exclusive scan of two counters per thread (blockDim.x a multiple of
// 32, <= 1024); totals in *tot.
__device__ int2 block_exclusive_scan2(int2 v, int2* warp_buf, int2* tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int2 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yx = __shfl_up_sync(0xffffffffu, x.x, o), yy = __shfl_up_sync(0xffffffffu, x.y, o);
        if (lane >= o) {
            x.x += yx;
            x.y += yy;
        }
    }
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int2 t = lane < nw ? warp_buf[lane] : make_int2(0, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yx = __shfl_up_sync(0xffffffffu, t.x, o), yy = __shfl_up_sync(0xffffffffu, t.y, o);
            if (lane >= o) {
                t.x += yx;
                t.y += yy;
            }
        }
        warp_buf[lane] = t;
    }
    __syncthreads();
    const int2 w0 = warp > 0 ? warp_buf[warp - 1] : make_int2(0, 0);
    *tot = warp_buf[nw - 1];
    __syncthreads();
    return make_int2(w0.x + x.x - v.x, w0.y + x.y - v.y);
}

struct ListItems {
    int ever[kListPer], last[kListPer], kr[kListPer];  // flags
    int kr_u[kListPer], kr_e[kListPer];
};

// Flags of this thread's items of chunk c: keys c*kListChunk + kListPer*tid + i (index
// order) and ranks likewise (rank order).
__device__ __forceinline__ void list_items(const int32_t* ex, const int32_t* p, int S, int n, int block, int c,
                                           ListItems& it, int* status)
{
    const int base = c * kListChunk + kListPer * (int)threadIdx.x;
    const int bs = block <= 1 ? 1 : block;
#pragma unroll
    for (int i = 0; i < kListPer; ++i) {
        const int j = base + i;
        const int e = j < S ? ex[j] : 0;
        const int ever = (j < S && top_lo(j, block) < e) ? 1 : 0;
        it.ever[i] = ever;
        it.last[i] = (ever && e >= S) ? 1 : 0;
        const int r = base + i;
        int u = -1, eu = 0, kr = 0;
        if (r < n) {
            u = p[r];
            if (u < 0 || u >= n) {
                set_status(status, DMA_ERR_DEVICE_CHECK);
            } else {
                eu = ex[(int64_t)u * bs];
                kr = top_lo(u * bs, block) < eu ? 1 : 0;
            }
        }
        it.kr[i] = kr;
        it.kr_u[i] = u;
        it.kr_e[i] = eu;
    }
}

// cnt[seg][chunk] = (ever, last, kr) counts of the chunk.
__global__ void __launch_bounds__(kListThreads) list_count_kernel(const int32_t* __restrict__ expiry,
                                                                  const int32_t* __restrict__ p, int S, int n,
                                                                  int block, int nlc, int4* __restrict__ cnt,
                                                                  int* status)
{
    __shared__ int4 red[kListThreads / 32];
    const int seg = blockIdx.y, c = blockIdx.x;
    ListItems it;
    list_items(expiry + (int64_t)seg * S, p + (int64_t)seg * n, S, n, block, c, it, status);
    int a = 0, l = 0, k = 0;
#pragma unroll
    for (int i = 0; i < kListPer; ++i) {
        a += it.ever[i];
        l += it.last[i];
        k += it.kr[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        l += __shfl_xor_sync(0xffffffffu, l, o);
        k += __shfl_xor_sync(0xffffffffu, k, o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = make_int4(a, l, k, 0);
    __syncthreads();
    if (threadIdx.x == 0) {
        int4 t = make_int4(0, 0, 0, 0);
        for (int w = 0; w < kListThreads / 32; ++w) {
            t.x += red[w].x;
            t.y += red[w].y;
            t.z += red[w].z;
        }
        cnt[(int64_t)seg * nlc + c] = t;
    }
}

__global__ void __launch_bounds__(kListThreads) list_write_kernel(
    const int32_t* __restrict__ expiry, const int32_t* __restrict__ p, int S, int n, int block, int nlc,
    const int4* __restrict__ cnt, int32_t* __restrict__ idx, int32_t* __restrict__ count,
    int32_t* __restrict__ top_idx, int32_t* __restrict__ top_count, int top_cap, int32_t* __restrict__ kr_u,
    int32_t* __restrict__ kr_e, int32_t* __restrict__ kr_n, int* status)
{
    __shared__ int2 warp_buf[32];
    __shared__ int4 off_s;
    const int seg = blockIdx.y, c = blockIdx.x;
    // offsets: the counts of the chunks before this one
    if (threadIdx.x < 32) {
        int a = 0, l = 0, k = 0;
        for (int q = threadIdx.x; q < c; q += 32) {
            const int4 v = cnt[(int64_t)seg * nlc + q];
            a += v.x;
            l += v.y;
            k += v.z;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            l += __shfl_xor_sync(0xffffffffu, l, o);
            k += __shfl_xor_sync(0xffffffffu, k, o);
        }
        if (threadIdx.x == 0) off_s = make_int4(a, l, k, 0);
    }
    ListItems it;
    list_items(expiry + (int64_t)seg * S, p + (int64_t)seg * n, S, n, block, c, it, status);
    int a = 0, l = 0, k = 0;
#pragma unroll
    for (int i = 0; i < kListPer; ++i) {
        a += it.ever[i];
        l += it.last[i];
        k += it.kr[i];
    }
    int2 tot;
    const int2 b_al = block_exclusive_scan2(make_int2(a, l), warp_buf, &tot);
    const int b_k = block_exclusive_scan2(make_int2(k, 0), warp_buf, &tot).x;
    const int4 off = off_s;
    const int base = c * kListChunk + kListPer * (int)threadIdx.x;
    int oa = off.x + b_al.x, ol = off.y + b_al.y, ok = off.z + b_k;
#pragma unroll
    for (int i = 0; i < kListPer; ++i) {
        const int j = base + i;
        if (it.ever[i]) idx[(int64_t)seg * S + oa++] = j;
        if (it.last[i] && top_idx) {
            if (ol < top_cap)
                top_idx[(int64_t)seg * top_cap + ol] = j;
            else
                set_status(status, DMA_ERR_DEVICE_CHECK);
            ++ol;
        }
        if (it.kr[i]) {
            kr_u[(int64_t)seg * n + ok] = it.kr_u[i];
            kr_e[(int64_t)seg * n + ok] = it.kr_e[i];
            ++ok;
        }
    }
    if (c == nlc - 1 && threadIdx.x == kListThreads - 1) {
        count[seg] = oa;
        if (top_count) top_count[seg] = min(ol, top_cap);
        kr_n[seg] = ok;
    }
}

// ---------------------------------------------------- super-group lists ---

// The entries of the rank-ordered ever-kept list that can reach a super group of
// sg_tiles consecutive query tiles (the same tile-range test as the per-tile lists),
// compacted in rank order.  Every per-tile list CTA of the super group then walks
// this list instead of the whole one: on long sequences most ever-kept units live
// for a short stretch of rows, so the super group's list is a fraction of the whole.
// An entry reaching the rows [R0, R1] is in the top set of row R0 or enters it at a
// later row, so a list holds at most k + (R1 - R0 + 1) entries (sg_cap).
constexpr int kSgThreads = 1024;
constexpr int kSgPer = 4;

template <bool kBlocks>
__global__ void __launch_bounds__(kSgThreads) sg_list_kernel(const int32_t* __restrict__ kr_u,
                                                            const int32_t* __restrict__ kr_e,
                                                            const int32_t* __restrict__ kr_n, int S, int n,
                                                            int block, int window, int n_qt, int sg_tiles,
                                                            int sg_cap, int32_t* __restrict__ sg_u,
                                                            int32_t* __restrict__ sg_e, int32_t* __restrict__ sg_n,
                                                            int* status)
{
    __shared__ int warp_buf[32];
    const int seg = blockIdx.y, sg = blockIdx.x, n_sg = gridDim.x;
    const int first = sg * sg_tiles, last = min(n_qt, first + sg_tiles) - 1;
    const int bs = kBlocks ? block : 1;
    const int32_t* ku = kr_u + (int64_t)seg * n;
    const int32_t* ke = kr_e + (int64_t)seg * n;
    int32_t* ou = sg_u + ((int64_t)seg * n_sg + sg) * sg_cap;
    int32_t* oe = sg_e + ((int64_t)seg * n_sg + sg) * sg_cap;
    const int m = min(max(kr_n[seg], 0), n);
    int out = 0;
    for (int base = 0; base < m; base += kSgThreads * kSgPer) {
        int u[kSgPer], e[kSgPer];
        unsigned keep = 0;
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kSgPer; ++i) {
            const int q = base + (int)threadIdx.x * kSgPer + i;
            u[i] = 0;
            e[i] = 0;
            if (q >= m) continue;
            u[i] = ku[q];
            e[i] = ke[q];
            const int j0 = u[i] * bs;
            if (u[i] < 0 || j0 >= S) {
                set_status(status, DMA_ERR_DEVICE_CHECK);
                continue;
            }
            if (e[i] <= 0) continue;
            const int lo = top_lo(j0, block);
            const int ta = max(lo / kQTile, window > 0 ? (j0 + window + kQTile - 1) / kQTile : j0 / kQTile);
            const int tb = min(n_qt - 1, (e[i] - 1) / kQTile);
            if (ta <= tb && ta <= last && tb >= first) {
                keep |= 1u << i;
                ++cnt;
            }
        }
        int tot;
        int o = out + block_exclusive_scan(cnt, warp_buf, &tot);
#pragma unroll
        for (int i = 0; i < kSgPer; ++i) {
            if (!((keep >> i) & 1u)) continue;
            if (o < sg_cap) {
                ou[o] = u[i];
                oe[o] = e[i];
            } else {
                set_status(status, DMA_ERR_DEVICE_CHECK);
            }
            ++o;
        }
        out += tot;
    }
    if (threadIdx.x == 0) sg_n[seg * n_sg + sg] = min(out, sg_cap);
}

// ----------------------------------------------------------- per-tile lists ---

constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileGroup = 8;          // consecutive query tiles per CTA
constexpr int kTilePartialCap = 1024;  // keys kept by only some rows of a tile (at most ~384 by construction)
constexpr int kTileOccSmem = 64 * 1024;  // largest shared-memory occupancy array (sequences up to 512K keys)
constexpr int kTilePartBytes = kTileGroup * kTilePartialCap * 4;

// For query tile [q0, q1]: keys j <= lim (lim = q0 - window, or q1 without a
// window) with lo_j <= q1 and expiry_j > q0.  The keys kept by every row of the
// tile (lo_j <= q0 and expiry_j > q1) come first, then the keys kept by only some
// of its rows; each group in rank order (best unit first; the keys of a block
// ascending), so that a consumer walking the list in blocks meets the keys most
// likely to hold a row's maximum first and finds the blocks that need a per-row
// mask at the end.  Also the bitmap of 64-key blocks holding a kept key
// (gathered keys and the window band).
//
// A CTA builds the lists of kTileGroup consecutive tiles of one segment.  Each
// warp owns a contiguous slice of the rank-ordered unit list and walks it twice,
// 32 entries at a time: once to count its keys per tile, once to write them at
// its offsets; order within a warp comes from ballots (token units: one key per
// entry) or warp scans (block units), across warps from one block-wide step.
// kr_u, kr_e, kr_n: the ever-kept units in rank order with their expiry, per list (list_stride
// entries apart) and their number; list l = seg * lists_per_seg + tile0 / tiles_per_list.
// Token units fit four CTAs per SM (one wave on long sequences); block units take more
// registers (the per-entry key counts): two CTAs per SM, which keeps them from spilling.
template <bool kBlocks>
__global__ void __launch_bounds__(kTileThreads, kBlocks ? 2 : 4) tile_list_kernel(
    const int32_t* __restrict__ kr_u, const int32_t* __restrict__ kr_e, const int32_t* __restrict__ kr_n,
    int list_stride, int lists_per_seg, int tiles_per_list, int S, int block, int window, int n_qt,
    int tile_stride, int bitmap_words, int32_t* __restrict__ tile_cnt, int32_t* __restrict__ tile_idx,
    uint32_t* __restrict__ bitmap, int* status)
{
    // one byte per (tile, 64-key block), set by plain stores and packed into the bitmap at the
    // end; for long sequences (occ_smem false) the bits go straight to the bitmap in global
    // memory with atomics instead
    // dynamic shared memory: the partial groups, then the occupancy bytes
    extern __shared__ __align__(16) unsigned char tl_smem[];
    auto part_s = reinterpret_cast<int(*)[kTilePartialCap]>(tl_smem);  // [kTileGroup]
    uint8_t* occ = tl_smem + kTilePartBytes;  // [kTileGroup][bitmap_words * 32] when occ_smem
    __shared__ int2 warp_cnt[kTileWarps][kTileGroup];
    const int seg = blockIdx.y, tile0 = blockIdx.x * kTileGroup;
    const int ntile = min(kTileGroup, n_qt - tile0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = lanemask_lt();
    const int bs = kBlocks ? block : 1;
    const int list = seg * lists_per_seg + tile0 / tiles_per_list;
    const int32_t* ku = kr_u + (int64_t)list * list_stride;
    const int32_t* ke = kr_e + (int64_t)list * list_stride;
    const int m = min(max(kr_n[list], 0), list_stride);
    const int occ_len = bitmap_words * 32;
    const bool occ_smem = kTileGroup * occ_len <= kTileOccSmem;
    if (bitmap) {
        if (occ_smem) {
            for (int t = threadIdx.x; t < kTileGroup * occ_len; t += kTileThreads) occ[t] = 0;
        } else {
            for (int t = threadIdx.x; t < ntile * bitmap_words; t += kTileThreads)
                bitmap[((int64_t)seg * n_qt + tile0) * bitmap_words + t] = 0;
            __syncthreads();
        }
    }
    auto mark = [&](int g, int b64) {
        if (occ_smem)
            occ[g * occ_len + b64] = 1;
        else
            atomicOr(&bitmap[((int64_t)seg * n_qt + tile0 + g) * bitmap_words + b64 / 32], 1u << (b64 & 31));
    };
    int tq0[kTileGroup], tq1[kTileGroup], tlim[kTileGroup];
#pragma unroll
    for (int g = 0; g < kTileGroup; ++g) {
        const int t = min(tile0 + g, n_qt - 1);
        tq0[g] = t * kQTile;
        tq1[g] = min(S, tq0[g] + kQTile) - 1;
        tlim[g] = window > 0 ? tq0[g] - window : tq1[g];
    }
    struct Ent {
        int j0, lo, e;
        bool valid;
    };
    auto load = [&](int q) -> Ent {
        Ent x{0, 0, 0, false};
        if (q < m) {
            const int u = ku[q];
            x.e = ke[q];
            x.j0 = u * bs;
            if (u < 0 || x.j0 >= S) {
                set_status(status, DMA_ERR_DEVICE_CHECK);
            } else {
                x.lo = top_lo(x.j0, block);
                x.valid = true;
            }
        }
        return x;
    };
    // bit g of `member`: the entry has keys in tile g's list; of `full`: they are kept by every row
    // of the tile.  Both are contiguous tile ranges: the entry is in the list of tiles ta..tb
    //   lo_j <= q1(t)   <=>  t >= lo / 128
    //   j0 <= lim(t)    <=>  t >= ceil((j0 + window) / 128)  (window > 0), t >= j0 / 128 otherwise
    //   expiry > q0(t)  <=>  t <= (expiry - 1) / 128
    // and kept by every row of tiles fa..fb within it
    //   lo_j <= q0(t)   <=>  t >= ceil(lo / 128)
    //   expiry > q1(t)  <=>  expiry == S  or  t <= expiry / 128 - 1
    const int last_tile = tile0 + ntile - 1;
    auto masks = [&](const Ent& x, uint32_t& member, uint32_t& full) {
        member = 0;
        full = 0;
        if (!x.valid || x.e <= 0) return;
        const int ta = max(x.lo / kQTile, window > 0 ? (x.j0 + window + kQTile - 1) / kQTile : x.j0 / kQTile);
        const int tb = min(n_qt - 1, (x.e - 1) / kQTile);
        const int fa = max(ta, (x.lo + kQTile - 1) / kQTile);
        const int fb = x.e >= S ? tb : min(tb, x.e / kQTile - 1);
        auto range = [&](int a, int b) -> uint32_t {
            a = max(a, tile0);
            b = min(b, last_tile);
            if (a > b) return 0u;
            return ((2u << (b - tile0)) - 1u) & ~((1u << (a - tile0)) - 1u);
        };
        member = range(ta, tb);
        full = member & range(fa, fb);
    };
    auto nkeys = [&](const Ent& x, int g) -> int { return kBlocks ? min(bs, tlim[g] - x.j0 + 1) : 1; };
    auto warp_excl = [&](int v, int& total) -> int {  // exclusive prefix over the warp, and its total
        if (!kBlocks) {
            const uint32_t bal = __ballot_sync(0xffffffffu, v != 0);
            total = __popc(bal);
            return __popc(bal & lt);
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        total = __shfl_sync(0xffffffffu, x, 31);
        return x - v;
    };
    // this warp's slice of the list, in multiples of 32 entries
    const int per = ((m + kTileWarps - 1) / kTileWarps + 31) / 32 * 32;
    const int w_begin = min(m, warp * per), w_end = min(m, w_begin + per);
    // pass 1: this lane's key counts per tile, then the warp's.  Token units have one key per
    // entry: the eight per-tile counts are byte lanes of one 64-bit word each for the two groups,
    // a member mask added with its bits spread into bytes (flushed before a byte can overflow).
    int2 cnt[kTileGroup];
#pragma unroll
    for (int g = 0; g < kTileGroup; ++g) cnt[g] = make_int2(0, 0);
    uint64_t acc_f = 0, acc_p = 0;
    int acc_n = 0;
    auto spread = [](uint32_t m8) -> uint64_t {  // bit g of m8 -> byte g
        uint64_t r = 0;
#pragma unroll
        for (int g = 0; g < kTileGroup; ++g) r |= (uint64_t)((m8 >> g) & 1u) << (8 * g);
        return r;
    };
    auto flush = [&]() {
#pragma unroll
        for (int g = 0; g < kTileGroup; ++g) {
            cnt[g].x += (int)((acc_f >> (8 * g)) & 0xffu);
            cnt[g].y += (int)((acc_p >> (8 * g)) & 0xffu);
        }
        acc_f = acc_p = 0;
        acc_n = 0;
    };
#pragma unroll 4
    for (int qb = w_begin; qb < w_end; qb += 32) {
        const Ent x = load(qb + lane < w_end ? qb + lane : m);
        uint32_t mem, full;
        masks(x, mem, full);
        if (!kBlocks) {
            acc_f += spread(full);
            acc_p += spread(mem & ~full);
            if (++acc_n == 255) flush();
            continue;
        }
        if (mem == 0) continue;
#pragma unroll
        for (int g = 0; g < kTileGroup; ++g) {
            const int c = (mem >> g) & 1u ? nkeys(x, g) : 0;
            if ((full >> g) & 1u)
                cnt[g].x += c;
            else
                cnt[g].y += c;
        }
    }
    if (!kBlocks) flush();
#pragma unroll
    for (int g = 0; g < kTileGroup; ++g) {
        const int vf = __reduce_add_sync(0xffffffffu, cnt[g].x);
        const int vp = __reduce_add_sync(0xffffffffu, cnt[g].y);
        if (lane == 0) warp_cnt[warp][g] = make_int2(vf, vp);
    }
    __syncthreads();
    int2 off[kTileGroup];
#pragma unroll
    for (int g = 0; g < kTileGroup; ++g) {
        off[g] = make_int2(0, 0);
        for (int w = 0; w < warp; ++w) {
            off[g].x += warp_cnt[w][g].x;
            off[g].y += warp_cnt[w][g].y;
        }
    }
    // pass 2: write at the warp's offsets, in entry order
#pragma unroll 2
    for (int qb = w_begin; qb < w_end; qb += 32) {
        const Ent x = load(qb + lane < w_end ? qb + lane : m);
        uint32_t mem, full;
        masks(x, mem, full);
        if (__ballot_sync(0xffffffffu, mem != 0) == 0) continue;
#pragma unroll
        for (int g = 0; g < kTileGroup; ++g) {
            const bool f = (full >> g) & 1u;
            const int c = (mem >> g) & 1u ? nkeys(x, g) : 0;
            int tf, tp;
            int of = off[g].x + warp_excl(f ? c : 0, tf);
            int op = off[g].y + warp_excl(f ? 0 : c, tp);
            off[g].x += tf;
            off[g].y += tp;
            if (c == 0) continue;
            int32_t* out = tile_idx + ((int64_t)seg * n_qt + tile0 + g) * tile_stride;
            for (int q = 0; q < c; ++q) {
                const int j = x.j0 + q;
                if (f) {
                    if (of < tile_stride)
                        out[of] = j;
                    else
                        set_status(status, DMA_ERR_DEVICE_CHECK);
                    ++of;
                } else {
                    if (op < kTilePartialCap)
                        part_s[g][op] = j;
                    else
                        set_status(status, DMA_ERR_DEVICE_CHECK);
                    ++op;
                }
            }
            if (bitmap)
                for (int b64 = x.j0 / kBitmapBlock; b64 <= (x.j0 + c - 1) / kBitmapBlock; ++b64) mark(g, b64);
        }
    }
    __syncthreads();  // part_s and occ complete
#pragma unroll
    for (int g = 0; g < kTileGroup; ++g) {
        if (g >= ntile) break;
        int tot_f = 0, tot_p = 0;
        for (int w = 0; w < kTileWarps; ++w) {
            tot_f += warp_cnt[w][g].x;
            tot_p += warp_cnt[w][g].y;
        }
        tot_p = min(tot_p, kTilePartialCap);
        const int tile = tile0 + g;
        int32_t* out = tile_idx + ((int64_t)seg * n_qt + tile) * tile_stride;
        for (int t = threadIdx.x; t < tot_p; t += kTileThreads) {
            const int o = tot_f + t;
            if (o < tile_stride)
                out[o] = part_s[g][t];
            else
                set_status(status, DMA_ERR_DEVICE_CHECK);
        }
        if (threadIdx.x == 0) tile_cnt[(int64_t)seg * n_qt + tile] = min(tot_f + tot_p, tile_stride);
        if (bitmap && window > 0) {
            const int band_lo = max(0, tq0[g] - window + 1);
            for (int b64 = band_lo / kBitmapBlock + threadIdx.x; b64 <= tq1[g] / kBitmapBlock; b64 += kTileThreads)
                mark(g, b64);
        }
    }
    if (bitmap && occ_smem) {
        __syncthreads();
        // warp w packs words w, w + 8, ... of every tile: lane l holds block 32 * word + l
        for (int g = 0; g < ntile; ++g) {
            uint32_t* bo = bitmap + ((int64_t)seg * n_qt + tile0 + g) * bitmap_words;
            for (int wd = warp; wd < bitmap_words; wd += kTileWarps) {
                const uint32_t bits = __ballot_sync(0xffffffffu, occ[g * occ_len + 32 * wd + lane] != 0);
                if (lane == 0) bo[wd] = bits;
            }
        }
    }
}

// ---------------------------------------------------------------- update ----

constexpr int kUpdateThreads = 1024;
// top set of row t = top-w(top set of row t-1 + key t), t = seq_len[b] - 1.
__global__ void __launch_bounds__(kUpdateThreads) update_kernel(const float* __restrict__ scores, int Hkv, int S,
                                                                const int32_t* __restrict__ seq_len,
                                                                int32_t* __restrict__ top_idx,
                                                                int32_t* __restrict__ top_count, int top_cap,
                                                                HeadBudget hb, int* status)
{
    extern __shared__ int32_t buf[];  // [budget]
    __shared__ uint32_t red_key[32];
    __shared__ int red_pos[32];
    __shared__ int worst_pos;
    const int seg = blockIdx.x;
    const int b = seg / Hkv;
    const int budget = seg_budget(hb, seg, status, threadIdx.x == 0);
    const int t = seq_len ? seq_len[b] - 1 : S - 1;
    const float* sc = scores + (int64_t)seg * S;
    int32_t* ti = top_idx + (int64_t)seg * top_cap;
    const int cnt = top_count[seg];
    if (t < 0 || t >= S || cnt < 0 || cnt > budget || (cnt > 0 && ti[cnt - 1] >= t)) {
        if (threadIdx.x == 0) set_status(status, DMA_ERR_DEVICE_CHECK);
        return;
    }
    if (budget == 0) return;
    if (cnt < budget) {
        if (threadIdx.x == 0) {
            ti[cnt] = t;
            top_count[seg] = cnt + 1;
        }
        return;
    }
    // worst member: largest ranking key, ties to the larger index (= later position in the list)
    uint32_t wk = 0;
    int wp = -1;
    for (int u = threadIdx.x; u < cnt; u += kUpdateThreads) {
        int j = ti[u];
        buf[u] = j;
        if (j < 0 || j >= S) {
            set_status(status, DMA_ERR_DEVICE_CHECK);
            j = 0;
        }
        uint32_t kk = rank_key(sc[j]);
        if (wp < 0 || kk > wk || (kk == wk && u > wp)) {
            wk = kk;
            wp = u;
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint32_t ok = __shfl_xor_sync(0xffffffffu, wk, o);
        int op = __shfl_xor_sync(0xffffffffu, wp, o);
        if (op >= 0 && (wp < 0 || ok > wk || (ok == wk && op > wp))) {
            wk = ok;
            wp = op;
        }
    }
    if (lane == 0) {
        red_key[warp] = wk;
        red_pos[warp] = wp;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t bk = 0;
        int bp = -1;
        for (int w = 0; w < kUpdateThreads / 32; ++w) {
            int op = red_pos[w];
            uint32_t ok = red_key[w];
            if (op >= 0 && (bp < 0 || ok > bk || (ok == bk && op > bp))) {
                bk = ok;
                bp = op;
            }
        }
        // the newest key has the largest index: it enters only with a strictly better score
        worst_pos = rank_key(sc[t]) < bk ? bp : -1;
    }
    __syncthreads();
    const int wpos = worst_pos;
    if (wpos < 0) return;
    for (int u = wpos + threadIdx.x; u < cnt - 1; u += kUpdateThreads) ti[u] = buf[u + 1];
    if (threadIdx.x == 0) ti[cnt - 1] = t;
}

}  // namespace

// ------------------------------------------------------------------- host ----

SelectPlan make_select_plan(int B, int Hkv, int S, int w, int block)
{
    SelectPlan pl{};
    pl.nseg = B * Hkv;
    pl.S = S;
    pl.n = block <= 1 ? S : S / block;
    pl.k = block <= 1 ? w : w / block;
    if (pl.k > pl.n) pl.k = pl.n;
    const int n = pl.n > 0 ? pl.n : 1;
    pl.nchunk = (n + kRadixChunk - 1) / kRadixChunk;
    // about 256 rank chunks per segment: the chunks right after rank k move the staircase at
    // nearly every rank, so short chunks keep the longest walk short
    pl.T = pl.X = std::max(64, pow2_ceil((n + 255) / 256));
    pl.nC = (n + pl.T - 1) / pl.T;
    pl.nX = (n + pl.X - 1) / pl.X;
    const size_t nu = (size_t)pl.nseg * n;
    size_t o = 0;
    for (int i = 0; i < 2; ++i) {
        pl.off_key[i] = o;
        o = align_up(o + nu * 4, 256);
        pl.off_val[i] = o;
        o = align_up(o + nu * 4, 256);
    }
    pl.off_hist = o;
    o = align_up(o + (size_t)pl.nseg * kRadixBins * pl.nchunk * 4, 256);
    pl.off_rank = o;
    o = align_up(o + nu * 4, 256);
    pl.off_tab = o;
    o = align_up(o + (size_t)pl.nseg * pl.nC * pl.nX * 4, 256);
    pl.off_f0 = o;
    o = align_up(o + (size_t)pl.nseg * pl.nC * 4, 256);
    pl.off_bval = o;
    pl.off_bexp = o;
    if (block > 1) {
        o = align_up(o + nu * 4, 256);
        pl.off_bexp = o;
        o = align_up(o + nu * 4, 256);
    }
    pl.nlc = (std::max(S, n) + kListChunk - 1) / kListChunk;
    pl.off_lcnt = o;
    o = align_up(o + (size_t)pl.nseg * pl.nlc * 16, 256);
    pl.off_krn = o;
    o = align_up(o + (size_t)pl.nseg * 4, 256);
    // super groups: at least 64 query tiles each (a multiple of the per-CTA group), at most 16
    // of them per segment
    const int n_qt = (S + kQTile - 1) / kQTile;
    pl.sg_tiles = std::max(64, (n_qt + 15) / 16);
    pl.sg_tiles = (pl.sg_tiles + kTileGroup - 1) / kTileGroup * kTileGroup;
    pl.n_sg = (n_qt + pl.sg_tiles - 1) / pl.sg_tiles;
    pl.sg_cap = (int)std::min<int64_t>(n, (int64_t)pl.k + (int64_t)pl.sg_tiles * kQTile + 1);
    if (pl.n_sg > 1) {
        const size_t nl = (size_t)pl.nseg * pl.n_sg;
        pl.off_sgu = o;
        o = align_up(o + nl * pl.sg_cap * 4, 256);
        pl.off_sge = o;
        o = align_up(o + nl * pl.sg_cap * 4, 256);
        pl.off_sgn = o;
        o = align_up(o + nl * 4, 256);
    } else {
        pl.off_sgu = pl.off_sge = pl.off_sgn = o;
    }
    pl.bytes = o;
    return pl;
}

cudaError_t launch_select_full(const float* scores, const SelectPlan& pl, const dma_kept_t* kept,
                               const int32_t* w_head, void* ws, int* status, cudaStream_t st)
{
    char* W = static_cast<char*>(ws);
    const int nseg = pl.nseg, n = pl.n, S = pl.S, block = kept->block;
    uint32_t* keyb[2] = {reinterpret_cast<uint32_t*>(W + pl.off_key[0]), reinterpret_cast<uint32_t*>(W + pl.off_key[1])};
    int32_t* valb[2] = {reinterpret_cast<int32_t*>(W + pl.off_val[0]), reinterpret_cast<int32_t*>(W + pl.off_val[1])};
    uint32_t* hist = reinterpret_cast<uint32_t*>(W + pl.off_hist);
    int32_t* rank = reinterpret_cast<int32_t*>(W + pl.off_rank);
    int32_t* tab = reinterpret_cast<int32_t*>(W + pl.off_tab);
    int32_t* f0 = reinterpret_cast<int32_t*>(W + pl.off_f0);
    float* bval = reinterpret_cast<float*>(W + pl.off_bval);
    int32_t* bexp = reinterpret_cast<int32_t*>(W + pl.off_bexp);
    cudaError_t e;

    const HeadBudget hb{w_head, kept->Hkv, block, kept->w, pl.k};
    const float* unit_values = scores;
    int32_t* E = kept->expiry;  // token units: the unit expiry is the key expiry
    if (block > 1) {
        unit_values = bval;
        E = bexp;
        if (n > 0) {
            block_max_kernel<<<dim3((n + 127) / 128, nseg), 128, 0, st>>>(scores, S, n, block, bval);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    if (n > 0) {
        // 1. sort units best-first
        for (int pass = 0; pass < 4; ++pass) {
            RadixIn in{};
            if (pass == 0) {
                in.values = unit_values;
            } else {
                in.key = keyb[(pass - 1) & 1];
                in.val = valb[(pass - 1) & 1];
            }
            const int shift = 8 * pass;
            dim3 grid(pl.nchunk, nseg);
            // few chunks per segment: every scatter CTA sums the counts itself (no scan launch)
            const bool counts = pl.nchunk <= kRadixFuseChunks;
            radix_hist_kernel<<<grid, kRadixThreads, 0, st>>>(in, n, pl.nchunk, shift, hist);
            if (!counts) radix_scan_kernel<<<nseg, 1024, 0, st>>>(hist, pl.nchunk);
            radix_scatter_kernel<<<grid, kRadixThreads, 0, st>>>(in, n, pl.nchunk, shift, hist, counts,
                                                                 keyb[pass & 1], valb[pass & 1],
                                                                 pass == 3 ? rank : nullptr, status);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        const int32_t* p = valb[1];
        // 2-3. unit expiry
        if (kept->mode == DMA_SEL_GLOBAL) {
            global_expiry_kernel<<<dim3((n + 255) / 256, nseg), 256, 0, st>>>(rank, n, hb, E, status);
        } else {
            count_table_kernel<<<dim3(pl.nC, nseg), 256, pl.nX * 4, st>>>(p, n, pl.T, pl.nC, pl.X, pl.nX, tab);
            count_prefix_kernel<<<dim3((pl.nX + 127) / 128, nseg), 128, 0, st>>>(tab, pl.nC, pl.nX);
            boundary_kernel<<<dim3(pl.nC, nseg), kBoundaryThreads, pl.nX * 4, st>>>(p, rank, tab, n, hb, pl.T,
                                                                                    pl.nC, pl.X, pl.nX, f0, status);
            if (n <= 65536) {
                const int smem = n * 2;
                if (smem > 48 * 1024 &&
                    (e = cudaFuncSetAttribute(walk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
                        cudaSuccess)
                    return e;
                walk_kernel<true><<<dim3((pl.nC + kWalkSmemWarps - 1) / kWalkSmemWarps, nseg), kWalkSmemWarps * 32,
                                    smem, st>>>(p, rank, f0, nseg, n, hb, pl.T, pl.nC, E, status);
            } else {
                const int walkers = nseg * pl.nC;
                walk_kernel<false><<<(walkers + kWalkWarps - 1) / kWalkWarps, kWalkWarps * 32, 0, st>>>(
                    p, rank, f0, nseg, n, hb, pl.T, pl.nC, E, status);
            }
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (block > 1) {
        expand_block_kernel<<<dim3((S + 255) / 256, nseg), 256, 0, st>>>(bexp, S, n, block, kept->expiry);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 4. lists: the ever-kept keys and the last row's top set (index order), the ever-kept units
    // in rank order (into the sort's key buffers, free by now), then the per-tile key lists
    {
        int4* lcnt = reinterpret_cast<int4*>(W + pl.off_lcnt);
        int32_t* kr_u = reinterpret_cast<int32_t*>(keyb[0]);
        int32_t* kr_e = reinterpret_cast<int32_t*>(keyb[1]);
        int32_t* kr_n = reinterpret_cast<int32_t*>(W + pl.off_krn);
        const int32_t* p = valb[1];
        dim3 grid(pl.nlc, nseg);
        list_count_kernel<<<grid, kListThreads, 0, st>>>(kept->expiry, p, S, n, block, pl.nlc, lcnt, status);
        list_write_kernel<<<grid, kListThreads, 0, st>>>(kept->expiry, p, S, n, block, pl.nlc, lcnt, kept->idx,
                                                         kept->count, kept->top_idx, kept->top_count, kept->top_cap,
                                                         kr_u, kr_e, kr_n, status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (kept->tile_idx) {
            const int occ = kTileGroup * kept->bitmap_words * 32;
            const int smem = kTilePartBytes + ((kept->bitmap && occ <= kTileOccSmem) ? occ : 0);
            auto kern = block > 1 ? tile_list_kernel<true> : tile_list_kernel<false>;
            if (smem > 48 * 1024 &&
                (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
                return e;
            const int32_t *lu = kr_u, *le = kr_e, *ln = kr_n;
            int stride = n, per_seg = 1, tiles = kept->n_qt;
            if (pl.n_sg > 1) {
                int32_t* sg_u = reinterpret_cast<int32_t*>(W + pl.off_sgu);
                int32_t* sg_e = reinterpret_cast<int32_t*>(W + pl.off_sge);
                int32_t* sg_n = reinterpret_cast<int32_t*>(W + pl.off_sgn);
                auto sgk = block > 1 ? sg_list_kernel<true> : sg_list_kernel<false>;
                sgk<<<dim3(pl.n_sg, nseg), kSgThreads, 0, st>>>(kr_u, kr_e, kr_n, S, n, block, kept->window,
                                                                kept->n_qt, pl.sg_tiles, pl.sg_cap, sg_u, sg_e,
                                                                sg_n, status);
                lu = sg_u;
                le = sg_e;
                ln = sg_n;
                stride = pl.sg_cap;
                per_seg = pl.n_sg;
                tiles = pl.sg_tiles;
            }
            kern<<<dim3((kept->n_qt + kTileGroup - 1) / kTileGroup, nseg), kTileThreads, smem, st>>>(
                lu, le, ln, stride, per_seg, tiles, S, block, kept->window, kept->n_qt, kept->tile_stride,
                kept->bitmap_words, kept->tile_cnt, kept->tile_idx, kept->bitmap, status);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_select_update(const float* scores, const dma_kept_t* kept, const int32_t* seq_len,
                                 const int32_t* w_head, int* status, cudaStream_t st)
{
    const int nseg = kept->B * kept->Hkv;
    const int budget = kept->w < kept->S ? kept->w : kept->S;
    const HeadBudget hb{w_head, kept->Hkv, 1, kept->w, budget};
    size_t smem = (size_t)(budget > 0 ? budget : 1) * 4;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    update_kernel<<<nseg, kUpdateThreads, smem, st>>>(scores, kept->Hkv, kept->S, seq_len, kept->top_idx,
                                                     kept->top_count, kept->top_cap, hb, status);
    return cudaGetLastError();
}

}  // namespace dma
