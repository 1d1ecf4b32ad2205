// Backward of the sparse attention on the 5th-generation tensor cores (bf16,
// D = 64 or 128): two kernels over the same per-query-tile key lists as the
// forward (the tile's gathered keys, then the window band (q0 - window, q1]).
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §四/§五/§七: gradients flow
// through the kept positions only; a skipped position has weight exactly 0 and
// gets exactly zero gradient, so pairs outside the kept sets are never formed.
// With p_ij = exp(scale <Q_i, K_j> + s_j - lse_i) over row i's kept set:
//   dP = dO V^T,  dx = p (dP - Delta_i),  dQ = scale dx K,
//   dK = scale dx^T Q,  dV = p^T dO,  ds_j = sum_i dx_ij.
//
// Row kernel (dQ).  One CTA = one (batch, KV head, query tile); the G query heads
// one after another (a "pass" each), the tile's key blocks inside a pass.  Per
// (head, block): S = Q K^T and dP = dO V^T (both operands in shared memory), then
// the elementwise warps form dx in bf16 over S in tensor memory, and
// dQ += dx K (dx from tensor memory, K in shared memory).  dQ stays in tensor
// memory for the whole pass and is written once (fp32).  S is double-buffered,
// so S of block k+2 is computed while the elementwise warps work on block k+1.
//
// Key kernel (dK, dV, ds).  Same CTA geometry, key blocks outside and the G heads
// inside, with the products transposed so that a tensor-memory lane is a KEY:
// S^T = K Q^T, dP^T = V dO^T; the elementwise warps write p^T and dx^T (bf16)
// back into tensor memory, where they are the A operand of dV += p^T dO and
// dK += dx^T Q; ds_j is a sum along the thread's own lane.  dK and dV of a block
// collect all G heads in tensor memory and are then added to global memory once
// per (query tile, key block) with 16-byte vector reductions, by a separate
// warpgroup while the next block proceeds.
//
// Tensor memory: row kernel dQ [0, D), S0 [128, 256), S1 [256, 384), dP [384, 512);
// key kernel S^T [0, 128), dP^T [128, 256), dK [256, 256 + D), dV [384, 384 + D).
// A (row, key) element lives in the lane of its row (row kernel) or key (key
// kernel); the 128 columns of one 128 x 128 product are split between two
// elementwise warps of the same lane quarter (columns [0, 64) and [64, 128)),
// which meet at a small mbarrier before either overwrites columns the other
// still reads.
//
// Delta_i: the row kernel forms dx with <dO_i, O_i> (the forward's output, rounded for
// bf16) and, from the same p and dP, sums Delta_i = sum_j p_ij dP_ij over the kept pairs
// (the two column halves of a row add into one zeroed array); the key kernel uses that
// summed form, so its sums over
// thousands of rows (dK, ds) carry no per-row error from the rounded O.
//
// Every wait is bounded (2 s by default); a wait that runs out sets
// DMA_ERR_TIMEOUT in the device status word and the CTA winds down.
#include <cmath>

#include "dma_internal.cuh"
#include "tc_primitives.cuh"

namespace dma {
namespace {

using namespace tc;

constexpr int kBN = 128;              // keys per block
constexpr int kRowsPerTile = kQTile;  // 128 query rows per tile
constexpr int kIdxStages = 4;         // depth of the key-metadata ring
constexpr int kEwWarps = 8;           // elementwise warps: 4 lane quarters x 2 column halves
constexpr int kCopyThreads = 64;
constexpr int kCopyChunks = 4;
constexpr float kLog2e = 1.4426950408889634f;

// ---- packed pairs of fp32 ----------------------------------------------------
struct f2 {
    uint64_t v;
};
__device__ __forceinline__ f2 mk2(float a, float b)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void split2(f2 a, float& x, float& y)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(a.v));
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b)
{
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
// 16 bytes added to global memory (fp32 x 4), without a return value.
__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ int fresh_ctaid()
{
    int v;
    asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(v));
    return v;
}

// ---- the CTA's work unit ------------------------------------------------------
// (batch, KV head) segment, query tile, and the tile's key list: gathered keys, then the window
// band.  Each role recomputes it from a block index read afresh, so that none of it stays live
// across role branches.
struct Geom {
    int b, h, seg, q0, q1, W, n_g, band_lo, n_all, nblk;
    const int32_t* gl;
    __device__ __forceinline__ int key_at(int u, int S, int* status) const
    {
        int j = -1;
        if (u < n_g) {
            j = gl[u];
            if (j < 0 || j >= S) {
                set_status(status, DMA_ERR_DEVICE_CHECK);
                j = -1;
            }
        } else if (u < n_all) {
            j = band_lo + (u - n_g);
        }
        return j;
    }
};

__device__ __forceinline__ Geom tile_geom(const BwdArgs& a, int unit)
{
    Geom g;
    const int nseg = a.B * a.Hkv;
    const int tile = a.n_qt - 1 - unit / nseg;  // longest tiles first
    g.seg = unit % nseg;
    g.b = g.seg / a.Hkv;
    g.h = g.seg % a.Hkv;
    g.q0 = tile * kRowsPerTile;
    g.q1 = min(a.S, g.q0 + kRowsPerTile) - 1;
    g.W = a.window;
    g.n_g = min(max(a.tile_cnt[(int64_t)g.seg * a.n_qt + tile], 0), a.tile_stride);
    g.gl = a.tile_idx + ((int64_t)g.seg * a.n_qt + tile) * a.tile_stride;
    g.band_lo = g.W > 0 ? max(0, g.q0 - g.W + 1) : g.q1 + 1;
    const int n_b = g.W > 0 ? g.q1 + 1 - g.band_lo : 0;
    g.n_all = g.n_g + n_b;
    g.nblk = (g.n_all + kBN - 1) / kBN;
    return g;
}

// Key-metadata ring slot: j[128] (key index, -1 past the end), bias[128] f32 (score in log2
// units, -inf past the end), jm[128] (window start), lo[128], tl[128] (top interval
// [lo, lo + tl)), then the flag "every row of the tile keeps every key of the block".
constexpr int kIdxSlot = 5 * kBN * 4 + 16;

// The metadata warp: fills slot t % kStages for steps t = 0 .. nt-1, where step t walks key
// block t % nblk.  `empty_base` / `full_base`: the ring's barrier slots.
template <int kStages, typename BarFn, typename WaitFn, typename SlotFn>
__device__ __forceinline__ void meta_loop(const BwdArgs& a, const Geom& g, int nt, int lane, BarFn bar,
                                          WaitFn wait_warp, SlotFn idx_slot, int full_base, int empty_base)
{
    const int q0 = g.q0, q1 = g.q1, W = g.W, nblk = g.nblk;
    const float* sc = a.scores + (int64_t)g.seg * a.S;
    const int32_t* ex = a.expiry + (int64_t)g.seg * a.S;
    int jc[4], jn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) jc[e] = g.key_at(4 * lane + e, a.S, a.status);
    for (int t = 0; t < nt; ++t) {
        const int r = t % kStages, use = t / kStages;
        if (use >= 1 && !wait_warp(empty_base + r, (use - 1) & 1)) break;
        float scv[4];
        int exv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            scv[e] = jc[e] >= 0 ? sc[jc[e]] : 0.f;
            exv[e] = jc[e] >= 0 ? ex[jc[e]] : 0;
        }
        const int kn = (t + 1) % nblk;
#pragma unroll
        for (int e = 0; e < 4; ++e) jn[e] = (t + 1 < nt) ? g.key_at(kn * kBN + 4 * lane + e, a.S, a.status) : -1;
        int* js = idx_slot(r);
        float* mb = reinterpret_cast<float*>(js + kBN);
        int* mj = js + 2 * kBN;
        int* mlo = js + 3 * kBN;
        int* mtl = js + 4 * kBN;
        bool full = true;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * lane + e, j = jc[e];
            float bias = -INFINITY;
            int jj = -(1 << 30), lo = 0, tl = 0;
            if (j >= 0) {
                bias = scv[e] * kLog2e;
                jj = j;
                lo = top_lo(j, a.block);
                tl = max(0, exv[e] - lo);
                const bool wfull = j <= q0 && j + W > q1;
                const bool tfull = lo <= q0 && lo + tl > q1;
                const bool ufull = tl > 0 && lo <= j + W && j <= q0 && max(j + W, lo + tl) > q1;
                full = full && (wfull || tfull || ufull);
            }
            js[c] = j;
            mb[c] = bias;
            mj[c] = jj;
            mlo[c] = lo;
            mtl[c] = tl;
        }
        const bool all_full = __all_sync(0xffffffffu, full);
        if (lane == 0) js[5 * kBN] = all_full ? 1 : 0;
        mbar_arrive(bar(full_base + r));
#pragma unroll
        for (int e = 0; e < 4; ++e) jc[e] = jn[e];
    }
}

// Copies 128 rows (indices js[row]; -1 = zero row) of D bf16 into the 128-byte-swizzled operand
// layout at `tile`: each of the 64 copy threads takes kCPT 16-byte chunks of every
// (64 / kTPR)-th row.
template <int D>
struct RowCopier {
    static constexpr int kCPR = D / 8;
    static constexpr int kCPT = kCopyChunks < kCPR ? kCopyChunks : kCPR;
    static constexpr int kTPR = kCPR / kCPT;
    static constexpr int kRowsPerSweep = kCopyThreads / kTPR;
    static constexpr int kSweeps = kBN / kRowsPerSweep;
    static constexpr int kHalf = kBN * 128;
    static_assert(kRowsPerSweep % 8 == 0 && kBN % kRowsPerSweep == 0, "copy sweep shape");
    int chunk0, r0;
    uint32_t ph;
    __device__ __forceinline__ explicit RowCopier(int ct) : chunk0(ct % kTPR), r0(ct / kTPR), ph((uint32_t)(ct / kTPR) & 7u) {}
    __device__ __forceinline__ uint32_t chunk_off(int i) const
    {
        const int c = chunk0 + kTPR * i;
        return (uint32_t)((c >> 3) * kHalf) + ((((uint32_t)c & 7u) ^ ph) << 4);
    }
    // gathered rows: base + js[row] * stride
    __device__ __forceinline__ void gather(uint32_t tile, const int* js, const __nv_bfloat16* base, int64_t stride) const
    {
#pragma unroll 4
        for (int m = 0; m < kSweeps; ++m) {
            const int row = r0 + kRowsPerSweep * m;
            const int j = js[row];
            const uint32_t rb = tile + row * 128;
            const __nv_bfloat16* src = base + chunk0 * 8 + (int64_t)(j >= 0 ? j : 0) * stride;
#pragma unroll
            for (int c = 0; c < kCPT; ++c) cp_async16(rb + chunk_off(c), src + 8 * kTPR * c, j >= 0);
        }
    }
    // consecutive rows first .. first + 127 (rows >= limit are zero)
    __device__ __forceinline__ void rows(uint32_t tile, int first, int limit, const __nv_bfloat16* base,
                                         int64_t stride) const
    {
#pragma unroll 4
        for (int m = 0; m < kSweeps; ++m) {
            const int row = r0 + kRowsPerSweep * m;
            const int i = first + row;
            const uint32_t rb = tile + row * 128;
            const __nv_bfloat16* src = base + chunk0 * 8 + (int64_t)min(i, limit - 1) * stride;
#pragma unroll
            for (int c = 0; c < kCPT; ++c) cp_async16(rb + chunk_off(c), src + 8 * kTPR * c, i < limit);
        }
    }
};

// Shared-memory operand descriptors (128-byte swizzle): K-major (rows x D, the reduction over D)
// and MN-major (rows are the reduction dimension, D the output columns); the k-th 16-element
// slab of the reduction is an offset added to the descriptor.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile) { return smem_desc_sw128(tile, 16, 1024); }
__device__ __forceinline__ uint32_t kmajor_step(int kk) { return (uint32_t)(((kk / 4) * (kBN * 128) + (kk % 4) * 32) >> 4); }
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile) { return smem_desc_sw128(tile, kBN * 128, 1024); }
__device__ __forceinline__ uint32_t mnmajor_step(int kk) { return (uint32_t)(kk * (2048 >> 4)); }

// =============================================================== row kernel (dQ)
// Q and dO of the pass's query head live in tensor memory as the A operand of S = Q K^T and
// dP = dO V^T, so shared memory holds only gathered K and V rows, three blocks of each in
// flight.  S and dP are single: S of the next block is computed as soon as the elementwise
// warps have read this block's S into registers; dx is written over dP once dP has been read,
// and is the A operand of dQ += dx K; the next dP follows that product.
constexpr int kDqThreads = 640;  // EW warps 0-15, MMA 16, metadata 17, copies 18-19
constexpr int kDqEwWarps = 16;   // 4 lane quarters x 4 column quarters
constexpr int kDqMma = 16, kDqMeta = 17, kDqCopy0 = 18;
constexpr int kDqStages = 3;     // K and V blocks in flight
constexpr int kDqIdxStages = 6;
// Registers per thread: 96 at launch (640 x 96 = 61,440); the control warps give registers to
// the elementwise warps: 512 * 104 + 128 * 64 = 640 * 96.
constexpr int kDqRegsEw = 104;
constexpr int kDqRegsCtl = 64;
static_assert(512 * kDqRegsEw + 128 * kDqRegsCtl <= kDqThreads * 96, "register split exceeds the launch's registers");

enum : int {
    kQBarKFull = 0,   // kDqStages
    kQBarKEmpty = 3,  // kDqStages
    kQBarVFull = 6,   // kDqStages
    kQBarVEmpty = 9,  // kDqStages
    kQBarQReady = 12, // Q and dO of the pass in tensor memory (and the previous pass's dQ read out)
    kQBarSFull = 13,
    kQBarSRead = 14,
    kQBarDPFull = 15,
    kQBarDsReady = 16,
    kQBarDQDone = 17,
    kQBarDrain = 18,
    kQBarQuad = 19,  // 4 (lane quarters)
    kQBarIdxFull = 23,
    kQBarIdxEmpty = 23 + kDqIdxStages,
    kQNumBars = 23 + 2 * kDqIdxStages
};

template <int D>
struct DqLayout {
    static constexpr int kTile = kBN * D * 2;
    static constexpr int kK = 0;
    static constexpr int kV = kDqStages * kTile;
    static constexpr int kIdx = 2 * kDqStages * kTile;
    static constexpr int kBars = kIdx + kDqIdxStages * kIdxSlot;
    static constexpr int kMisc = kBars + 8 * kQNumBars;
    static constexpr int kEnd = kMisc + 16;
    static constexpr int kSmemBytes = kEnd + 1024;
};
static_assert(DqLayout<128>::kSmemBytes <= 227 * 1024, "row kernel shared memory");

// tensor-memory columns of the row kernel
constexpr uint32_t kTmDQ = 0, kTmQ = 128, kTmDO = 192, kTmS = 256, kTmDP = 384;

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1) bwd_dq_tc_kernel(const BwdArgs a, const uint64_t wait_ns)
{
    using L = DqLayout<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    auto idx_slot = [&](int r) { return reinterpret_cast<int*>(sm + L::kIdx + r * kIdxSlot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);
    auto bar = [&](int i) { return sbase + L::kBars + 8 * i; };
    auto wait_warp = [&](int i, int parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, wait_ns));
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.H / a.Hkv;
    {
        const Geom g = tile_geom(a, blockIdx.x);
        if (g.nblk == 0) {
            // nothing kept by any row of the tile: dQ = 0
            for (int t = threadIdx.x; t < kRowsPerTile * G; t += kDqThreads) {
                const int r = t % kRowsPerTile, gq = t / kRowsPerTile, i = g.q0 + r;
                if (i > g.q1) continue;
                float4* dq = reinterpret_cast<float4*>(a.dQ + (((int64_t)g.b * a.S + i) * a.H + g.h * G + gq) * D);
                for (int c = 0; c < D / 4; ++c) dq[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            return;
        }
    }
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < kQNumBars; ++i) mbar_init(bar(i), 1);
        for (int s = 0; s < kDqStages; ++s) {
            mbar_init(bar(kQBarKFull + s), kCopyThreads);
            mbar_init(bar(kQBarVFull + s), kCopyThreads);
        }
        mbar_init(bar(kQBarQReady), 32 * kDqEwWarps);
        mbar_init(bar(kQBarSRead), 32 * kDqEwWarps);
        mbar_init(bar(kQBarDsReady), 32 * kDqEwWarps);
        for (int q = 0; q < 4; ++q) mbar_init(bar(kQBarQuad + q), 4);
        for (int r = 0; r < kDqIdxStages; ++r) {
            mbar_init(bar(kQBarIdxFull + r), 32);
            mbar_init(bar(kQBarIdxEmpty + r), kDqEwWarps + 2);  // EW warps and the two copy warps
        }
        mbar_init_fence();
    }
    if (warp == kDqMma) tmem_alloc<512>(smem_u32(tmem_slot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kDqMeta) {
        regs_decrease<kDqRegsCtl>();
        const Geom g = tile_geom(a, fresh_ctaid());
        meta_loop<kDqIdxStages>(a, g, G * g.nblk, lane, bar, wait_warp, idx_slot, kQBarIdxFull, kQBarIdxEmpty);
    } else if (warp >= kDqCopy0) {
        regs_decrease<kDqRegsCtl>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int n = G * g.nblk;
        const RowCopier<D> cp(threadIdx.x - kDqCopy0 * 32);
        const int64_t kv_stride = (int64_t)a.Hkv * D;
        const __nv_bfloat16* Kh = static_cast<const __nv_bfloat16*>(a.K) + ((int64_t)g.b * a.S * a.Hkv + g.h) * D;
        const __nv_bfloat16* Vh = static_cast<const __nv_bfloat16*>(a.V) + ((int64_t)g.b * a.S * a.Hkv + g.h) * D;
        bool ok = true;
        for (int u = 0; u < n && ok; ++u) {
            const int r = u % kDqIdxStages, st = u % kDqStages, use = u / kDqStages;
            if (!(ok = wait_warp(kQBarIdxFull + r, (u / kDqIdxStages) & 1))) break;
            if (use >= 1 && !(ok = wait_warp(kQBarKEmpty + st, (use - 1) & 1))) break;
            cp.gather(sbase + L::kK + st * L::kTile, idx_slot(r), Kh, kv_stride);
            cp_async_arrive(bar(kQBarKFull + st));
            if (use >= 1 && !(ok = wait_warp(kQBarVEmpty + st, (use - 1) & 1))) break;
            cp.gather(sbase + L::kV + st * L::kTile, idx_slot(r), Vh, kv_stride);
            cp_async_arrive(bar(kQBarVFull + st));
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kQBarIdxEmpty + r));
        }
        cp_async_wait_all();
    } else if (warp == kDqMma) {
        regs_decrease<kDqRegsCtl>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk;
        const uint32_t tm = *tmem_slot;
        const bool leader = lane == 0;
        constexpr uint32_t idS = idesc_bf16_f32(128, kBN, false);
        constexpr uint32_t idQ = idesc_bf16_f32(128, D, true);
        auto commit = [&](int barid) {
            if (leader) mma_commit(bar(barid));
        };
        // S(u) = Q K(u)^T and dP(u) = dO V(u)^T: A from tensor memory, B K-major in shared memory
        auto start_s = [&](int u) -> bool {
            const int st = u % kDqStages;
            if (!wait_warp(kQBarKFull + st, (u / kDqStages) & 1)) return false;
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t dk = kmajor_desc(sbase + L::kK + st * L::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                if (leader) mma_ts(tm + kTmS, tm + kTmQ + kk * 8, dk + kmajor_step(kk), idS, kk > 0);
            commit(kQBarSFull);
            return true;
        };
        auto start_dp = [&](int u) -> bool {
            const int st = u % kDqStages;
            if (!wait_warp(kQBarVFull + st, (u / kDqStages) & 1)) return false;
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t dv = kmajor_desc(sbase + L::kV + st * L::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                if (leader) mma_ts(tm + kTmDP, tm + kTmDO + kk * 8, dv + kmajor_step(kk), idS, kk > 0);
            commit(kQBarDPFull);
            commit(kQBarVEmpty + st);
            return true;
        };
        bool ok = true;
        for (int gq = 0; gq < G && ok; ++gq) {
            const int u0 = gq * nblk;
            // this pass's Q and dO are in tensor memory (the previous pass's dQ has been read out)
            if (!(ok = wait_warp(kQBarQReady, gq & 1))) break;
            tc_fence_after();
            if (!(ok = start_s(u0) && start_dp(u0))) break;
            for (int k = 0; k < nblk; ++k) {
                const int u = u0 + k;
                if (k + 1 < nblk) {
                    // the next S as soon as this one has been read
                    if (!(ok = wait_warp(kQBarSRead, u & 1))) break;
                    if (!(ok = start_s(u + 1))) break;
                }
                if (!(ok = wait_warp(kQBarDsReady, u & 1))) break;
                tc_fence_after();
                const uint64_t dk = mnmajor_desc(sbase + L::kK + (u % kDqStages) * L::kTile);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    if (leader)
                        mma_ts(tm + kTmDQ, tm + kTmDP + kk * 8, dk + mnmajor_step(kk), idQ, (k == 0 && kk == 0) ? 0u : 1u);
                commit(kQBarKEmpty + u % kDqStages);
                if (k + 1 < nblk && !(ok = start_dp(u + 1))) break;
            }
            if (!ok) break;
            commit(kQBarDQDone);
        }
        commit(kQBarDrain);
        if (leader) mbar_wait_drain(bar(kQBarDrain), 0, wait_ns);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise
        // Thread = query row r (tensor-memory lane) and key columns [32 cq, 32 cq + 32) of a block.
        regs_increase<kDqRegsEw>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk, q0 = g.q0, W = g.W;
        const uint32_t tm = *tmem_slot;
        const int quarter = warp & 3, cq = warp >> 2;
        const int r = quarter * 32 + lane, i = q0 + r;
        const bool valid = i < a.S;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const f2 cc2 = mk2(a.scale * kLog2e, a.scale * kLog2e);
        constexpr int kQC = D / 8;  // packed Q (and dO) columns of this thread: D / 4 elements
        bool ok = true;
        for (int gq = 0; gq < G && ok; ++gq) {
            const int hq = g.h * G + gq;
            // Q and dO of the pass into tensor memory (bf16 pairs, the A operand layout)
            {
                const int64_t qo = (((int64_t)g.b * a.S + min(i, a.S - 1)) * a.H + hq) * D + cq * (D / 4);
                const uint4* qs = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.Q) + qo);
                const uint4* gs = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dO) + qo);
                uint32_t qv[kQC], gv[kQC];
#pragma unroll
                for (int c = 0; c < kQC / 4; ++c) {
                    const uint4 x = valid ? __ldg(qs + c) : make_uint4(0, 0, 0, 0);
                    const uint4 y = valid ? __ldg(gs + c) : make_uint4(0, 0, 0, 0);
                    qv[4 * c] = x.x; qv[4 * c + 1] = x.y; qv[4 * c + 2] = x.z; qv[4 * c + 3] = x.w;
                    gv[4 * c] = y.x; gv[4 * c + 1] = y.y; gv[4 * c + 2] = y.z; gv[4 * c + 3] = y.w;
                }
                if constexpr (kQC == 16) {
                    tmem_st16(tm + kTmQ + lane_off + cq * kQC, qv);
                    tmem_st16(tm + kTmDO + lane_off + cq * kQC, gv);
                } else {
                    tmem_st8(tm + kTmQ + lane_off + cq * kQC, qv);
                    tmem_st8(tm + kTmDO + lane_off + cq * kQC, gv);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kQBarQReady));
            }
            const int64_t rs = ((int64_t)g.b * a.H + hq) * a.S + i;
            float lse_l2 = valid ? a.lse[rs] * kLog2e : INFINITY;
            if (lse_l2 == -INFINITY) lse_l2 = INFINITY;  // a row that keeps nothing contributes nothing
            const float dl = valid ? a.delta[rs] : 0.f;
            const f2 nl2 = mk2(-lse_l2, -lse_l2), dl2 = mk2(dl, dl);
            f2 dsum2 = mk2(0.f, 0.f);  // sum of p dP over this thread's keys: the summed form of Delta
            for (int k = 0; k < nblk; ++k) {
                const int u = gq * nblk + k, ridx = u % kDqIdxStages;
                ok = wait_warp(kQBarIdxFull + ridx, (u / kDqIdxStages) & 1) && wait_warp(kQBarSFull, u & 1);
                if (!ok) break;
                tc_fence_after();
                const int* js = idx_slot(ridx);
                const float* mb = reinterpret_cast<const float*>(js + kBN) + 32 * cq;
                const int* mj = js + 2 * kBN + 32 * cq;
                const int* mlo = js + 3 * kBN + 32 * cq;
                const int* mtl = js + 4 * kBN + 32 * cq;
                const bool all_full = js[5 * kBN] != 0;
                float p[32];
                tmem_ld32f(tm + kTmS + lane_off + 32 * cq, p);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(bar(kQBarSRead));
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 bb = *reinterpret_cast<const float4*>(mb + c);
                    f2 x01 = add2(fma2(mk2(p[c], p[c + 1]), cc2, mk2(bb.x, bb.y)), nl2);
                    f2 x23 = add2(fma2(mk2(p[c + 2], p[c + 3]), cc2, mk2(bb.z, bb.w)), nl2);
                    float x0, x1, x2, x3;
                    split2(x01, x0, x1);
                    split2(x23, x2, x3);
                    p[c] = ex2(x0);
                    p[c + 1] = ex2(x1);
                    p[c + 2] = ex2(x2);
                    p[c + 3] = ex2(x3);
                    if (!all_full) {
                        // kept iff j <= i < j + window  or  lo_j <= i < expiry_j
                        const int4 jj = *reinterpret_cast<const int4*>(mj + c);
                        const int4 lo = *reinterpret_cast<const int4*>(mlo + c);
                        const int4 tl = *reinterpret_cast<const int4*>(mtl + c);
                        if (!((unsigned)(i - jj.x) < (unsigned)W || (unsigned)(i - lo.x) < (unsigned)tl.x)) p[c] = 0.f;
                        if (!((unsigned)(i - jj.y) < (unsigned)W || (unsigned)(i - lo.y) < (unsigned)tl.y)) p[c + 1] = 0.f;
                        if (!((unsigned)(i - jj.z) < (unsigned)W || (unsigned)(i - lo.z) < (unsigned)tl.z)) p[c + 2] = 0.f;
                        if (!((unsigned)(i - jj.w) < (unsigned)W || (unsigned)(i - lo.w) < (unsigned)tl.w)) p[c + 3] = 0.f;
                    }
                }
                if (!(ok = wait_warp(kQBarDPFull, u & 1))) break;
                tc_fence_after();
                float dp[32];
                tmem_ld32f(tm + kTmDP + lane_off + 32 * cq, dp);
                tmem_ld_wait();
                // the four column quarters of this lane quarter have read dP before any writes dx
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kQBarQuad + quarter));
                if (!(ok = wait_warp(kQBarQuad + quarter, u & 1))) break;
                tc_fence_after();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const f2 p2 = mk2(p[e], p[e + 1]), dp2 = mk2(dp[e], dp[e + 1]);
                    dsum2 = fma2(p2, dp2, dsum2);
                    float d0, d1;
                    split2(mul2(p2, sub2(dp2, dl2)), d0, d1);
                    pk[e / 2] = pack_bf16(d0, d1);
                }
                tmem_st16(tm + kTmDP + lane_off + 16 * cq, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kQBarDsReady));
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kQBarIdxEmpty + ridx));
            }
            if (!ok) break;
            if (valid) {
                float d0, d1;
                split2(dsum2, d0, d1);
                atomicAdd(a.delta_x + rs, d0 + d1);  // the four column quarters of the row
            }
            // the pass's dQ: scale * accumulator, fp32
            if (!(ok = wait_warp(kQBarDQDone, gq & 1))) break;
            tc_fence_after();
            float* dq = a.dQ + (((int64_t)g.b * a.S + min(i, a.S - 1)) * a.H + hq) * D + cq * (D / 4);
            if constexpr (D == 128) {
                float v[32];
                tmem_ld32f(tm + kTmDQ + lane_off + cq * 32, v);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dq + e) =
                            make_float4(a.scale * v[e], a.scale * v[e + 1], a.scale * v[e + 2], a.scale * v[e + 3]);
                }
            } else {
                uint32_t v[16];
                tmem_ld16(tm + kTmDQ + lane_off + cq * 16, v);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4*>(dq + e) =
                            make_float4(a.scale * __uint_as_float(v[e]), a.scale * __uint_as_float(v[e + 1]),
                                        a.scale * __uint_as_float(v[e + 2]), a.scale * __uint_as_float(v[e + 3]));
                }
            }
            tc_fence_before();
        }
    }

    if (threadIdx.x == 0 && *abort_flag) set_status(a.status, DMA_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kDqMma) tmem_dealloc<512>(*tmem_slot);
}

// =============================================================== key kernel (dK, dV, ds)
constexpr int kDkvThreads = 512;  // EW warps 0-7, flush 8-11, MMA 12, metadata 13, copies 14-15
constexpr int kKvFlush0 = 8, kKvMma = 12, kKvMeta = 13, kKvCopy0 = 14;
constexpr int kRegsEw = 168;
constexpr int kRegsOther = 88;
static_assert(8 * 32 * kRegsEw + 8 * 32 * kRegsOther <= kDkvThreads * 128, "register split exceeds the launch's registers");

enum : int {
    kKBarKVFull = 0,
    kKBarKVEmpty = 1,
    kKBarQFull = 2,   // 2 stages
    kKBarQEmpty = 4,  // 2 stages
    kKBarSFull = 6,
    kKBarSRead = 7,
    kKBarDPFull = 8,
    kKBarPdsReady = 9,
    kKBarKVDone = 10,
    kKBarKVFree = 11,
    kKBarDrain = 12,
    kKBarPair = 13,  // 4
    kKBarIdxFull = 17,
    kKBarIdxEmpty = 17 + kIdxStages,
    kKNumBars = 17 + 2 * kIdxStages
};

template <int D>
struct DkvLayout {
    static constexpr int kTile = kBN * D * 2;
    static constexpr int kK = 0;
    static constexpr int kV = kTile;
    static constexpr int kQ = 2 * kTile;       // 2 stages
    static constexpr int kdO = 4 * kTile;      // 2 stages
    static constexpr int kRows = 6 * kTile;    // [stage][lse 128 | Delta 128] f32
    static constexpr int kRowsStage = 2 * kRowsPerTile * 4;
    static constexpr int kIdx = kRows + 2 * kRowsStage;
    static constexpr int kXpose = kIdx + kIdxStages * kIdxSlot;  // per flush warp: 32 rows x 32 f32
    static constexpr int kBars = kXpose + 4 * 32 * 32 * 4;
    static constexpr int kMisc = kBars + 8 * kKNumBars;
    static constexpr int kEnd = kMisc + 16;
    static constexpr int kSmemBytes = kEnd + 1024;
};
static_assert(DkvLayout<128>::kSmemBytes <= 227 * 1024, "key kernel shared memory");

// bits [lo, hi) of a 64-bit mask, both clipped to [0, 64]
__device__ __forceinline__ uint64_t range_mask(int lo, int hi)
{
    lo = max(lo, 0);
    hi = min(hi, 64);
    if (hi <= lo) return 0ull;
    const uint64_t upto_hi = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
    return upto_hi & ~((1ull << lo) - 1ull);
}

template <int D>
__global__ void __launch_bounds__(kDkvThreads, 1) bwd_dkv_tc_kernel(const BwdArgs a, const uint64_t wait_ns)
{
    using L = DkvLayout<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    auto idx_slot = [&](int r) { return reinterpret_cast<int*>(sm + L::kIdx + r * kIdxSlot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);
    auto bar = [&](int i) { return sbase + L::kBars + 8 * i; };
    auto wait_warp = [&](int i, int parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, wait_ns));
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.H / a.Hkv;
    {
        const Geom g = tile_geom(a, blockIdx.x);
        if (g.nblk == 0) return;  // nothing kept by the tile: no gradient to add
    }
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < kKNumBars; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(kKBarKVFull), kCopyThreads);
        for (int s = 0; s < 2; ++s) mbar_init(bar(kKBarQFull + s), kCopyThreads);
        mbar_init(bar(kKBarSRead), 32 * kEwWarps);
        mbar_init(bar(kKBarPdsReady), 32 * kEwWarps);
        mbar_init(bar(kKBarKVFree), 128);
        for (int q = 0; q < 4; ++q) mbar_init(bar(kKBarPair + q), 2);
        for (int r = 0; r < kIdxStages; ++r) {
            mbar_init(bar(kKBarIdxFull + r), 32);
            mbar_init(bar(kKBarIdxEmpty + r), kEwWarps + 4 + 2);  // EW, flush and copy warps
        }
        mbar_init_fence();
    }
    if (warp == kKvMma) tmem_alloc<512>(smem_u32(tmem_slot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kKvMeta) {
        regs_decrease<kRegsOther>();
        const Geom g = tile_geom(a, fresh_ctaid());
        meta_loop<kIdxStages>(a, g, g.nblk, lane, bar, wait_warp, idx_slot, kKBarIdxFull, kKBarIdxEmpty);
    } else if (warp >= kKvCopy0) {
        regs_decrease<kRegsOther>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk;
        const int ct = threadIdx.x - kKvCopy0 * 32;
        const RowCopier<D> cp(ct);
        const int64_t kv_stride = (int64_t)a.Hkv * D;
        const __nv_bfloat16* Kh = static_cast<const __nv_bfloat16*>(a.K) + ((int64_t)g.b * a.S * a.Hkv + g.h) * D;
        const __nv_bfloat16* Vh = static_cast<const __nv_bfloat16*>(a.V) + ((int64_t)g.b * a.S * a.Hkv + g.h) * D;
        const int64_t q_stride = (int64_t)a.H * D;
        bool ok = true;
        for (int k = 0; k < nblk && ok; ++k) {
            const int r = k % kIdxStages;
            if (!(ok = wait_warp(kKBarIdxFull + r, (k / kIdxStages) & 1))) break;
            if (k > 0 && !(ok = wait_warp(kKBarKVEmpty, (k - 1) & 1))) break;
            cp.gather(sbase + L::kK, idx_slot(r), Kh, kv_stride);
            cp.gather(sbase + L::kV, idx_slot(r), Vh, kv_stride);
            cp_async_arrive(bar(kKBarKVFull));
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kKBarIdxEmpty + r));
            for (int gq = 0; gq < G; ++gq) {
                const int u = k * G + gq, s = u & 1;
                if (u >= 2 && !(ok = wait_warp(kKBarQEmpty + s, ((u >> 1) - 1) & 1))) break;
                const int hq = g.h * G + gq;
                const int64_t off = ((int64_t)g.b * a.S * a.H + hq) * D;
                cp.rows(sbase + L::kQ + s * L::kTile, g.q0, a.S, static_cast<const __nv_bfloat16*>(a.Q) + off, q_stride);
                cp.rows(sbase + L::kdO + s * L::kTile, g.q0, a.S, static_cast<const __nv_bfloat16*>(a.dO) + off, q_stride);
                // lse and the summed Delta of the tile's rows (zero past the end: those columns are
                // masked)
                const int64_t rs = ((int64_t)g.b * a.H + hq) * a.S;
                const uint32_t rows_s = sbase + L::kRows + s * L::kRowsStage;
                for (int t = ct; t < 2 * kRowsPerTile; t += kCopyThreads) {
                    const int row = t % kRowsPerTile, i = g.q0 + row;
                    const float* src = (t < kRowsPerTile ? a.lse : a.delta_x) + rs + min(i, a.S - 1);
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(rows_s + 4 * t), "l"(src),
                                 "r"(i < a.S ? 4 : 0)
                                 : "memory");
                }
                cp_async_arrive(bar(kKBarQFull + s));
            }
        }
        cp_async_wait_all();
    } else if (warp == kKvMma) {
        regs_decrease<kRegsOther>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk, n = nblk * G;
        const uint32_t tm = *tmem_slot;
        const uint32_t tS = tm, tDP = tm + 128, tDK = tm + 256, tDV = tm + 384;
        const bool leader = lane == 0;
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, false);
        constexpr uint32_t idD = idesc_bf16_f32(128, D, true);
        auto commit = [&](int barid) {
            if (leader) mma_commit(bar(barid));
        };
        auto issue_s = [&](int u) {  // S^T = K Q^T
            const uint64_t dk = kmajor_desc(sbase + L::kK);
            const uint64_t dq = kmajor_desc(sbase + L::kQ + (u & 1) * L::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                if (leader) mma_ss(tS, dk + kmajor_step(kk), dq + kmajor_step(kk), idS, kk > 0);
        };
        auto issue_dp = [&](int u) {  // dP^T = V dO^T
            const uint64_t dv = kmajor_desc(sbase + L::kV);
            const uint64_t dg = kmajor_desc(sbase + L::kdO + (u & 1) * L::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                if (leader) mma_ss(tDP, dv + kmajor_step(kk), dg + kmajor_step(kk), idS, kk > 0);
        };
        auto issue_dvdk = [&](int u, bool first) {  // dV += p^T dO, dK += dx^T Q
            const uint64_t dg = mnmajor_desc(sbase + L::kdO + (u & 1) * L::kTile);
            const uint64_t dq = mnmajor_desc(sbase + L::kQ + (u & 1) * L::kTile);
#pragma unroll
            for (int kk = 0; kk < kRowsPerTile / 16; ++kk)
                if (leader) mma_ts(tDV, tDP + kk * 8, dg + mnmajor_step(kk), idD, (first && kk == 0) ? 0u : 1u);
#pragma unroll
            for (int kk = 0; kk < kRowsPerTile / 16; ++kk)
                if (leader) mma_ts(tDK, tDP + 64 + kk * 8, dq + mnmajor_step(kk), idD, (first && kk == 0) ? 0u : 1u);
        };
        auto operands = [&]() {
            fence_proxy_async_smem();
            tc_fence_after();
        };
        bool ok = wait_warp(kKBarKVFull, 0) && wait_warp(kKBarQFull + 0, 0);
        if (ok) {
            operands();
            issue_s(0);
            commit(kKBarSFull);
            issue_dp(0);
            commit(kKBarDPFull);
            if (G == 1) commit(kKBarKVEmpty);  // block 0's K and V have no further reader
        }
        for (int u = 0; u < n && ok; ++u) {
            const int k = u / G, gq = u % G;
            if (gq < G - 1) {
                // the next head of this block: its S^T as soon as this head's S^T has been read
                ok = wait_warp(kKBarSRead, u & 1) && wait_warp(kKBarQFull + ((u + 1) & 1), ((u + 1) >> 1) & 1);
                if (!ok) break;
                operands();
                issue_s(u + 1);
                commit(kKBarSFull);
                if (!(ok = wait_warp(kKBarPdsReady, u & 1))) break;
                if (gq == 0 && k > 0 && !(ok = wait_warp(kKBarKVFree, (k - 1) & 1))) break;
                tc_fence_after();
                issue_dvdk(u, gq == 0);
                commit(kKBarQEmpty + (u & 1));
                issue_dp(u + 1);
                commit(kKBarDPFull);
                if (gq + 1 == G - 1) commit(kKBarKVEmpty);  // the block's last S^T and dP^T are issued
            } else {
                if (!(ok = wait_warp(kKBarPdsReady, u & 1))) break;
                if (gq == 0 && k > 0 && !(ok = wait_warp(kKBarKVFree, (k - 1) & 1))) break;
                tc_fence_after();
                issue_dvdk(u, gq == 0);
                commit(kKBarQEmpty + (u & 1));
                commit(kKBarKVDone);
                if (u + 1 < n) {
                    ok = wait_warp(kKBarKVFull, (k + 1) & 1) && wait_warp(kKBarQFull + ((u + 1) & 1), ((u + 1) >> 1) & 1);
                    if (!ok) break;
                    operands();
                    issue_s(u + 1);
                    commit(kKBarSFull);
                    issue_dp(u + 1);
                    commit(kKBarDPFull);
                    if (G == 1) commit(kKBarKVEmpty);
                }
            }
        }
        commit(kKBarDrain);
        if (leader) mbar_wait_drain(bar(kKBarDrain), 0, wait_ns);
        __syncwarp();
    } else if (warp >= kKvFlush0) {
        // ------------------------------------------------------------------ flush
        // Thread = key lane r: the block's dK (times scale) and dV rows added to global memory.
        // Each 32-column chunk of the warp's 32 rows is turned around in shared memory so that one
        // 16-byte reduction instruction covers four rows x 128 contiguous bytes (4 L2 requests,
        // against 32 when every lane adds to its own row).
        regs_decrease<kRegsOther>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk;
        const uint32_t tm = *tmem_slot;
        const int quarter = warp & 3, r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sc = a.scale;
        // [row][8 groups of 4 f32], group q of row x stored at position q ^ (x & 7)
        float* xb = reinterpret_cast<float*>(sm + L::kXpose) + (warp - kKvFlush0) * 32 * 32;
        const int64_t seg_row0 = (int64_t)g.b * a.S * a.Hkv + g.h;  // row (b, j, h) = seg_row0 + j * Hkv
        auto put_row = [&](const float* v, float mul) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(xb + lane * 32 + ((q ^ (lane & 7)) * 4)) =
                    make_float4(mul * v[4 * q], mul * v[4 * q + 1], mul * v[4 * q + 2], mul * v[4 * q + 3]);
            __syncwarp();
        };
        auto add_rows = [&](float* out, int c, int j) {
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int x = 4 * it + (lane >> 3), q = lane & 7;
                const int jx = __shfl_sync(0xffffffffu, j, x);
                const float4 w = *reinterpret_cast<const float4*>(xb + x * 32 + ((q ^ (x & 7)) * 4));
                if (jx >= 0) red_add4(out + (seg_row0 + (int64_t)jx * a.Hkv) * D + c + 4 * q, w.x, w.y, w.z, w.w);
            }
            __syncwarp();
        };
        bool ok = true;
        for (int k = 0; k < nblk && ok; ++k) {
            const int ridx = k % kIdxStages;
            if (!(ok = wait_warp(kKBarIdxFull + ridx, (k / kIdxStages) & 1))) break;
            const int j = idx_slot(ridx)[r];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kKBarIdxEmpty + ridx));
            if (!(ok = wait_warp(kKBarKVDone, k & 1))) break;
            tc_fence_after();
            // dK chunks (tensor-memory columns 256..), then dV chunks (384..); the MMA may overwrite
            // both accumulators once the last chunk is in registers
#pragma unroll 1
            for (int t = 0; t < 2 * (D / 32); ++t) {
                const int c = (t % (D / 32)) * 32;
                const bool is_v = t >= D / 32;
                float v[32];
                tmem_ld32f(tm + (is_v ? 384 : 256) + lane_off + c, v);
                tmem_ld_wait();
                if (t == 2 * (D / 32) - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(kKBarKVFree));
                }
                put_row(v, is_v ? 1.f : sc);
                add_rows(is_v ? a.dV : a.dK, c, j);
            }
        }
    } else {
        // ------------------------------------------------------------ elementwise
        // Thread = key lane r of the block; query-row columns [64 hh, 64 hh + 64) of the tile.
        regs_increase<kRegsEw>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk, q0 = g.q0, W = min(g.W, a.S);
        const int nrows = g.q1 - q0 + 1;
        const uint32_t tm = *tmem_slot;
        const int quarter = warp & 3, hh = warp >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float c_log2 = a.scale * kLog2e;
        const f2 ml2 = mk2(-kLog2e, -kLog2e);
        bool ok = true;
        for (int k = 0; k < nblk && ok; ++k) {
            const int ridx = k % kIdxStages;
            if (!(ok = wait_warp(kKBarIdxFull + ridx, (k / kIdxStages) & 1))) break;
            const int* js = idx_slot(ridx);
            const int j = js[r];
            const float bias = reinterpret_cast<const float*>(js + kBN)[r];
            const int lo = js[3 * kBN + r], tl = js[4 * kBN + r];
            const bool all_full = js[5 * kBN] != 0;
            // the columns (rows q0 + c) of this half that keep key j
            const int c0 = q0 + 64 * hh;
            uint64_t keep = range_mask(0, nrows - 64 * hh);
            if (j < 0)
                keep = 0ull;
            else if (!all_full)
                keep &= range_mask(j - c0, j + W - c0) | range_mask(lo - c0, lo + tl - c0);
            const f2 bias2 = mk2(bias, bias), cc2 = mk2(c_log2, c_log2);
            float dsa = 0.f;
            for (int gq = 0; gq < G; ++gq) {
                const int u = k * G + gq;
                ok = wait_warp(kKBarQFull + (u & 1), (u >> 1) & 1) && wait_warp(kKBarSFull, u & 1);
                if (!ok) break;
                tc_fence_after();
                const float* lse_s = reinterpret_cast<const float*>(sm + L::kRows + (u & 1) * L::kRowsStage) + 64 * hh;
                const float* dl_s = lse_s + kRowsPerTile;
                float p[64];
                tmem_ld32f(tm + lane_off + 64 * hh, p);
                tmem_ld32f(tm + lane_off + 64 * hh + 32, p + 32);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(bar(kKBarSRead));
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 ls = *reinterpret_cast<const float4*>(lse_s + c);
                    f2 x01 = fma2(mk2(ls.x, ls.y), ml2, fma2(mk2(p[c], p[c + 1]), cc2, bias2));
                    f2 x23 = fma2(mk2(ls.z, ls.w), ml2, fma2(mk2(p[c + 2], p[c + 3]), cc2, bias2));
                    float x0, x1, x2, x3;
                    split2(x01, x0, x1);
                    split2(x23, x2, x3);
                    p[c] = ((keep >> c) & 1ull) ? ex2(x0) : 0.f;
                    p[c + 1] = ((keep >> (c + 1)) & 1ull) ? ex2(x1) : 0.f;
                    p[c + 2] = ((keep >> (c + 2)) & 1ull) ? ex2(x2) : 0.f;
                    p[c + 3] = ((keep >> (c + 3)) & 1ull) ? ex2(x3) : 0.f;
                }
                if (!(ok = wait_warp(kKBarDPFull, u & 1))) break;
                tc_fence_after();
                float dp[64];
                tmem_ld32f(tm + 128 + lane_off + 64 * hh, dp);
                tmem_ld32f(tm + 128 + lane_off + 64 * hh + 32, dp + 32);
                tmem_ld_wait();
                // both column halves of this lane quarter have read dP^T before either writes
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kKBarPair + quarter));
                if (!(ok = wait_warp(kKBarPair + quarter, u & 1))) break;
                tc_fence_after();
                uint32_t pp[32], pd[32];
                f2 acc = mk2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float2 dl = *reinterpret_cast<const float2*>(dl_s + c);
                    const f2 d = mul2(mk2(p[c], p[c + 1]), sub2(mk2(dp[c], dp[c + 1]), mk2(dl.x, dl.y)));
                    acc = add2(acc, d);
                    float d0, d1;
                    split2(d, d0, d1);
                    pp[c / 2] = pack_bf16(p[c], p[c + 1]);
                    pd[c / 2] = pack_bf16(d0, d1);
                }
                {
                    float a0, a1;
                    split2(acc, a0, a1);
                    dsa += a0 + a1;
                }
                tmem_st32(tm + 128 + lane_off + 32 * hh, pp);
                tmem_st32(tm + 128 + lane_off + 64 + 32 * hh, pd);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kKBarPdsReady));
            }
            if (!ok) break;
            if (j >= 0 && dsa != 0.f) atomicAdd(a.ds + (int64_t)g.seg * a.S + j, dsa);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kKBarIdxEmpty + ridx));
        }
    }

    if (threadIdx.x == 0 && *abort_flag) set_status(a.status, DMA_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kKvMma) tmem_dealloc<512>(*tmem_slot);
}

template <int D>
cudaError_t launch_typed(const BwdArgs& a, uint64_t wait_ns, cudaStream_t st)
{
    const int64_t grid = (int64_t)a.n_qt * a.B * a.Hkv;
    int smem = DqLayout<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    bwd_dq_tc_kernel<D><<<(unsigned)grid, kDqThreads, smem, st>>>(a, wait_ns);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    smem = DkvLayout<D>::kSmemBytes;
    e = cudaFuncSetAttribute(bwd_dkv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    bwd_dkv_tc_kernel<D><<<(unsigned)grid, kDkvThreads, smem, st>>>(a, wait_ns);
    return cudaGetLastError();
}

}  // namespace

bool bwd_tc_supported(dma_dtype_t dt, int D) { return dt == DMA_BF16 && (D == 64 || D == 128); }

cudaError_t launch_bwd_tc(const BwdArgs& a, int D, uint64_t wait_ns, cudaStream_t st)
{
    return D == 128 ? launch_typed<128>(a, wait_ns, st) : launch_typed<64>(a, wait_ns, st);
}

}  // namespace dma
