// Sparse attention prefill on the 5th-generation tensor cores (bf16, D = 64 or
// 128): tcgen05 MMAs with fp32 accumulators in tensor memory, kept K/V rows
// gathered into shared memory by TMA (tile::gather4).
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §四/§五: masked positions are
// skipped outright -- no query-key product is formed for them -- and since their
// weight would be exactly 0 the result equals the full masked softmax.  For the
// query tile [q0, q1] of 128 rows the only keys touched are the tile's gathered
// list (keys outside the window band whose top-set interval meets the tile) and
// the window band (q0 - window, q1].  Key j is kept by row i iff
//     j <= i < j + window   or   lo_j <= i < expiry_j,
// and the kept logit is scale * <Q_i, K_j> + s_j.
//
// One CTA = one (batch, KV head, query tile); it serves all G = H / Hkv query
// heads of the KV head, two at a time (two "M-tiles" of 128 rows), so each
// gathered K/V block is fetched once per pair of query heads.  Roles:
//   warps 0-3 / 4-7  softmax of M-tile A / B: thread = one query row (= one
//                    tensor-memory lane); S from tensor memory, masked online
//                    softmax in the log2 domain, P (bf16) written back over S
//   warp 8           MMA issue (one thread): S = Q K^T (both operands in shared
//                    memory), O += P V (P from tensor memory, V in shared memory)
//   warp 9           producer: Q tiles, K and V blocks of 128 gathered rows
//                    (4 rows per gather4 per lane), per-key bias and mask data
//   warps 10-11      idle (they complete the third warpgroup, which hands its
//                    registers to the softmax warpgroups)
// Tensor memory (512 columns): O_A, O_B at columns 0 and 128; S_A, S_B at 256
// and 384.  The MMA order S_A(k+1) after PV_A(k), then PV_B(k), S_B(k+1) lets
// one softmax warpgroup work while the tensor core serves the other.
//
// Exponents are always taken against the exact running maximum of the row, so
// the largest weight seen so far is exactly 1.0 in bf16.  (Keeping an older
// maximum until it is exceeded by a wide margin would save rescaling O in
// tensor memory, but then the dominant weight of a peaked row is 2^f with a
// fractional f, and its bf16 rounding alone moves O by up to 2^-9 |V|.)
// Every wait is bounded (2 s); a wait that runs out sets DMA_ERR_TIMEOUT in the
// device status word and the CTA winds down without further work.
#include <cmath>

#include <cudaTypedefs.h>

#include "dma_internal.cuh"
#include "tc_primitives.cuh"

namespace dma {
namespace {

using namespace tc;

constexpr int kBN = 128;            // keys per block
constexpr int kRowsPerTile = kQTile;  // 128 query rows per M-tile
constexpr int kTcThreads = 384;  // three warpgroups
constexpr int kMmaWarp = 8;
constexpr int kProdWarp = 9;
// Registers per thread: 168 at launch (384 threads); the third warpgroup (MMA,
// producer, two idle warps) gives registers to the two softmax warpgroups:
// 128 * 88 + 256 * 208 = 384 * 168.
constexpr int kRegsControl = 88;
constexpr int kRegsSoftmax = 208;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 0.f;  // rescale whenever the row maximum rises
// One exponential pair in kPolyEvery is computed by ex2_poly (0: none).
constexpr int kPolyEvery = 0;

// barrier slots
enum : int {
    kBarQFull = 0,
    kBarQEmpty = 1,
    kBarKFull = 2,      // 2 stages
    kBarKEmpty = 4,     // 2 stages
    kBarVFull = 6,      // 2 stages
    kBarVEmpty = 8,     // 2 stages
    kBarMetaFull = 10,  // 2 stages
    kBarSFull = 12,     // per M-tile
    kBarPFull = 14,     // per M-tile
    kBarOFull = 16,     // per M-tile
    kBarDrain = 18,
    kNumBars = 19
};

template <int D>
struct Layout {
    static constexpr int kTile = kBN * D * 2;  // bytes of one 128-row bf16 tile
    static constexpr int kHalf = kBN * 128;    // bytes of one 64-column half of a tile
    static constexpr int kQ = 0;               // Q_A, Q_B
    static constexpr int kK = 2 * kTile;       // K stages 0, 1
    static constexpr int kV = 4 * kTile;       // V stages 0, 1
    static constexpr int kMeta = 6 * kTile;    // per stage: bias[128] f32, j[128], lo[128], tl[128]
    static constexpr int kMetaStage = 4 * kBN * 4;
    static constexpr int kFlags = kMeta + 2 * kMetaStage;  // per stage: all-full flag
    static constexpr int kBars = kFlags + 64;
    static constexpr int kMisc = kBars + 8 * kNumBars;  // tmem base, abort flag
    static constexpr int kEnd = kMisc + 16;
    static constexpr int kSmemBytes = kEnd + 1024;  // slack for 1024-byte alignment
};

struct TcArgs {
    const float* scores;     // [B][Hkv][S]
    const int32_t* expiry;   // [B][Hkv][S]
    const int32_t* tile_cnt; // [B][Hkv][n_qt]
    const int32_t* tile_idx; // [B][Hkv][n_qt][tile_stride]
    __nv_bfloat16* O;        // [B][S][H][D]
    float* lse;              // [B][H][S] or null
    int* status;
    int B, S, H, Hkv, G, n_qt, tile_stride, window, block;
    float c_log2;            // scale * log2(e)
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^x on the FMA pipe, for x <= 8 (x may be -inf): Cody-Waite range reduction
// x = j + f with j = round(x) and f in [-1/2, 1/2] (the integer j is read out of
// the mantissa of x + 1.5 * 2^23), then a degree-3 polynomial for 2^f whose
// coefficients minimise the relative error on [-1/2, 1/2] (about 7.5e-5, far
// below the bf16 rounding of P), and j is added to the exponent bits.  Results
// below 2^-126 come out as tiny or zero values.
__device__ __forceinline__ float ex2_poly(float x)
{
    x = fmaxf(x, -126.f);
    const float t = x + 12582912.f;  // 1.5 * 2^23: round to an integer in the low mantissa bits
    const float j = t - 12582912.f;
    const float f = x - j;
    float p = fmaf(0.0551711433f, f, 0.242609963f);
    p = fmaf(p, f, 0.693260968f);
    p = fmaf(p, f, 0.999928117f);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcArgs a)
{
    using L = Layout<D>;
    constexpr int kHalves = D / 64;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    float* meta_bias = reinterpret_cast<float*>(sm + L::kMeta);  // [stage][4][128]
    int* flags = reinterpret_cast<int*>(sm + L::kFlags);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);
    auto bar = [&](int i) { return sbase + L::kBars + 8 * i; };
    // A wait whose outcome is the same for every lane of the warp, so that warp-collective
    // instructions after it are never reached by only part of the warp.
    auto wait_warp = [&](int i, int parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, kWaitNs));
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nseg = a.B * a.Hkv;
    const int unit = blockIdx.x;
    const int tile = a.n_qt - 1 - unit / nseg;  // longest tiles first
    const int seg = unit % nseg;
    const int b = seg / a.Hkv, h = seg % a.Hkv;
    const int q0 = tile * kRowsPerTile;
    const int q1 = min(a.S, q0 + kRowsPerTile) - 1;
    const int W = a.window;

    int n_g = a.tile_cnt[(int64_t)seg * a.n_qt + tile];
    n_g = min(max(n_g, 0), a.tile_stride);
    const int32_t* gl = a.tile_idx + ((int64_t)seg * a.n_qt + tile) * a.tile_stride;
    const int band_lo = W > 0 ? max(0, q0 - W + 1) : q1 + 1;
    const int n_b = W > 0 ? q1 + 1 - band_lo : 0;
    const int n_all = n_g + n_b;
    const int nblk = (n_all + kBN - 1) / kBN;
    const int npass = (a.G + 1) / 2;

    if (nblk == 0) {
        // nothing kept for any row of the tile: O = 0, lse = -inf
        for (int t = threadIdx.x; t < kRowsPerTile * a.G; t += kTcThreads) {
            const int r = t % kRowsPerTile, g = t / kRowsPerTile, i = q0 + r;
            if (i > q1) continue;
            const int hq = h * a.G + g;
            uint4* op = reinterpret_cast<uint4*>(a.O + (((int64_t)b * a.S + i) * a.H + hq) * D);
            for (int c = 0; c < D / 8; ++c) op[c] = make_uint4(0, 0, 0, 0);
            if (a.lse) a.lse[((int64_t)b * a.H + hq) * a.S + i] = -INFINITY;
        }
        return;
    }

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(kBarMetaFull + 0), 32);
        mbar_init(bar(kBarMetaFull + 1), 32);
        mbar_init(bar(kBarPFull + 0), 128);
        mbar_init(bar(kBarPFull + 1), 128);
        mbar_init_fence();
    }
    if (warp == kMmaWarp) tmem_alloc<512>(smem_u32(tmem_slot));
    if (warp == kProdWarp && lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // key at position u of the tile's list (gathered keys, then the band); -1 past the end
    auto key_at = [&](int u) -> int {
        int j = -1;
        if (u < n_g) {
            j = gl[u];
            if (j < 0 || j >= a.S) {
                set_status(a.status, DMA_ERR_DEVICE_CHECK);
                j = -1;
            }
        } else if (u < n_all) {
            j = band_lo + (u - n_g);
        }
        return j;
    };

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ producer
        regs_decrease<kRegsControl>();
        const int64_t kv_row0 = (int64_t)b * a.S * a.Hkv + h;  // row of (b, j = 0, h)
        int t_issued_k = -1, t_issued_v = -1;
        auto load_k = [&](int t, int k) -> bool {
            const int s = t & 1, use = t >> 1;
            if (use >= 1 && !wait_warp(kBarKEmpty + s, (use - 1) & 1)) return false;
            if (lane == 0) mbar_arrive_expect_tx(bar(kBarKFull + s), L::kTile);
            __syncwarp();
            int rr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = key_at(k * kBN + 4 * lane + e);
                rr[e] = j >= 0 ? (int)(kv_row0 + (int64_t)j * a.Hkv) : -1;
            }
#pragma unroll
            for (int hf = 0; hf < kHalves; ++hf)
                tma_gather4(sbase + L::kK + s * L::kTile + hf * L::kHalf + 4 * lane * 128, &kmap, 64 * hf, rr[0],
                            rr[1], rr[2], rr[3], bar(kBarKFull + s));
            t_issued_k = t;
            return true;
        };
        auto load_v = [&](int t, int k) -> bool {
            const int s = t & 1, use = t >> 1;
            if (use >= 1 && !wait_warp(kBarVEmpty + s, (use - 1) & 1)) return false;
            float* mb = meta_bias + s * 4 * kBN;
            int* mj = reinterpret_cast<int*>(mb + kBN);
            int* mlo = mj + kBN;
            int* mtl = mlo + kBN;
            int rr[4];
            bool full = true;
            const float* sc = a.scores + (int64_t)seg * a.S;
            const int32_t* ex = a.expiry + (int64_t)seg * a.S;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = 4 * lane + e;
                const int j = key_at(k * kBN + c);
                rr[e] = j >= 0 ? (int)(kv_row0 + (int64_t)j * a.Hkv) : -1;
                float bias = -INFINITY;
                int jj = -(1 << 30), lo = 0, tl = 0;
                if (j >= 0) {
                    bias = sc[j] * kLog2e;
                    jj = j;
                    lo = top_lo(j, a.block);
                    tl = max(0, ex[j] - lo);
                    // is the key kept by every row of the tile?
                    const bool wfull = j <= q0 && j + W > q1;
                    const bool tfull = lo <= q0 && lo + tl > q1;
                    const bool ufull = tl > 0 && lo <= j + W && j <= q0 && max(j + W, lo + tl) > q1;
                    full = full && (wfull || tfull || ufull);
                }
                mb[c] = bias;
                mj[c] = jj;
                mlo[c] = lo;
                mtl[c] = tl;
            }
            const bool all_full = __all_sync(0xffffffffu, full);
            if (lane == 0) flags[s] = all_full ? 1 : 0;
            mbar_arrive(bar(kBarMetaFull + s));
            if (lane == 0) mbar_arrive_expect_tx(bar(kBarVFull + s), L::kTile);
            __syncwarp();
#pragma unroll
            for (int hf = 0; hf < kHalves; ++hf)
                tma_gather4(sbase + L::kV + s * L::kTile + hf * L::kHalf + 4 * lane * 128, &vmap, 64 * hf, rr[0],
                            rr[1], rr[2], rr[3], bar(kBarVFull + s));
            t_issued_v = t;
            return true;
        };

        bool ok = true;
        for (int p = 0; p < npass && ok; ++p) {
            const int nm = (2 * p + 1 < a.G) ? 2 : 1;
            if (p >= 1 && !wait_warp(kBarQEmpty, (p - 1) & 1)) break;
            if (lane == 0) mbar_arrive_expect_tx(bar(kBarQFull), nm * L::kTile);
            __syncwarp();
            for (int x = 0; x < nm; ++x) {
                const int hq = h * a.G + 2 * p + x;
                int rr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = q0 + 4 * lane + e;
                    rr[e] = i < a.S ? (int)(((int64_t)b * a.S + i) * a.H + hq) : -1;
                }
#pragma unroll
                for (int hf = 0; hf < kHalves; ++hf)
                    tma_gather4(sbase + L::kQ + x * L::kTile + hf * L::kHalf + 4 * lane * 128, &qmap, 64 * hf, rr[0],
                                rr[1], rr[2], rr[3], bar(kBarQFull));
            }
            const int t0 = p * nblk;
            ok = load_k(t0, 0);
            for (int k = 0; k < nblk && ok; ++k) {
                if (k + 1 < nblk) ok = load_k(t0 + k + 1, k + 1);
                if (ok) ok = load_v(t0 + k, k);
            }
        }
        if (*abort_flag) {
            // let the loads already issued land before the CTA's shared memory goes away
            if (t_issued_k >= 0) mbar_wait_drain(bar(kBarKFull + (t_issued_k & 1)), (t_issued_k >> 1) & 1, kWaitNs);
            if (t_issued_v >= 0) mbar_wait_drain(bar(kBarVFull + (t_issued_v & 1)), (t_issued_v >> 1) & 1, kWaitNs);
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        regs_decrease<kRegsControl>();
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, kBN, false);
            constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
            auto issue_s = [&](int x, int s) {
                const uint32_t qa = sbase + L::kQ + x * L::kTile, ka = sbase + L::kK + s * L::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * L::kHalf + (kk % 4) * 32;
                    mma_ss(tmem + 256 + 128 * x, smem_desc_sw128(qa + off, 16, 1024),
                           smem_desc_sw128(ka + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int x, int s, bool first) {
                const uint32_t va = sbase + L::kV + s * L::kTile;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tmem + 128 * x, tmem + 256 + 128 * x + kk * 8, smem_desc_sw128(va + kk * 2048, L::kHalf, 1024),
                           idO, (first && kk == 0) ? 0u : 1u);
            };
            bool ok = true;
            for (int p = 0; p < npass && ok; ++p) {
                const int nm = (2 * p + 1 < a.G) ? 2 : 1;
                if (!(ok = mbar_wait(bar(kBarQFull), p & 1, abort_flag, kWaitNs))) break;
                const int t0 = p * nblk;
                if (!(ok = mbar_wait(bar(kBarKFull + (t0 & 1)), (t0 >> 1) & 1, abort_flag, kWaitNs))) break;
                tc_fence_after();
                issue_s(0, t0 & 1);
                mma_commit(bar(kBarSFull + 0));
                if (nm == 2) {
                    issue_s(1, t0 & 1);
                    mma_commit(bar(kBarSFull + 1));
                }
                mma_commit(bar(kBarKEmpty + (t0 & 1)));
                for (int k = 0; k < nblk; ++k) {
                    const int t = t0 + k, s = t & 1;
                    const int t1 = t + 1, s1 = t1 & 1;
                    if (!(ok = mbar_wait(bar(kBarVFull + s), (t >> 1) & 1, abort_flag, kWaitNs))) break;
                    if (!(ok = mbar_wait(bar(kBarPFull + 0), t & 1, abort_flag, kWaitNs))) break;
                    tc_fence_after();
                    issue_pv(0, s, k == 0);
                    if (k + 1 < nblk) {
                        if (!(ok = mbar_wait(bar(kBarKFull + s1), (t1 >> 1) & 1, abort_flag, kWaitNs))) break;
                        tc_fence_after();
                        issue_s(0, s1);
                        mma_commit(bar(kBarSFull + 0));
                    } else {
                        mma_commit(bar(kBarOFull + 0));
                    }
                    if (nm == 2) {
                        if (!(ok = mbar_wait(bar(kBarPFull + 1), t & 1, abort_flag, kWaitNs))) break;
                        tc_fence_after();
                        issue_pv(1, s, k == 0);
                    }
                    mma_commit(bar(kBarVEmpty + s));
                    if (k + 1 < nblk) {
                        if (nm == 2) {
                            issue_s(1, s1);
                            mma_commit(bar(kBarSFull + 1));
                        }
                        mma_commit(bar(kBarKEmpty + s1));
                    } else if (nm == 2) {
                        mma_commit(bar(kBarOFull + 1));
                    }
                }
                if (ok) mma_commit(bar(kBarQEmpty));
            }
            // every MMA issued so far has completed before tensor memory is released
            mma_commit(bar(kBarDrain));
            mbar_wait_drain(bar(kBarDrain), 0, kWaitNs);
        }
        __syncwarp();
    } else if (warp >= 8) {
        regs_decrease<kRegsControl>();  // the idle warps of the third warpgroup
    } else {
        // ------------------------------------------------------------- softmax
        regs_increase<kRegsSoftmax>();
        const int x = warp >> 2;      // M-tile (warpgroup)
        const int quarter = warp & 3;  // tensor-memory lane quarter
        const int r = quarter * 32 + lane;
        const int i = q0 + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + 256 + 128 * x + lane_off;
        const uint32_t tO = tmem + 128 * x + lane_off;
        bool ok = true;
        for (int p = 0; p < npass && ok; ++p) {
            const int nm = (2 * p + 1 < a.G) ? 2 : 1;
            if (x >= nm) break;
            const int hq = h * a.G + 2 * p + x;
            float m_used = -INFINITY, l = 0.f;
            for (int k = 0; k < nblk; ++k) {
                const int t = p * nblk + k, s = t & 1;
                if (!(ok = wait_warp(kBarMetaFull + s, (t >> 1) & 1))) break;
                if (!(ok = wait_warp(kBarSFull + x, t & 1))) break;
                tc_fence_after();
                const float* mb = meta_bias + s * 4 * kBN;
                const int all_full = flags[s];
                float xv[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t rg[32];
                    tmem_ld32(tS + 32 * c, rg);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) xv[32 * c + e] = __uint_as_float(rg[e]);
                }
                float mx[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) mx[e] = -INFINITY;
                if (all_full) {
#pragma unroll
                    for (int c = 0; c < kBN; c += 4) {
                        const float4 bb = *reinterpret_cast<const float4*>(mb + c);
                        xv[c + 0] = fmaf(xv[c + 0], a.c_log2, bb.x);
                        xv[c + 1] = fmaf(xv[c + 1], a.c_log2, bb.y);
                        xv[c + 2] = fmaf(xv[c + 2], a.c_log2, bb.z);
                        xv[c + 3] = fmaf(xv[c + 3], a.c_log2, bb.w);
                        mx[(c / 4) & 3] = fmaxf(mx[(c / 4) & 3], fmaxf(fmaxf(xv[c], xv[c + 1]), fmaxf(xv[c + 2], xv[c + 3])));
                    }
                } else {
                    // per-column keep bits for this row, then the masked logits
                    const int* mj = reinterpret_cast<const int*>(mb + kBN);
                    const int* mlo = mj + kBN;
                    const int* mtl = mlo + kBN;
                    uint32_t kbits[kBN / 32];
#pragma unroll
                    for (int w32 = 0; w32 < kBN / 32; ++w32) {
                        uint32_t bits = 0;
#pragma unroll 1
                        for (int cc = 0; cc < 32; ++cc) {
                            const int c = 32 * w32 + cc;
                            const bool kept =
                                (unsigned)(i - mj[c]) < (unsigned)W || (unsigned)(i - mlo[c]) < (unsigned)mtl[c];
                            bits |= (kept ? 1u : 0u) << cc;
                        }
                        kbits[w32] = bits;
                    }
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        const bool kept = (kbits[c / 32] >> (c % 32)) & 1u;
                        xv[c] = kept ? fmaf(xv[c], a.c_log2, mb[c]) : -INFINITY;
                        mx[c & 3] = fmaxf(mx[c & 3], xv[c]);
                    }
                }
                const float m_blk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                // The maximum of a row moved up: rescale what it has accumulated.  tcgen05.ld/st
                // are warp-collective, so the warp rescales together whenever one of its rows
                // needs it (factor 1 for the others).
                const bool raise = m_blk > m_used + kRescaleThreshold;
                const bool rescale = raise && k > 0 && m_used != -INFINITY;
                const float alpha = rescale ? ex2(m_used - m_blk) : 1.f;
                if (raise) m_used = m_blk;
                if (__any_sync(0xffffffffu, rescale)) {
                    l *= alpha;
#pragma unroll 1
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t rg[16];
                        tmem_ld16(tO + 16 * c, rg);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e) rg[e] = __float_as_uint(__uint_as_float(rg[e]) * alpha);
                        tmem_st16(tO + 16 * c, rg);
                    }
                }
                const float m_eff = m_used == -INFINITY ? 0.f : m_used;
                float ls[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) ls[e] = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        // a share of the exponentials goes to the FMA pipe, the rest to the MUFU
                        const bool poly = kPolyEvery > 0 && (e % (kPolyEvery > 0 ? kPolyEvery : 1)) == kPolyEvery - 1;
                        const float p0 = poly ? ex2_poly(xv[c0 + 2 * e] - m_eff) : ex2(xv[c0 + 2 * e] - m_eff);
                        const float p1 = poly ? ex2_poly(xv[c0 + 2 * e + 1] - m_eff) : ex2(xv[c0 + 2 * e + 1] - m_eff);
                        ls[e & 3] += p0 + p1;
                        pk[e] = pack_bf16(p0, p1);
                    }
                    tmem_st16(tS + c0 / 2, pk);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + x));
            }
            if (!ok) break;
            // epilogue: O = accumulator / l
            if (!(ok = wait_warp(kBarOFull + x, p & 1))) break;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* op = a.O + (((int64_t)b * a.S + min(i, a.S - 1)) * a.H + hq) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rg[32];
                tmem_ld32(tO + 32 * c, rg);
                tmem_ld_wait();
                if (i < a.S) {
                    uint4* o4 = reinterpret_cast<uint4*>(op + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(rg[8 * v + 0]) * inv, __uint_as_float(rg[8 * v + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(rg[8 * v + 2]) * inv, __uint_as_float(rg[8 * v + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(rg[8 * v + 4]) * inv, __uint_as_float(rg[8 * v + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(rg[8 * v + 6]) * inv, __uint_as_float(rg[8 * v + 7]) * inv);
                        o4[v] = w;
                    }
                }
            }
            if (a.lse && i < a.S)
                a.lse[((int64_t)b * a.H + hq) * a.S + i] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
            tc_fence_before();
        }
    }

    if (threadIdx.x == 0 && *abort_flag) set_status(a.status, DMA_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc<512>(tmem);
}

// cuTensorMapEncodeTiled, looked up through the runtime so that the library
// does not link the driver library directly (it loads on machines without one).
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 2-D view (rows x D) of a [.., D] bf16 tensor, one-row box of 64 columns, 128-byte swizzle.
bool make_row_map(CUtensorMap* m, const void* base, int64_t rows, int D)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, 1};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_typed(const void* Q, const void* K, const void* V, int B, int S, int H, int Hkv,
                         const float* scores, const dma_kept_t* kept, float scale, void* O, float* lse, int* status,
                         cudaStream_t st)
{
    CUtensorMap qm, km, vm;
    if (!make_row_map(&qm, Q, (int64_t)B * S * H, D) || !make_row_map(&km, K, (int64_t)B * S * Hkv, D) ||
        !make_row_map(&vm, V, (int64_t)B * S * Hkv, D))
        return cudaErrorInvalidValue;
    TcArgs a;
    a.scores = scores;
    a.expiry = kept->expiry;
    a.tile_cnt = kept->tile_cnt;
    a.tile_idx = kept->tile_idx;
    a.O = static_cast<__nv_bfloat16*>(O);
    a.lse = lse;
    a.status = status;
    a.B = B;
    a.S = S;
    a.H = H;
    a.Hkv = Hkv;
    a.G = H / Hkv;
    a.n_qt = kept->n_qt;
    a.tile_stride = kept->tile_stride;
    a.window = kept->window;
    a.block = kept->block;
    a.c_log2 = scale * kLog2e;
    const int smem = Layout<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)kept->n_qt * B * Hkv;
    prefill_tc_kernel<D><<<(unsigned)grid, kTcThreads, smem, st>>>(qm, km, vm, a);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(dma_dtype_t dt, int B, int S, int H, int Hkv, int D)
{
    if (dt != DMA_BF16 || (D != 64 && D != 128)) return false;
    // row coordinates of the tensor maps are 32-bit
    return (int64_t)B * S * H < ((int64_t)1 << 31) && (int64_t)B * S * Hkv < ((int64_t)1 << 31);
}

cudaError_t launch_prefill_tc(const void* Q, const void* K, const void* V, int B, int S, int H, int Hkv, int D,
                              const float* scores, const dma_kept_t* kept, float scale, void* O, float* lse,
                              int* status, cudaStream_t st)
{
    if (D == 128) return launch_typed<128>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, status, st);
    return launch_typed<64>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, status, st);
}

}  // namespace dma
