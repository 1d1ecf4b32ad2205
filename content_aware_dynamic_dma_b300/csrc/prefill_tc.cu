// Sparse attention prefill on the 5th-generation tensor cores (bf16, D = 64 or
// 128): tcgen05 MMAs with fp32 accumulators in tensor memory, kept K/V rows
// gathered into shared memory with cp.async.
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
// gathered K/V block is fetched once per pair of query heads.  Roles (512
// threads, four warpgroups):
//   warps 0-3 / 4-7  softmax of M-tile A / B: a thread owns one query row (= one
//                    tensor-memory lane): S from tensor memory, masked online
//                    softmax in the log2 domain, P (bf16) written back over S
//   warps 8-11       correction: rescales a row's O accumulator in tensor memory
//                    when its running maximum rises (while the softmax computes
//                    the exponentials), and writes O / row sum and lse at the end
//                    of a pass
//   warp 12          MMA issue (one thread): S = Q K^T (both operands in shared
//                    memory), O += P V (P from tensor memory, V in shared memory)
//   warp 13          key metadata: runs up to eight blocks ahead, filling a ring
//                    with each block's key indices, bias (score, log2 units),
//                    keep intervals and an "every row keeps every key" flag
//   warps 14-15      copies: Q tiles and the K and V rows of each block,
//                    gathered with 16-byte cp.async into the 128-byte-swizzled
//                    operand layout (a TMA tile::gather4 moves only about 8
//                    bytes per cycle per SM, a quarter of what this needs)
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

#include "dma_internal.cuh"
#include "tc_primitives.cuh"

namespace dma {
namespace {

using namespace tc;

constexpr int kBN = 128;              // keys per block
constexpr int kRowsPerTile = kQTile;  // 128 query rows per M-tile
constexpr int kTcThreads = 512;       // four warpgroups
constexpr int kCorrWarp0 = 8;         // warps 8-11
constexpr int kMmaWarp = 12;
constexpr int kMetaWarp = 13;
constexpr int kCopyWarp0 = 14;  // warps 14 and 15
constexpr int kSoftmaxWarps = 8;
constexpr int kCopyThreads = 64;
// 16-byte chunks of a row that one copy thread takes, and the depth of the key-metadata ring.
// Measured on the 16K and both 64K workloads against (4, 4): (2, 8) is 1.8% faster at 16K, the
// same at 64K in token units and 7% faster in 64-key block units.
constexpr int kCopyChunks = 2;
constexpr int kIdxStages = 8;
// Registers per thread: 128 at launch (512 threads x 128 = the whole register
// file); the correction and control warpgroups give registers to the two softmax
// warpgroups: 256 * 192 + 128 * 64 + 128 * 64 = 512 * 128.
constexpr int kRegsSoftmax = 192;
constexpr int kRegsCorr = 64;
constexpr int kRegsControl = 64;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsCorr + 128 * kRegsControl <= kTcThreads * 128,
              "register split exceeds the launch's registers");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// barrier slots
enum : int {
    kBarQFull = 0,
    kBarQEmpty = 1,
    kBarK0Full = 2,   // the K rows of a pass's first block have landed
    kBarKEmpty = 4,   // 2 stages
    kBarBlkFull = 6,  // 2 stages (block t: t & 1): the V rows of block t and the K rows of block t + 1
    kBarVEmpty = 8,   // 2 stages
    kBarSFull = 10,   // per M-tile: S of a block is in tensor memory
    kBarPFull = 12,   // per M-tile: P of a block is in tensor memory (softmax) and O is rescaled
                      // for it, or read out by the previous pass's epilogue (correction)
    kBarOFull = 14,   // per M-tile: the last PV of a pass has completed
    kBarDrain = 16,
    kBarAFull = 17,   // per M-tile: the rescale factors of a block are in shared memory
    kBarStats = 21,   // per (M-tile, pass parity): the row sums of a pass are in shared memory
    kBarIdxFull = 25,  // kIdxStages slots
    kBarIdxEmpty = 25 + kIdxStages,
    kNumBars = 25 + 2 * kIdxStages
};

template <int D>
struct Layout {
    static constexpr int kTile = kBN * D * 2;  // bytes of one 128-row bf16 tile
    static constexpr int kHalf = kBN * 128;    // bytes of one 64-column half of a tile
    static constexpr int kQ = 0;               // Q_A, Q_B
    static constexpr int kK = 2 * kTile;       // K stages 0, 1
    static constexpr int kV = 4 * kTile;       // V stages 0, 1
    // key-metadata ring, per slot: j[128] (key index, -1 past the end), bias[128] f32 (log2 units,
    // -inf past the end), jm[128] (window start), lo[128], tl[128] (top interval [lo, lo + tl)),
    // then the all-full flag
    static constexpr int kIdx = 6 * kTile;
    static constexpr int kIdxSlot = 5 * kBN * 4 + 16;
    static constexpr int kAlpha = kIdx + kIdxStages * kIdxSlot;    // [M-tile][row] f32
    static constexpr int kStats = kAlpha + 2 * kRowsPerTile * 4;   // [parity][M-tile][row] f32 row sums
    static constexpr int kBars = kStats + 2 * 2 * kRowsPerTile * 4;
    static constexpr int kMisc = kBars + 8 * kNumBars;  // tmem base, abort flag
    static constexpr int kEnd = kMisc + 16;
    static constexpr int kSmemBytes = kEnd + 1024;  // slack for 1024-byte alignment
};

struct TcArgs {
    const __nv_bfloat16* Q;  // [B][S][H][D]
    const __nv_bfloat16* K;  // [B][S][Hkv][D]
    const __nv_bfloat16* V;  // [B][S][Hkv][D]
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

// Packed pairs of fp32 (one instruction for two lanes of arithmetic).
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
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The CTA's work unit: (batch, KV head) segment and query tile, and the tile's key list
// (gathered keys, then the window band).  Every role computes it for itself, from a block
// index read afresh, so that none of it stays live across the role branches (the roles run
// with different register budgets).
struct Geom {
    int b, h, seg, q0, q1, W, n_g, band_lo, n_all, nblk, npass;
    const int32_t* gl;

    // key at position u of the tile's list; -1 past the end (and for an out-of-range gathered
    // index, which is recorded as DMA_ERR_DEVICE_CHECK)
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

__device__ __forceinline__ int fresh_ctaid()
{
    int v;
    asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(v));
    return v;
}

__device__ __forceinline__ Geom tile_geom(const TcArgs& a, int unit)
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
    g.npass = (a.G + 1) / 2;
    return g;
}

// kFaultTest: the wait limit comes from the arguments and the drop-arrive injection is
// compiled in; the launches of normal use run the kernel without either (fixed 2 s limit).
template <int D, bool kFaultTest>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const TcArgs a, const uint64_t test_wait_ns, const int test_drop_arrive)
{
    // (test_*: used only by the fault-test instantiation: the wait limit, and whether CTA 0
    // withholds the copy warps' signal for the K rows of its first block)
    const uint64_t wait_ns = kFaultTest ? test_wait_ns : kDefaultWaitNs;
    using L = Layout<D>;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic so that the compiler keeps every access
    // through it in the shared state space (ld/st.shared, not generic loads)
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    auto idx_slot = [&](int r) { return reinterpret_cast<int*>(sm + L::kIdx + r * L::kIdxSlot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);
    float* alpha_sm = reinterpret_cast<float*>(sm + L::kAlpha);
    float* stats_sm = reinterpret_cast<float*>(sm + L::kStats);
    auto bar = [&](int i) { return sbase + L::kBars + 8 * i; };
    // A wait whose outcome is the same for every lane of the warp, so that warp-collective
    // instructions after it are never reached by only part of the warp.
    auto wait_warp = [&](int i, int parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, wait_ns));
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    {
        const Geom g = tile_geom(a, blockIdx.x);
        if (g.nblk == 0) {
            // nothing kept for any row of the tile: O = 0, lse = -inf
            for (int t = threadIdx.x; t < kRowsPerTile * a.G; t += kTcThreads) {
                const int r = t % kRowsPerTile, gq = t / kRowsPerTile, i = g.q0 + r;
                if (i > g.q1) continue;
                const int hq = g.h * a.G + gq;
                uint4* op = reinterpret_cast<uint4*>(a.O + (((int64_t)g.b * a.S + i) * a.H + hq) * D);
                for (int c = 0; c < D / 8; ++c) op[c] = make_uint4(0, 0, 0, 0);
                if (a.lse) a.lse[((int64_t)g.b * a.H + hq) * a.S + i] = -INFINITY;
            }
            return;
        }
    }

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        for (int i = 0; i < kIdxStages; ++i) {
            mbar_init(bar(kBarIdxFull + i), 32);
            // the softmax warps and the two copy warps (in a pass with one M-tile, the warps of
            // M-tile A arrive twice)
            mbar_init(bar(kBarIdxEmpty + i), kSoftmaxWarps + 2);
        }
        mbar_init(bar(kBarQFull), kCopyThreads);
        mbar_init(bar(kBarK0Full), kCopyThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarBlkFull + i), kCopyThreads);
            mbar_init(bar(kBarPFull + i), 2 * kRowsPerTile);
            mbar_init(bar(kBarAFull + i), kRowsPerTile);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar(kBarStats + i), kRowsPerTile);
        mbar_init_fence();
    }
    if (warp == kMmaWarp) tmem_alloc<512>(smem_u32(tmem_slot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMetaWarp) {
        // -------------------------------------------------------- key metadata
        regs_decrease<kRegsControl>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int seg = g.seg, q0 = g.q0, q1 = g.q1, W = g.W, nblk = g.nblk, npass = g.npass;
        auto key_at = [&](int u) { return g.key_at(u, a.S, a.status); };
        const float* sc = a.scores + (int64_t)seg * a.S;
        const int32_t* ex = a.expiry + (int64_t)seg * a.S;
        const int nt = npass * nblk;  // blocks over all passes (every pass walks the same keys)
        int jc[4], jn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) jc[e] = key_at(4 * lane + e);
        for (int t = 0; t < nt; ++t) {
            const int r = t % kIdxStages, use = t / kIdxStages;
            if (use >= 1 && !wait_warp(kBarIdxEmpty + r, (use - 1) & 1)) break;
            // this block's scores and expiries, and the next block's indices, in flight together
            float scv[4];
            int exv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                scv[e] = jc[e] >= 0 ? sc[jc[e]] : 0.f;
                exv[e] = jc[e] >= 0 ? ex[jc[e]] : 0;
            }
            const int kn = (t + 1) % nblk;
#pragma unroll
            for (int e = 0; e < 4; ++e) jn[e] = (t + 1 < nt) ? key_at(kn * kBN + 4 * lane + e) : -1;
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
                    // is the key kept by every row of the tile?
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
            mbar_arrive(bar(kBarIdxFull + r));
#pragma unroll
            for (int e = 0; e < 4; ++e) jc[e] = jn[e];
        }
    } else if (warp >= kCopyWarp0) {
        // -------------------------------------------------------------- copies
        regs_decrease<kRegsControl>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int b = g.b, h = g.h, q0 = g.q0, nblk = g.nblk, npass = g.npass;
        // Each thread copies kCPT 16-byte chunks of a row (one index load and one address
        // computation per row for all of them): chunks c0, c0 + kTPR, c0 + 2 kTPR, ... so that the
        // kTPR threads of a row read kTPR adjacent chunks in each instruction (whole 32-byte
        // sectors).  A sweep covers kRowsPerSweep rows, a multiple of 8, so the swizzle phase (row
        // mod 8) of a thread's rows never changes.
        constexpr int kCPR = D / 8;  // 16-byte chunks per row
        constexpr int kCPT = kCopyChunks < kCPR ? kCopyChunks : kCPR;
        constexpr int kTPR = kCPR / kCPT;  // threads per row
        constexpr int kRowsPerSweep = kCopyThreads / kTPR;
        constexpr int kSweeps = kBN / kRowsPerSweep;
        static_assert(kRowsPerSweep % 8 == 0 && kBN % kRowsPerSweep == 0, "copy sweep shape");
        const int ct = threadIdx.x - kCopyWarp0 * 32;
        const int chunk0 = ct % kTPR, r0 = ct / kTPR;
        const uint32_t ph = (uint32_t)r0 & 7u;  // swizzle phase of every row this thread copies
        // shared-memory offset of chunk i of this thread within its row
        auto chunk_off = [&](int i) -> uint32_t {
            const int c = chunk0 + kTPR * i;
            return (uint32_t)((c >> 3) * L::kHalf) + ((((uint32_t)c & 7u) ^ ph) << 4);
        };
        const __nv_bfloat16* Kh = a.K + ((int64_t)b * a.S * a.Hkv + h) * D + chunk0 * 8;
        const __nv_bfloat16* Vh = a.V + ((int64_t)b * a.S * a.Hkv + h) * D + chunk0 * 8;
        const int64_t kv_stride = (int64_t)a.Hkv * D;
        // Copies never wait for their own completion: each group ends with an arrival that the
        // barrier receives once the thread's copies have landed.  The consumer (the MMA thread)
        // orders them for the tensor core's reads with a proxy fence after its wait.
        auto acquire = [&](int barid, int parity) -> bool { return wait_warp(barid, parity); };
        auto committed = [&](int barid) { cp_async_arrive(bar(barid)); };
        auto copy_rows = [&](uint32_t tile, const int* js, const __nv_bfloat16* base) {
#pragma unroll 4
            for (int m = 0; m < kSweeps; ++m) {
                const int row = r0 + kRowsPerSweep * m;
                const int j = js[row];
                const uint32_t rb = tile + row * 128;
                const __nv_bfloat16* src = base + (int64_t)(j >= 0 ? j : 0) * kv_stride;
#pragma unroll
                for (int c = 0; c < kCPT; ++c) cp_async16(rb + chunk_off(c), src + 8 * kTPR * c, j >= 0);
            }
        };
        bool ok = true;
        for (int p = 0; p < npass && ok; ++p) {
            const int nm = (2 * p + 1 < a.G) ? 2 : 1;
            if (p >= 1 && !(ok = acquire(kBarQEmpty, (p - 1) & 1))) break;
            for (int x = 0; x < nm; ++x) {
                const int hq = h * a.G + 2 * p + x;
                const uint32_t tile = sbase + L::kQ + x * L::kTile;
#pragma unroll 4
                for (int m = 0; m < kSweeps; ++m) {
                    const int row = r0 + kRowsPerSweep * m;
                    const int i = q0 + row;
                    const uint32_t rb = tile + row * 128;
                    const __nv_bfloat16* src = a.Q + (((int64_t)b * a.S + min(i, a.S - 1)) * a.H + hq) * D + chunk0 * 8;
#pragma unroll
                    for (int c = 0; c < kCPT; ++c) cp_async16(rb + chunk_off(c), src + 8 * kTPR * c, i < a.S);
                }
            }
            committed(kBarQFull);
            const int t0 = p * nblk;
            // copies of the K rows of block t into stage t & 1 (no completion signal of their own)
            auto load_k = [&](int t) -> bool {
                const int s = t & 1, use = t >> 1, r = t % kIdxStages;
                if (!acquire(kBarIdxFull + r, (t / kIdxStages) & 1)) return false;
                if (use >= 1 && !acquire(kBarKEmpty + s, (use - 1) & 1)) return false;
                copy_rows(sbase + L::kK + s * L::kTile, idx_slot(r), Kh);
                return true;
            };
            auto load_v = [&](int t) -> bool {
                const int s = t & 1, use = t >> 1, r = t % kIdxStages;
                if (use >= 1 && !acquire(kBarVEmpty + s, (use - 1) & 1)) return false;
                copy_rows(sbase + L::kV + s * L::kTile, idx_slot(r), Vh);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarIdxEmpty + r));  // done with this slot's indices
                return true;
            };
            ok = load_k(t0);
            // (fault injection for tests: the MMA warp's wait for these rows then runs out)
            if (ok && !(kFaultTest && test_drop_arrive && blockIdx.x == 0 && p == 0)) committed(kBarK0Full);
            // V of a block is needed (by PV) before K of the next one (by the next S); one
            // completion signal covers both
            for (int k = 0; k < nblk && ok; ++k) {
                ok = load_v(t0 + k);
                if (ok && k + 1 < nblk) ok = load_k(t0 + k + 1);
                if (ok) committed(kBarBlkFull + ((t0 + k) & 1));
            }
        }
        cp_async_wait_all();  // the copies already issued land before shared memory goes away
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        // The whole warp runs the issue loop with warp-uniform values (the descriptors and
        // tensor-memory addresses then live in uniform registers) and lane 0 issues each
        // tcgen05.mma and commit: issuing from a single-thread branch was measured to take about
        // 110 cycles per MMA, more than the tensor core needs to execute it.
        regs_decrease<kRegsControl>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int nblk = g.nblk, npass = g.npass;
        const uint32_t tmem = *tmem_slot;
        const bool leader = lane == 0;
        constexpr uint32_t idS = idesc_bf16_f32(128, kBN, false);
        constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
        // (a descriptor's start address is its low 14 bits, in 16-byte units: the step to the next
        // 16-element slab is added to the descriptor itself, which never carries out of that field
        // since shared memory ends below 256 KB)
        auto issue_s = [&](int x, int s) {
            const uint64_t dq = smem_desc_sw128(sbase + L::kQ + x * L::kTile, 16, 1024);
            const uint64_t dk = smem_desc_sw128(sbase + L::kK + s * L::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * L::kHalf + (kk % 4) * 32) >> 4;
                if (leader) mma_ss(tmem + 256 + 128 * x, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int x, int s, bool first) {
            const uint64_t dv = smem_desc_sw128(sbase + L::kV + s * L::kTile, L::kHalf, 1024);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                if (leader)
                    mma_ts(tmem + 128 * x, tmem + 256 + 128 * x + kk * 8, dv + (uint32_t)(kk * (2048 >> 4)), idO,
                           (first && kk == 0) ? 0u : 1u);
        };
        auto commit = [&](int barid) {
            if (leader) mma_commit(bar(barid));
        };
        // PV of M-tile x for block t: P written by the softmax and O rescaled (or, for a pass's
        // first block, read out by the previous pass's epilogue) by the correction warps
        auto wait_pv = [&](int x, int t) -> bool { return wait_warp(kBarPFull + x, t & 1); };
        bool ok = true;
        for (int p = 0; p < npass && ok; ++p) {
            const int nm = (2 * p + 1 < a.G) ? 2 : 1;
            if (!(ok = wait_warp(kBarQFull, p & 1))) break;
            const int t0 = p * nblk;
            if (!(ok = wait_warp(kBarK0Full, p & 1))) break;
            fence_proxy_async_smem();  // the cp.async writes (generic proxy) before the MMA reads them
            tc_fence_after();
            issue_s(0, t0 & 1);
            commit(kBarSFull + 0);
            if (nm == 2) {
                issue_s(1, t0 & 1);
                commit(kBarSFull + 1);
            }
            commit(kBarKEmpty + (t0 & 1));
            for (int k = 0; k < nblk; ++k) {
                const int t = t0 + k, s = t & 1;
                const int t1 = t + 1, s1 = t1 & 1;
                // this block's V and the next block's K (both copied by cp.async), then one proxy
                // fence for both: their writes must be ordered before the tensor core's reads
                if (!(ok = wait_warp(kBarBlkFull + s, (t >> 1) & 1))) break;
                fence_proxy_async_smem();
                if (!(ok = wait_pv(0, t))) break;
                tc_fence_after();
                issue_pv(0, s, k == 0);
                if (k + 1 < nblk) {
                    issue_s(0, s1);
                    commit(kBarSFull + 0);
                } else {
                    commit(kBarOFull + 0);
                }
                if (nm == 2) {
                    if (!(ok = wait_pv(1, t))) break;
                    tc_fence_after();
                    issue_pv(1, s, k == 0);
                }
                commit(kBarVEmpty + s);
                if (k + 1 < nblk) {
                    if (nm == 2) {
                        issue_s(1, s1);
                        commit(kBarSFull + 1);
                    }
                    commit(kBarKEmpty + s1);
                } else if (nm == 2) {
                    commit(kBarOFull + 1);
                }
            }
            if (ok) commit(kBarQEmpty);
        }
        // every MMA issued so far has completed before tensor memory is released
        commit(kBarDrain);
        if (leader) mbar_wait_drain(bar(kBarDrain), 0, wait_ns);
        __syncwarp();
    } else if (warp >= kCorrWarp0) {
        // ---------------------------------------------------------- correction
        // Thread = row r of both M-tiles.  Per block: wait for the softmax's rescale factor of
        // the row (posted as soon as the block maximum is known), scale the row's O accumulator
        // in tensor memory when any row of the warp needs it, and release the block's PV.  At the
        // end of a pass: O / row sum to global memory (bf16) and lse.
        regs_decrease<kRegsCorr>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int b = g.b, h = g.h, q0 = g.q0, nblk = g.nblk, npass = g.npass;
        const uint32_t tmem = *tmem_slot;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int i = q0 + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        bool ok = true;
        for (int p = 0; p < npass && ok; ++p) {
            const int nm = (2 * p + 1 < a.G) ? 2 : 1;
            for (int k = 0; k < nblk && ok; ++k) {
                const int t = p * nblk + k;
                for (int x = 0; x < nm; ++x) {
                    if (!(ok = wait_warp(kBarAFull + x, t & 1))) break;
                    if (k > 0) {
                        const float alpha = alpha_sm[x * kRowsPerTile + r];
                        if (__any_sync(0xffffffffu, alpha != 1.f)) {
                            // PV of the previous block has completed: the softmax saw this block's S,
                            // committed after it
                            tc_fence_after();
                            const uint32_t tO = tmem + 128 * x + lane_off;
                            const f2 al2 = mk2(alpha, alpha);
#pragma unroll
                            for (int c0 = 0; c0 < D; c0 += 16) {
                                uint32_t o0[16];
                                tmem_ld16(tO + c0, o0);
                                tmem_ld_wait();
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    float y0, y1;
                                    split2(mul2(mk2(__uint_as_float(o0[e]), __uint_as_float(o0[e + 1])), al2), y0, y1);
                                    o0[e] = __float_as_uint(y0);
                                    o0[e + 1] = __float_as_uint(y1);
                                }
                                tmem_st16(tO + c0, o0);
                            }
                            tmem_st_wait();
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(bar(kBarPFull + x));
                }
            }
            if (!ok) break;
            // epilogue of the pass: O = accumulator / row sum
            for (int x = 0; x < nm; ++x) {
                const int par = p & 1;
                ok = wait_warp(kBarStats + 2 * x + par, (p >> 1) & 1) && wait_warp(kBarOFull + x, p & 1);
                if (!ok) break;
                tc_fence_after();
                const float l_row = stats_sm[(par * 2 + x) * kRowsPerTile + r];
                const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                const int hq = h * a.G + 2 * p + x;
                const uint32_t tO = tmem + 128 * x + lane_off;
                __nv_bfloat16* op = a.O + (((int64_t)b * a.S + min(i, a.S - 1)) * a.H + hq) * D;
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t rg[16];
                    tmem_ld16(tO + 16 * c, rg);
                    tmem_ld_wait();
                    if (i < a.S) {
                        uint4* o4 = reinterpret_cast<uint4*>(op + 16 * c);
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(rg[8 * v + 0]) * inv, __uint_as_float(rg[8 * v + 1]) * inv);
                            w.y = pack_bf16(__uint_as_float(rg[8 * v + 2]) * inv, __uint_as_float(rg[8 * v + 3]) * inv);
                            w.z = pack_bf16(__uint_as_float(rg[8 * v + 4]) * inv, __uint_as_float(rg[8 * v + 5]) * inv);
                            w.w = pack_bf16(__uint_as_float(rg[8 * v + 6]) * inv, __uint_as_float(rg[8 * v + 7]) * inv);
                            o4[v] = w;
                        }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------- softmax
        // Thread = one query row of M-tile x (tensor-memory lane r): the 128 logits of a block
        // in registers, the exact block maximum, the rescale factor posted for the correction
        // warps, then the exponentials written back as bf16 P over S.
        regs_increase<kRegsSoftmax>();
        const Geom g = tile_geom(a, fresh_ctaid());
        const int q0 = g.q0, W = g.W, nblk = g.nblk, npass = g.npass;
        const uint32_t tmem = *tmem_slot;
        const int x = warp >> 2;  // M-tile
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int i = q0 + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + 256 + 128 * x + lane_off;
        const f2 cc2 = mk2(a.c_log2, a.c_log2);
        bool ok = true;
        for (int p = 0; p < npass && ok; ++p) {
            const int nm = (2 * p + 1 < a.G) ? 2 : 1;
            if (x >= nm) break;  // M-tile B has no query head in the last pass of an odd group
            const uint32_t idx_arrivals = nm == 1 ? 2u : 1u;  // M-tile A then arrives for both
            float m_used = -INFINITY, l = 0.f;
            for (int k = 0; k < nblk; ++k) {
                const int t = p * nblk + k;
                const int ridx = t % kIdxStages;
                ok = wait_warp(kBarIdxFull + ridx, (t / kIdxStages) & 1) && wait_warp(kBarSFull + x, t & 1);
                if (!ok) break;
                tc_fence_after();
                const int* js = idx_slot(ridx);
                const float* mb = reinterpret_cast<const float*>(js + kBN);
                const int all_full = js[5 * kBN];
                float xv[kBN];
                tmem_ld32f(tS + 0, xv);
                tmem_ld32f(tS + 32, xv + 32);
                tmem_ld32f(tS + 64, xv + 64);
                tmem_ld32f(tS + 96, xv + 96);
                tmem_ld_wait();
                // logits in log2 units: x = S * scale * log2(e) + bias * log2(e)
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (all_full) {
#pragma unroll
                    for (int c = 0; c < kBN; c += 4) {
                        const float4 bb = *reinterpret_cast<const float4*>(mb + c);
                        f2 x01 = fma2(mk2(xv[c], xv[c + 1]), cc2, mk2(bb.x, bb.y));
                        f2 x23 = fma2(mk2(xv[c + 2], xv[c + 3]), cc2, mk2(bb.z, bb.w));
                        split2(x01, xv[c], xv[c + 1]);
                        split2(x23, xv[c + 2], xv[c + 3]);
                        const int q = (c / 4) & 3;
                        mx[q] = max3(mx[q], xv[c], xv[c + 1]);
                        mx[q] = max3(mx[q], xv[c + 2], xv[c + 3]);
                    }
                } else {
                    // kept iff j <= i < j + window  or  lo_j <= i < expiry_j
                    const int* mj = js + 2 * kBN;
                    const int* mlo = js + 3 * kBN;
                    const int* mtl = js + 4 * kBN;
#pragma unroll
                    for (int c = 0; c < kBN; c += 4) {
                        const float4 bb = *reinterpret_cast<const float4*>(mb + c);
                        const int4 jj = *reinterpret_cast<const int4*>(mj + c);
                        const int4 lo = *reinterpret_cast<const int4*>(mlo + c);
                        const int4 tl = *reinterpret_cast<const int4*>(mtl + c);
                        f2 x01 = fma2(mk2(xv[c], xv[c + 1]), cc2, mk2(bb.x, bb.y));
                        f2 x23 = fma2(mk2(xv[c + 2], xv[c + 3]), cc2, mk2(bb.z, bb.w));
                        split2(x01, xv[c], xv[c + 1]);
                        split2(x23, xv[c + 2], xv[c + 3]);
                        if (!((unsigned)(i - jj.x) < (unsigned)W || (unsigned)(i - lo.x) < (unsigned)tl.x)) xv[c] = -INFINITY;
                        if (!((unsigned)(i - jj.y) < (unsigned)W || (unsigned)(i - lo.y) < (unsigned)tl.y)) xv[c + 1] = -INFINITY;
                        if (!((unsigned)(i - jj.z) < (unsigned)W || (unsigned)(i - lo.z) < (unsigned)tl.z)) xv[c + 2] = -INFINITY;
                        if (!((unsigned)(i - jj.w) < (unsigned)W || (unsigned)(i - lo.w) < (unsigned)tl.w)) xv[c + 3] = -INFINITY;
                        const int q = (c / 4) & 3;
                        mx[q] = max3(mx[q], xv[c], xv[c + 1]);
                        mx[q] = max3(mx[q], xv[c + 2], xv[c + 3]);
                    }
                }
                const float m_blk = max3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
                // The maximum of the row moved up: what O has accumulated is rescaled by the
                // correction warps while the exponentials are computed here.
                const bool raise = m_blk > m_used;
                const bool rescale = raise && k > 0 && m_used != -INFINITY;
                const float alpha = rescale ? ex2(m_used - m_blk) : 1.f;
                if (raise) m_used = m_blk;
                alpha_sm[x * kRowsPerTile + r] = alpha;
                tc_fence_before();
                mbar_arrive(bar(kBarAFull + x));
                const float m_eff = m_used == -INFINITY ? 0.f : m_used;
                const f2 me2 = mk2(m_eff, m_eff);
                f2 ls[4] = {mk2(0.f, 0.f), mk2(0.f, 0.f), mk2(0.f, 0.f), mk2(0.f, 0.f)};
#pragma unroll
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float a0, a1;
                        split2(sub2(mk2(xv[c0 + 2 * e], xv[c0 + 2 * e + 1]), me2), a0, a1);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        ls[e & 3] = add2(ls[e & 3], mk2(p0, p1));
                        pk[e] = pack_bf16(p0, p1);
                    }
                    tmem_st16(tS + c0 / 2, pk);
                }
                {
                    const f2 tt = add2(add2(ls[0], ls[1]), add2(ls[2], ls[3]));
                    float t0, t1;
                    split2(tt, t0, t1);
                    l = l * alpha + (t0 + t1);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + x));
                __syncwarp();
                if (lane == 0) mbar_arrive_cnt(bar(kBarIdxEmpty + ridx), idx_arrivals);  // done with the metadata
            }
            if (!ok) break;
            // the pass's row sum for the correction warps' epilogue, and lse
            stats_sm[((p & 1) * 2 + x) * kRowsPerTile + r] = l;
            mbar_arrive(bar(kBarStats + 2 * x + (p & 1)));
            if (a.lse && i < a.S)
                a.lse[((int64_t)g.b * a.H + g.h * a.G + 2 * p + x) * a.S + i] =
                    l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
        }
    }

    if (threadIdx.x == 0 && *abort_flag) set_status(a.status, DMA_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc<512>(*tmem_slot);
}

template <int D>
cudaError_t launch_typed(const void* Q, const void* K, const void* V, int B, int S, int H, int Hkv,
                         const float* scores, const dma_kept_t* kept, float scale, void* O, float* lse, int* status,
                         uint64_t wait_ns, int fault_mode, cudaStream_t st)
{
    TcArgs a;
    const int drop_arrive = fault_mode == DMA_FAULT_DROP_ARRIVE ? 1 : 0;
    a.Q = static_cast<const __nv_bfloat16*>(Q);
    a.K = static_cast<const __nv_bfloat16*>(K);
    a.V = static_cast<const __nv_bfloat16*>(V);
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
    const bool fault_test = wait_ns != kDefaultWaitNs || drop_arrive;
    auto kernel = fault_test ? prefill_tc_kernel<D, true> : prefill_tc_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)kept->n_qt * B * Hkv;
    kernel<<<(unsigned)grid, kTcThreads, smem, st>>>(a, wait_ns, drop_arrive);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(dma_dtype_t dt, int B, int S, int H, int Hkv, int D)
{
    (void)B;
    (void)S;
    (void)H;
    (void)Hkv;
    return dt == DMA_BF16 && (D == 64 || D == 128);
}

cudaError_t launch_prefill_tc(const void* Q, const void* K, const void* V, int B, int S, int H, int Hkv, int D,
                              const float* scores, const dma_kept_t* kept, float scale, void* O, float* lse,
                              int* status, uint64_t wait_ns, int fault_mode, cudaStream_t st)
{
    if (D == 128)
        return launch_typed<128>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, status, wait_ns, fault_mode, st);
    return launch_typed<64>(Q, K, V, B, S, H, Hkv, scores, kept, scale, O, lse, status, wait_ns, fault_mode, st);
}

}  // namespace dma
