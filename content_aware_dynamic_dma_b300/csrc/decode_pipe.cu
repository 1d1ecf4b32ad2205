// Sparse attention decode, bf16: a pipelined split-K kernel over the kept rows.
//
// Dynamic Mask Attention summary (lsdiaocha.cn), §七: the full KV cache stays
// resident and only the selection changes; row L-1 of a cache of length L
// attends to the top set of that row united with the window {L-window .. L-1}.
// Skipped rows are never read (§四).
//
// HBM-bound: the algorithmic traffic is 2 * D * 2 bytes of K and V per kept row
// per KV head.  One CTA takes a contiguous part of one (sequence, KV head)
// kept list and walks it in stages of 64 keys.  All four warps gather the K and
// V rows of a stage with 16-byte cp.async copies (a TMA tile::gather4 moves only
// about 8 bytes per cycle per SM, a quarter of what these row gathers need),
// three stages in flight, into a 128-byte-swizzled layout.  Each warp then
// takes 16 keys of the stage: logits of all G = H / Hkv query heads of the
// group with mma.sync (query heads padded to 16 rows, keys as the 8-wide N
// dimension), an online softmax in the log2 domain in registers, and
// O += P V with P taken straight from the logit accumulators.  The warps'
// partial results are merged in shared memory and written as one
// (max, sum, O) partial per (sequence, query head, split); a second kernel
// merges the splits by log-sum-exp.
#include <algorithm>
#include <cmath>

#include "dma_internal.cuh"
#include "tc_primitives.cuh"

namespace dma {
namespace {

using namespace tc;

constexpr int kStageKeys = 64;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kMaxSplitKeys = 8192;  // longest key list of one split (32 KB of shared memory)
constexpr int kPipeThreads = kConsumerWarps * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct PipeLayout {
    static constexpr int kTile = kStageKeys * D * 2;    // K or V rows of one stage
    static constexpr int kStage = 2 * kTile;            // K then V
    static constexpr int kBias = kStages * kStage;      // [stage][64] f32
    static constexpr int kMerge = 0;  // [warp][16][D + 2] f32, over the stages once the pipeline is drained
    static_assert(kConsumerWarps * 16 * (D + 2) * 4 <= kBias, "merge area must fit in the stages");
    static constexpr int kKeys = kBias + kStages * kStageKeys * 4;  // the split's key list (runtime length)
    // bytes of shared memory for a split of at most `max_keys` keys, then (paged cache) the
    // sequence's `bt_entries` block-table entries (1024 of slack for alignment)
    static constexpr int smem_bytes(int max_keys, int bt_entries = 0) { return kKeys + (max_keys + bt_entries) * 4 + 1024; }
};

struct PipeArgs {
    const __nv_bfloat16* q;     // [B][H][D]
    const int32_t* cache_len;   // [B] or null
    const float* scores;        // [B][Hkv][Lmax]
    const int32_t* top_idx;     // [B][Hkv][top_cap]
    const int32_t* top_count;   // [B][Hkv]
    float* part_o;              // [B * H][nsplit][D]
    float* part_ml;             // [B * H][nsplit][2]  (max in log2 units, sum)
    int B, Lmax, H, Hkv, G, top_cap, window, nsplit;
    float c_log2;               // scale * log2(e)
    // paged cache: K/V pages [n_pages][1 << pshift][Hkv][D], block_table [B][max_pages]
    const int32_t* block_table;
    int n_pages, max_pages, pshift;
    int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D (16x8, f32) += A (16x16, bf16, row) * B (16x8, bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk `chunk` (8 elements) of row r in a
// 128-byte-swizzled tile of 64 rows.
__device__ __forceinline__ uint32_t sw_off(int r, int chunk)
{
    return (uint32_t)((chunk >> 3) * (kStageKeys * 128) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

// Entry u of the (sequence, KV head) list: top-set keys outside the window,
// then the window band; -1 for an entry that contributes nothing.
__device__ __forceinline__ int list_key(int u, const int32_t* top, int n_top, int L, int window)
{
    if (u < n_top) {
        const int j = top[u];
        return (j >= 0 && j < L - window && j <= L - 1) ? j : -1;
    }
    const int j = L - window + (u - n_top);
    return (j >= 0 && j <= L - 1) ? j : -1;
}

// kPaged: Kc and Vc are K/V pages; key j of sequence b is row
// (block_table[b][j >> pshift] << pshift) + (j & (page size - 1)) of them.
template <int D, bool kPaged>
__global__ void __launch_bounds__(kPipeThreads, 2) decode_pipe_kernel(const __nv_bfloat16* __restrict__ Kc,
                                                                      const __nv_bfloat16* __restrict__ Vc,
                                                                      const PipeArgs a)
{
    using L_ = PipeLayout<D>;
    constexpr int kNT = D / 8;       // 8-wide output tiles
    constexpr int kCPR = D / 8;      // 16-byte chunks per row
    constexpr int kRowsPerPass = kPipeThreads / kCPR;  // rows covered by one sweep of the CTA
    constexpr int kSweeps = kStageKeys / kRowsPerPass;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base, by pointer arithmetic so that accesses through it stay ld/st.shared
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    float* bias_s = reinterpret_cast<float*>(sm + L_::kBias);
    float* merge_s = reinterpret_cast<float*>(sm + L_::kMerge);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The merge kernel may be scheduled once every CTA of this grid has started; it waits for
    // this grid's completion (and its memory) before reading the partials.
    asm volatile("griddepcontrol.launch_dependents;");
    const int seg = blockIdx.y, split = blockIdx.x;
    const int b = seg / a.Hkv, h = seg % a.Hkv;
    const int G = a.G;
    // cache lengths outside [1, Lmax] are clamped so that no row outside the cache is read
    const int L = a.cache_len ? min(max(a.cache_len[b], 1), a.Lmax) : a.Lmax;
    const int n_top = min(max(a.top_count[seg], 0), a.top_cap);
    const int n_all = n_top + a.window;
    // the list's stages of 64 keys, shared out evenly: split s takes stages
    // [s * n / nsplit, (s + 1) * n / nsplit)
    const int nst_all = (n_all + kStageKeys - 1) / kStageKeys;
    const int st_begin = (int)((int64_t)split * nst_all / a.nsplit);
    const int st_end = (int)((int64_t)(split + 1) * nst_all / a.nsplit);
    const int u_begin = min(n_all, st_begin * kStageKeys), u_end = min(n_all, st_end * kStageKeys);
    const int nst = st_end - st_begin;
    const int32_t* top = a.top_idx + (int64_t)seg * a.top_cap;
    const float* sc = a.scores + (int64_t)seg * a.Lmax;
    const int64_t row_stride = (int64_t)a.Hkv * D;
    const __nv_bfloat16* Kh = Kc + (kPaged ? (int64_t)h * D : ((int64_t)b * a.Lmax * a.Hkv + h) * D);
    const __nv_bfloat16* Vh = Vc + (kPaged ? (int64_t)h * D : ((int64_t)b * a.Lmax * a.Hkv + h) * D);

    // Key indices: the whole split's key list is read into shared memory once, before the first
    // copies (a per-stage index load would put its latency into every stage); the copies (chunk
    // `part` of rows r0 + kRowsPerPass * m of a stage) read their row indices from there.
    int* keys_s = reinterpret_cast<int*>(sm + L_::kKeys);
    const int n_keys = u_end - u_begin;
    for (int i = threadIdx.x; i < n_keys; i += kPipeThreads)
        keys_s[i] = list_key(u_begin + i, top, n_top, L, a.window);
    // paged cache: the sequence's block-table entries for pages 0 .. (L - 1) >> pshift (an entry
    // outside [0, n_pages) marks its page's rows as unreadable: recorded, and read as zeros)
    int* bt_s = keys_s + n_keys;
    if constexpr (kPaged) {
        const int n_pg = ((L - 1) >> a.pshift) + 1;
        for (int i = threadIdx.x; i < n_pg; i += kPipeThreads) {
            int phys = a.block_table[(int64_t)b * a.max_pages + i];
            if (phys < 0 || phys >= a.n_pages) {
                set_status(a.status, DMA_ERR_DEVICE_CHECK);
                phys = -1;
            }
            bt_s[i] = phys;
        }
    }
    // the row of key j in Kh / Vh, or -1
    auto key_row = [&](int j) -> int64_t {
        if constexpr (kPaged) {
            if (j < 0) return -1;
            const int phys = bt_s[j >> a.pshift];
            return phys < 0 ? -1 : ((int64_t)phys << a.pshift) + (j & ((1 << a.pshift) - 1));
        } else {
            return j;
        }
    };
    const int part = threadIdx.x % kCPR, r0 = threadIdx.x / kCPR;
    auto key_at = [&](int st, int r) -> int {
        const int i = st * kStageKeys + r;
        return i < n_keys ? keys_s[i] : -1;
    };
    auto issue = [&](int st) {
        if (st < nst) {
            const int s = st % kStages;
            const uint32_t kt = sbase + s * L_::kStage, vt = kt + L_::kTile;
#pragma unroll
            for (int m = 0; m < kSweeps; ++m) {
                const int r = r0 + kRowsPerPass * m;
                const int64_t row = key_row(key_at(st, r));
                const bool ok = row >= 0;
                const int64_t off = (ok ? row : 0) * row_stride + part * 8;
                cp_async16(kt + sw_off(r, part), Kh + off, ok);
                cp_async16(vt + sw_off(r, part), Vh + off, ok);
            }
            if (threadIdx.x < kStageKeys) {
                const int j = key_at(st, threadIdx.x);
                float* bd = bias_s + s * kStageKeys + threadIdx.x;
                if (j >= 0)
                    cp_async4(smem_u32(bd), sc + j);
                else
                    *bd = -INFINITY;
            }
        }
        cp_async_commit();  // one group per stage slot, possibly empty, so the group count stays uniform
    };

    const int g = lane >> 2, t = lane & 3;
    // query fragments (A operand, heads as rows): rows g and g + 8, dims 16 kk + 2 t (+1, +8, +9)
    uint32_t qa[D / 16][4];
    {
        const __nv_bfloat16* qb = a.q + ((int64_t)b * a.H + (int64_t)h * G) * D;
        auto qv = [&](int row, int d) -> uint32_t {
            if (row >= G) return 0u;
            return *reinterpret_cast<const uint32_t*>(qb + (int64_t)row * D + d);
        };
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa[kk][0] = qv(g, 16 * kk + 2 * t);
            qa[kk][1] = qv(g + 8, 16 * kk + 2 * t);
            qa[kk][2] = qv(g, 16 * kk + 2 * t + 8);
            qa[kk][3] = qv(g + 8, 16 * kk + 2 * t + 8);
        }
    }
    float o[kNT][4];
#pragma unroll
    for (int n = 0; n < kNT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads g, g + 8
    const int kr = 16 * warp;  // this warp's 16 keys of each stage

    __syncthreads();  // the key list is in shared memory
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) issue(st);
    for (int st = 0; st < nst; ++st) {
        cp_async_wait<kStages - 2>();  // this thread's copies of stage st have landed
        __syncthreads();               // everyone's have; everyone is done with stage st - 1
        issue(st + kStages - 1);       // into the slot of stage st - 1
        const int s = st % kStages;
        const uint32_t kt = sbase + s * L_::kStage, vt = kt + L_::kTile;
        // logits: two 8-key tiles
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        {
            // even and odd k-steps in separate accumulators: two short dependency chains
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            const int mi = lane >> 3, ri = lane & 7;
            const int key = kr + 8 * (mi >> 1) + ri;
#pragma unroll
            for (int kk = 0; kk < D / 16; kk += 2) {
                uint32_t b0, b1, b2, b3, e0, e1, e2, e3;
                ldsm_x4(kt + sw_off(key, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                ldsm_x4(kt + sw_off(key, 2 * kk + 2 + (mi & 1)), e0, e1, e2, e3);
                mma16816(c0, qa[kk], b0, b1);
                mma16816(c1, qa[kk], b2, b3);
                mma16816(d0, qa[kk + 1], e0, e1);
                mma16816(d1, qa[kk + 1], e2, e3);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                c0[e] += d0[e];
                c1[e] += d1[e];
            }
        }
        const float* bs = bias_s + s * kStageKeys + kr;
        const float bb0 = bs[2 * t], bb1 = bs[2 * t + 1], bb2 = bs[8 + 2 * t], bb3 = bs[8 + 2 * t + 1];
        // x for head g: c0[0], c0[1], c1[0], c1[1]; head g + 8: c0[2], c0[3], c1[2], c1[3]
        float x0 = fmaf(c0[0], a.c_log2, bb0 * kLog2e), x1 = fmaf(c0[1], a.c_log2, bb1 * kLog2e);
        float x2 = fmaf(c1[0], a.c_log2, bb2 * kLog2e), x3 = fmaf(c1[1], a.c_log2, bb3 * kLog2e);
        float y0 = fmaf(c0[2], a.c_log2, bb0 * kLog2e), y1 = fmaf(c0[3], a.c_log2, bb1 * kLog2e);
        float y2 = fmaf(c1[2], a.c_log2, bb2 * kLog2e), y3 = fmaf(c1[3], a.c_log2, bb3 * kLog2e);
        float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3)), my = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
        my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
        const float mn0 = fmaxf(m0, mx), mn1 = fmaxf(m1, my);
        const float e0 = mn0 == -INFINITY ? 0.f : mn0, e1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = ex2(m0 - e0), al1 = ex2(m1 - e1);  // 0 while nothing was kept
        m0 = mn0;
        m1 = mn1;
        x0 = ex2(x0 - e0);
        x1 = ex2(x1 - e0);
        x2 = ex2(x2 - e0);
        x3 = ex2(x3 - e0);
        y0 = ex2(y0 - e1);
        y1 = ex2(y1 - e1);
        y2 = ex2(y2 - e1);
        y3 = ex2(y3 - e1);
        float s0 = (x0 + x1) + (x2 + x3), s1 = (y0 + y1) + (y2 + y3);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        l0 = l0 * al0 + s0;
        l1 = l1 * al1 + s1;
        const uint32_t pa[4] = {pack_bf16(x0, x1), pack_bf16(y0, y1), pack_bf16(x2, x3), pack_bf16(y2, y3)};
        // O += P V: V fragments by transposed 8x8 loads, two 8-wide output tiles per load
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int key = kr + 8 * (mi & 1) + ri;
#pragma unroll
            for (int n = 0; n < kNT; n += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt + sw_off(key, n + (mi >> 1)), b0, b1, b2, b3);
                o[n][0] *= al0;
                o[n][1] *= al0;
                o[n][2] *= al1;
                o[n][3] *= al1;
                o[n + 1][0] *= al0;
                o[n + 1][1] *= al0;
                o[n + 1][2] *= al1;
                o[n + 1][3] *= al1;
                mma16816(o[n], pa, b0, b1);
                mma16816(o[n + 1], pa, b2, b3);
            }
        }
    }
    cp_async_wait<0>();
    // every warp is done with the stages before they are reused for the merge
    __syncthreads();
    {
        float* mw = merge_s + warp * 16 * (D + 2);
        if (t == 0) {
            mw[g * (D + 2) + D] = m0;
            mw[g * (D + 2) + D + 1] = l0;
            mw[(g + 8) * (D + 2) + D] = m1;
            mw[(g + 8) * (D + 2) + D + 1] = l1;
        }
#pragma unroll
        for (int n = 0; n < kNT; ++n) {
            mw[g * (D + 2) + 8 * n + 2 * t] = o[n][0];
            mw[g * (D + 2) + 8 * n + 2 * t + 1] = o[n][1];
            mw[(g + 8) * (D + 2) + 8 * n + 2 * t] = o[n][2];
            mw[(g + 8) * (D + 2) + 8 * n + 2 * t + 1] = o[n][3];
        }
    }
    __syncthreads();
    // merge the warps and write this split's partial for each query head
    for (int e = threadIdx.x; e < G * (D + 2); e += kPipeThreads) {
        const int hg = e / (D + 2), c = e % (D + 2);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, merge_s[(w * 16 + hg) * (D + 2) + D]);
        float acc = 0.f;
        if (M != -INFINITY) {
            const int cc = c == D ? D + 1 : c;  // the max slot merges the sums
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = merge_s[(w * 16 + hg) * (D + 2) + D];
                if (mw != -INFINITY) acc = fmaf(merge_s[(w * 16 + hg) * (D + 2) + cc], ex2(mw - M), acc);
            }
        }
        const int64_t pi = ((int64_t)b * a.H + (int64_t)h * G + hg) * a.nsplit + split;
        if (c < D)
            a.part_o[pi * D + c] = acc;
        else if (c == D)
            a.part_ml[pi * 2 + 1] = acc;
        else
            a.part_ml[pi * 2] = M;
    }
}

template <int D>
__global__ void __launch_bounds__(D) decode_pipe_merge_kernel(int nsplit, const float* __restrict__ part_o,
                                                              const float* __restrict__ part_ml,
                                                              __nv_bfloat16* __restrict__ o, float* __restrict__ lse)
{
    // launched as a programmatic dependent of the partial kernel: wait until that grid has
    // completed and its writes are visible (returns at once without such a dependency)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int bh = blockIdx.x, d = threadIdx.x;
    const float* ml = part_ml + (int64_t)bh * nsplit * 2;
    float M = -INFINITY;
    for (int c = 0; c < nsplit; ++c) M = fmaxf(M, ml[2 * c]);
    float Ls = 0.f, acc = 0.f;
    if (M != -INFINITY) {
        for (int c = 0; c < nsplit; ++c) {
            const float mc = ml[2 * c];
            if (mc == -INFINITY) continue;
            const float wgt = ex2(mc - M);
            Ls = fmaf(ml[2 * c + 1], wgt, Ls);
            acc = fmaf(part_o[((int64_t)bh * nsplit + c) * D + d], wgt, acc);
        }
    }
    o[(int64_t)bh * D + d] = __float2bfloat16_rn(Ls > 0.f ? acc / Ls : 0.f);
    if (lse && d == 0) lse[bh] = Ls > 0.f ? (M + __log2f(Ls)) * kLn2 : -INFINITY;
}

// The kept lists and, for a paged cache, its geometry (block_table null: contiguous cache).
struct PipeLists {
    const int32_t* top_idx;
    const int32_t* top_count;
    int top_cap, window;
    const int32_t* block_table;
    int n_pages, max_pages, pshift;
};

template <int D>
cudaError_t launch_typed(const void* q, const void* Kc, const void* Vc, int B, int Lmax, const int32_t* cache_len,
                         int H, int Hkv, const float* scores, const PipeLists& kl, float scale, void* o,
                         float* lse, void* ws, int nsplit, int* status, cudaStream_t st)
{
    PipeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.cache_len = cache_len;
    a.scores = scores;
    a.top_idx = kl.top_idx;
    a.top_count = kl.top_count;
    a.part_o = static_cast<float*>(ws);
    a.part_ml = a.part_o + (size_t)B * H * nsplit * D;
    a.B = B;
    a.Lmax = Lmax;
    a.H = H;
    a.Hkv = Hkv;
    a.G = H / Hkv;
    a.top_cap = kl.top_cap;
    a.window = kl.window;
    a.nsplit = nsplit;
    a.c_log2 = scale * kLog2e;
    a.block_table = kl.block_table;
    a.n_pages = kl.n_pages;
    a.max_pages = kl.max_pages;
    a.pshift = kl.pshift;
    a.status = status;
    const bool paged = kl.block_table != nullptr;
    // the longest split's key list: ceil(stages / nsplit) stages of 64 keys
    const int max_stages = std::max(1, (kl.top_cap + kl.window + kStageKeys - 1) / kStageKeys);
    const int smem = PipeLayout<D>::smem_bytes(((max_stages + nsplit - 1) / nsplit) * kStageKeys,
                                               paged ? kl.max_pages : 0);
    auto kernel = paged ? decode_pipe_kernel<D, true> : decode_pipe_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3(nsplit, B * Hkv), kPipeThreads, smem, st>>>(static_cast<const __nv_bfloat16*>(Kc),
                                                              static_cast<const __nv_bfloat16*>(Vc), a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the merge launches while the partial kernel's last wave runs (programmatic dependent
    // launch), so the gap between the two kernels is hidden
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B * H);
    cfg.blockDim = dim3(D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_pipe_merge_kernel<D>, nsplit, static_cast<const float*>(a.part_o),
                              static_cast<const float*>(a.part_ml), static_cast<__nv_bfloat16*>(o), lse);
}

cudaError_t launch_lists(const void* q, const void* Kc, const void* Vc, int B, int Lmax, const int32_t* cache_len,
                         int H, int Hkv, int D, const float* scores, const PipeLists& kl, float scale, void* o,
                         float* lse, void* ws, int* status, cudaStream_t st)
{
    // splits: the policy's, or more when a split's key list would not fit its shared-memory bound
    const int max_stages = std::max(1, (kl.top_cap + kl.window + kStageKeys - 1) / kStageKeys);
    const int nsplit = std::max(decode_pipe_splits(B, Hkv, kl.top_cap, kl.window),
                                (max_stages * kStageKeys + kMaxSplitKeys - 1) / kMaxSplitKeys);
    if (D == 128)
        return launch_typed<128>(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, scores, kl, scale, o, lse, ws, nsplit, status,
                                 st);
    return launch_typed<64>(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, scores, kl, scale, o, lse, ws, nsplit, status, st);
}

}  // namespace

bool decode_pipe_supported(dma_dtype_t dt, int B, int Lmax, int H, int Hkv, int D)
{
    return dt == DMA_BF16 && (D == 64 || D == 128) && H / Hkv <= 16 && (int64_t)B * Lmax * Hkv < ((int64_t)1 << 31);
}

// Splits per (sequence, KV head): the fewest that still give about one and a half
// waves of resident CTAs (two per SM).  Every CTA pays for reading its key list
// and for filling and draining its copy pipeline, so fewer, longer CTAs win until
// the grid gets too short to keep the machine busy: on 64 sequences x 8 KV heads
// with lists of 33 stages, 1 split took 0.114 ms, 2 splits 0.118 ms, 4 splits
// 0.120 ms and 6 splits 0.130 ms per step.  Never more than the 64-row stages of
// the longest list (the workspace is sized for that many).
int decode_pipe_splits(int B, int Hkv, int top_cap, int window)
{
    const int max_split = std::max(1, (top_cap + window + 63) / 64);
    const int slots = 2 * 148;
    const int segs = B * Hkv;
    const int want = std::max(1, (3 * slots + 2 * segs - 1) / (2 * segs));  // ceil(1.5 * slots / segs)
    return std::min(max_split, want);
}

cudaError_t launch_decode_pipe(const void* q, const void* Kc, const void* Vc, int B, int Lmax,
                               const int32_t* cache_len, int H, int Hkv, int D, const float* scores,
                               const dma_kept_t* kept, float scale, void* o, float* lse, void* ws, int* status,
                               cudaStream_t st)
{
    const PipeLists kl{kept->top_idx, kept->top_count, kept->top_cap, kept->window, nullptr, 0, 0, 0};
    return launch_lists(q, Kc, Vc, B, Lmax, cache_len, H, Hkv, D, scores, kl, scale, o, lse, ws, status, st);
}

cudaError_t launch_decode_paged(const void* q, const void* Kp, const void* Vp, const int32_t* block_table,
                                int n_pages, int B, int max_pages, int pshift, const int32_t* cache_len, int H,
                                int Hkv, int D, const float* scores, const int32_t* top_idx,
                                const int32_t* top_count, int top_cap, int window, float scale, void* o, float* lse,
                                void* ws, int* status, cudaStream_t st)
{
    const PipeLists kl{top_idx, top_count, top_cap, window, block_table, n_pages, max_pages, pshift};
    return launch_lists(q, Kp, Vp, B, max_pages << pshift, cache_len, H, Hkv, D, scores, kl, scale, o, lse, ws,
                        status, st);
}

}  // namespace dma
