// k_prefill_tc.cu -- causal GQA prefill on the fifth-generation tensor core
// (tcgen05, TMEM accumulators, TMA-staged operands), bf16 in, fp32
// accumulate, d_h = 128.
//
// What it computes ("第二章 Prefill：整层状态演化与 KV 建立", section 2.3):
// for query head h of KV group g = floor(h*H_kv/H_q) and a query row at
// absolute position p, the softmax over the finite scores
// <q, k_j>/sqrt(d_h), j = 0..p, applied to V.  Keys before this call's
// rows come from the paged cache through the block table ("KV Cache 与
// Prefill/Decode 推理路径", PagedAttention), so a prefill over an existing
// prefix (incremental prefill: the old prefix fully visible, the new block
// lower-triangular) and a fresh prefill are the same loop.  This call's own
// rows either were stored by a cache-write launch before this kernel, or
// (fused write, section 2.6's write-then-attend done in one kernel) are read
// from the call's k and v and each new page is stored to the pool by the
// one CTA whose query rows begin on it.
//
// Mapping to the hardware.
//  * A CTA owns two 128-row query tiles of one (batch entry, KV head).  A
//    tile's rows are (position, head) pairs -- 128/g positions times the g
//    query heads of the group -- so one TMA box fills it and every K/V tile
//    staged in shared memory serves all g heads (GQA shares K/V, it is not
//    duplicated; the KV head is indexed).
//  * Key tiles are 128 tokens = 8 pages, aligned to absolute position 0;
//    the CTA visits only tiles that hold a key some of its rows may see:
//    tiles wholly above the diagonal are skipped ("KV Cache 与 Prefill/
//    Decode 推理路径", causal tile skipping).  Diagonal tiles are masked per
//    element.
//  * Warp roles: warps 0 and 3 issue TMA (warp 0 Q once per item and K per
//    key tile, warp 3 V per key tile; one 4 KB box per page block through
//    the block table, eight lanes at once, two stages each); warp 1 owns
//    TMEM and issues the S MMAs, warp 2 the PV MMAs; warpgroups 1 and 2
//    (warps 4-7, 8-11) run the softmax, one per query tile, thread = row.
//  * Persistent: one CTA per SM walks its own run of items, assigned on the
//    host longest-first to the least-loaded CTA; both MMA streams run on
//    across items, so the next item's first S = Q K^T is issued as soon as
//    its Q and K have landed and the S buffer is free.
//  * TMEM (512 columns): S | P0 | P1 | O0 | O1.  S = Q K^T (fp32, 128
//    columns) is computed into a buffer the two query tiles take in turn;
//    the softmax warps read their row of it and release it at once, then
//    write P = exp2(S*c - m) as bf16 into their tile's P columns, and the
//    PV MMA takes P straight from TMEM as its A operand: O += P V.  The S
//    MMAs (one issuing warp) and the PV MMAs (another) form two independent
//    streams; a softmax has about four MMA groups of time before its PV is
//    due.
//  * Online softmax (the FlashAttention recurrence): a running row max m and
//    sum l; O is rescaled in TMEM only when the max grows by more than 2^8,
//    otherwise the stale max stays the reference (exact in real arithmetic).
//  * Epilogue: O / l in fp32 -> bf16, staged per 64-column half in a 16 KB
//    shared-memory buffer per query tile (128-byte swizzle, so the row-per-
//    thread writes are conflict-free) and written by one TMA store per half;
//    padding rows of the tile are written as zeros (with the fused write,
//    padding rows no tile covers are cleared by the producer warps).
// Every wait is bounded; on a timeout the CTA raises GQA_DEVERR_TIMEOUT,
// drains what it has in flight (bounded) and exits cleanly.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <type_traits>
#include <atomic>

#include "kernels.cuh"
#include "sm100.cuh"

namespace gqa {

using namespace sm100;

namespace {

// Every GQA_EXP2_POLY_EVERY-th pair of exponentials is evaluated by a
// polynomial on the FMA pipe instead of the MUFU unit (0 = never), to keep
// the MUFU unit from bounding the softmax.
#ifndef GQA_EXP2_POLY_EVERY
#define GQA_EXP2_POLY_EVERY 0
#endif

constexpr int kPolyEvery = GQA_EXP2_POLY_EVERY > 0 ? GQA_EXP2_POLY_EVERY : 1;
constexpr bool kPoly = GQA_EXP2_POLY_EVERY > 0;
constexpr int D = 128;
// K and V have pipelines of their own: a V stage is held from PV of the
// first query tile to the end of PV of the second, so V wants one stage more
// than K to hide the load latency (about 2 us under full load).
#ifndef GQA_K_STAGES
#define GQA_K_STAGES 2
#endif
#ifndef GQA_V_STAGES
#define GQA_V_STAGES 2
#endif
constexpr int kKStages = GQA_K_STAGES;
#ifndef GQA_PV_ORDER
#define GQA_PV_ORDER 1
#endif
constexpr bool kPvOrder = GQA_PV_ORDER != 0;
// Programmatic dependent launch: the kernel may start while the cache write
// that precedes it finishes; only the K/V loads wait for that grid.
#ifndef GQA_PDL
#define GQA_PDL 1
#endif
constexpr int kVStages = GQA_V_STAGES;
constexpr int kThreads = 384;     // warpgroup 0: TMA + MMA; warpgroups 1, 2: softmax
constexpr uint32_t kTileBytes = 128 * 64 * 2;        // one 128-row x 64-column bf16 half tile
constexpr int kPageElems = kPageTokens * D;           // one page block of one head (4 KB)
// TMEM columns: one S buffer (fp32, 128 keys) shared by the two query tiles,
// P of each tile (bf16 pairs, 64 columns) and O of each tile (fp32, 128).
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;

struct __align__(1024) TcSmem {
    __nv_bfloat16 q[2][2][128 * 64];                   // [query tile][column half]
    __nv_bfloat16 k[kKStages][2][128 * 64];
    __nv_bfloat16 v[kVStages][2][128 * 64];
    __nv_bfloat16 o[2][128 * 64];                      // epilogue staging, one column half per query tile
    uint64_t bar_q, q_empty, q_rot[2];
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t k_land[kKStages], v_land[kVStages];       // Q8: a stage's codes have landed
    uint64_t s_full[2], s_free, p_full[2], pv_done[2], fin[2];
    uint64_t fix_bar[2];                               // fused write: a K (V) tile that needs its tail cleared landed
    uint32_t tmem;
    int abort_;
    int last_;                                         // this CTA completed a split group
    float mrg_m[128], mrg_inv[128];                    // split merge: max and 1 / sum per row
    int s_issued[2];                                   // S MMAs of tile 0 / 1 issued so far (monotonic)
};

static_assert(sizeof(TcSmem) + 1024 <= 227 * 1024, "shared memory per CTA");

struct TcParams {
    const SeqDesc *seqs;
    const TcItem *items;      // grouped by CTA: CTA c takes items[item_start[c] .. item_start[c + 1])
    const int32_t *item_start;
    const int32_t *tables;
    void *pool;               // page pool (bf16), for the appended rows below
    int32_t stride;
    int32_t num_pages;
    int32_t H_kv;
    int32_t H_q;
    int32_t n;          // padded rows per batch entry
    int32_t G;          // query heads per KV head
    int32_t rows_pos;   // positions per query tile (128 / G)
    __nv_bfloat16 *out; // [B, n, H_q, 128]
    int32_t *err;
    float scale_log2;   // log2(e) / sqrt(d_h)
    const float2 *rope; // rotary (cos, sin) [position][64], or null
    int32_t window;     // sliding window (0 = none)
    float *ws_o;        // split items' partial O, m, l (TcSplitWs)
    float2 *ws_ml;
    int32_t *counters;
    int32_t slot_rows;
    const __nv_bfloat16 *app_k;   // fused append: this call's one new K and V row per entry
    const __nv_bfloat16 *app_v;   // ([B, H_kv, 128]), written at position past; null = none
    const float *scales;          // Q8: per-row scales of the FP8 E4M3 pool (block * 16 + slot)
    int32_t fused;                // 1: rows of this call are read from k / v and written to their pages here
    int32_t B;
    const int64_t *zero_start;    // fused: CTA c clears padding units zero_start[c] .. zero_start[c + 1] - 1
};

// The parameters of a launch that carries its descriptors (the kernel's INL
// form): byte offsets into inl of seqs, items, item_start, zero_start and
// tables (-1: the pointer in TcParams is used).  Only these launches pay
// for the large parameter block.
struct TcParamsInl : TcParams {
    int32_t inl_off[5];
    alignas(16) unsigned char inl[kTcInlineBytes];
};
static_assert(sizeof(TcParamsInl) + 7 * sizeof(CUtensorMap) <= 32764, "kernel parameter space");

// Two FP8 E4M3 codes (low byte first) dequantised with their row's scale:
// decode (exact, through f16), times the scale in fp32, rounded to a bf16
// pair for the tensor cores.
__device__ __forceinline__ uint32_t e4m3x2_bf16x2(uint32_t pair, float2 sc)
{
    const float2 f =
        __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(pair & 0xffffu), __NV_E4M3)));
    const float2 x = fma2(f, sc, make_float2(0.f, 0.f));
    return pack_bf16x2(x.x, x.y);
}

__device__ __forceinline__ void abort_with(TcSmem &s, int32_t *err, int32_t bit)
{
    s.abort_ = 1;
    atomicOr(err, bit);
}

// Persistent: CTA c takes the host-assigned run of items item_start[c] ..
// item_start[c + 1] - 1 in order.  Barrier phases run on
// across items (global tile counter gt), so the next item's Q and first K/V
// tile load while the current item's last tiles and epilogue run.
// ROPE: queries rotated in-kernel (p.rope is the table); WIN: items may start
// past key tile 0 (a sliding window, whose keys before the window are
// masked, or split items); Q8: the pool holds FP8 E4M3 codes with a scale
// per row (mKV then maps the code bytes).  All are template flags so the
// plain path carries none of their instructions.
template <bool ROPE, bool WIN, bool Q8, bool INL = false>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKV,
                  const __grid_constant__ CUtensorMap mO, const __grid_constant__ CUtensorMap mKt,
                  const __grid_constant__ CUtensorMap mVt, const __grid_constant__ CUtensorMap mKp,
                  const __grid_constant__ CUtensorMap mVp,
                  const __grid_constant__ typename std::conditional<INL, TcParamsInl, TcParams>::type p)
{
    extern __shared__ unsigned char smem_raw[];
    TcSmem &s = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The descriptors, from the parameters when the launch carries them.
    auto inl_or = [&](int which, const void *ptr) -> const void * {
        if constexpr (INL)
            return p.inl_off[which] >= 0 ? static_cast<const void *>(p.inl + p.inl_off[which]) : ptr;
        else
            return ptr;
    };
    const SeqDesc *seqs = static_cast<const SeqDesc *>(inl_or(0, p.seqs));
    const TcItem *items = static_cast<const TcItem *>(inl_or(1, p.items));
    const int32_t *item_start = static_cast<const int32_t *>(inl_or(2, p.item_start));
    const int64_t *zero_start = static_cast<const int64_t *>(inl_or(3, p.zero_start));
    const int32_t *tables = static_cast<const int32_t *>(inl_or(4, p.tables));
    const int i_begin = item_start[blockIdx.x], i_end = item_start[blockIdx.x + 1];

    if (warp == 1) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    // Rows G*rows_pos..127 of each query tile are never written by the Q box
    // (G not dividing 128); zero them once so they hold finite values.
    {
        const int box_rows = p.G * p.rows_pos;
        const int extra = (128 - box_rows) * 128 / 16;  // 16-byte units per tile half
        for (int u = threadIdx.x; u < 4 * extra; u += blockDim.x) {
            const int th = u / extra, r = u % extra;    // th = tile * 2 + half
            reinterpret_cast<uint4 *>(s.q[th >> 1][th & 1] + box_rows * 64)[r] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        s.abort_ = 0;
        s.s_issued[0] = s.s_issued[1] = 0;
        mbar_init(&s.bar_q, 1);
        mbar_init(&s.q_rot[0], 4);                     // rotary: a tile's 4 softmax warps, per item
        mbar_init(&s.q_rot[1], 4);
        mbar_init(&s.q_empty, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.k_empty[i], 1);
            mbar_init(&s.k_land[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.v_empty[i], 1);
            mbar_init(&s.v_land[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s.s_full[t], 1);
            mbar_init(&s.p_full[t], 4);
            mbar_init(&s.pv_done[t], 1);
        }
        mbar_init(&s.s_free, 4);
        mbar_init(&s.fin[0], 1);
        mbar_init(&s.fin[1], 1);
        mbar_init(&s.fix_bar[0], 1);
        mbar_init(&s.fix_bar[1], 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s.tmem;

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------------------ TMA producers
        // Warp 0 loads Q and K, warp 3 loads V: with one producer a V stage
        // that frees late held up the next K tile behind it.  Each is a
        // whole warp: lane 0 keeps the barriers, and a tile's copies are
        // issued one per lane, 8 at once, one 4 KB box per page block (a
        // page block of one head holds the tile's 16 rows in operand order;
        // the TMA engine's cost is mostly per box).
        const bool vside = warp == 3;
        if (lane == 0) {
            if (!vside)
                prefetch_tmap(&mQ);
            prefetch_tmap(&mKV);
            if (p.fused) {
                prefetch_tmap(vside ? &mVt : &mKt);
                prefetch_tmap(vside ? &mVp : &mKp);
            }
        }
        const int stages = vside ? kVStages : kKStages;
        const uint32_t q_bytes = 2u * 2u * (uint32_t)(p.G * p.rows_pos) * 64u * 2u;
        const int my_pg = lane & 7;
        const bool boxer = lane < 8;
        const int blk_page = 2 * p.H_kv;                  // blocks per page
        uint32_t gt = 0;                                  // tiles issued so far by this warp
        int k = 0, q_issued = 0;
        bool ok = true;
        // Lane 0 waits; the warp learns the outcome from it.
        auto wait0 = [&](uint64_t *bar, uint32_t parity) -> bool {
            int w = 1;
            if (lane == 0)
                w = mbar_wait(bar, parity, &s.abort_) ? 1 : 0;
            return __shfl_sync(0xffffffffu, w, 0) != 0;
        };
        auto load_q = [&](const TcItem &it) {
            if (lane == 0)
                mbar_arrive_expect_tx(&s.bar_q, q_bytes);
            __syncwarp();
            if (lane < 4)                                 // lane = query tile * 2 + column half
                tma_load_4d(&mQ, &s.bar_q, s.q[lane >> 1][lane & 1], 64 * (lane & 1), it.kvh * p.G,
                            it.i0 + (lane >> 1) * p.rows_pos, it.b);
        };
        // Fused append (decode, count = 1): the warp writes this call's K
        // (warp 0) or V (warp 3) row of head kvh at position past into its
        // page slot, with the rotation of the cache write for K under ROPE
        // (pairs (e, e + 64) rotated by the position, each product, sum and
        // difference rounded to fp32), then orders the writes before the
        // TMA load that reads them.  Lane l holds elements 4l .. 4l + 3.
        auto append_row = [&](const TcItem &it, const SeqDesc &sd) {
            const int pos = sd.past;
            const int pg = tables[(size_t)sd.row * p.stride + pos / kPageTokens];
            if (pg < 0 || pg >= p.num_pages) {
                if (lane == 0)
                    atomicOr(p.err, kErrPageId);
                return;
            }
            const __nv_bfloat16 *src = (vside ? p.app_v : p.app_k) + ((size_t)it.b * p.H_kv + it.kvh) * D;
            uint2 val = reinterpret_cast<const uint2 *>(src)[lane];
            if (ROPE && !vside) {
                uint2 oth;
                oth.x = __shfl_xor_sync(0xffffffffu, val.x, 16);
                oth.y = __shfl_xor_sync(0xffffffffu, val.y, 16);
                const bool first = lane < 16;            // elements < 64: the x of each pair
                const float2 *cs = p.rope + (size_t)pos * (D / 2) + 4 * (lane & 15);
                const __nv_bfloat16 *a = reinterpret_cast<const __nv_bfloat16 *>(&val);
                const __nv_bfloat16 *b2 = reinterpret_cast<const __nv_bfloat16 *>(&oth);
                uint2 res;
                __nv_bfloat16 *rr = reinterpret_cast<__nv_bfloat16 *>(&res);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = __bfloat162float(first ? a[e] : b2[e]);
                    const float y = __bfloat162float(first ? b2[e] : a[e]);
                    const float2 tcs = __ldg(cs + e);
                    const float o = first ? __fsub_rn(__fmul_rn(x, tcs.x), __fmul_rn(y, tcs.y))
                                          : __fadd_rn(__fmul_rn(x, tcs.y), __fmul_rn(y, tcs.x));
                    rr[e] = __float2bfloat16_rn(o);
                }
                val = res;
            }
            const int slot = pos & (kPageTokens - 1), bo = lane * 8;
            char *blk = reinterpret_cast<char *>(p.pool) +
                        ((size_t)(pg * 2 + (vside ? 1 : 0)) * p.H_kv + it.kvh) * (size_t)(kPageElems * 2);
            *reinterpret_cast<uint2 *>(blk + (((slot >> 3) * 2 + (bo >> 7)) << 10) + ((slot & 7) << 7) + (bo & 127)) = val;
            fence_proxy_async_global();
            __syncwarp();
        };
        // Q8: the codes of a stage's 8 page blocks land in its upper half
        // (block pg at byte 16384 + 2048 pg: [16 rows][128 codes]); the warp
        // rewrites the stage in place as the bf16 operand (block pg at 4096 pg:
        // [8-row group][column half][8 rows][64 elements], 128-byte rows with
        // the 16-byte chunks swizzled by row), each code dequantised with its
        // row's scale (fp32 product, rounded to bf16).  Block pg's output
        // overlaps only blocks below pg and its own input, which the warp has
        // read in full before it writes.  Then the stage is marked full.
        // The scales of the lane's row in each of the tile's 8 pages are
        // loaded when the tile is issued, so they are in registers by the
        // time the tile is converted.
        bool pending = false;                             // Q8: a landed tile still to convert
        int pend_st = 0;
        uint32_t pend_use = 0;
        float pend_sc[8];
        auto convert = [&](int st, uint32_t use, const float (&scl)[8]) -> bool {
            if (!wait0(vside ? &s.v_land[st] : &s.k_land[st], use & 1))
                return false;
            unsigned char *base = reinterpret_cast<unsigned char *>(vside ? s.v[st][0] : s.k[st][0]);
            const int r = lane >> 1, h = lane & 1;        // this lane's row (slot) and column half
#pragma unroll
            for (int pg = 0; pg < 8; ++pg) {
                const float2 sc2 = make_float2(scl[pg], scl[pg]);
                const uint4 *src = reinterpret_cast<const uint4 *>(base + 16384 + 2048 * pg + r * 128 + h * 64);
                uint4 c4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    c4[i] = src[i];
                __syncwarp();
                unsigned char *dst = base + 4096 * pg + (r >> 3) * 2048 + h * 1024 + (r & 7) * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {             // chunk c: elements 8c .. 8c + 7 of the half
                    const uint32_t w0 = (c & 1) ? c4[c >> 1].z : c4[c >> 1].x;
                    const uint32_t w1 = (c & 1) ? c4[c >> 1].w : c4[c >> 1].y;
                    uint4 o;
                    o.x = e4m3x2_bf16x2(w0, sc2);
                    o.y = e4m3x2_bf16x2(w0 >> 16, sc2);
                    o.z = e4m3x2_bf16x2(w1, sc2);
                    o.w = e4m3x2_bf16x2(w1 >> 16, sc2);
                    *reinterpret_cast<uint4 *>(dst + ((c ^ (r & 7)) << 4)) = o;
                }
                __syncwarp();
            }
            fence_proxy_async_smem();                     // the MMA reads the stage through the async proxy
            __syncwarp();
            if (lane == 0)
                mbar_arrive(vside ? &s.v_full[st] : &s.k_full[st]);
            return true;
        };
        // Fused calls: the padding rows of out that no item stores (rows
        // zero_from .. n-1 of each entry, all heads) are cleared by the two
        // producer warps once their loads are issued; the host gives the
        // least-loaded CTAs the largest shares.
        const int64_t row_units = (int64_t)p.H_q * (D * 2 / 16);   // 16-byte units of one output row
        int64_t z_next = 0, z_end = 0, zb_start = 0, zb_end = 0;
        int zb = -1;
        uint4 *zb_base = nullptr;                         // out row zero_from of entry zb
        if (p.fused) {
            const int64_t c0 = zero_start[blockIdx.x], c1 = zero_start[blockIdx.x + 1];
            const int64_t mid = c0 + (c1 - c0) / 2;
            z_next = vside ? mid : c0;
            z_end = vside ? c1 : mid;
        }
        auto zero_some = [&](int64_t units) {
            const int64_t stop = min(z_end, z_next + units);
            for (int64_t u = z_next + lane; u < stop; u += 32) {
                // Each lane's units increase: the entry changes rarely.
                while (u >= zb_end) {
                    ++zb;
                    zb_start = zb_end;
                    zb_end = zb_start + (int64_t)(p.n - seqs[zb].zero_from) * row_units;
                    zb_base = reinterpret_cast<uint4 *>(p.out) +
                              ((size_t)zb * p.n + seqs[zb].zero_from) * (size_t)row_units;
                }
                zb_base[u - zb_start] = make_uint4(0, 0, 0, 0);
            }
            z_next = stop;
        };
        // Fused write (p.fused; every entry's past is a multiple of 16, so
        // each page holds old rows only or this call's rows only).  Pages at
        // positions >= past are read from this call's k / v, not from the
        // pool: a tile wholly past `past` as one 32 KB box (mKt / mVt), a
        // tile that straddles it page by page (mKp / mVp for the new pages).
        // Both maps view k / v [B, n, H_kv, 128] as [H_kv][8-row group]
        // [column half][8 rows][64], so a box lands in exactly the layout a
        // page box from the pool lands in.  Rows past the entry's valid
        // length (padding, or the next entry's rows) are cleared in shared
        // memory after landing, before the stage is marked full.  The item
        // whose query rows include a new page's first position owns that
        // page: once the tile has landed (checked when its stage is next
        // refilled) lane pg stores page block pg to the pool with one TMA
        // store, so every new page is written exactly once and no CTA reads
        // a page this launch writes.
        int own_blk[2] = {-1, -1};                        // per stage: pool block this lane stores, or -1
        bool stores_out = false;                          // this lane has bulk stores in flight
        uint32_t fix_uses = 0;
        auto flush_stores = [&](int st, uint32_t parity) -> bool {
            uint64_t *full = vside ? &s.v_full[st] : &s.k_full[st];
            if (!__any_sync(0xffffffffu, own_blk[st] >= 0))
                return true;
            if (!wait0(full, parity))                     // the tile has landed (and been fixed up)
                return false;
            if (own_blk[st] >= 0) {
                const __nv_bfloat16 *src = (vside ? s.v[st][0] : s.k[st][0]) + my_pg * kPageElems;
                tma_store_3d(&mKV, src, 0, 0, own_blk[st]);
                tma_store_commit();
                stores_out = true;
            }
            own_blk[st] = -1;
            return true;
        };
        // Loads this warp's half (K or V) of key tile j of an item into
        // stage gt % stages once its last readers are done.
        auto load_tile = [&](const TcItem &it, const SeqDesc &sd, int j) -> bool {
            const int st = gt % stages;
            const uint32_t use = gt / stages;
            int ph = p.num_pages;                         // out of range: the box reads zeros
            const int seq_pages = (sd.past + sd.count + kPageTokens - 1) / kPageTokens;
            if (boxer) {
                const int lp = 8 * j + my_pg;
                if (lp < seq_pages) {
                    ph = tables[(size_t)sd.row * p.stride + lp];
                    if (ph < 0)                            // released by the sliding window: never visible
                        ph = p.num_pages;
                    else if (ph >= p.num_pages) {
                        if (!vside)
                            atomicOr(p.err, kErrPageId);
                        ph = p.num_pages;
                    }
                }
            }
            uint64_t *empty = vside ? &s.v_empty[st] : &s.k_empty[st];
            uint64_t *full = vside ? &s.v_full[st] : &s.k_full[st];
            __nv_bfloat16 *dst = vside ? s.v[st][0] : s.k[st][0];
            // Q8: the previous tile (landed in the other stage) is converted
            // first, so that its conversion overlaps the MMAs still reading
            // this stage.
            if (Q8 && pending) {
                if (!convert(pend_st, pend_use, pend_sc))
                    return false;
                pending = false;
            }
            // Owned pages of the stage's previous tile go to the pool first;
            // their reads of the stage must end before it is refilled.
            if (!Q8 && p.fused && use > 0 && !flush_stores(st, (use - 1) & 1))
                return false;
            if (use > 0 && !wait0(empty, (use - 1) & 1))
                return false;
            if (!Q8 && p.fused) {
                if (stores_out)
                    tma_store_wait_read();
                stores_out = false;
                __syncwarp();
            }
            if (!Q8 && p.app_k && j == it.nt - 1 && (sd.past >> 7) == j)
                append_row(it, sd);                       // the tile holds this call's new token: write it first
            if (Q8) {
                // Codes (2 KB per page block) into the stage's upper half; the
                // rows' scales are pulled into L1 for the softmax warps.
                uint64_t *land = vside ? &s.v_land[st] : &s.k_land[st];
                if (lane == 0)
                    mbar_arrive_expect_tx(land, kTileBytes);
                __syncwarp();
                const int blk = ph * blk_page + (vside ? p.H_kv : 0) + it.kvh;
                if (boxer) {
                    tma_load_3d(&mKV, land, reinterpret_cast<unsigned char *>(dst) + 16384 + 2048 * my_pg, 0, 0, blk);
                    if (ph < p.num_pages)
                        asm volatile("prefetch.global.L1 [%0];" ::"l"(p.scales + (size_t)blk * kPageTokens));
                }
                ++gt;
                float nsc[8];                             // this tile's scales of row lane / 2
                const int my_blk = boxer && ph < p.num_pages ? blk : -1;
#pragma unroll
                for (int pg = 0; pg < 8; ++pg) {
                    const int b2 = __shfl_sync(0xffffffffu, my_blk, pg);
                    nsc[pg] = b2 >= 0 ? __ldg(p.scales + (size_t)b2 * kPageTokens + (lane >> 1)) : 0.0f;
                }
                pending = true, pend_st = st, pend_use = use;
#pragma unroll
                for (int pg = 0; pg < 8; ++pg)
                    pend_sc[pg] = nsc[pg];
                return true;
            }
            // 0: every page from the pool; 1: the whole tile from k / v;
            // 2: old pages from the pool, new ones from k / v.
            int mode = 0;
            if (p.fused && 128 * (j + 1) > sd.past)
                mode = 128 * j >= sd.past ? 1 : 2;
            const int l_end = sd.past + sd.count;
            const bool fix = mode != 0 && 128 * (j + 1) > l_end;   // rows past the valid length to clear
            uint64_t *bar = fix ? &s.fix_bar[vside ? 1 : 0] : full;
            if (lane == 0)
                mbar_arrive_expect_tx(bar, 2 * kTileBytes);
            __syncwarp();
            const int blk0 = (vside ? p.H_kv : 0) + it.kvh;
            const int grow0 = it.b * p.n - sd.past;      // row of k / v (over all entries) of position 0
            if (mode == 1) {
                if (lane == 0)
                    tma_load_5d(vside ? &mVt : &mKt, bar, dst, 0, 0, 0, (grow0 + 128 * j) >> 3, it.kvh);
            } else if (boxer) {
                const int lp = 8 * j + my_pg;
                if (mode == 2 && 16 * lp >= sd.past && lp < seq_pages)
                    tma_load_5d(vside ? &mVp : &mKp, bar, dst + my_pg * kPageElems, 0, 0, 0, (grow0 + 16 * lp) >> 3,
                                it.kvh);
                else
                    tma_load_3d(&mKV, bar, dst + my_pg * kPageElems, 0, 0, ph * blk_page + blk0);
            }
            if (mode != 0) {
                const int lp = 8 * j + my_pg, r0 = 16 * lp - sd.past;
                own_blk[st] = (boxer && r0 >= 0 && lp < seq_pages && r0 >= it.i0 && r0 < it.i0 + 2 * p.rows_pos &&
                               ph < p.num_pages)
                                  ? ph * blk_page + blk0
                                  : -1;
            }
            if (fix) {
                if (!wait0(&s.fix_bar[vside ? 1 : 0], fix_uses & 1))
                    return false;
                ++fix_uses;
                // Whole rows are cleared, so the 128-byte swizzle inside a
                // row does not matter: row r is slot r % 16 of page block
                // r / 16, its column halves 1 KB apart within the 8-row group.
                unsigned char *base = reinterpret_cast<unsigned char *>(dst);
                const int r_lo = l_end - 128 * j > 0 ? l_end - 128 * j : 0;
                for (int u = r_lo * 16 + lane; u < 128 * 16; u += 32) {
                    const int r = u >> 4, c = u & 15;
                    *reinterpret_cast<uint4 *>(base + (r >> 4) * 4096 + ((r >> 3) & 1) * 2048 + (c >> 3) * 1024 +
                                               (r & 7) * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(full);
            }
            ++gt;                                         // this tile is in flight from here on
            return true;
        };
        // The first item's Q load is issued before the K loop.
        bool first_q_issued = false;
        if (!vside && i_begin < i_end) {
            load_q(items[i_begin]);
            first_q_issued = true;
        }
#if GQA_PDL
        // The pages are written by the preceding cache-write grid: its
        // writes are complete and visible once this returns (at once when
        // no grid precedes).  Q above does not depend on it.
        asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
        for (int idx = i_begin; ok && idx < i_end; ++idx, ++k) {
            const TcItem it = items[idx];
            const SeqDesc sd = seqs[it.b];
            // The first K tile only needs a free stage; issue it before
            // waiting for the previous item to release the Q buffers.
            if (!load_tile(it, sd, WIN ? it.j0 : 0)) {
                ok = false;
                break;
            }
            if (!vside) {
                if (k > 0) {
                    if (!wait0(&s.q_empty, (k - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    load_q(it);
                }
                ++q_issued;
            }
            for (int j = (WIN ? it.j0 : 0) + 1; j < it.nt; ++j) {
                if (!load_tile(it, sd, j)) {
                    ok = false;
                    break;
                }
            }
        }
        if (z_next < z_end)
            zero_some(z_end - z_next);
        // The stages' last tiles: their owned pages go to the pool now.
        if (!Q8 && p.fused && ok) {
            for (uint32_t g = (gt > (uint32_t)stages ? gt - stages : 0); ok && g < gt; ++g)
                ok = flush_stores(g % stages, (g / stages) & 1);
        }
        if (!Q8 && p.fused)
            tma_store_wait_all();                         // every store has completed before the CTA exits
        if (Q8 && ok && pending && !convert(pend_st, pend_use, pend_sc))   // the last tile
            ok = false;
        if (lane == 0) {
            if (!ok)
                abort_with(s, p.err, kErrTimeout);
            // Drain: every issued copy lands before the CTA exits.
            int never = 0;
            for (uint32_t g = (gt > (uint32_t)stages ? gt - stages : 0); g < gt; ++g) {
                uint64_t *full = Q8 ? (vside ? &s.v_land[g % stages] : &s.k_land[g % stages])
                                    : (vside ? &s.v_full[g % stages] : &s.k_full[g % stages]);
                if (!mbar_wait(full, (g / stages) & 1, &never))
                    atomicOr(p.err, kErrTimeout);
            }
            if (first_q_issued && q_issued == 0)
                q_issued = 1;
            if (q_issued > 0 && !mbar_wait(&s.bar_q, (q_issued - 1) & 1, &never))
                atomicOr(p.err, kErrTimeout);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues every S = Q K^T, warp 2 every O += P V.  The two
        // streams depend on each other only through the softmax warps, and
        // a thread issuing MMAs spends most of its time stalled behind the
        // tensor pipe: with both streams queued, one stream's waits and
        // bookkeeping no longer leave the pipe idle.
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S = Q K^T: both K-major
            const uint32_t id_o = idesc_bf16(128, 128, 0, 1);   // O += P V: V is N-major
            // Descriptors are built once; an MMA then costs two adds and the
            // instruction itself.  Q tile t, K stage st and V stage sv start
            // 2 * kTileBytes apart; a column half is kTileBytes further.
            constexpr uint32_t kHalf = kTileBytes >> 4, kStage = 2 * kTileBytes >> 4;
            // Q tile: [column half][128 rows][64], 8-row atoms 1 KB apart.
            // K and V stages: 8 page blocks of 4 KB, each [8-token group]
            // [column half][8 tokens][64]: 8-token atoms 2 KB apart, the
            // second column half 1 KB after the first.
            const uint32_t hi_q = desc_sw128_hi(1024), hi_kv = desc_sw128_hi(2048);
            const uint32_t q_lo = desc_sw128_lo(smem_u32(s.q[0][0]), 16);
            const uint32_t k_lo = desc_sw128_lo(smem_u32(s.k[0][0]), 16);
            const uint32_t v_lo = desc_sw128_lo(smem_u32(s.v[0][0]), 1024);   // N-major: halves 1 KB apart
            auto issue_s = [&](int t, int st) {
                const uint32_t a0 = q_lo + t * kStage, b0 = k_lo + st * kStage;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {   // 16 columns = 32 bytes per k-step
                    const uint32_t qoff = (ks / 4) * kHalf + (ks % 4) * 2, koff = (ks / 4) * 64 + (ks % 4) * 2;
                    mma_ss(tm + kColS, desc_join(a0 + qoff, hi_q), desc_join(b0 + koff, hi_kv), id_s, ks > 0);
                }
            };
            auto issue_o = [&](int t, int sv, bool acc) {
                const uint32_t b0 = v_lo + sv * kStage;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)   // 16 keys = two 8-token atoms = 4 KB per k-step
                    mma_ts(tm + kColO + 128 * t, tm + kColP + 64 * t + ks * 8, desc_join(b0 + ks * 256, hi_kv), id_o,
                           (acc || ks > 0) ? 1u : 0u);
            };
            // One flat stream of key tiles over this CTA's items: tile g is
            // tile j of item k.  The S buffer takes S0(g), S1(g), S0(g+1), ...
            // (S1 only for items whose second query tile holds a valid row):
            // each S waits until the softmax warps have read the one before
            // it, s_free completing once per S read.
            bool ok = true;
            uint32_t g = 0, ns = 0, g1 = 0;                 // key tiles, S MMAs, tile-1 PVs
            int k = 0;
            if (warp == 1) {
                for (int idx = i_begin; ok && idx < i_end; ++idx, ++k) {
                    const int nt = items[idx].nt, j0 = WIN ? items[idx].j0 : 0;
                    const bool two = items[idx].tiles > 1;
                    for (int j = j0; j < nt; ++j, ++g) {
                        const int st = g % kKStages;
                        ok = (ns == 0 || mbar_wait(&s.s_free, (ns - 1) & 1, &s.abort_)) &&
                             (j > j0 || mbar_wait(ROPE ? &s.q_rot[0] : &s.bar_q, k & 1, &s.abort_)) &&
                             mbar_wait(&s.k_full[st], (g / kKStages) & 1, &s.abort_);
                        if (!ok)
                            break;
                        tc_fence_after();
                        issue_s(0, st);
                        mma_commit(&s.s_full[0]);
                        *(volatile int *)&s.s_issued[0] = (int)g + 1;
                        ++ns;
                        // The second tile's rotation is awaited once per item
                        // either way, which keeps q_rot[1]'s phases in step.
                        ok = (j > j0 || !ROPE || mbar_wait(&s.q_rot[1], k & 1, &s.abort_));
                        if (ok && two) {
                            ok = mbar_wait(&s.s_free, (ns - 1) & 1, &s.abort_);
                            if (ok) {
                                tc_fence_after();
                                issue_s(1, st);
                                mma_commit(&s.s_full[1]);
                                *(volatile int *)&s.s_issued[1] = (int)g + 1;
                                ++ns;
                            }
                        }
                        if (!ok)
                            break;
                        mma_commit(&s.k_empty[st]);
                        if (j + 1 == nt)
                            mma_commit(&s.q_empty);      // the last S of the item has read Q
                    }
                }
            } else {
                // PV_t(g) goes into the tensor pipe right behind S_t(g+1): the
                // S MMAs, on which the softmax warps wait, then run alone, and
                // PV_t(g) runs while the softmax warps read S_t(g+1) and the
                // next S is issued.  A bounded poll on the S issuer's count;
                // it orders issue only (the barriers carry every dependency),
                // and is skipped for an item's last tile.
                auto after_s = [&](int t, uint32_t count) {
                    const uint64_t t0 = globaltimer();
                    for (int it = 0; *(volatile int *)&s.s_issued[t] < (int)count; ++it)
                        if ((it & 63) == 63 && globaltimer() - t0 > 20000)
                            break;
                };
                for (int idx = i_begin; ok && idx < i_end; ++idx, ++k) {
                    const int nt = items[idx].nt, j0 = WIN ? items[idx].j0 : 0;
                    const bool two = items[idx].tiles > 1;
                    for (int j = j0; j < nt; ++j, ++g) {
                        const int sv = g % kVStages;
                        const bool order = kPvOrder && j + 1 < nt;
                        ok = mbar_wait(&s.p_full[0], g & 1, &s.abort_) &&
                             mbar_wait(&s.v_full[sv], (g / kVStages) & 1, &s.abort_);
                        if (!ok)
                            break;
                        if (order)
                            after_s(0, g + 2);
                        tc_fence_after();
                        issue_o(0, sv, j > j0);
                        mma_commit(&s.pv_done[0]);
                        if (two) {
                            ok = mbar_wait(&s.p_full[1], g1 & 1, &s.abort_);
                            if (!ok)
                                break;
                            if (order)
                                after_s(1, g + 2);
                            tc_fence_after();
                            issue_o(1, sv, j > j0);
                            mma_commit(&s.pv_done[1]);
                            ++g1;
                        }
                        mma_commit(&s.v_empty[sv]);
                    }
                }
            }
            if (!ok)
                abort_with(s, p.err, kErrTimeout);
            // Every MMA this thread issued completes before TMEM is released.
            int never = 0;
            mma_commit(&s.fin[warp - 1]);
            if (!mbar_wait(&s.fin[warp - 1], 0, &never))
                atomicOr(p.err, kErrTimeout);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp >> 2) - 1;                  // query tile of this warpgroup: 0 or 1
        const int quarter = warp & 3;                   // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;              // row of the tile
        const uint32_t lane_addr = tm + ((uint32_t)(quarter * 32) << 16);
        const uint32_t tS = lane_addr + kColS, tP = lane_addr + kColP + 64 * t, tO = lane_addr + kColO + 128 * t;
        const float c = p.scale_log2;
        const float2 cc = make_float2(c, c);
        uint32_t gt = 0;
        int k = 0;
        bool ok = true;
        // Rotary mechanism: rotate this thread's row of an item's Q tile in
        // place once the tile has landed; the S issuer waits for all eight
        // warps.  Pair (e, e + 64) sits at the same swizzled offset of the
        // two column halves.  Rows without a valid position stay as they are
        // (their outputs are discarded).  Done for the next item right after
        // this item's last softmax, so the next item's first S overlaps the
        // epilogue.
        auto rotate_q = [&](const TcItem &iq, uint32_t parity) -> bool {
            const SeqDesc sq = seqs[iq.b];
            const int relq = iq.i0 + t * p.rows_pos + r / p.G;
            if (!mbar_wait(&s.bar_q, parity, &s.abort_))
                return false;
            if (r < p.G * p.rows_pos && relq < sq.count) {
                unsigned char *h0 = reinterpret_cast<unsigned char *>(s.q[t][0]) + r * 128;
                unsigned char *h1 = reinterpret_cast<unsigned char *>(s.q[t][1]) + r * 128;
                const float4 *cs4 = reinterpret_cast<const float4 *>(p.rope + (size_t)(sq.past + relq) * (D / 2));
                // Two rounds of four 16-byte chunks: every table load of a
                // round is issued before any shared-memory store (read-only
                // loads), so a round costs one trip to L2.
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float4 cv[16];
                    uint4 a[4], b[4];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        cv[i] = __ldg(cs4 + 16 * half + i);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int off = ((4 * half + c4) ^ (r & 7)) << 4;
                        a[c4] = *reinterpret_cast<const uint4 *>(h0 + off);
                        b[c4] = *reinterpret_cast<const uint4 *>(h1 + off);
                    }
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t *aw = reinterpret_cast<uint32_t *>(&a[c4]), *bw = reinterpret_cast<uint32_t *>(&b[c4]);
#pragma unroll
                        for (int w2 = 0; w2 < 4; ++w2) {          // elements 8*chunk + 2*w2, +1
                            const float4 c = cv[4 * c4 + w2];         // (cos, sin) of both elements
                            const float x0 = __uint_as_float(aw[w2] << 16), x1 = __uint_as_float(aw[w2] & 0xffff0000u);
                            const float y0 = __uint_as_float(bw[w2] << 16), y1 = __uint_as_float(bw[w2] & 0xffff0000u);
                            aw[w2] = pack_bf16x2(x0 * c.x - y0 * c.y, x1 * c.z - y1 * c.w);
                            bw[w2] = pack_bf16x2(x0 * c.y + y0 * c.x, x1 * c.w + y1 * c.z);
                        }
                        const int off = ((4 * half + c4) ^ (r & 7)) << 4;
                        *reinterpret_cast<uint4 *>(h0 + off) = a[c4];
                        *reinterpret_cast<uint4 *>(h1 + off) = b[c4];
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s.q_rot[t]);
            return true;
        };
        auto prefetch_rows = [&](const TcItem &iq) {
            const SeqDesc sq = seqs[iq.b];
            const int relq = iq.i0 + t * p.rows_pos + r / p.G;
            if (r < p.G * p.rows_pos && relq < sq.count) {
                const char *row = reinterpret_cast<const char *>(p.rope + (size_t)(sq.past + relq) * (D / 2));
#pragma unroll
                for (int ln = 0; ln < 4; ++ln)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 128 * ln));
            }
        };
        if (ROPE && i_begin < i_end)
            prefetch_rows(items[i_begin]);
        if (ROPE && i_begin < i_end && !rotate_q(items[i_begin], 0)) {
            ok = false;
            abort_with(s, p.err, kErrTimeout);
        }
        for (int idx = i_begin; ok && idx < i_end; ++idx, ++k) {
            const TcItem it = items[idx];
            const SeqDesc sd = seqs[it.b];
            if (ROPE && idx + 1 < i_end)
                prefetch_rows(items[idx + 1]);         // the next item's table rows into L2
            if (t == 1 && it.tiles < 2) {
                // No valid row in this item's second tile: nothing is issued
                // for it (its rows are padding, zeroed with the cache write).
                // Only the next item's rotation, which the S issuer awaits
                // once per item, is this warpgroup's part.
                if (ROPE && idx + 1 < i_end && !rotate_q(items[idx + 1], (k + 1) & 1)) {
                    ok = false;
                    break;
                }
                continue;
            }
            const int nt = it.nt;
            const bool row_in_box = r < p.G * p.rows_pos;
            const int rel = it.i0 + t * p.rows_pos + r / p.G;   // row within the batch entry
            const bool valid = row_in_box && rel < sd.count;
            const int qpos = sd.past + rel;             // absolute position: sees keys qlo..qpos
            const int qlo = WIN ? window_start(qpos, p.window) : 0;
            const int j0 = WIN ? it.j0 : 0;
            float m = -INFINITY, l = 0.0f;
            for (int j = j0; j < nt; ++j) {
                const uint32_t g = gt + (j - j0);
                if (!mbar_wait(&s.s_full[t], g & 1, &s.abort_)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                __syncwarp();                            // tcgen05.ld is warp-collective
                uint32_t su[128];
                tmem_ld128(tS, su);                      // this row of S (fp32), waited for
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s.s_free);              // the MMA may overwrite S now
                __syncwarp();
                const int key0 = 128 * j;
                if (key0 + 127 > qpos || (WIN && key0 < qlo)) {  // diagonal or window edge: mask keys outside qlo..qpos
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (key0 + i > qpos || (WIN && key0 + i < qlo))
                            su[i] = 0xff800000u;         // -inf
                }
                // Row max: four independent 3-input max chains of depth 16.
                float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < 128; i += 8) {
                    a0 = max3(a0, __uint_as_float(su[i]), __uint_as_float(su[i + 1]));
                    a1 = max3(a1, __uint_as_float(su[i + 2]), __uint_as_float(su[i + 3]));
                    a2 = max3(a2, __uint_as_float(su[i + 4]), __uint_as_float(su[i + 5]));
                    a3 = max3(a3, __uint_as_float(su[i + 6]), __uint_as_float(su[i + 7]));
                }
                const float mx = max3(fmaxf(a0, a1), a2, a3);
                const float m_new = fmaxf(m, mx * c);
                const bool grow = m_new > m + 8.0f;      // rescale only when the max grows by > 2^8
                float alpha = 1.0f;
                if (grow) {
                    alpha = ex2(m - m_new);              // 0 on the first visible tile
                    l *= alpha;
                    m = m_new;
                }
                // The O rescale below touches TMEM with warp-collective loads
                // and stores: do it for the whole warp when any row needs it
                // (alpha = 1 for the others).
                const bool rescale_o = __any_sync(0xffffffffu, grow && j > j0);
                __syncwarp();
                const float m_use = (m == -INFINITY) ? 0.0f : m;
                const float2 mm = make_float2(-m_use, -m_use);
                // P of this warpgroup's previous tile and O must have been
                // consumed by PV(g-1) before P is overwritten or O rescaled.
                if (g > 0 && !mbar_wait(&s.pv_done[t], (g - 1) & 1, &s.abort_)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                __syncwarp();
                // P = 2^(S c - m), bf16, into this warpgroup's P columns.
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 32 * q4 + 2 * i;
                        const float2 x =
                            fma2(make_float2(__uint_as_float(su[e]), __uint_as_float(su[e + 1])), cc, mm);
                        float2 pr;
                        if (kPoly && (i % kPolyEvery) == kPolyEvery - 1)
                            pr = exp2_poly2(x);
                        else
                            pr = make_float2(ex2(x.x), ex2(x.y));
                        acc[i & 3] = add2(acc[i & 3], pr);
                        pk[i] = pack_bf16x2(pr.x, pr.y);
                    }
                    tmem_st16(tP + 16 * q4, pk);
                }
                const float2 s01 = add2(acc[0], acc[1]), s23 = add2(acc[2], acc[3]);
                l += (s01.x + s01.y) + (s23.x + s23.y);
                if (rescale_o) {                         // O (PV of tile g-1 is complete) *= alpha
#pragma unroll 1
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t u[32];
                        tmem_ld32(tO + 32 * q4, u);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                        tmem_st32(tO + 32 * q4, u);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s.p_full[t]);
                __syncwarp();
            }
            if (!ok)
                break;
            if (ROPE && idx + 1 < i_end && !rotate_q(items[idx + 1], (k + 1) & 1)) {
                ok = false;
                break;
            }
            // ---- epilogue: O / l -> bf16, staged one 64-column half at a time in
            // shared memory (128-byte swizzle, the layout of the tensor map) and
            // written by one TMA store per half.  Rows past the valid length
            // are written as zeros; positions past n are clipped by the store.
            // The named barriers below need every thread of the warpgroup, so
            // a timeout is agreed on by all of them before anyone leaves.
            if (named_bar_any(1 + t, 128, !mbar_wait(&s.pv_done[t], (gt + (nt - j0) - 1) & 1, &s.abort_))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (WIN && it.part >= 0) {
                // Split item: this range's unnormalised O row and its (m, l)
                // go to workspace slot it.part; the CTA that completes the
                // group's last split merges the group's slots into out.
                const bool mine = valid && r < p.slot_rows;
                float4 *po = reinterpret_cast<float4 *>(p.ws_o + ((size_t)it.part * p.slot_rows + r) * D);
#pragma unroll 1
                for (int h = 0; h < 4; ++h) {
                    uint32_t u[32];
                    __syncwarp();
                    tmem_ld32(tO + 32 * h, u);
                    if (mine) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            __stcg(po + 8 * h + i, make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                                               __uint_as_float(u[4 * i + 2]),
                                                               __uint_as_float(u[4 * i + 3])));
                    }
                }
                if (mine)
                    __stcg(p.ws_ml + (size_t)it.part * p.slot_rows + r, make_float2(m, l));
                __threadfence();
                tc_fence_before();
                named_bar_sync(1 + t, 128);
                const int first = it.part - it.split;
                if (r == 0)
                    s.last_ = atomicAdd(p.counters + first, 1) == it.nsplit - 1;
                named_bar_sync(1 + t, 128);
                if (s.last_) {
                    // O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, M = max_s m_s (a
                    // split without a visible key for a row has m = -inf, l = 0).  The
                    // merge is a chain of loads from L2, kept short: each thread first
                    // issues the loads of its first two rows' partial columns over
                    // eight splits, then every (m, l) pair of the group goes to this
                    // warpgroup's staging buffer in one round; per row M and 1 / sum
                    // come from there, and the weights 2^(m_s - M) / sum are formed as
                    // the columns are summed, eight splits and two rows per round.
                    __threadfence();
                    const int rows = min(p.slot_rows, sd.count * p.G);
                    const int nsp = it.nsplit;
                    const float2 *ml = p.ws_ml + (size_t)first * p.slot_rows;
                    float2 *sml = reinterpret_cast<float2 *>(s.o[t]);   // (m, l) of split q, row rr at q * rows + rr
                    const bool fit = nsp * rows <= (int)(sizeof(s.o[0]) / sizeof(float2));
                    auto ml_at = [&](int q2, int rr) {
                        return fit ? sml[q2 * rows + rr] : __ldcg(ml + (size_t)q2 * p.slot_rows + rr);
                    };
                    // Thread r: columns 4 * (r % 32) .. + 3 of rows r / 32 and r / 32 + 4,
                    // then + 8, ...
                    const int c4 = r & 31, sub = r >> 5;
                    const float4 *o4 = reinterpret_cast<const float4 *>(p.ws_o) + c4;
                    float4 va[8], vb[8];
                    auto load8 = [&](int q0, int ra, int rb) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const size_t sl = (size_t)(first + q0 + i) * p.slot_rows;
                            va[i] = q0 + i < nsp && ra < rows ? __ldcg(o4 + (sl + ra) * (D / 4))
                                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                            vb[i] = q0 + i < nsp && rb < rows ? __ldcg(o4 + (sl + rb) * (D / 4))
                                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    };
                    load8(0, sub, sub + 4);                  // in flight over the (m, l) round below
                    if (r == 0)
                        tma_store_wait_read();               // earlier stores have left the buffer
                    named_bar_sync(1 + t, 128);
                    if (fit)
                        for (int f = r; f < nsp * rows; f += 128) {
                            const int q2 = f / rows, rr = f - q2 * rows;
                            sml[f] = __ldcg(ml + (size_t)q2 * p.slot_rows + rr);
                        }
                    named_bar_sync(1 + t, 128);
                    if (r < rows) {
                        float M = -INFINITY;
                        for (int q2 = 0; q2 < nsp; ++q2)
                            M = fmaxf(M, ml_at(q2, r).x);
                        if (M == -INFINITY)                  // no visible key at all: zeros, not NaN
                            M = 0.0f;
                        float Lsum = 0.0f;
                        for (int q2 = 0; q2 < nsp; ++q2) {
                            const float2 v2 = ml_at(q2, r);
                            Lsum += ex2(v2.x - M) * v2.y;
                        }
                        s.mrg_m[r] = M;
                        s.mrg_inv[r] = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
                    }
                    named_bar_sync(1 + t, 128);
                    for (int ra = sub; ra < rows; ra += 8) {
                        const int rb = ra + 4;                  // second row of the pair (if < rows)
                        float4 acc_a = make_float4(0.f, 0.f, 0.f, 0.f), acc_b = acc_a;
                        for (int q0 = 0; q0 < nsp; q0 += 8) {
                            if (ra != sub || q0 != 0)            // the first round is already in flight
                                load8(q0, ra, rb);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                if (q0 + i >= nsp)
                                    break;
                                const int q2 = q0 + i;
                                const float wa = ex2(ml_at(q2, ra).x - s.mrg_m[ra]) * s.mrg_inv[ra];
                                acc_a.x += wa * va[i].x, acc_a.y += wa * va[i].y;
                                acc_a.z += wa * va[i].z, acc_a.w += wa * va[i].w;
                                if (rb < rows) {
                                    const float wb = ex2(ml_at(q2, rb).x - s.mrg_m[rb]) * s.mrg_inv[rb];
                                    acc_b.x += wb * vb[i].x, acc_b.y += wb * vb[i].y;
                                    acc_b.z += wb * vb[i].z, acc_b.w += wb * vb[i].w;
                                }
                            }
                        }
                        auto put = [&](int rr, const float4 &a) {
                            __nv_bfloat16 *o = p.out +
                                (((size_t)it.b * p.n + it.i0 + rr / p.G) * p.H_q + it.kvh * p.G + rr % p.G) * D + 4 * c4;
                            *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
                        };
                        put(ra, acc_a);
                        if (rb < rows)
                            put(rb, acc_b);
                    }
                    named_bar_sync(1 + t, 128);              // the staging buffer is free again
                    if (r == 0)
                        p.counters[first] = 0;               // ready for the next launch
                }
                gt += nt - j0;
                continue;
            }
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            unsigned char *stage = reinterpret_cast<unsigned char *>(s.o[t]) + r * 128;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t u0[32], u1[32];
                __syncwarp();
                tmem_ld32(tO + 64 * h, u0);
                tmem_ld32(tO + 64 * h + 32, u1);
                if (r == 0)
                    tma_store_wait_read();               // the previous store has left the buffer
                named_bar_sync(1 + t, 128);
                if (row_in_box) {
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint32_t *u = cc < 4 ? u0 + 8 * cc : u1 + 8 * (cc - 4);
                        uint4 v4;
                        v4.x = pack_bf16x2(__uint_as_float(u[0]) * inv_l, __uint_as_float(u[1]) * inv_l);
                        v4.y = pack_bf16x2(__uint_as_float(u[2]) * inv_l, __uint_as_float(u[3]) * inv_l);
                        v4.z = pack_bf16x2(__uint_as_float(u[4]) * inv_l, __uint_as_float(u[5]) * inv_l);
                        v4.w = pack_bf16x2(__uint_as_float(u[6]) * inv_l, __uint_as_float(u[7]) * inv_l);
                        if (!valid)                      // padding row: zeros, whatever O holds
                            v4 = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(stage + ((cc ^ (r & 7)) << 4)) = v4;
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(1 + t, 128);
                if (r == 0 && it.i0 + t * p.rows_pos < p.n) {
                    tma_store_4d(&mO, s.o[t], 64 * h, it.kvh * p.G, it.i0 + t * p.rows_pos, it.b);
                    tma_store_commit();
                }
            }
            tc_fence_before();
            gt += nt - j0;
        }
        if (!ok)
            abort_with(s, p.err, kErrTimeout);
        if (r == 0)
            tma_store_wait_all();                       // every store has landed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

// The bounded wait every kernel here uses, on a barrier phase that nothing
// completes: it gives up after limit_ns and records a timeout in the error
// word, as a pipeline wait would.  Exercises the failure path without a
// fault.
__global__ void wait_probe_kernel(int32_t *err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_ = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_for(&bar, 0, &abort_, limit_ns))
        atomicOr(err, kErrTimeout);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    }
    return fn;
}

bool encode_tmap(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
                 const cuuint32_t *box, bool bytes, bool bytes_swizzled)
{
    auto fn = encoder();
    if (!fn)
        return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    // bytes: FP8 code blocks, copied as they are (the tensor-core kernel lays
    // them out itself) or 128-byte swizzled (read by ldmatrix).
    return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
              const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              bytes && !bytes_swizzled ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_wait_probe(int32_t *err, uint64_t limit_ns, cudaStream_t st)
{
    wait_probe_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

namespace {

// Byte offsets of the host descriptors in TcParams::inl (16-byte aligned),
// and the bytes they need.
size_t inline_layout(const TcHostDesc &h, int32_t (&off)[5])
{
    const size_t bytes[5] = {(size_t)h.n_seqs * sizeof(SeqDesc), (size_t)h.n_items * sizeof(TcItem),
                             (size_t)h.n_start * sizeof(int32_t), (size_t)h.n_zero * sizeof(int64_t),
                             h.n_tables * sizeof(int32_t)};
    const bool given[5] = {h.seqs != nullptr, h.items != nullptr, h.item_start != nullptr, h.zero_start != nullptr,
                           h.tables != nullptr};
    size_t at = 0;
    for (int i = 0; i < 5; ++i) {
        off[i] = -1;
        if (!given[i])
            continue;
        at = (at + 15) & ~(size_t)15;
        off[i] = (int32_t)std::min<size_t>(at, INT32_MAX);
        at += bytes[i];
    }
    return at;
}

}  // namespace

bool prefill_tc_inline_fits(const TcHostDesc &h)
{
    int32_t off[5];
    return h.seqs && h.items && h.item_start && inline_layout(h, off) <= kTcInlineBytes;
}

bool prefill_tc_supported(int group, int H_kv) { return group >= 1 && group <= 128 && H_kv >= 1; }

int prefill_tc_rows_per_tile(int group) { return 128 / group; }

cudaError_t launch_prefill_tc(const PoolView &pv, const SeqDesc *d_seqs, const TcItem *d_items,
                              const int32_t *d_item_start, int grid, int B, int n, int H_q, const void *q, void *out,
                              const TcSplitWs &ws, cudaStream_t st, cudaEvent_t ev_start, const void *app_k,
                              const void *app_v, const void *fused_k, const void *fused_v,
                              const int64_t *d_zero_start, const TcHostDesc *host)
{
    if (pv.d != D || grid <= 0)
        return grid <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    const int G = H_q / pv.H_kv;
    const int rows_pos = 128 / G;
    if (G < 1 || rows_pos < 1 || grid < 1)
        return cudaErrorInvalidValue;
    CUtensorMap mq, mkv, mo;
    const cuuint64_t qdims[4] = {(cuuint64_t)D, (cuuint64_t)H_q, (cuuint64_t)n, (cuuint64_t)B};
    const cuuint64_t qstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)H_q * D * 2, (cuuint64_t)n * H_q * D * 2};
    const cuuint32_t qbox[4] = {64, (cuuint32_t)G, (cuuint32_t)rows_pos, 1};
    // The pool as 128-byte lines: [block][32 lines][64 elements]; a box is
    // one page block (4 KB).
    const cuuint64_t kvdims[3] = {64, 32, (cuuint64_t)pv.num_pages * 2 * pv.H_kv};
    const cuuint64_t kvstr[2] = {128, 32 * 128};
    const cuuint32_t kvbox[3] = {64, 32, 1};
    // FP8 E4M3 pool: a block is [16 rows][128 code bytes]; one 2 KB box each.
    const bool q8 = pv.dtype == kDtypeFp8;
    const cuuint64_t kv8dims[3] = {128, 16, (cuuint64_t)pv.num_pages * 2 * pv.H_kv};
    const cuuint64_t kv8str[2] = {128, 16 * 128};
    const cuuint32_t kv8box[3] = {128, 16, 1};
    if (q8 && (pv.rope || app_k || !pv.scales))
        return cudaErrorInvalidValue;
    // out has the shape and layout of q: the same box serves the stores.
    if (!encode_tmap(&mq, 4, q, qdims, qstr, qbox) ||
        !(q8 ? encode_tmap(&mkv, 3, pv.pool, kv8dims, kv8str, kv8box, true) : encode_tmap(&mkv, 3, pv.pool, kvdims, kvstr, kvbox)) ||
        !encode_tmap(&mo, 4, out, qdims, qstr, qbox))
        return cudaErrorInvalidValue;
    // Fused write: k and v [B, n, H_kv, 128] as [H_kv][B * n / 8 row groups]
    // [column half][8 rows][64 elements] (n a multiple of 8), boxes of one
    // key tile (16 groups, 32 KB) and of one page (2 groups, 4 KB).
    const bool fused = fused_k != nullptr;
    CUtensorMap mkt, mvt, mkp, mvp;
    if (fused) {
        if (q8 || pv.rope || app_k || !fused_v || !d_zero_start || n % 8 != 0)
            return cudaErrorInvalidValue;
        const cuuint64_t fdims[5] = {64, 8, 2, (cuuint64_t)B * n / 8, (cuuint64_t)pv.H_kv};
        const cuuint64_t fstr[4] = {(cuuint64_t)pv.H_kv * D * 2, 128, (cuuint64_t)8 * pv.H_kv * D * 2, (cuuint64_t)D * 2};
        const cuuint32_t tbox[5] = {64, 8, 2, 16, 1}, pbox[5] = {64, 8, 2, 2, 1};
        if (!encode_tmap(&mkt, 5, fused_k, fdims, fstr, tbox) || !encode_tmap(&mvt, 5, fused_v, fdims, fstr, tbox) ||
            !encode_tmap(&mkp, 5, fused_k, fdims, fstr, pbox) || !encode_tmap(&mvp, 5, fused_v, fdims, fstr, pbox))
            return cudaErrorInvalidValue;
    } else {
        mkt = mvt = mkp = mvp = mkv;               // unused
    }
    // The INL form when the caller hands over host descriptors; the caller
    // has skipped the upload of the device copies, so a form that cannot
    // carry them is an error, not a fallback.
    const bool inl = host != nullptr;
    if (inl && (!prefill_tc_inline_fits(*host) || q8 || pv.rope))
        return cudaErrorInvalidValue;
    TcParamsInl prmi;
    TcParams &prm = prmi;
    prm.seqs = d_seqs;
    prm.items = d_items;
    prm.item_start = d_item_start;
    prm.tables = pv.tables;
    prm.pool = pv.pool;
    prm.app_k = (const __nv_bfloat16 *)app_k;
    prm.app_v = (const __nv_bfloat16 *)app_v;
    prm.scales = pv.scales;
    prm.stride = pv.stride;
    prm.num_pages = pv.num_pages;
    prm.H_kv = pv.H_kv;
    prm.H_q = H_q;
    prm.n = n;
    prm.G = G;
    prm.rows_pos = rows_pos;
    prm.out = (__nv_bfloat16 *)out;
    prm.err = pv.err;
    prm.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    prm.rope = pv.rope;
    prm.window = pv.window;
    prm.ws_o = ws.o;
    prm.ws_ml = ws.ml;
    prm.counters = ws.counters;
    prm.slot_rows = ws.slot_rows;
    prm.fused = fused ? 1 : 0;
    prm.B = B;
    prm.zero_start = d_zero_start;
    if (inl) {
        inline_layout(*host, prmi.inl_off);
        const void *src[5] = {host->seqs, host->items, host->item_start, host->zero_start, host->tables};
        const size_t bytes[5] = {(size_t)host->n_seqs * sizeof(SeqDesc), (size_t)host->n_items * sizeof(TcItem),
                                 (size_t)host->n_start * sizeof(int32_t), (size_t)host->n_zero * sizeof(int64_t),
                                 host->n_tables * sizeof(int32_t)};
        for (int i = 0; i < 5; ++i)
            if (prmi.inl_off[i] >= 0 && bytes[i])
                memcpy(prmi.inl + prmi.inl_off[i], src[i], bytes[i]);
    }
    const int smem = (int)sizeof(TcSmem) + 1024;
    // The shared-memory opt-in is per device: remember it per device.
    constexpr int kMaxDev = 64;
    static std::atomic<bool> attr_set[kMaxDev][8];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return cudaErrorInvalidDevice;
    const bool win = pv.window > 0 || ws.ranged;
    const int which = inl ? 6 + (win ? 1 : 0) : q8 ? 4 + (win ? 1 : 0) : (pv.rope ? 1 : 0) + (win ? 2 : 0);
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                          TcParams);
    using KernInl = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                             CUtensorMap, TcParamsInl);
    const Kern kern[6] = {prefill_tc_kernel<false, false, false>, prefill_tc_kernel<true, false, false>,
                          prefill_tc_kernel<false, true, false>,  prefill_tc_kernel<true, true, false>,
                          prefill_tc_kernel<false, false, true>,  prefill_tc_kernel<false, true, true>};
    const KernInl kern_inl[2] = {prefill_tc_kernel<false, false, false, true>,
                                 prefill_tc_kernel<false, true, false, true>};
    const void *fn = inl ? (const void *)kern_inl[which - 6] : (const void *)kern[which];
    if (!attr_set[dev][which].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_set[dev][which].store(true, std::memory_order_release);
    }
    if (ev_start)
        cudaEventRecord(ev_start, st);       // after the host-side preparation above
#if GQA_PDL
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (inl)
        return cudaLaunchKernelEx(&cfg, kern_inl[which - 6], mq, mkv, mo, mkt, mvt, mkp, mvp, prmi);
    return cudaLaunchKernelEx(&cfg, kern[which], mq, mkv, mo, mkt, mvt, mkp, mvp, prm);
#else
    if (inl)
        kern_inl[which - 6]<<<grid, kThreads, smem, st>>>(mq, mkv, mo, mkt, mvt, mkp, mvp, prmi);
    else
        kern[which]<<<grid, kThreads, smem, st>>>(mq, mkv, mo, mkt, mvt, mkp, mvp, prm);
    return cudaGetLastError();
#endif
}

}  // namespace gqa
