// k_decode_cluster.cu -- single-token decode of a small batch over the paged
// cache (bf16, d_h = 128): each (batch entry, KV head) is served by one
// thread-block cluster whose CTAs split its pages, and the CTAs' partial
// softmax states are merged inside the cluster through distributed shared
// memory.
//
// What it computes ("KV Cache 与 Prefill/Decode 推理路径", decode lesson: the
// single new query reads every cached key, its own included; the
// PagedAttention section: keys are found through the block table;
// "第二章 Prefill：整层状态演化与 KV 建立" section 2.3 for the scores and the
// softmax): for query head h of KV group g,
//     out[b,h] = sum_t softmax_t(<q[b,h], K[t,g]>/sqrt(128)) V[t,g]
// over the visible positions t (every cached one, or the last W of them with
// a sliding window).
//
// Why a kernel of its own: with few sequences (B * H_kv well below the SM
// count) each (entry, head) holds many bytes but there are few of them, so
// its keys are split across SMs and the parts merged.  The persistent
// tensor-core kernel merges through a global workspace and the CTA that
// finishes last, which puts a fence, an atomic and two rounds of L2 reads
// after the data has streamed, and its per-CTA set-up (TMEM, twelve warps)
// and 128-key tile chain add more.  Here:
//  * grid (cs, H_kv, B) in clusters of cs CTAs along x: CTA r of the cluster
//    of (b, kvh) takes pages [r P / cs, (r + 1) P / cs) of the P pages that
//    hold visible keys;
//  * eight producer lanes request the CTA's pages up front, as far as a
//    ring of kStages stages allows: a stage is the page's K block and V
//    block, one TMA box (8 KB, 128-byte swizzled: the two blocks are the
//    kv = 0, 1 neighbours of a [2 page + kv][head] view of the pool),
//    completed on an mbarrier.  Lane p issues pages p, p + 8, ...: the
//    copies of eight pages are issued at once, since one thread issuing them
//    in turn leaves the SM's copy engine idle between boxes, and one box per
//    page rather than one per block halves the engine's per-copy cost;
//  * kWarps consumer warps take the pages round robin.  The group's g heads
//    are the rows of a 16-row mma.sync m16n8k16 tile (bf16 operands, fp32
//    accumulation; rows past g hold zeros): S = Q K^T over the page's 16 keys
//    (8 k-steps x 2 n-tiles, K fragments by ldmatrix from the swizzled
//    stage), an online softmax per row in exp2 units, then O += P V with P
//    rounded to bf16 as the A operand straight from the score registers and
//    V fragments by ldmatrix.trans;
//  * the warps' (m, l, O) meet in shared memory; then each CTA stores its
//    (m, l) into every CTA of the cluster and column slice j (columns
//    j * 128 / cs .. (j + 1) * 128 / cs - 1) of its summed O into CTA j
//    (distributed shared memory), one cluster barrier makes the stores
//    visible, and CTA j merges the slices it holds and writes those columns
//    of out.  Cluster sizes need not be powers of two: 12-CTA clusters, for
//    instance, put 96 SMs on eight (entry, head) pairs where 16-CTA ones do
//    not all fit on the GPU at once.  (Stores of each warp's own partial
//    straight into the merging CTAs, skipping the combine in shared memory,
//    measured slower: eight times the remote stores and a merge over
//    eight times the partials.)  Nothing goes through global memory but q, the pages
//    and out, and no CTA waits on a flag another one sets.
// Decode with append (app_k / app_v): the warp that holds the page of
// position past writes the new K/V row into the landed stage, before reading
// it, and into the pool.
#include <cuda_bf16.h>

#include <atomic>

#include "kernels.cuh"
#include "sm100.cuh"

namespace gqa {

namespace {

using namespace sm100;

constexpr int D = 128;
// Consumer warps: 8 for the wide form (16 MMA rows of heads; 64 accumulator
// registers a lane), 12 for the narrow form (g <= 8: 16 keys or dims as MMA
// rows and the heads as the 8 columns; 32 accumulator registers a lane, so
// more warps fit and hide more latency).  One producer warp on top.
template <bool NARROW> struct DcCfg {
    static constexpr int kWarps = NARROW ? 12 : 8;
    static constexpr int kThreads = (kWarps + 1) * 32;
};
constexpr int kStages = 24;
constexpr int kIssuePages = 8;                     // pages whose copies are issued at once
// A stage is refilled by the lane that filled it (page i and i + kStages
// have one issuing lane), so a lane's final wait on a stage is for its own
// last copy into it; and by the warp that read it (page i and i + kStages
// have one consumer warp), so stages free in each warp's own order.
static_assert(kStages % kIssuePages == 0, "a stage must be refilled by the lane that filled it");
static_assert(kStages % DcCfg<false>::kWarps == 0 && kStages % DcCfg<true>::kWarps == 0,
              "a stage must be read by one consumer warp");
constexpr int kBlockBytes = kPageTokens * D * 2;   // one page of one head: 4 KB
constexpr int kMaxCluster = 16;
constexpr int kRows = 16;                          // MMA rows: the group's heads, zero-padded

constexpr int kRedStride = D + 4;                  // warp-combine rows, padded against bank conflicts
// CTA j of a cluster of cs merges columns [lo(j), lo(j + 1)), lo(j) =
// j * 128 / cs; cs times the widest slice is at most 140 for cs <= 16.
constexpr int kInStride = 144;
__host__ __device__ constexpr int slice_lo(int j, int cs) { return j * D / cs; }
// The CTA whose slice holds column col.
__device__ __forceinline__ int slice_owner(int col, int cs) { return ((col + 1) * cs - 1) / D; }
constexpr int kInline = 16;                        // entries whose descriptors travel in the parameters
template <int W>
struct __align__(1024) DcSmem {
    unsigned char ring[kStages][2 * kBlockBytes];  // stage: K block, then V block
    // Received from the cluster's CTAs (rank r): unnormalised O rows,
    // columns [r * w, (r + 1) * w) = this CTA's slice of w columns as CTA r
    // holds it; and (m, l) per row.
    float in_o[kRows][kInStride];
    float in_m[kMaxCluster][kRows], in_l[kMaxCluster][kRows];
    float wm[W][kRows], wl[W][kRows];              // per consumer warp
    uint64_t full[kStages], empty[kStages];
    int abort_;
};
static_assert(DcCfg<true>::kWarps * kRows * kRedStride * sizeof(float) <= sizeof(DcSmem<12>::ring),
              "the warp combine reuses the ring");

struct DcParams {
    const SeqDesc *seqs;                           // device descriptors, or null: inl[] holds them
    SeqDesc inl[kInline];
    const int32_t *tables;
    unsigned char *pool;
    int32_t *err;
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    const __nv_bfloat16 *app_k, *app_v;
    const float *scales;                           // FP8 E4M3: scale of (block, slot) at block * 16 + slot
    int stride, num_pages, H_kv, H_q, G, window;
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_ncta()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: writes before it are visible to
// the cluster's reads after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Store v into the shared memory of cluster CTA `rank`, at the offset
// `local` has in this CTA's.
__device__ __forceinline__ void st_cluster(float *local, uint32_t rank, float v)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// E4M3 codes 0, 1 of w as an f16 pair (lo) and codes 2, 3 (hi), the lower
// code in the lower half: every E4M3 value is exact in f16.
__device__ __forceinline__ void e4m3x4_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t prmt2(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// FP8 E4M3 stage: a page block is 16 slots of 128 code bytes, one 128-byte
// line each, swizzled by the TMA copy: 16-byte unit c of slot s sits at
// s * 128 + (c xor (s % 8)) * 16.  K codes at 0, V codes at 2048, then the
// 16 K and the 16 V row scales.
constexpr int kQ8Block = kPageTokens * D;          // 2 KB
__device__ __forceinline__ uint32_t q8_off(int s, int c) { return (uint32_t)(s << 7) + (uint32_t)(((c ^ (s & 7)) << 4)); }

// Byte offset, within a landed page block, of 16-byte unit c (columns
// 8c .. 8c + 7) of slot s: the pool's block layout (two groups of 8 slots,
// each stored 128-byte chunk by chunk) as the 128-byte swizzle of the TMA
// copy places it: line (s / 8) * 16 + (c / 8) * 8 + s % 8, unit (c % 8) xor (s % 8).
__device__ __forceinline__ uint32_t stage_off(int s, int c)
{
    return (uint32_t)((((s >> 3) << 4) + ((c >> 3) << 3) + (s & 7)) << 7) + (uint32_t)(((c & 7) ^ (s & 7)) << 4);
}

// Q8: the pool holds FP8 E4M3 codes and row scales.  Codes convert exactly
// to f16, so both products run on f16 mma.sync: each lane's ldmatrix
// register holds four consecutive codes of a key row (dims 4j .. 4j + 3 of a
// 16-dim k-step), which is the B fragment of k indices 2j, 2j + 1 and
// 2j + 8, 2j + 9 -- a fixed permutation of the dims inside each k-step that
// q's A fragments follow (the contraction does not depend on the order).  q
// enters f16 after an exact power-of-two scaling per head (undone, with the
// key row's scale, on the fp32 score).  For O += P V the value scales are
// folded into P: P' = P s_v / R, R the largest value scale the warp has met
// (O is rescaled when R grows, as for the softmax maximum, and multiplied by
// R at the end); ldmatrix.trans plus a byte permute give the key pairs of
// the B fragments, whose n columns are the even and the odd dims of a
// 16-dim unit (undone when O is combined).
template <bool Q8, bool NARROW>
__global__ void __launch_bounds__(DcCfg<NARROW>::kThreads, 1)
decode_cluster_kernel(const __grid_constant__ CUtensorMap mKV, const __grid_constant__ CUtensorMap mSc,
                      const DcParams p)
{
    constexpr int kWarps = DcCfg<NARROW>::kWarps;
    extern __shared__ unsigned char smem_raw[];
    DcSmem<kWarps> &s =
        *reinterpret_cast<DcSmem<kWarps> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y;
    const uint32_t rank = cluster_rank(), cs = cluster_ncta();
    const SeqDesc sd = p.seqs ? p.seqs[b] : p.inl[b];
    const int past = sd.past;                              // the query's position (L - 1)
    const int L = past + 1;
    const int ws = window_start(past, p.window);           // first visible key
    const int pfirst = decode_first_token(L, p.window) / kPageTokens;
    const int P = (L - pfirst * kPageTokens + kPageTokens - 1) / kPageTokens;
    const int i_lo = (int)((int64_t)rank * P / cs), i_hi = (int)((int64_t)(rank + 1) * P / cs);
    const int npg = i_hi - i_lo;
    const int32_t *tab = p.tables + (size_t)sd.row * p.stride + pfirst + i_lo;
    const int G = p.G;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        s.abort_ = 0;
        fence_barrier_init();
    }
    // Launched as a programmatic dependent of the kernel before it in the
    // stream (often the previous decode step): the set-up above overlaps
    // that kernel's end; q, the pool, the tables and out are touched only
    // after it has completed.  The next launch may be scheduled once every
    // CTA of this one is resident.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    __syncthreads();

    const int r0 = lane >> 2, qc = (lane & 3) * 2;         // fragment row / column pair of this lane
    float o[D / 8][4];                                     // O rows r0, r0 + 8; columns 8j + qc, + 1 (narrow: tiles 0-7)
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows r0, r0 + 8 (narrow: heads 2 c4, + 1)
    float R = 0.f;                                         // Q8: largest value scale met so far (O is in units of R)

    if (warp == kWarps) {
        // ---- producer ---------------------------------------------------
        if (lane < kIssuePages) {
            if (lane == 0) {
                prefetch_tmap(&mKV);
                if (Q8)
                    prefetch_tmap(&mSc);
            }
            int issued = 0;                                // pages lane issued: lane, lane + 8, ...
            for (int i = lane; i < npg; i += kIssuePages) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(&s.empty[st], ((i / kStages) - 1) & 1, &s.abort_)) {
                    s.abort_ = 1;
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
                int page = tab[i];
                if ((unsigned)page >= (unsigned)p.num_pages) {
                    atomicOr(p.err, kErrPageId);
                    page = p.num_pages;                    // out of range: the boxes read zeros
                }
                // One box holds the page's K block and V block (block
                // indices (2 page + kv) H_kv + head, kv = 0, 1); FP8 adds
                // one for their two rows of scales.
                if constexpr (Q8) {
                    mbar_arrive_expect_tx(&s.full[st], 2 * kQ8Block + 2 * kPageTokens * 4);
                    tma_load_4d(&mKV, &s.full[st], s.ring[st], 0, 0, kvh, 2 * page);
                    tma_load_3d(&mSc, &s.full[st], s.ring[st] + 2 * kQ8Block, 0, kvh, 2 * page);
                } else {
                    mbar_arrive_expect_tx(&s.full[st], 2 * kBlockBytes);
                    tma_load_4d(&mKV, &s.full[st], s.ring[st], 0, 0, kvh, 2 * page);
                }
                issued = i + 1;
            }
            // Every issued copy lands before the ring is reused or the CTA
            // ends (copies of earlier uses of a stage were waited for by
            // their consumers before the stage was issued again).
            const int never = 0;
            for (int i = lane; i < issued; i += kIssuePages)
                if (i + kStages >= issued && !mbar_wait(&s.full[i % kStages], (i / kStages) & 1, &never)) {
                    s.abort_ = 1;
                    atomicOr(p.err, kErrTimeout);
                }
        }
        __syncwarp();                                      // the warp meets the block barrier converged
    } else if constexpr (NARROW) {
        // ---- consumers, narrow form (g <= 8) ------------------------------
        // S^T = K Q^T: the page's 16 keys are the MMA rows, the group's heads
        // the 8 columns (none wasted for g = 8); O^T += V^T P^T: 16 dims as
        // the rows of each of 8 MMA tiles.  This lane: keys (and dims) r4,
        // r4 + 8 of a tile, heads 2 c4, 2 c4 + 1; m0 / m1, l0 / l1 are the
        // running maximum and sum of those two heads.
        const int r4 = lane >> 2, c4 = lane & 3;
        const float kScale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
        float qs0 = kScale, qs1 = kScale;                  // score factor of heads 2 c4, 2 c4 + 1
        // Q^T as the B operand of k-step kk: head r4 (zero past g).
        uint32_t qb[D / 16][2];
        if constexpr (!Q8) {
            const uint32_t *qh = reinterpret_cast<const uint32_t *>(p.q + ((size_t)b * p.H_q + kvh * G + r4) * D);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qb[kk][0] = r4 < G ? qh[8 * kk + c4] : 0u;          // dims 16 kk + 2 c4, + 1
                qb[kk][1] = r4 < G ? qh[8 * kk + 4 + c4] : 0u;      // dims 16 kk + 8 + 2 c4, + 1
            }
        } else {
            // Dims 16 kk + 4 c4 .. + 3 (the code layout's permutation of the
            // k-step); scaled by 2^e so the head's largest |q| lies in
            // [2^14, 2^15), then rounded to f16.
            const uint2 *qh = reinterpret_cast<const uint2 *>(p.q + ((size_t)b * p.H_q + kvh * G + r4) * D) + c4;
            float a = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                if (r4 < G) {
                    const uint2 u = qh[4 * kk];
                    a = fmaxf(fmaxf(a, fmaxf(fabsf(__uint_as_float(u.x << 16)), fabsf(__uint_as_float(u.x & 0xffff0000u)))),
                              fmaxf(fabsf(__uint_as_float(u.y << 16)), fabsf(__uint_as_float(u.y & 0xffff0000u))));
                }
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            int e = 0;                                     // a * 2^e in [2^14, 2^15), clamped
            if (a > 0.f)
                e = max(-126, min(126, 14 - ((int)((__float_as_uint(a) >> 23) & 0xff) - 127)));
            const float f = __uint_as_float((uint32_t)(e + 127) << 23);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint2 u = r4 < G ? qh[4 * kk] : make_uint2(0u, 0u);
                qb[kk][0] = pack_f16x2(__uint_as_float(u.x << 16) * f, __uint_as_float(u.x & 0xffff0000u) * f);
                qb[kk][1] = pack_f16x2(__uint_as_float(u.y << 16) * f, __uint_as_float(u.y & 0xffff0000u) * f);
            }
            const float qsh = kScale * __uint_as_float((uint32_t)(127 - e) << 23);   // head r4's factor
            qs0 = __shfl_sync(0xffffffffu, qsh, 8 * c4);          // head 2 c4 sits in lanes 8 c4 ..
            qs1 = __shfl_sync(0xffffffffu, qsh, 8 * c4 + 4);      // head 2 c4 + 1 in lanes 8 c4 + 4 ..
        }
#pragma unroll
        for (int j = 0; j < D / 16; ++j)
            o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;           // ldmatrix: matrix and row this lane addresses
        const uint32_t ring0 = smem_u32(s.ring[0]);
        for (int i = warp; i < npg; i += kWarps) {
            const int st = i % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&s.full[st], (i / kStages) & 1, &s.abort_))) {
                if (lane == 0) {
                    s.abort_ = 1;
                    atomicOr(p.err, kErrTimeout);
                }
                break;
            }
            const uint32_t kb = ring0 + (uint32_t)st * (2 * kBlockBytes), vb = kb + (Q8 ? kQ8Block : kBlockBytes);
            const int pos0 = (pfirst + i_lo + i) * kPageTokens;    // position of the page's slot 0
            if (!Q8 && p.app_k && pos0 <= past && past < pos0 + kPageTokens) {
                // The appended row: lanes 0-15 its K units, 16-31 its V units.
                const int slot = past - pos0, kv = lane >> 4, c = lane & 15;
                const __nv_bfloat16 *src = (kv ? p.app_v : p.app_k) + ((size_t)b * p.H_kv + kvh) * D + 8 * c;
                const uint4 val = *reinterpret_cast<const uint4 *>(src);
                *reinterpret_cast<uint4 *>(s.ring[st] + kv * kBlockBytes + stage_off(slot, c)) = val;
                const int page = tab[i];
                if ((unsigned)page < (unsigned)p.num_pages)
                    *reinterpret_cast<uint4 *>(p.pool + (((size_t)page * 2 + kv) * p.H_kv + kvh) * kBlockBytes +
                                               pool_in_block(2, slot, 16 * c)) = val;
                __syncwarp();
            }
            // S^T: two accumulators (even and odd k-steps) halve the chain.
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            float k0s = 1.f, k1s = 1.f, v0s = 1.f, v1s = 1.f;   // Q8: scales of keys r4, r4 + 8
            if constexpr (!Q8) {
                // Matrices of one ldmatrix: (keys 0-7, dims 16 kk ..), (keys
                // 8-15, same), (keys 0-7, dims 16 kk + 8 ..), (keys 8-15, same).
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(kb + stage_off(8 * (mi & 1) + rr, 2 * kk + (mi >> 1)), a[0], a[1], a[2], a[3]);
                    mma_bf16((kk & 1) ? sb : sa, a, qb[kk][0], qb[kk][1]);
                }
            } else {
                // Matrices: (keys 0-7, unit 2h), (keys 8-15, 2h), (keys 0-7,
                // 2h + 1), (keys 8-15, 2h + 1); a register's four codes are
                // dims 4 c4 .. + 3 of its key: k indices 2 c4, + 1 (lo) and
                // 8 + 2 c4, + 1 (hi).
#pragma unroll
                for (int h = 0; h < D / 32; ++h) {
                    uint32_t w0, w1, w2, w3, l0_, h0_, l1_, h1_;
                    ldsm_x4(kb + q8_off(8 * (mi & 1) + rr, 2 * h + (mi >> 1)), w0, w1, w2, w3);
                    e4m3x4_f16(w0, l0_, h0_);
                    e4m3x4_f16(w1, l1_, h1_);
                    const uint32_t ae[4] = {l0_, l1_, h0_, h1_};
                    mma_f16(sa, ae, qb[2 * h][0], qb[2 * h][1]);
                    e4m3x4_f16(w2, l0_, h0_);
                    e4m3x4_f16(w3, l1_, h1_);
                    const uint32_t ao[4] = {l0_, l1_, h0_, h1_};
                    mma_f16(sb, ao, qb[2 * h + 1][0], qb[2 * h + 1][1]);
                }
                const float *ksc = reinterpret_cast<const float *>(s.ring[st] + 2 * kQ8Block);
                k0s = ksc[r4];
                k1s = ksc[8 + r4];
                v0s = ksc[kPageTokens + r4];
                v1s = ksc[kPageTokens + 8 + r4];
            }
            // Visible keys only, in exp2 units: sc = [key r4 | r4 + 8][head 2 c4 | + 1].
            const int t0 = pos0 + r4, t1 = pos0 + 8 + r4;
            const bool vis0 = t0 <= past && t0 >= ws, vis1 = t1 <= past && t1 >= ws;
            float sc[4];
            sc[0] = vis0 ? (sa[0] + sb[0]) * qs0 * k0s : -INFINITY;
            sc[1] = vis0 ? (sa[1] + sb[1]) * qs1 * k0s : -INFINITY;
            sc[2] = vis1 ? (sa[2] + sb[2]) * qs0 * k1s : -INFINITY;
            sc[3] = vis1 ? (sa[3] + sb[3]) * qs1 * k1s : -INFINITY;
            // Column maxima: the two keys here, then the 8 lanes of the same c4.
            float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
            }
            const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
            const float f0 = n0 == -INFINITY ? 0.f : n0, f1 = n1 == -INFINITY ? 0.f : n1;
            float a0 = ex2(m0 - f0), a1 = ex2(m1 - f1);   // 0 while nothing was visible
            m0 = n0;
            m1 = n1;
            float pr[4] = {ex2(sc[0] - f0), ex2(sc[1] - f1), ex2(sc[2] - f0), ex2(sc[3] - f1)};
            l0 = l0 * a0 + (pr[0] + pr[2]);                // this lane's keys; lanes summed at the end
            l1 = l1 * a1 + (pr[1] + pr[3]);
            if constexpr (Q8) {
                // P' = P s_v / R, R the largest value scale met (all 16 keys
                // of the page: max over the lanes of one c4).
                float vm = fmaxf(v0s, v1s);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
                    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                if (vm > R) {                              // the same in every lane; O = 0 while R = 0
                    a0 *= R / vm;
                    a1 *= R / vm;
                    R = vm;
                }
                const float invR = R > 0.f ? 1.f / R : 0.f;
                pr[0] *= v0s * invR;
                pr[1] *= v0s * invR;
                pr[2] *= v1s * invR;
                pr[3] *= v1s * invR;
            }
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    o[j][0] *= a0;
                    o[j][1] *= a1;
                    o[j][2] *= a0;
                    o[j][3] *= a1;
                }
            }
            // P^T as the B operand for head r4: keys 2 c4, + 1 (b0) and
            // 8 + 2 c4, + 1 (b1).  Key k of head h sits in lane 4 (k % 8) +
            // h / 2; each lane sends its two heads as (key r4, key r4 + 8)
            // pairs, and the two lanes holding keys 2 c4 and 2 c4 + 1 of this
            // head give b0, b1 by a byte permute.
            const uint32_t ph0 = Q8 ? pack_f16x2(pr[0], pr[2]) : pack_bf16x2(pr[0], pr[2]);
            const uint32_t ph1 = Q8 ? pack_f16x2(pr[1], pr[3]) : pack_bf16x2(pr[1], pr[3]);
            const int sA = 8 * c4 + (r4 >> 1), sB = sA + 4;
            const uint32_t xa0 = __shfl_sync(0xffffffffu, ph0, sA), xa1 = __shfl_sync(0xffffffffu, ph1, sA);
            const uint32_t xb0 = __shfl_sync(0xffffffffu, ph0, sB), xb1 = __shfl_sync(0xffffffffu, ph1, sB);
            const uint32_t X = (r4 & 1) ? xa1 : xa0, Y = (r4 & 1) ? xb1 : xb0;
            const uint32_t pb0 = prmt2(X, Y, 0x5410), pb1 = prmt2(X, Y, 0x7632);
            if constexpr (!Q8) {
                // V^T of dims 16 j .. + 15: matrices (keys 0-7, dims 16 j ..),
                // (keys 0-7, dims 16 j + 8 ..), (keys 8-15, 16 j ..), (keys
                // 8-15, 16 j + 8 ..), transposed.
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    uint32_t a[4];
                    ldsm_x4_t(vb + stage_off(8 * (mi >> 1) + rr, 2 * j + (mi & 1)), a[0], a[1], a[2], a[3]);
                    mma_bf16(o[j], a, pb0, pb1);
                }
            } else {
                // Matrices (keys 0-7, unit 2h), (keys 0-7, 2h + 1), (keys
                // 8-15, 2h), (keys 8-15, 2h + 1), transposed as code pairs; a
                // byte permute makes key pairs per dim.  Tile 2h + par: rows
                // r, r + 8 = dims 32h + 2r + par, 32h + 16 + 2r + par.
#pragma unroll
                for (int h = 0; h < D / 32; ++h) {
                    uint32_t w0, w1, w2, w3, e0[2], e1[2], e2[2], e3[2];
                    ldsm_x4_t(vb + q8_off(8 * (mi >> 1) + rr, 2 * h + (mi & 1)), w0, w1, w2, w3);
                    e4m3x4_f16(prmt(w0, 0x3120), e0[0], e0[1]);
                    e4m3x4_f16(prmt(w1, 0x3120), e1[0], e1[1]);
                    e4m3x4_f16(prmt(w2, 0x3120), e2[0], e2[1]);
                    e4m3x4_f16(prmt(w3, 0x3120), e3[0], e3[1]);
#pragma unroll
                    for (int par = 0; par < 2; ++par) {
                        const uint32_t a[4] = {e0[par], e1[par], e2[par], e3[par]};
                        mma_f16(o[2 * h + par], a, pb0, pb1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s.empty[st]);
        }
        // Column sums over the 8 lanes of one c4.
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (r4 == 0) {
            s.wm[warp][2 * c4] = m0;
            s.wm[warp][2 * c4 + 1] = m1;
            s.wl[warp][2 * c4] = l0;
            s.wl[warp][2 * c4 + 1] = l1;
        }
    } else {
        // ---- consumers --------------------------------------------------
        // Q as the A operand of each k-step: rows r0 / r0 + 8 (zero past g),
        // columns 16 kk + qc, + 1 and 16 kk + 8 + qc, + 1.
        uint32_t qa[D / 16][4];
        const float kScale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
        float qs0 = kScale, qs1 = kScale;                  // score factor of rows r0, r0 + 8
        if constexpr (!Q8) {
            const uint32_t *q0 = reinterpret_cast<const uint32_t *>(p.q + ((size_t)b * p.H_q + kvh * G + r0) * D);
            const uint32_t *q1 = q0 + 8 * D / 2;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qa[kk][0] = r0 < G ? q0[8 * kk + qc / 2] : 0u;
                qa[kk][1] = r0 + 8 < G ? q1[8 * kk + qc / 2] : 0u;
                qa[kk][2] = r0 < G ? q0[8 * kk + 4 + qc / 2] : 0u;
                qa[kk][3] = r0 + 8 < G ? q1[8 * kk + 4 + qc / 2] : 0u;
            }
        } else {
            // Rows r0 / r0 + 8, dims 16 kk + 4j .. + 3 (j = lane % 4): one
            // 8-byte load each; scaled by 2^e so the row's largest |q| lies
            // in [2^14, 2^15), then rounded to f16.
            const uint2 *q0 = reinterpret_cast<const uint2 *>(p.q + ((size_t)b * p.H_q + kvh * G + r0) * D) + (lane & 3);
            const uint2 *q1 = q0 + 8 * D / 4;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (r0 < G) {
                    const uint2 u = q0[4 * kk];
                    a0 = fmaxf(fmaxf(a0, fmaxf(fabsf(__uint_as_float(u.x << 16)), fabsf(__uint_as_float(u.x & 0xffff0000u)))),
                               fmaxf(fabsf(__uint_as_float(u.y << 16)), fabsf(__uint_as_float(u.y & 0xffff0000u))));
                }
                if (r0 + 8 < G) {
                    const uint2 u = q1[4 * kk];
                    a1 = fmaxf(fmaxf(a1, fmaxf(fabsf(__uint_as_float(u.x << 16)), fabsf(__uint_as_float(u.x & 0xffff0000u)))),
                               fmaxf(fabsf(__uint_as_float(u.y << 16)), fabsf(__uint_as_float(u.y & 0xffff0000u))));
                }
            }
            a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, 1));
            a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
            a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, 2));
            a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 2));
            auto pow2_exp = [](float a) {                  // e with a * 2^e in [2^14, 2^15), clamped
                if (!(a > 0.f))
                    return 0;
                const int E = (int)((__float_as_uint(a) >> 23) & 0xff) - 127;
                return max(-126, min(126, 14 - E));
            };
            const int e0 = pow2_exp(a0), e1 = pow2_exp(a1);
            const float f0 = __uint_as_float((uint32_t)(e0 + 127) << 23), f1 = __uint_as_float((uint32_t)(e1 + 127) << 23);
            qs0 = kScale * __uint_as_float((uint32_t)(127 - e0) << 23);
            qs1 = kScale * __uint_as_float((uint32_t)(127 - e1) << 23);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint2 u0 = r0 < G ? q0[4 * kk] : make_uint2(0u, 0u);
                const uint2 u1 = r0 + 8 < G ? q1[4 * kk] : make_uint2(0u, 0u);
                qa[kk][0] = pack_f16x2(__uint_as_float(u0.x << 16) * f0, __uint_as_float(u0.x & 0xffff0000u) * f0);
                qa[kk][2] = pack_f16x2(__uint_as_float(u0.y << 16) * f0, __uint_as_float(u0.y & 0xffff0000u) * f0);
                qa[kk][1] = pack_f16x2(__uint_as_float(u1.x << 16) * f1, __uint_as_float(u1.x & 0xffff0000u) * f1);
                qa[kk][3] = pack_f16x2(__uint_as_float(u1.y << 16) * f1, __uint_as_float(u1.y & 0xffff0000u) * f1);
            }
        }
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;           // ldmatrix: matrix and row this lane addresses
        const uint32_t ring0 = smem_u32(s.ring[0]);
        for (int i = warp; i < npg; i += kWarps) {
            const int st = i % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&s.full[st], (i / kStages) & 1, &s.abort_))) {
                if (lane == 0) {
                    s.abort_ = 1;
                    atomicOr(p.err, kErrTimeout);
                }
                break;
            }
            const uint32_t kb = ring0 + (uint32_t)st * (2 * kBlockBytes), vb = kb + (Q8 ? kQ8Block : kBlockBytes);
            const int pos0 = (pfirst + i_lo + i) * kPageTokens;    // position of the page's slot 0
            if (!Q8 && p.app_k && pos0 <= past && past < pos0 + kPageTokens) {
                // The appended row: lanes 0-15 its K units, 16-31 its V units.
                const int slot = past - pos0, kv = lane >> 4, c = lane & 15;
                const __nv_bfloat16 *src = (kv ? p.app_v : p.app_k) + ((size_t)b * p.H_kv + kvh) * D + 8 * c;
                const uint4 val = *reinterpret_cast<const uint4 *>(src);
                *reinterpret_cast<uint4 *>(s.ring[st] + kv * kBlockBytes + stage_off(slot, c)) = val;
                const int page = tab[i];
                if ((unsigned)page < (unsigned)p.num_pages)
                    *reinterpret_cast<uint4 *>(p.pool + (((size_t)page * 2 + kv) * p.H_kv + kvh) * kBlockBytes +
                                               pool_in_block(2, slot, 16 * c)) = val;
                __syncwarp();
            }
            // S = Q K^T: n-tile 0 = keys 0-7, n-tile 1 = keys 8-15.
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float mul[2][2];                               // score factor per (n-tile, key of the lane)
            float vsk[2][2];                               // Q8: value scale of those keys
            if constexpr (!Q8) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + stage_off(8 * (mi >> 1) + rr, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                    mma_bf16(sc[0], qa[kk], b0, b1);
                    mma_bf16(sc[1], qa[kk], b2, b3);
                }
                mul[0][0] = mul[0][1] = mul[1][0] = mul[1][1] = 1.f;
            } else {
                // Matrices of one ldmatrix: (keys 0-7, k-step 2h), (keys
                // 0-7, 2h + 1), (keys 8-15, 2h), (keys 8-15, 2h + 1).
#pragma unroll
                for (int h = 0; h < D / 32; ++h) {
                    uint32_t w0, w1, w2, w3, lo, hi;
                    ldsm_x4(kb + q8_off(8 * (mi >> 1) + rr, 2 * h + (mi & 1)), w0, w1, w2, w3);
                    e4m3x4_f16(w0, lo, hi);
                    mma_f16(sc[0], qa[2 * h], lo, hi);
                    e4m3x4_f16(w1, lo, hi);
                    mma_f16(sc[0], qa[2 * h + 1], lo, hi);
                    e4m3x4_f16(w2, lo, hi);
                    mma_f16(sc[1], qa[2 * h], lo, hi);
                    e4m3x4_f16(w3, lo, hi);
                    mma_f16(sc[1], qa[2 * h + 1], lo, hi);
                }
                const float *ksc = reinterpret_cast<const float *>(s.ring[st] + 2 * kQ8Block);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        mul[nt][e] = ksc[8 * nt + qc + e];
                        vsk[nt][e] = ksc[kPageTokens + 8 * nt + qc + e];
                    }
            }
            // Visible keys only, in exp2 units.
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = pos0 + 8 * nt + qc + (e & 1);
                    sc[nt][e] = (t <= past && t >= ws) ? sc[nt][e] * (e < 2 ? qs0 : qs1) * mul[nt][e & 1] : -INFINITY;
                }
            float x0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            float x1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
            const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
            const float f0 = n0 == -INFINITY ? 0.f : n0, f1 = n1 == -INFINITY ? 0.f : n1;
            float a0 = ex2(m0 - f0), a1 = ex2(m1 - f1);   // 0 while nothing was visible
            m0 = n0;
            m1 = n1;
            float pr[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pr[nt][e] = ex2(sc[nt][e] - (e < 2 ? f0 : f1));
            l0 = l0 * a0 + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
            l1 = l1 * a1 + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
            float invR = 1.f;
            if constexpr (Q8) {
                // The page's largest value scale (all 16 keys: the quad holds them).
                float vm = fmaxf(fmaxf(vsk[0][0], vsk[0][1]), fmaxf(vsk[1][0], vsk[1][1]));
                vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 1));
                vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 2));
                if (vm > R) {                              // the same in every lane; O = 0 while R = 0
                    a0 *= R / vm;
                    a1 *= R / vm;
                    R = vm;
                }
                invR = R > 0.f ? 1.f / R : 0.f;
            }
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    o[j][0] *= a0;
                    o[j][1] *= a0;
                    o[j][2] *= a1;
                    o[j][3] *= a1;
                }
            }
            if constexpr (!Q8) {
                // O += P V: P (16 rows x 16 keys) is the A operand as the
                // score fragments hold it; n-tile j = columns 8j .. 8j + 7.
                const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                                        pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + stage_off(8 * (mi & 1) + rr, 2 * j + (mi >> 1)), b0, b1, b2, b3);
                    mma_bf16(o[2 * j], pa, b0, b1);
                    mma_bf16(o[2 * j + 1], pa, b2, b3);
                }
            } else {
                // P' = P s_v / R in f16.  Matrices of one ldmatrix.trans:
                // (keys 0-7, unit 2h), (keys 8-15, 2h), (keys 0-7, 2h + 1),
                // (keys 8-15, 2h + 1); a register holds the codes of dims
                // 16u + 2(lane / 4), + 1 for keys 2(lane % 4), + 1; a byte
                // permute makes key pairs per dim.  n-tile 2u + par = the
                // dims 16u + 2n + par.
                const float s00 = vsk[0][0] * invR, s01 = vsk[0][1] * invR;
                const float s10 = vsk[1][0] * invR, s11 = vsk[1][1] * invR;
                const uint32_t pa[4] = {pack_f16x2(pr[0][0] * s00, pr[0][1] * s01), pack_f16x2(pr[0][2] * s00, pr[0][3] * s01),
                                        pack_f16x2(pr[1][0] * s10, pr[1][1] * s11), pack_f16x2(pr[1][2] * s10, pr[1][3] * s11)};
#pragma unroll
                for (int h = 0; h < D / 32; ++h) {
                    uint32_t w0, w1, w2, w3, e0lo, e0hi, e1lo, e1hi;
                    ldsm_x4_t(vb + q8_off(8 * (mi & 1) + rr, 2 * h + (mi >> 1)), w0, w1, w2, w3);
                    e4m3x4_f16(prmt(w0, 0x3120), e0lo, e0hi);
                    e4m3x4_f16(prmt(w1, 0x3120), e1lo, e1hi);
                    mma_f16(o[4 * h], pa, e0lo, e1lo);
                    mma_f16(o[4 * h + 1], pa, e0hi, e1hi);
                    e4m3x4_f16(prmt(w2, 0x3120), e0lo, e0hi);
                    e4m3x4_f16(prmt(w3, 0x3120), e1lo, e1hi);
                    mma_f16(o[4 * h + 2], pa, e0lo, e1lo);
                    mma_f16(o[4 * h + 3], pa, e0hi, e1hi);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s.empty[st]);
        }
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if ((lane & 3) == 0) {
            s.wm[warp][r0] = m0;
            s.wm[warp][r0 + 8] = m1;
            s.wl[warp][r0] = l0;
            s.wl[warp][r0 + 8] = l1;
        }
    }
    __syncthreads();          // the ring is idle: every copy landed and was read

    // ---- the CTA's partial: warps combined -----------------------------------
    const bool ok = s.abort_ == 0;
    float *red = reinterpret_cast<float *>(s.ring[0]);     // [kWarps][kRows][kRedStride]
    if constexpr (NARROW) {
        if (warp < kWarps && ok) {
            const int r4 = lane >> 2, c4 = lane & 3;
            float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                M0 = fmaxf(M0, s.wm[w][2 * c4]);
                M1 = fmaxf(M1, s.wm[w][2 * c4 + 1]);
            }
            const float rs = Q8 ? R : 1.f;                 // Q8: O is in units of R
            const float c0 = m0 == -INFINITY ? 0.f : ex2(m0 - M0) * rs, c1 = m1 == -INFINITY ? 0.f : ex2(m1 - M1) * rs;
            float *w0 = red + ((size_t)warp * kRows + 2 * c4) * kRedStride, *w1 = w0 + kRedStride;
            const bool h0 = 2 * c4 < G, h1 = 2 * c4 + 1 < G;
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
                // bf16: tile j rows r, r + 8 = dims 16j + r, + 8; FP8: tile
                // 2h + par rows = dims 32h + 2r + par, + 16.
                const int d0 = Q8 ? 32 * (j >> 1) + 2 * r4 + (j & 1) : 16 * j + r4;
                const int d1 = d0 + (Q8 ? 16 : 8);
                if (h0) {
                    w0[d0] = o[j][0] * c0;
                    w0[d1] = o[j][2] * c0;
                }
                if (h1) {
                    w1[d0] = o[j][1] * c1;
                    w1[d1] = o[j][3] * c1;
                }
            }
        }
    } else if (warp < kWarps && ok) {

        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            M0 = fmaxf(M0, s.wm[w][r0]);
            M1 = fmaxf(M1, s.wm[w][r0 + 8]);
        }
        const float rs = Q8 ? R : 1.f;                     // Q8: O is in units of R
        const float c0 = m0 == -INFINITY ? 0.f : ex2(m0 - M0) * rs, c1 = m1 == -INFINITY ? 0.f : ex2(m1 - M1) * rs;
        float *w0 = red + ((size_t)warp * kRows + r0) * kRedStride, *w1 = w0 + 8 * kRedStride;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            if constexpr (!Q8) {
                if (r0 < G)
                    *reinterpret_cast<float2 *>(w0 + 8 * j + qc) = make_float2(o[j][0] * c0, o[j][1] * c0);
                if (r0 + 8 < G)
                    *reinterpret_cast<float2 *>(w1 + 8 * j + qc) = make_float2(o[j][2] * c1, o[j][3] * c1);
            } else {
                // n-tile j = 2u + par, column c: dim 16u + 2c + par.
                const int d0 = 16 * (j >> 1) + 2 * qc + (j & 1);
                if (r0 < G) {
                    w0[d0] = o[j][0] * c0;
                    w0[d0 + 2] = o[j][1] * c0;
                }
                if (r0 + 8 < G) {
                    w1[d0] = o[j][2] * c1;
                    w1[d0 + 2] = o[j][3] * c1;
                }
            }
        }
    }
    __syncthreads();
    // ---- into the cluster: column slice j of every row goes to CTA j ----------
    if (ok) {
        for (int e = threadIdx.x; e < G * D; e += DcCfg<NARROW>::kThreads) {
            const int row = e >> 7, col = e & (D - 1);
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w)              // a fixed order
                a += red[((size_t)w * kRows + row) * kRedStride + col];
            const int j = slice_owner(col, (int)cs), lo = slice_lo(j, (int)cs);
            st_cluster(&s.in_o[row][rank * (slice_lo(j + 1, (int)cs) - lo) + (col - lo)], (uint32_t)j, a);
        }
    }
    for (int t = threadIdx.x; t < G * (int)cs; t += DcCfg<NARROW>::kThreads) {
        const int j = t / G, row = t - j * G;
        float M = -INFINITY, l = 0.f;
        for (int w = 0; w < kWarps; ++w)
            M = fmaxf(M, s.wm[w][row]);
        for (int w = 0; w < kWarps; ++w)
            if (s.wm[w][row] != -INFINITY)
                l += s.wl[w][row] * ex2(s.wm[w][row] - M);
        st_cluster(&s.in_m[rank][row], (uint32_t)j, ok ? M : -INFINITY);
        st_cluster(&s.in_l[rank][row], (uint32_t)j, ok ? l : 0.f);
    }
    cluster_sync();           // every CTA's stores into this one are visible

    // ---- the merge of this CTA's columns [lo, lo + w) ---------------------------
    const int lo = slice_lo((int)rank, (int)cs), w = slice_lo((int)rank + 1, (int)cs) - lo;
    if (threadIdx.x < G) {
        // Weights 2^(m_r - M) / sum_r 2^(m_r - M) l_r, in cluster rank order.
        const int row = threadIdx.x;
        float M = -INFINITY, den = 0.f;
        for (uint32_t r = 0; r < cs; ++r)
            M = fmaxf(M, s.in_m[r][row]);
        for (uint32_t r = 0; r < cs; ++r) {
            const float w = s.in_m[r][row] == -INFINITY ? 0.f : ex2(s.in_m[r][row] - M);
            s.in_m[r][row] = w;
            den += w * s.in_l[r][row];
        }
        const float inv = 1.0f / den;
        for (uint32_t r = 0; r < cs; ++r)
            s.in_m[r][row] *= inv;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * w; e += DcCfg<NARROW>::kThreads) {
        const int row = e / w, c = e - row * w;
        float a = 0.f;
        for (uint32_t r = 0; r < cs; ++r)
            a = fmaf(s.in_m[r][row], s.in_o[row][r * w + c], a);
        p.out[((size_t)b * p.H_q + kvh * G + row) * D + lo + c] = __float2bfloat16_rn(a);
    }
}

constexpr int kSmemBytes =
    (int)(sizeof(DcSmem<12>) > sizeof(DcSmem<8>) ? sizeof(DcSmem<12>) : sizeof(DcSmem<8>)) + 1024;
constexpr int kMaxDev = 64;

// The shared-memory and cluster-size opt-ins are per device.
cudaError_t configure(int dev)
{
    static std::atomic<bool> done[kMaxDev];
    if (dev < 0 || dev >= kMaxDev)
        return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    cudaError_t e = cudaSuccess;
    for (auto k : {decode_cluster_kernel<false, false>, decode_cluster_kernel<true, false>,
                   decode_cluster_kernel<false, true>, decode_cluster_kernel<true, true>}) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    if (e == cudaSuccess)
        done[dev].store(true, std::memory_order_release);
    return e;
}

}  // namespace

bool decode_cluster_supported(int group) { return group >= 1 && group <= kRows; }

int decode_cluster_inline() { return kInline; }

int decode_cluster_capacity(int cluster)
{
    // Looked up once per device and size.
    static std::atomic<int> cap[kMaxDev][kMaxCluster + 1];
    int dev = 0;
    const int k = cluster;
    if (k < 1 || k > kMaxCluster || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev ||
        configure(dev) != cudaSuccess)
        return 0;
    int v = cap[dev][k].load(std::memory_order_acquire);
    if (v != 0)
        return v < 0 ? 0 : v;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster, 1, 1);
    cfg.blockDim = dim3(DcCfg<true>::kThreads);
    cfg.dynamicSmemBytes = (size_t)kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    // Every instantiation holds one CTA per SM (shared memory); the widest
    // block stands for them all.
    if (cudaOccupancyMaxActiveClusters(&n, decode_cluster_kernel<false, true>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cap[dev][k].store(n > 0 ? n : -1, std::memory_order_release);
    return n;
}

cudaError_t launch_decode_cluster(const PoolView &pv, const ClusterDecodeLaunch &a, cudaStream_t st,
                                  cudaEvent_t ev_start)
{
    const int G = pv.H_kv > 0 ? a.H_q / pv.H_kv : 0;
    const bool q8 = pv.dtype == kDtypeFp8;
    if (pv.d != D || (pv.dtype != kDtypeBf16 && !q8) || pv.rope || !decode_cluster_supported(G) || a.cluster < 1 ||
        a.cluster > kMaxCluster || a.B < 1 || a.B > 65535 || pv.H_kv > 65535 || (q8 && (a.app_k || !pv.scales)))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || (e = configure(dev)) != cudaSuccess)
        return e;
    // The pool as [2 page + kv][head][lines][line bytes]: bf16 blocks of
    // 32 lines of 64 elements, FP8 blocks of 16 slots of 128 codes; a box is
    // one head's K and V blocks of a page (8 KB, 4 KB).  FP8 scales as
    // [2 page + kv][head][16 floats, as 64 bytes]: a box holds both rows.
    CUtensorMap mkv, msc;
    const cuuint64_t H = (cuuint64_t)pv.H_kv, kvp = (cuuint64_t)pv.num_pages * 2;
    const cuuint64_t kvdims[4] = {64, 32, H, kvp}, kv8dims[4] = {128, 16, H, kvp}, scdims[3] = {64, H, kvp};
    const cuuint64_t kvstr[3] = {128, 4096, H * 4096}, kv8str[3] = {128, 2048, H * 2048}, scstr[2] = {64, H * 64};
    const cuuint32_t kvbox[4] = {64, 32, 1, 2}, kv8box[4] = {128, 16, 1, 2}, scbox[3] = {64, 1, 2};
    if (!(q8 ? encode_tmap(&mkv, 4, pv.pool, kv8dims, kv8str, kv8box, true, true) &&
                   encode_tmap(&msc, 3, pv.scales, scdims, scstr, scbox, true, false)
             : encode_tmap(&mkv, 4, pv.pool, kvdims, kvstr, kvbox)))
        return cudaErrorInvalidValue;
    if (!q8)
        msc = mkv;                                         // unused
    DcParams prm;
    if (a.host_seqs && a.B <= kInline) {
        prm.seqs = nullptr;
        for (int i = 0; i < a.B; ++i)
            prm.inl[i] = a.host_seqs[i];
    } else if (a.seqs) {
        prm.seqs = a.seqs;
    } else {
        return cudaErrorInvalidValue;
    }
    prm.tables = pv.tables;
    prm.pool = (unsigned char *)pv.pool;
    prm.err = pv.err;
    prm.q = (const __nv_bfloat16 *)a.q;
    prm.out = (__nv_bfloat16 *)a.out;
    prm.app_k = (const __nv_bfloat16 *)a.app_k;
    prm.app_v = (const __nv_bfloat16 *)a.app_v;
    prm.scales = pv.scales;
    prm.stride = pv.stride;
    prm.num_pages = pv.num_pages;
    prm.H_kv = pv.H_kv;
    prm.H_q = a.H_q;
    prm.G = G;
    prm.window = pv.window;
    if (ev_start)
        cudaEventRecord(ev_start, st);
    cudaLaunchConfig_t cfg = {};
    const bool narrow = G <= 8;
    cfg.gridDim = dim3((unsigned)a.cluster, (unsigned)pv.H_kv, (unsigned)a.B);
    cfg.blockDim = dim3(narrow ? DcCfg<true>::kThreads : DcCfg<false>::kThreads);
    cfg.dynamicSmemBytes = (size_t)kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (narrow)
        return q8 ? cudaLaunchKernelEx(&cfg, decode_cluster_kernel<true, true>, mkv, msc, prm)
                  : cudaLaunchKernelEx(&cfg, decode_cluster_kernel<false, true>, mkv, msc, prm);
    return q8 ? cudaLaunchKernelEx(&cfg, decode_cluster_kernel<true, false>, mkv, msc, prm)
              : cudaLaunchKernelEx(&cfg, decode_cluster_kernel<false, false>, mkv, msc, prm);
}

}  // namespace gqa
