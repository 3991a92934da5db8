// k_prefill_tc.cu -- causal GQA prefill on the fifth-generation tensor core
// (tcgen05, TMEM accumulators, TMA-staged operands), bf16 in, fp32
// accumulate, d_h = 128.
//
// What it computes ("第二章 Prefill：整层状态演化与 KV 建立", section 2.3):
// for query head h of KV group g = floor(h*H_kv/H_q) and a query row at
// absolute position p, the softmax over the finite scores
// <q, k_j>/sqrt(d_h), j = 0..p, applied to V.  Keys come from the paged
// cache through the block table ("KV Cache 与 Prefill/Decode 推理路径",
// PagedAttention): the cache write kernel has already stored this call's new
// rows, so a prefill over an existing prefix (incremental prefill: the old
// prefix fully visible, the new block lower-triangular) and a fresh prefill
// are the same loop.
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
//  * Warp roles: warp 0 issues TMA (Q once; K and V per key tile, one 16-
//    token page box at a time through the block table, two stages); warp 1
//    owns TMEM and issues the MMAs; warps 2-5 and 6-9 are two softmax
//    warpgroups, one per query tile, thread = row.
//  * TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  S = Q K^T
//    is computed into TMEM; the softmax warps read their row, write
//    P = exp2(S*c - m) back as bf16 over the first 64 columns of S, and the
//    PV MMA takes P straight from TMEM as its A operand: O += P V.
//  * Online softmax (the FlashAttention recurrence): a running row max m and
//    sum l; O is rescaled in TMEM only when the max grows by more than 2^8,
//    otherwise the stale max stays the reference (exact in real arithmetic).
//  * Epilogue: O / l in fp32 -> bf16, staged in shared memory over the
//    query tile and written with one TMA store per 64-column half; padding
//    rows are written as zeros.
// Every wait is bounded; on a timeout the CTA raises GQA_DEVERR_TIMEOUT,
// drains what it has in flight (bounded) and exits cleanly.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "sm100.cuh"

namespace gqa {

using namespace sm100;

namespace {

constexpr int D = 128;
constexpr int kStages = 2;
constexpr int kThreads = 320;
constexpr uint32_t kTileBytes = 128 * 64 * 2;        // one 128-row x 64-column bf16 half tile

struct __align__(1024) TcSmem {
    __nv_bfloat16 q[2][2][128 * 64];                   // [query tile][column half]
    __nv_bfloat16 k[kStages][2][128 * 64];
    __nv_bfloat16 v[kStages][2][128 * 64];
    uint64_t bar_q;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], p_full[2], o_full[2], fin;
    uint32_t tmem;
    int abort_;
};

struct TcParams {
    const SeqDesc *seqs;
    const TcItem *items;
    const int32_t *tables;
    int32_t stride;
    int32_t num_pages;
    int32_t H_kv;
    int32_t G;          // query heads per KV head
    int32_t rows_pos;   // positions per query tile (128 / G)
    int32_t *err;
    float scale_log2;   // log2(e) / sqrt(d_h)
};

__device__ __forceinline__ void abort_with(TcSmem &s, int32_t *err, int32_t bit)
{
    s.abort_ = 1;
    atomicOr(err, bit);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mO,
                  const __grid_constant__ CUtensorMap mKV, const TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    TcSmem &s = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const TcItem it = p.items[blockIdx.x];
    const SeqDesc sd = p.seqs[it.b];
    const int nt = it.nt;

    if (warp == 1) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        s.abort_ = 0;
        mbar_init(&s.bar_q, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.kv_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s.s_full[t], 1);
            mbar_init(&s.p_full[t], 4);
            mbar_init(&s.o_full[t], 1);
        }
        mbar_init(&s.fin, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s.tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&mQ);
            prefetch_tmap(&mKV);
            const uint32_t q_bytes = 2u * 2u * (uint32_t)(p.G * p.rows_pos) * 64u * 2u;
            mbar_arrive_expect_tx(&s.bar_q, q_bytes);
            for (int t = 0; t < 2; ++t)
                for (int c = 0; c < 2; ++c)
                    tma_load_4d(&mQ, &s.bar_q, s.q[t][c], 64 * c, it.kvh * p.G, it.i0 + t * p.rows_pos, it.b);
            const int32_t *tab = p.tables + (size_t)sd.row * p.stride;
            const int seq_pages = (sd.past + sd.count + kPageTokens - 1) / kPageTokens;
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int st = j % kStages;
                if (j >= kStages && !mbar_wait(&s.kv_empty[st], ((j / kStages) - 1) & 1, &s.abort_)) {
                    abort_with(s, p.err, kErrTimeout);
                    break;
                }
                int page[8];
#pragma unroll
                for (int pg = 0; pg < 8; ++pg) {
                    const int lp = 8 * j + pg;
                    int ph = p.num_pages;                 // out of range: the box reads zeros
                    if (lp < seq_pages) {
                        ph = tab[lp];
                        if ((unsigned)ph >= (unsigned)p.num_pages) {
                            atomicOr(p.err, kErrPageId);
                            ph = p.num_pages;
                        }
                    }
                    page[pg] = ph;
                }
                mbar_arrive_expect_tx(&s.k_full[st], 2 * kTileBytes);
#pragma unroll
                for (int pg = 0; pg < 8; ++pg)
                    for (int c = 0; c < 2; ++c)
                        tma_load_4d(&mKV, &s.k_full[st], s.k[st][c] + pg * 16 * 64, 64 * c, 0, it.kvh, page[pg]);
                mbar_arrive_expect_tx(&s.v_full[st], 2 * kTileBytes);
#pragma unroll
                for (int pg = 0; pg < 8; ++pg)
                    for (int c = 0; c < 2; ++c)
                        tma_load_4d(&mKV, &s.v_full[st], s.v[st][c] + pg * 16 * 64, 64 * c, 0, p.H_kv + it.kvh,
                                    page[pg]);
                ++issued;
            }
            // Drain: every issued copy must land before the CTA exits.
            int never = 0;
            for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
                const int st = j % kStages;
                if (!mbar_wait(&s.k_full[st], (j / kStages) & 1, &never) ||
                    !mbar_wait(&s.v_full[st], (j / kStages) & 1, &never))
                    atomicOr(p.err, kErrTimeout);
            }
            if (!mbar_wait(&s.bar_q, 0, &never))
                atomicOr(p.err, kErrTimeout);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S = Q K^T: both K-major
            const uint32_t id_o = idesc_bf16(128, 128, 0, 1);   // O += P V: V is N-major
            auto issue_s = [&](int t, int st) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = desc_sw128(smem_u32(s.q[t][ks / 4]) + (ks % 4) * 32, 16, 1024);
                    const uint64_t b = desc_sw128(smem_u32(s.k[st][ks / 4]) + (ks % 4) * 32, 16, 1024);
                    mma_ss(tm + 128 * t, a, b, id_s, ks > 0);
                }
            };
            auto issue_o = [&](int t, int st, bool acc) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t b = desc_sw128(smem_u32(s.v[st][0]) + ks * 2048, kTileBytes, 1024);
                    mma_ts(tm + 256 + 128 * t, tm + 128 * t + ks * 8, b, id_o, (acc || ks > 0) ? 1u : 0u);
                }
            };
            bool ok = nt > 0 && mbar_wait(&s.bar_q, 0, &s.abort_) && mbar_wait(&s.k_full[0], 0, &s.abort_);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                mma_commit(&s.s_full[0]);
                issue_s(1, 0);
                mma_commit(&s.s_full[1]);
            }
            for (int j = 0; ok && j < nt; ++j) {
                const int st = j % kStages, st2 = (j + 1) % kStages;
                ok = mbar_wait(&s.p_full[0], j & 1, &s.abort_) && mbar_wait(&s.v_full[st], (j / kStages) & 1, &s.abort_);
                if (!ok)
                    break;
                tc_fence_after();
                issue_o(0, st, j > 0);
                if (j == nt - 1)
                    mma_commit(&s.o_full[0]);
                if (j + 1 < nt) {
                    ok = mbar_wait(&s.k_full[st2], ((j + 1) / kStages) & 1, &s.abort_);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_s(0, st2);
                    mma_commit(&s.s_full[0]);
                }
                ok = mbar_wait(&s.p_full[1], j & 1, &s.abort_);
                if (!ok)
                    break;
                tc_fence_after();
                issue_o(1, st, j > 0);
                mma_commit(&s.kv_empty[st]);
                if (j == nt - 1)
                    mma_commit(&s.o_full[1]);
                if (j + 1 < nt) {
                    issue_s(1, st2);
                    mma_commit(&s.s_full[1]);
                }
            }
            if (!ok && nt > 0)
                abort_with(s, p.err, kErrTimeout);
            // Every issued MMA completes before TMEM is released.
            int never = 0;
            mma_commit(&s.fin);
            if (!mbar_wait(&s.fin, 0, &never))
                atomicOr(p.err, kErrTimeout);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 2) >> 2;                  // query tile of this warpgroup
        const int quarter = warp & 3;                   // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;              // row of the tile
        const bool row_in_box = r < p.G * p.rows_pos;
        const int rel = it.i0 + t * p.rows_pos + r / p.G;   // row index within the batch entry
        const bool valid = row_in_box && rel < sd.count;
        const int qpos = sd.past + rel;                 // absolute position: sees keys 0..qpos
        const uint32_t lane_addr = tm + ((uint32_t)(quarter * 32) << 16);
        const uint32_t tS = lane_addr + 128 * t, tO = lane_addr + 256 + 128 * t;
        const float c = p.scale_log2;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;

        for (int j = 0; j < nt; ++j) {
            if (!mbar_wait(&s.s_full[t], j & 1, &s.abort_)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float sv[128];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t u[32];
                tmem_ld32(tS + 32 * q4, u);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    sv[32 * q4 + i] = __uint_as_float(u[i]);
            }
            const int key0 = 128 * j;
            if (key0 + 127 > qpos) {                     // diagonal (or beyond): mask keys > qpos
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (key0 + i > qpos)
                        sv[i] = -INFINITY;
            }
            float mx = sv[0];
#pragma unroll
            for (int i = 1; i < 128; ++i)
                mx = fmaxf(mx, sv[i]);
            const float m_new = fmaxf(m, mx * c);
            if (m_new > m + 8.0f) {                      // rescale only when the max grows by > 2^8
                const float alpha = ex2(m - m_new);      // 0 on the first visible tile
                if (j > 0) {
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
                l *= alpha;
                m = m_new;
            }
            const float m_use = (m == -INFINITY) ? 0.0f : m;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ex2(fmaf(sv[32 * q4 + 2 * i], c, -m_use));
                    const float p1 = ex2(fmaf(sv[32 * q4 + 2 * i + 1], c, -m_use));
                    l += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tS + 16 * q4, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s.p_full[t]);
        }

        // ---- epilogue: O / l -> bf16 -> shared memory (over this Q tile) -> TMA store
        ok = ok && (nt == 0 || mbar_wait(&s.o_full[t], 0, &s.abort_));
        if (!ok)
            abort_with(s, p.err, kErrTimeout);
        if (ok) {
            tc_fence_after();
            const float inv_l = (valid && l > 0.0f) ? 1.0f / l : 0.0f;
            unsigned char *stage_base = reinterpret_cast<unsigned char *>(s.q[t][0]);
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t u[32];
                if (nt > 0)
                    tmem_ld32(tO + 32 * q4, u);
                else
                    for (int i = 0; i < 32; ++i)
                        u[i] = 0;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = valid ? pack_bf16x2(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l)
                                  : 0u;                  // padding rows are written as zeros
                // Columns 32*q4 .. +31 = half q4/2, 16-byte units 4*(q4%2) .. +3 of row r,
                // placed with the 128-byte swizzle the store's tensor map expects.
                unsigned char *row = stage_base + (q4 >> 1) * kTileBytes + r * 128;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const int unit = 4 * (q4 & 1) + k4;
                    *reinterpret_cast<uint4 *>(row + ((unit ^ (r & 7)) * 16)) =
                        make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        named_bar_sync(1 + t, 128);
        if (ok && warp == 2 + 4 * t && lane == 0) {
            for (int h2 = 0; h2 < 2; ++h2)
                tma_store_4d(&mO, s.q[t][h2], 64 * h2, it.kvh * p.G, it.i0 + t * p.rows_pos, it.b);
            tma_store_commit();
            tma_store_wait_read();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
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

bool encode4(CUtensorMap *m, const void *base, const cuuint64_t dims[4], const cuuint64_t strides[3],
             const cuuint32_t box[4])
{
    auto fn = encoder();
    if (!fn)
        return false;
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(int group, int H_kv) { return group >= 1 && group <= 128 && H_kv >= 1; }

int prefill_tc_rows_per_tile(int group) { return 128 / group; }

cudaError_t launch_prefill_tc(const PoolView &pv, const SeqDesc *d_seqs, const TcItem *d_items, int n_items, int B,
                              int n, int H_q, const void *q, void *out, cudaStream_t st)
{
    if (pv.d != D || n_items <= 0)
        return n_items <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    const int G = H_q / pv.H_kv;
    const int rows_pos = 128 / G;
    if (G < 1 || rows_pos < 1)
        return cudaErrorInvalidValue;
    CUtensorMap mq, mo, mkv;
    const cuuint64_t qdims[4] = {(cuuint64_t)D, (cuuint64_t)H_q, (cuuint64_t)n, (cuuint64_t)B};
    const cuuint64_t qstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)H_q * D * 2, (cuuint64_t)n * H_q * D * 2};
    const cuuint32_t qbox[4] = {64, (cuuint32_t)G, (cuuint32_t)rows_pos, 1};
    const cuuint64_t kvdims[4] = {(cuuint64_t)D, (cuuint64_t)kPageTokens, (cuuint64_t)2 * pv.H_kv,
                                  (cuuint64_t)pv.num_pages};
    const cuuint64_t kvstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)kPageTokens * D * 2,
                                 (cuuint64_t)2 * pv.H_kv * kPageTokens * D * 2};
    const cuuint32_t kvbox[4] = {64, (cuuint32_t)kPageTokens, 1, 1};
    if (!encode4(&mq, q, qdims, qstr, qbox) || !encode4(&mo, out, qdims, qstr, qbox) ||
        !encode4(&mkv, pv.pool, kvdims, kvstr, kvbox))
        return cudaErrorInvalidValue;
    TcParams prm;
    prm.seqs = d_seqs;
    prm.items = d_items;
    prm.tables = pv.tables;
    prm.stride = pv.stride;
    prm.num_pages = pv.num_pages;
    prm.H_kv = pv.H_kv;
    prm.G = G;
    prm.rows_pos = rows_pos;
    prm.err = pv.err;
    prm.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    const int smem = (int)sizeof(TcSmem) + 1024;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    prefill_tc_kernel<<<n_items, kThreads, smem, st>>>(mq, mo, mkv, prm);
    return cudaGetLastError();
}

}  // namespace gqa
