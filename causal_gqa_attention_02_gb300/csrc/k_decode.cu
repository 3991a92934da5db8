// k_decode.cu -- single-token decode over the paged cache, bf16, d_h = 128:
// split-K partials, then a combine pass.
//
// What it computes ("KV Cache 与 Prefill/Decode 推理路径", decode lesson: the
// single new query reads every cached key, old ones and its own; the
// PagedAttention section: keys are found through the block table; and
// "第二章 Prefill：整层状态演化与 KV 建立" section 2.3 for the scores and the
// softmax): for each query head h of KV group g,
//     out[b,h] = sum_t softmax_t(<q[b,h], K[t,g]>/sqrt(128)) V[t,g].
//
// Decode reads every cached K/V byte once and does ~1 flop per byte per
// query head, so it is bound by HBM bandwidth.  Design for that:
//  * one CTA per (batch entry, token chunk, KV head): all g = H_q/H_kv query
//    heads of the group are served from one read of the group's K/V (the
//    KV head is indexed, never duplicated);
//  * K pass: a warp takes one 16-token page (4 KiB, contiguous); lane pair
//    (2t, 2t+1) reads token t's row as eight 16-byte loads each, dots it
//    with q held in shared memory, and one shuffle joins the two halves;
//  * softmax of the chunk is exact (chunk max, then exp2 and sum), kept as
//    (max, sum) for the combine;
//  * V pass: a warp takes a page; lane l owns output elements 4l..4l+3 and
//    reads them for all 16 tokens with 8-byte loads (a warp covers one
//    256-byte row per load: coalesced);
//  * partials (max, sum, unnormalised o[g][128]) go to a workspace; the
//    combine kernel merges a sequence's chunks in a fixed order:
//        M = max_s m_s,  out = sum_s 2^(m_s-M) o_s / sum_s 2^(m_s-M) l_s.
// Scores are carried in log2 units (q pre-scaled by log2(e)/sqrt(128)) so
// every exponential is one ex2.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace gqa {

namespace {

constexpr int D = 128;
constexpr int kWarps = 4;
constexpr int kMaxChunk = 512;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float x)
{
    for (int o = 16; o > 0; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int G>
__global__ void __launch_bounds__(kWarps * 32)
decode_split_kernel(PoolView pv, const SeqDesc *__restrict__ seqs, const DecodeItem *__restrict__ items,
                    int chunk, int H_q, const __nv_bfloat16 *__restrict__ q, float *__restrict__ ws_o,
                    float *__restrict__ ws_ml)
{
    // q split in two halves of 64, the second offset by 68 floats so the two
    // halves' broadcasts fall in different banks.
    __shared__ __align__(16) float qs[G][2][68];
    __shared__ float sc[G][kMaxChunk];
    __shared__ __align__(16) float red[kWarps][G][D];
    __shared__ float ml[G][2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DecodeItem it = items[blockIdx.x];
    const int kvh = blockIdx.y;
    const int H_kv = pv.H_kv;
    const SeqDesc sd = seqs[it.b];
    const int L = sd.past + 1;
    const int t0 = it.split * chunk;
    const int nt = min(chunk, L - t0);
    const int npages = (nt + kPageTokens - 1) / kPageTokens;
    const int32_t *tab = pv.tables + (size_t)sd.row * pv.stride + t0 / kPageTokens;
    const __nv_bfloat16 *pool = (const __nv_bfloat16 *)pv.pool;
    const size_t page_elems = (size_t)2 * H_kv * kPageTokens * D;

    const float qscale = 1.4426950408889634f / sqrtf((float)D);   // log2(e) / sqrt(d_h)
    for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
        const int h = idx / D, e = idx % D;
        qs[h][e / 64][e % 64] = __bfloat162float(q[((size_t)it.b * H_q + kvh * G + h) * D + e]) * qscale;
    }
    __syncthreads();

    // ---- K pass: scores of the chunk -------------------------------------
    {
        const int tok = lane >> 1, half = lane & 1;
        for (int pg = warp; pg < npages; pg += kWarps) {
            const int page = tab[pg];
            const bool ok = (unsigned)page < (unsigned)pv.num_pages;
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h)
                acc[h] = 0.0f;
            if (ok) {
                const uint4 *kr = reinterpret_cast<const uint4 *>(pool + (size_t)page * page_elems +
                                                                  (size_t)kvh * kPageTokens * D) +
                                  tok * 16 + half * 8;
                uint4 kk[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    kk[j] = kr[j];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float f[8] = {bf_lo(kk[j].x), bf_hi(kk[j].x), bf_lo(kk[j].y), bf_hi(kk[j].y),
                                        bf_lo(kk[j].z), bf_hi(kk[j].z), bf_lo(kk[j].w), bf_hi(kk[j].w)};
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 qa = *reinterpret_cast<const float4 *>(&qs[h][half][j * 8]);
                        const float4 qb = *reinterpret_cast<const float4 *>(&qs[h][half][j * 8 + 4]);
                        float a = acc[h];
                        a = fmaf(f[0], qa.x, a); a = fmaf(f[1], qa.y, a);
                        a = fmaf(f[2], qa.z, a); a = fmaf(f[3], qa.w, a);
                        a = fmaf(f[4], qb.x, a); a = fmaf(f[5], qb.y, a);
                        a = fmaf(f[6], qb.z, a); a = fmaf(f[7], qb.w, a);
                        acc[h] = a;
                    }
                }
            } else if (lane == 0) {
                atomicOr(pv.err, kErrPageId);
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
                acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
            const int tl = pg * kPageTokens + tok;
            if (half == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    sc[h][tl] = (ok && tl < nt) ? acc[h] : -INFINITY;
            }
        }
    }
    __syncthreads();

    // ---- exact softmax over the chunk, per head --------------------------
    const int nslots = npages * kPageTokens;
    for (int h = warp; h < G; h += kWarps) {
        float mx = -INFINITY;
        for (int t = lane; t < nslots; t += 32)
            mx = fmaxf(mx, sc[h][t]);
        mx = warp_max(mx);
        float sum = 0.0f;
        for (int t = lane; t < nslots; t += 32) {
            const float s = sc[h][t];
            const float p = (s == -INFINITY) ? 0.0f : ex2(s - mx);
            sc[h][t] = p;
            sum += p;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            ml[h][0] = mx;
            ml[h][1] = sum;
        }
    }
    __syncthreads();

    // ---- V pass: o[h][4*lane .. 4*lane+3] ---------------------------------
    float o[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
        o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.0f;
    for (int pg = warp; pg < npages; pg += kWarps) {
        const int page = tab[pg];
        if ((unsigned)page >= (unsigned)pv.num_pages)
            continue;
        const uint2 *vr = reinterpret_cast<const uint2 *>(pool + (size_t)page * page_elems +
                                                          (size_t)(H_kv + kvh) * kPageTokens * D) + lane;
        uint2 vv[kPageTokens];
#pragma unroll
        for (int tk = 0; tk < kPageTokens; ++tk)
            vv[tk] = vr[tk * (D / 4)];
#pragma unroll
        for (int tk = 0; tk < kPageTokens; ++tk) {
            const int tl = pg * kPageTokens + tk;
            if (tl < nt) {
                const float f0 = bf_lo(vv[tk].x), f1 = bf_hi(vv[tk].x);
                const float f2 = bf_lo(vv[tk].y), f3 = bf_hi(vv[tk].y);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float p = sc[h][tl];
                    o[h][0] = fmaf(p, f0, o[h][0]);
                    o[h][1] = fmaf(p, f1, o[h][1]);
                    o[h][2] = fmaf(p, f2, o[h][2]);
                    o[h][3] = fmaf(p, f3, o[h][3]);
                }
            }
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
        *reinterpret_cast<float4 *>(&red[warp][h][4 * lane]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    __syncthreads();

    float *wo = ws_o + ((size_t)blockIdx.x * H_kv + kvh) * G * D;
    for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
        const int h = idx / D, e = idx % D;
        float s = red[0][h][e];
#pragma unroll
        for (int w = 1; w < kWarps; ++w)
            s += red[w][h][e];
        wo[idx] = s;
    }
    if (threadIdx.x < G) {
        float *wm = ws_ml + (((size_t)blockIdx.x * H_kv + kvh) * G + threadIdx.x) * 2;
        wm[0] = ml[threadIdx.x][0];
        wm[1] = ml[threadIdx.x][1];
    }
}

// One CTA per (query head, batch entry); thread e owns output element e.
__global__ void __launch_bounds__(D)
decode_combine_kernel(const int32_t *__restrict__ item_start, int H_q, int H_kv,
                      const float *__restrict__ ws_o, const float *__restrict__ ws_ml,
                      __nv_bfloat16 *__restrict__ out)
{
    const int h = blockIdx.x, b = blockIdx.y, e = threadIdx.x;
    const int G = H_q / H_kv, kvh = h / G, hh = h % G;
    const int i0 = item_start[b], i1 = item_start[b + 1];
    float M = -INFINITY;
    for (int i = i0; i < i1; ++i)
        M = fmaxf(M, ws_ml[(((size_t)i * H_kv + kvh) * G + hh) * 2]);
    float den = 0.0f, acc = 0.0f;
    for (int i = i0; i < i1; ++i) {
        const float *m = ws_ml + (((size_t)i * H_kv + kvh) * G + hh) * 2;
        const float w = ex2(m[0] - M);
        den = fmaf(w, m[1], den);
        acc = fmaf(w, ws_o[(((size_t)i * H_kv + kvh) * G + hh) * D + e], acc);
    }
    out[((size_t)b * H_q + h) * D + e] = __float2bfloat16_rn(acc / den);
}

template <int G>
cudaError_t launch_g(const PoolView &pv, const SeqDesc *d_seqs, const DecodeItem *d_items, int n_items,
                     int chunk, int H_q, const void *q, float *ws_o, float *ws_ml, cudaStream_t st)
{
    dim3 grid((unsigned)n_items, (unsigned)pv.H_kv);
    decode_split_kernel<G><<<grid, kWarps * 32, 0, st>>>(pv, d_seqs, d_items, chunk, H_q,
                                                        (const __nv_bfloat16 *)q, ws_o, ws_ml);
    return cudaGetLastError();
}

}  // namespace

bool decode_split_supported(int group) { return group >= 1 && group <= 8; }

cudaError_t launch_decode_split(const PoolView &pv, const SeqDesc *d_seqs, const DecodeItem *d_items,
                                int n_items, int chunk, int H_q, const void *q, float *ws_o,
                                float *ws_ml, cudaStream_t st)
{
    if (pv.d != D || chunk <= 0 || chunk > kMaxChunk || chunk % kPageTokens != 0)
        return cudaErrorInvalidValue;
    if (n_items <= 0)
        return cudaSuccess;
    switch (H_q / pv.H_kv) {
    case 1: return launch_g<1>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 2: return launch_g<2>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 3: return launch_g<3>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 4: return launch_g<4>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 5: return launch_g<5>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 6: return launch_g<6>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 7: return launch_g<7>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    case 8: return launch_g<8>(pv, d_seqs, d_items, n_items, chunk, H_q, q, ws_o, ws_ml, st);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_decode_combine(const int32_t *d_item_start, int B, int H_q, int H_kv,
                                  const float *ws_o, const float *ws_ml, void *out, cudaStream_t st)
{
    if (B <= 0)
        return cudaSuccess;
    dim3 grid((unsigned)H_q, (unsigned)B);
    decode_combine_kernel<<<grid, D, 0, st>>>(d_item_start, H_q, H_kv, ws_o, ws_ml,
                                              (__nv_bfloat16 *)out);
    return cudaGetLastError();
}

}  // namespace gqa
