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
//  * K pass: a warp takes one 16-token page (4 KiB, contiguous); each
//    half-warp reads a whole 256-byte token row per 16-byte-per-lane load
//    (512 contiguous bytes per instruction), dots its 8 columns with q held
//    in registers (packed fp32 pairs), and a transpose-reduce over the 16
//    lanes of a row (token set halved at each exchange) forms the scores;
//  * softmax of the chunk is exact (chunk max, then exp2 and sum), kept as
//    (max, sum) for the combine;
//  * V pass: the same lane layout; each lane accumulates its 8 columns over
//    its half-warp's tokens with probabilities broadcast from shared memory,
//    then the half-warps and the warps are summed;
//  * partials (max, sum, unnormalised o[g][128]) go to a workspace; the last
//    CTA of a (sequence, KV head) to finish merges its chunks in a fixed
//    order: M = max_s m_s, out = sum_s 2^(m_s-M) o_s / sum_s 2^(m_s-M) l_s.
// Scores are carried in log2 units (q pre-scaled by log2(e)/sqrt(128)) so
// every exponential is one ex2.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

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

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// A bf16 pair (low half = lower index) as two floats.
__device__ __forceinline__ float2 bf2(uint32_t x) { return make_float2(bf_lo(x), bf_hi(x)); }

// Two FP8 E4M3 codes (low byte = lower index) as two floats (exact).
__device__ __forceinline__ float2 e4m3x2(uint32_t x)
{
    return __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(x & 0xffffu), __NV_E4M3)));
}

// Eight consecutive row elements of this lane as float pairs: a 16-byte
// load of bf16, or an 8-byte load of E4M3 codes (the row's scale is applied
// by the caller).
template <bool Q8>
struct RowLoad;
template <>
struct RowLoad<false> {
    using T = uint4;
    static __device__ __forceinline__ void pairs(const T &x, float2 (&f)[4])
    {
        f[0] = bf2(x.x), f[1] = bf2(x.y), f[2] = bf2(x.z), f[3] = bf2(x.w);
    }
};
template <>
struct RowLoad<true> {
    using T = uint2;
    static __device__ __forceinline__ void pairs(const T &x, float2 (&f)[4])
    {
        f[0] = e4m3x2(x.x), f[1] = e4m3x2(x.x >> 16), f[2] = e4m3x2(x.y), f[3] = e4m3x2(x.y >> 16);
    }
};

// Lane layout for both passes over a 16-token page: lane l covers tokens
// 2i + l/16 (i = 0..7) and columns 8(l%16)..8(l%16)+7, so one 16-byte load
// per lane reads two whole 256-byte token rows: 512 contiguous bytes.  Q8:
// the pool holds FP8 E4M3 codes (a page block is [16 slots][128 bytes]) and
// a scale per row; one 8-byte load per lane reads two 128-byte rows, and a
// row's scale multiplies its score (K) or its probability (V).
template <int G, bool ROPE, bool Q8>
__global__ void __launch_bounds__(kWarps * 32)
decode_split_kernel(PoolView pv, const SeqDesc *__restrict__ seqs, const DecodeItem *__restrict__ items,
                    const int32_t *__restrict__ item_start, int chunk, int H_q,
                    const __nv_bfloat16 *__restrict__ q, float *__restrict__ ws_o, float *__restrict__ ws_ml,
                    int32_t *__restrict__ counters, __nv_bfloat16 *__restrict__ out)
{
    __shared__ __align__(16) float sc[kMaxChunk][G];     // scores, then probabilities (token-major)
    __shared__ __align__(16) float red[kWarps][G][D];
    __shared__ float ml[G][2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DecodeItem it = items[blockIdx.x];
    const int kvh = blockIdx.y;
    const int H_kv = pv.H_kv;
    const SeqDesc sd = seqs[it.b];
    const int L = sd.past + 1;
    const int ws = window_start(L - 1, pv.window);       // first visible key
    const int t0 = decode_first_token(L, pv.window) + it.split * chunk;
    const int nt = min(chunk, L - t0);
    const int npages = (nt + kPageTokens - 1) / kPageTokens;
    const int32_t *tab = pv.tables + (size_t)sd.row * pv.stride + t0 / kPageTokens;
    using RL = RowLoad<Q8>;
    using LT = typename RL::T;
    const LT *pool = (const LT *)pv.pool;
    // bf16: a page block (one head) is 256 uint4; lane l reads token 2i +
    // half, columns col..col+7, i.e. 128-byte chunk (l >> 3) & 1 of that row,
    // at uint4 offset (i / 4) * 128 + chunk * 64 + ((2i + half) % 8) * 8 + l % 8.
    // E4M3: a page block is 256 uint2, token t's row at uint2 offset 16 t.
    constexpr size_t kBlk = (size_t)kPageTokens * D * (Q8 ? 1 : 2) / sizeof(LT);
    const int half = lane >> 4, col = 8 * (lane & 15);
    const int lane_off = Q8 ? half * 16 + (lane & 15) : ((lane >> 3) & 1) * 64 + half * 8 + (lane & 7);
    auto row_at = [](int i) { return Q8 ? i * 32 : (i >> 2) * 128 + (i & 3) * 16; };   // token 2i + half

    // This lane's eight q columns of every head of the group, pre-scaled by
    // log2(e)/sqrt(d_h) so scores come out in exp2 units.
    const float qscale = 1.4426950408889634f / sqrtf((float)D);
    float2 qr[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 qv = *reinterpret_cast<const uint4 *>(q + ((size_t)it.b * H_q + kvh * G + h) * D + col);
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
            qr[h][u] = make_float2(bf_lo(w[u]) * qscale, bf_hi(w[u]) * qscale);
    }
    if (ROPE) {
        // Rotate q by its position L - 1: column c pairs with c + 64, held by
        // lane ^ 8 at the same register.
        const float4 *cs4 = reinterpret_cast<const float4 *>(pv.rope + (size_t)sd.past * (D / 2) + 8 * (lane & 7));
        const bool first = (lane & 8) == 0;
        float2 cs[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 t = cs4[j];
            cs[2 * j] = make_float2(t.x, t.y);
            cs[2 * j + 1] = make_float2(t.z, t.w);
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float ox = __shfl_xor_sync(0xffffffffu, qr[h][u].x, 8);
                const float oy = __shfl_xor_sync(0xffffffffu, qr[h][u].y, 8);
                const float2 c0 = cs[2 * u], c1 = cs[2 * u + 1];
                if (first)
                    qr[h][u] = make_float2(qr[h][u].x * c0.x - ox * c0.y, qr[h][u].y * c1.x - oy * c1.y);
                else
                    qr[h][u] = make_float2(ox * c0.y + qr[h][u].x * c0.x, oy * c1.y + qr[h][u].y * c1.x);
            }
    }

    // ---- K pass: scores of the chunk -------------------------------------
    for (int pg = warp; pg < npages; pg += kWarps) {
        const int page = tab[pg];
        const bool ok = (unsigned)page < (unsigned)pv.num_pages;
        float v[8][G];
        if (ok) {
            const LT *kr = pool + ((size_t)page * 2 * H_kv + kvh) * kBlk + lane_off;
            LT kk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                kk[i] = kr[row_at(i)];                       // token 2i + half, columns col..col+7
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float2 w[4];
                RL::pairs(kk[i], w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 a = make_float2(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        a = fma2(w[u], qr[h][u], a);
                    v[i][h] = a.x + a.y;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int h = 0; h < G; ++h)
                    v[i][h] = 0.f;
            if (lane == 0)
                atomicOr(pv.err, kErrPageId);
        }
        // Sum each token's 16 column slices: halve the token set at every
        // exchange (xor 8, 4, 2), then finish the last pair (xor 1).
        const int b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float send = b3 ? v[i][h] : v[i + 4][h];
                const float keep = b3 ? v[i + 4][h] : v[i][h];
                v[i][h] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float send = b2 ? v[i][h] : v[i + 2][h];
                const float keep = b2 ? v[i + 2][h] : v[i][h];
                v[i][h] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float send = b1 ? v[0][h] : v[1][h];
            const float keep = b1 ? v[1][h] : v[0][h];
            v[0][h] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
            v[0][h] += __shfl_xor_sync(0xffffffffu, v[0][h], 1);
        // Lane pair (l, l^1) now holds token 2(4 b3 + 2 b2 + b1) + half.
        const int tl = pg * kPageTokens + 2 * (4 * b3 + 2 * b2 + b1) + half;
        if ((lane & 1) == 0) {
            const float ks = (Q8 && ok) ? pv.scales[((size_t)page * 2 * H_kv + kvh) * kPageTokens + tl % kPageTokens]
                                        : 1.0f;
#pragma unroll
            for (int h = 0; h < G; ++h)
                sc[tl][h] = (ok && tl < nt && t0 + tl >= ws) ? (Q8 ? v[0][h] * ks : v[0][h]) : -INFINITY;
        }
    }
    __syncthreads();

    // ---- exact softmax over the chunk, per head --------------------------
    const int nslots = npages * kPageTokens;
    for (int h = warp; h < G; h += kWarps) {
        float mx = -INFINITY;
        for (int t = lane; t < nslots; t += 32)
            mx = fmaxf(mx, sc[t][h]);
        mx = warp_max(mx);
        float sum = 0.0f;
        for (int t = lane; t < nslots; t += 32) {
            const float s2 = sc[t][h];
            const float pr = (s2 == -INFINITY) ? 0.0f : ex2(s2 - mx);
            sc[t][h] = pr;
            sum += pr;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            ml[h][0] = mx;
            ml[h][1] = sum;
        }
    }
    __syncthreads();

    // ---- V pass: o[h][col..col+7] over this half-warp's tokens -----------
    float2 o[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int u = 0; u < 4; ++u)
            o[h][u] = make_float2(0.f, 0.f);
    for (int pg = warp; pg < npages; pg += kWarps) {
        const int page = tab[pg];
        if ((unsigned)page >= (unsigned)pv.num_pages)
            continue;
        const LT *vr = pool + ((size_t)page * 2 * H_kv + H_kv + kvh) * kBlk + lane_off;
        const float *vsc = Q8 ? pv.scales + ((size_t)page * 2 * H_kv + H_kv + kvh) * kPageTokens : nullptr;
        LT vv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            vv[i] = vr[row_at(i)];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int tl = pg * kPageTokens + 2 * i + half;   // probabilities are 0 past nt
            float2 w[4];
            RL::pairs(vv[i], w);
            const float vs = Q8 ? vsc[2 * i + half] : 1.0f;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pr = Q8 ? sc[tl][h] * vs : sc[tl][h];
                const float2 pp = make_float2(pr, pr);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    o[h][u] = fma2(pp, w[u], o[h][u]);
            }
        }
    }
    // Join the two half-warps (different tokens, same columns), then the warps.
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            o[h][u].x += __shfl_xor_sync(0xffffffffu, o[h][u].x, 16);
            o[h][u].y += __shfl_xor_sync(0xffffffffu, o[h][u].y, 16);
        }
    if (half == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4 *dst = reinterpret_cast<float4 *>(&red[warp][h][col]);
            dst[0] = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
            dst[1] = make_float4(o[h][2].x, o[h][2].y, o[h][3].x, o[h][3].y);
        }
    }
    __syncthreads();

    // ---- merge the chunks ----------------------------------------------------
    // A single chunk is the whole sequence: write out directly.  Otherwise
    // each CTA leaves its partial (max, sum, o) in the workspace and bumps the
    // (entry, KV head) counter; the CTA that arrives last merges all chunks in
    // chunk order -- M = max m_s, out = sum 2^(m_s-M) o_s / sum 2^(m_s-M) l_s --
    // and resets the counter for the next call.  No CTA waits on another.
    const int i0 = item_start[it.b];
    const int ns = item_start[it.b + 1] - i0;
    const int e = threadIdx.x;                         // one output column per thread (128 = d_h)
    if (ns == 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float acc = red[0][h][e];
#pragma unroll
            for (int w = 1; w < kWarps; ++w)
                acc += red[w][h][e];
            out[((size_t)it.b * H_q + kvh * G + h) * D + e] = __float2bfloat16_rn(acc / ml[h][1]);
        }
        return;
    }
    float *wo = ws_o + ((size_t)blockIdx.x * H_kv + kvh) * G * D;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float acc = red[0][h][e];
#pragma unroll
        for (int w = 1; w < kWarps; ++w)
            acc += red[w][h][e];
        wo[h * D + e] = acc;
    }
    if (threadIdx.x < G) {
        float *wm = ws_ml + (((size_t)blockIdx.x * H_kv + kvh) * G + threadIdx.x) * 2;
        wm[0] = ml[threadIdx.x][0];
        wm[1] = ml[threadIdx.x][1];
    }
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(&counters[(size_t)it.b * H_kv + kvh], 1);
        s_last = prev == ns - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    // The merge reads ns partials per head; with many chunks (a long
    // sequence in a small batch) one thread walking them in turn would wait
    // out an L2 round trip per chunk, so the loads are spread: warp w takes
    // chunks w, w + 4, ..., lane l columns 4l..4l+3 of every head, and the
    // four warps' sums meet in shared memory.
    const size_t stride = (size_t)H_kv * G;            // between consecutive chunks' partials
    const float *ml0 = ws_ml + ((size_t)i0 * H_kv + kvh) * G * 2;
    const float *po0 = ws_o + ((size_t)i0 * H_kv + kvh) * G * D;
    __shared__ float sM[G], sden[kWarps][G];
    for (int h = warp; h < G; h += kWarps) {           // M = max over chunks of m
        float M = -INFINITY;
        for (int i = lane; i < ns; i += 32)
            M = fmaxf(M, __ldcg(ml0 + (i * stride + h) * 2));
#pragma unroll
        for (int o = 16; o; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if (lane == 0)
            sM[h] = M;
    }
    __syncthreads();
    float4 acc[G];
    float den[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
        den[h] = 0.f;
    }
#pragma unroll 1
    for (int i = warp; i < ns; i += kWarps) {          // a fixed order per warp
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float2 mlv = __ldcg(reinterpret_cast<const float2 *>(ml0 + (i * stride + h) * 2));
            const float4 o4 = __ldcg(reinterpret_cast<const float4 *>(po0 + (i * stride + h) * D) + lane);
            const float w = ex2(mlv.x - sM[h]);
            den[h] = fmaf(w, mlv.y, den[h]);
            acc[h].x = fmaf(w, o4.x, acc[h].x);
            acc[h].y = fmaf(w, o4.y, acc[h].y);
            acc[h].z = fmaf(w, o4.z, acc[h].z);
            acc[h].w = fmaf(w, o4.w, acc[h].w);
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        *reinterpret_cast<float4 *>(&red[warp][h][4 * lane]) = acc[h];
        if (lane == 0)
            sden[warp][h] = den[h];
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float a = 0.f, dn = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {             // warps in a fixed order
            a += red[w][h][e];
            dn += sden[w][h];
        }
        out[((size_t)it.b * H_q + kvh * G + h) * D + e] = __float2bfloat16_rn(a / dn);
    }
    if (threadIdx.x == 0)
        counters[(size_t)it.b * H_kv + kvh] = 0;
}

template <int G>
cudaError_t launch_g(const PoolView &pv, const DecodeLaunch &a, cudaStream_t st)
{
    dim3 grid((unsigned)a.n_items, (unsigned)pv.H_kv);
    // The rotating and the quantised kernels are separate instantiations, so
    // that a plain bf16 cache runs the plain one.
    const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q;
    __nv_bfloat16 *out = (__nv_bfloat16 *)a.out;
    if (pv.dtype == kDtypeFp8)
        decode_split_kernel<G, false, true><<<grid, kWarps * 32, 0, st>>>(pv, a.seqs, a.items, a.item_start, a.chunk,
                                                                         a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
    else if (pv.rope)
        decode_split_kernel<G, true, false><<<grid, kWarps * 32, 0, st>>>(pv, a.seqs, a.items, a.item_start, a.chunk,
                                                                         a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
    else
        decode_split_kernel<G, false, false><<<grid, kWarps * 32, 0, st>>>(pv, a.seqs, a.items, a.item_start, a.chunk,
                                                                          a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
    return cudaGetLastError();
}

}  // namespace

bool decode_split_supported(int group) { return group >= 1 && group <= 8; }

cudaError_t launch_decode_split(const PoolView &pv, const DecodeLaunch &a, cudaStream_t st)
{
    if (pv.d != D || a.chunk <= 0 || a.chunk > kMaxChunk || a.chunk % kPageTokens != 0)
        return cudaErrorInvalidValue;
    if (a.n_items <= 0)
        return cudaSuccess;
    switch (a.H_q / pv.H_kv) {
    case 1: return launch_g<1>(pv, a, st);
    case 2: return launch_g<2>(pv, a, st);
    case 3: return launch_g<3>(pv, a, st);
    case 4: return launch_g<4>(pv, a, st);
    case 5: return launch_g<5>(pv, a, st);
    case 6: return launch_g<6>(pv, a, st);
    case 7: return launch_g<7>(pv, a, st);
    case 8: return launch_g<8>(pv, a, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace gqa
