// k_decode.cu -- single-token decode over the paged cache, d_h = 128, bf16 or
// FP8 E4M3 cache: split-K partials, then a combine pass.
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
//  * FP8 E4M3 cache: half the bytes, but the FMA form above issues ~600
//    instructions per page, which bounds it (measured: the same time as the
//    bf16 cache), so both passes run as f16 mma.sync contractions instead
//    (q8_scores, q8_values: ~125 instructions per page);
//  * partials (max, sum, unnormalised o[g][128]) go to a workspace; the last
//    CTA of a (sequence, KV head) to finish merges its chunks in a fixed
//    order: M = max_s m_s, out = sum_s 2^(m_s-M) o_s / sum_s 2^(m_s-M) l_s.
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

// Eight consecutive bf16 row elements (one 16-byte load) as float pairs.
__device__ __forceinline__ void bf16x8(const uint4 &x, float2 (&f)[4])
{
    f[0] = bf2(x.x), f[1] = bf2(x.y), f[2] = bf2(x.z), f[3] = bf2(x.w);
}

// ---- FP8 E4M3 cache: both passes on mma.sync (m16n8k16, f16 operands,
// fp32 accumulation).  An E4M3 code is exact in f16 (one cvt per pair), so
// the score pass, S^T = K Q^T with the 16 tokens of a page as the M rows and
// the group's heads as the N columns, multiplies exact values; the value
// pass is O^T = V^T P'^T with 16 output columns as M rows and the page's
// tokens as K.  Both contractions may take the d_h axis in any order as long
// as the two operands agree, so each lane's K (V) loads are whole 16-byte
// pieces of rows and the fragments are assembled from them in registers:
// per page a lane issues four 16-byte loads, 32 conversions and 8 MMAs per
// pass, against ~300 instructions per pass for the FMA form of the bf16
// kernel.  Fragment coordinates follow the m16n8k16 layout: lane = 4 g + c;
// A rows g, g + 8 and B column g; A/B k-pairs 2c, 2c + 1 and 2c + 8, 2c + 9.

// Codes 0, 1 of w as an f16 pair (lo), codes 2, 3 (hi); the lower code in the
// lower half.
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi) : "r"(w));
}

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word(const uint4 &u, int i)
{
    return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w;
}

// One warp step of either E4M3 pass covers a pair of pages (chunk pages
// pg0, pg0 + 1): the page ids (-1 past the chunk) and this lane's four
// 16-byte pieces of each.  Score pass: rows g, g + 8, bytes 16c .. and
// 64 + 16c ..; value pass: rows 2c, 2c + 1, 2c + 8, 2c + 9, bytes 16g ...
// Score-pass steps also carry the row scales the step needs (K rows g,
// g + 8; V row "lane" for lanes < 16): they live at random addresses like
// the codes, so loading them at use would put a memory round trip inside
// every step.  Steps are loaded one ahead of their use, so a warp always has
// a step's bytes in flight while it computes.
struct Q8Pair {
    int page[2];
    uint4 r[2][4];
    float ks[2][2], vs[2];
};

template <bool VSIDE>
__device__ __forceinline__ void q8_load(const PoolView &pv, int kvh, const int32_t *__restrict__ tab, int npages,
                                        int pg0, int lane, Q8Pair &x)
{
    const int g = lane >> 2, c = lane & 3;
    constexpr size_t kBlk = (size_t)kPageTokens * D;    // bytes of one page block
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        x.page[pp] = pg0 + pp < npages ? tab[pg0 + pp] : -1;
        if ((unsigned)x.page[pp] < (unsigned)pv.num_pages) {
            const unsigned char *blk = reinterpret_cast<const unsigned char *>(pv.pool) +
                                       ((size_t)x.page[pp] * 2 * pv.H_kv + (VSIDE ? pv.H_kv : 0) + kvh) * kBlk;
            if (VSIDE) {
                blk += 16 * g;
                x.r[pp][0] = *reinterpret_cast<const uint4 *>(blk + (2 * c) * D);
                x.r[pp][1] = *reinterpret_cast<const uint4 *>(blk + (2 * c + 1) * D);
                x.r[pp][2] = *reinterpret_cast<const uint4 *>(blk + (2 * c + 8) * D);
                x.r[pp][3] = *reinterpret_cast<const uint4 *>(blk + (2 * c + 9) * D);
            } else {
                x.r[pp][0] = *reinterpret_cast<const uint4 *>(blk + g * D + 16 * c);
                x.r[pp][1] = *reinterpret_cast<const uint4 *>(blk + g * D + 64 + 16 * c);
                x.r[pp][2] = *reinterpret_cast<const uint4 *>(blk + (g + 8) * D + 16 * c);
                x.r[pp][3] = *reinterpret_cast<const uint4 *>(blk + (g + 8) * D + 64 + 16 * c);
                const float *scl = pv.scales + ((size_t)x.page[pp] * 2 * pv.H_kv + kvh) * kPageTokens;
                x.ks[pp][0] = scl[g];
                x.ks[pp][1] = scl[g + 8];
                x.vs[pp] = lane < kPageTokens ? scl[(size_t)pv.H_kv * kPageTokens + lane] : 0.0f;
            }
        }
    }
}

// Score pass over an E4M3 chunk.  Lane (g, c) loads, per page, bytes 16c ..
// 16c + 15 and 64 + 16c .. 64 + 16c + 15 of token rows g and g + 8: its 32
// codes per row, taken four per k-step (k-step s: codes 4s .. 4s + 3, i.e.
// dims 16c + 4s .. for s < 4 and 64 + 16c + 4(s - 4) .. after), which is the
// order in which q enters as the B operand.  q of head g is rounded to f16
// after an exact power-of-two scaling that puts its largest element in
// [2^14, 2^15) (bf16 values are then exact in f16); the factor is undone,
// together with log2(e)/sqrt(d_h) and the key row's scale, on the fp32
// score.  Also copies each page's V scales to vs and leaves their maximum
// (per warp) in vmax_w.
template <int G>
__device__ __forceinline__ void q8_scores(const PoolView &pv, const __nv_bfloat16 *__restrict__ qg, int kvh,
                                          const int32_t *__restrict__ tab, int npages, int nt, int t0, int ws,
                                          float (*sc)[G], float *vs, float *vmax_w, int warp, int lane)
{
    const int g = lane >> 2, c = lane & 3;
    uint32_t qf[8][2];
    float fac;                                          // 2^-k log2(e)/sqrt(d_h) of head g
    {
        float qv[32];
        if (g < G) {
            const uint4 *q4 = reinterpret_cast<const uint4 *>(qg + (size_t)g * D);
            const uint4 u[4] = {q4[2 * c], q4[2 * c + 1], q4[8 + 2 * c], q4[9 + 2 * c]};
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    qv[8 * j + 2 * i] = bf_lo(word(u[j], i));
                    qv[8 * j + 2 * i + 1] = bf_hi(word(u[j], i));
                }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                qv[i] = 0.0f;
        }
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            mx = fmaxf(mx, fabsf(qv[i]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // mx in [2^(E-127), 2^(E-126)): scale by 2^k, k = 141 - E, kept in
        // [-113, 100] so that both 2^k and 2^-k are normal floats.
        const int E = max((int)((__float_as_uint(mx) >> 23) & 0xffu), 1);
        const int k = min(max(141 - E, -113), 100);
        const float up = __uint_as_float((uint32_t)(127 + k) << 23);
        fac = __uint_as_float((uint32_t)(127 - k) << 23) * (1.4426950408889634f / sqrtf((float)D));
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            qf[s][0] = f16x2_rn(qv[4 * s] * up, qv[4 * s + 1] * up);
            qf[s][1] = f16x2_rn(qv[4 * s + 2] * up, qv[4 * s + 3] * up);
        }
    }
    __syncwarp();
    const float fac0 = __shfl_sync(0xffffffffu, fac, (8 * c) & 31);        // head 2c
    const float fac1 = __shfl_sync(0xffffffffu, fac, (8 * c + 4) & 31);    // head 2c + 1
    float vmax = 0.0f;
    Q8Pair cur, nxt;
    if (2 * warp < npages)
        q8_load<false>(pv, kvh, tab, npages, 2 * warp, lane, cur);
    for (int pg0 = 2 * warp; pg0 < npages; pg0 += 2 * kWarps) {
        if (pg0 + 2 * kWarps < npages)
            q8_load<false>(pv, kvh, tab, npages, pg0 + 2 * kWarps, lane, nxt);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            const int pg = pg0 + pp, page = cur.page[pp];
            if (pg >= npages)
                break;
            const bool ok = (unsigned)page < (unsigned)pv.num_pages;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            float ks0 = 0.f, ks1 = 0.f;
            if (ok) {
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    uint32_t a0, a1, a2, a3;
                    e4m3x4_f16x2(word(cur.r[pp][s >> 2], s & 3), a0, a2);
                    e4m3x4_f16x2(word(cur.r[pp][2 + (s >> 2)], s & 3), a1, a3);
                    mma_f16(d, a0, a1, a2, a3, qf[s][0], qf[s][1]);
                }
                ks0 = cur.ks[pp][0];
                ks1 = cur.ks[pp][1];
                if (lane < kPageTokens) {
                    vs[pg * kPageTokens + lane] = cur.vs[pp];
                    vmax = fmaxf(vmax, cur.vs[pp]);
                }
            } else if (lane == 0) {
                atomicOr(pv.err, kErrPageId);
            }
            // d: S^T rows g, g + 8 (tokens), columns 2c, 2c + 1 (heads).
            const int ta = pg * kPageTokens + g, tb = ta + 8;
            const bool va = ok && ta < nt && t0 + ta >= ws, vb = ok && tb < nt && t0 + tb >= ws;
            if (2 * c < G) {
                sc[ta][2 * c] = va ? d[0] * fac0 * ks0 : -INFINITY;
                sc[tb][2 * c] = vb ? d[2] * fac0 * ks1 : -INFINITY;
            }
            if (2 * c + 1 < G) {
                sc[ta][2 * c + 1] = va ? d[1] * fac1 * ks0 : -INFINITY;
                sc[tb][2 * c + 1] = vb ? d[3] * fac1 * ks1 : -INFINITY;
            }
            __syncwarp();                               // converged for the next page's MMAs
        }
        cur = nxt;
    }
    vmax = warp_max(vmax);
    if (lane == 0)
        vmax_w[warp] = vmax;
}

// Value pass over an E4M3 chunk (after the softmax): lane (g, c) loads bytes
// 16g .. 16g + 15 of token rows 2c, 2c + 1, 2c + 8, 2c + 9 of each page, so
// M-tile m's rows g, g + 8 are output columns 16g + m and 16g + 8 + m; a
// byte permute pairs the two tokens of a k-pair before each conversion.  The
// B operand is P'[h][t] = P[h][t] vs[t] / vmax in [0, 1], rounded to f16; the
// accumulated O^T is multiplied back by vmax and written to this warp's
// slice of red (heads 2c, 2c + 1, columns 16g .. 16g + 15).
template <int G>
__device__ __forceinline__ void q8_values(const PoolView &pv, int kvh, const int32_t *__restrict__ tab, int npages,
                                          const float (*sc)[G], const float *vs, float vmax, float (*red)[D],
                                          int warp, int lane, Q8Pair cur)
{
    const int g = lane >> 2, c = lane & 3;
    const float inv = vmax > 0.0f ? 1.0f / vmax : 0.0f;
    float o[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[m][i] = 0.0f;
    Q8Pair nxt;                                         // cur: the first step, loaded before the softmax
    for (int pg0 = 2 * warp; pg0 < npages; pg0 += 2 * kWarps) {
        if (pg0 + 2 * kWarps < npages)
            q8_load<true>(pv, kvh, tab, npages, pg0 + 2 * kWarps, lane, nxt);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            if ((unsigned)cur.page[pp] >= (unsigned)pv.num_pages)
                continue;                               // past the chunk, or a bad id (flagged in the score pass)
            uint32_t b0 = 0u, b1 = 0u;
            if (g < G) {
                const int t = (pg0 + pp) * kPageTokens + 2 * c;
                b0 = f16x2_rn(sc[t][g] * (vs[t] * inv), sc[t + 1][g] * (vs[t + 1] * inv));
                b1 = f16x2_rn(sc[t + 8][g] * (vs[t + 8] * inv), sc[t + 9][g] * (vs[t + 9] * inv));
            }
            __syncwarp();                               // converged for the MMAs
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                // Words w (columns 16g + 4w ..) and w + 2 (16g + 8 + 4w ..);
                // selector 0x5140 pairs bytes 0, 1 of two tokens, 0x7362 bytes 2, 3.
                uint32_t a[4][4];                       // [m - 4w][fragment register]
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int x = r & 2 ? 2 : 0;        // token pair: (2c, 2c + 1) or (2c + 8, 2c + 9)
                    const int wi = r & 1 ? w + 2 : w;   // fragment rows g (a0, a2) or g + 8 (a1, a3)
                    const int reg = (r & 1) | (r & 2);  // a0, a1, a2, a3
                    const uint32_t lo = prmt(word(cur.r[pp][x], wi), word(cur.r[pp][x + 1], wi), 0x5140u);
                    const uint32_t hi = prmt(word(cur.r[pp][x], wi), word(cur.r[pp][x + 1], wi), 0x7362u);
                    e4m3x4_f16x2(lo, a[0][reg], a[1][reg]);
                    e4m3x4_f16x2(hi, a[2][reg], a[3][reg]);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    mma_f16(o[4 * w + m], a[m][0], a[m][1], a[m][2], a[m][3], b0, b1);
            }
        }
        cur = nxt;
    }
    // o[m]: O^T rows g, g + 8 of M-tile m = output columns 16g + m, 16g + 8 + m;
    // columns 2c, 2c + 1 = heads.
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * c + hh;
        if (h < G) {
            float4 *dst = reinterpret_cast<float4 *>(&red[h][16 * g]);
            dst[0] = make_float4(o[0][hh] * vmax, o[1][hh] * vmax, o[2][hh] * vmax, o[3][hh] * vmax);
            dst[1] = make_float4(o[4][hh] * vmax, o[5][hh] * vmax, o[6][hh] * vmax, o[7][hh] * vmax);
            dst[2] = make_float4(o[0][2 + hh] * vmax, o[1][2 + hh] * vmax, o[2][2 + hh] * vmax, o[3][2 + hh] * vmax);
            dst[3] = make_float4(o[4][2 + hh] * vmax, o[5][2 + hh] * vmax, o[6][2 + hh] * vmax, o[7][2 + hh] * vmax);
        }
    }
}

// bf16 lane layout for both passes over a 16-token page: lane l covers
// tokens 2i + l/16 (i = 0..7) and columns 8(l%16)..8(l%16)+7, so one 16-byte
// load per lane reads two whole 256-byte token rows: 512 contiguous bytes.
// Q8: the pool holds FP8 E4M3 codes (a page block is [16 slots][128 bytes])
// and a scale per row, and both passes run on mma.sync (q8_scores,
// q8_values); the softmax and the merge are shared.
// KPRE (with ROPE): the pool holds keys before the rotation; each key row is
// rotated by its position as it is read (column c pairs with c + 64, held by
// lane ^ 8; cos/sin of the token's table row), in fp32.
template <int G, bool ROPE, bool Q8, bool KPRE>
__global__ void __launch_bounds__(kWarps * 32)
decode_split_kernel(PoolView pv, const SeqDesc *__restrict__ seqs, const DecodeItem *__restrict__ items,
                    const int32_t *__restrict__ item_start, int chunk, int H_q,
                    const __nv_bfloat16 *__restrict__ q, float *__restrict__ ws_o, float *__restrict__ ws_ml,
                    int32_t *__restrict__ counters, __nv_bfloat16 *__restrict__ out)
{
    __shared__ __align__(16) float sc[kMaxChunk][G];     // scores, then probabilities (token-major)
    __shared__ __align__(16) float red[kWarps][G][D];
    __shared__ float ml[G][2];
    __shared__ __align__(16) float q8_vs[Q8 ? kMaxChunk : 1];   // Q8: V row scales of the chunk
    __shared__ float q8_vmax[kWarps];

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
    // bf16: a page block (one head) is 256 uint4; lane l reads token 2i +
    // half, columns col..col+7, i.e. 128-byte chunk (l >> 3) & 1 of that row,
    // at uint4 offset (i / 4) * 128 + chunk * 64 + ((2i + half) % 8) * 8 + l % 8.
    const uint4 *pool = (const uint4 *)pv.pool;
    constexpr size_t kBlk = (size_t)kPageTokens * D * 2 / sizeof(uint4);
    const int half = lane >> 4, col = 8 * (lane & 15);
    const int lane_off = ((lane >> 3) & 1) * 64 + half * 8 + (lane & 7);
    auto row_at = [](int i) { return (i >> 2) * 128 + (i & 3) * 16; };   // token 2i + half

    Q8Pair q8_first;
    if constexpr (Q8) {
        q8_scores<G>(pv, q + ((size_t)it.b * H_q + kvh * G) * D, kvh, tab, npages, nt, t0, ws, sc, q8_vs, q8_vmax,
                     warp, lane);
        if (2 * warp < npages)                          // the value pass's first step, in flight over the softmax
            q8_load<true>(pv, kvh, tab, npages, 2 * warp, lane, q8_first);
    } else {
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
            const uint4 *kr = pool + ((size_t)page * 2 * H_kv + kvh) * kBlk + lane_off;
            uint4 kk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                kk[i] = kr[row_at(i)];                       // token 2i + half, columns col..col+7
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float2 w[4];
                bf16x8(kk[i], w);
                if (KPRE) {
                    const int pos = t0 + pg * kPageTokens + 2 * i + half;
                    const float4 *cs4 = reinterpret_cast<const float4 *>(pv.rope + (size_t)pos * (D / 2) + (col & 63));
                    const bool first = (lane & 8) == 0;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 c2 = __ldg(cs4 + u);     // (cos, sin) of columns 2u, 2u + 1 of the pair half
                        const float ox = __shfl_xor_sync(0xffffffffu, w[u].x, 8);
                        const float oy = __shfl_xor_sync(0xffffffffu, w[u].y, 8);
                        if (first)
                            w[u] = make_float2(w[u].x * c2.x - ox * c2.y, w[u].y * c2.z - oy * c2.w);
                        else
                            w[u] = make_float2(ox * c2.y + w[u].x * c2.x, oy * c2.w + w[u].y * c2.z);
                    }
                }
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
#pragma unroll
            for (int h = 0; h < G; ++h)
                sc[tl][h] = (ok && tl < nt && t0 + tl >= ws) ? v[0][h] : -INFINITY;
        }
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
    if constexpr (Q8) {
        float vmax = q8_vmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w)
            vmax = fmaxf(vmax, q8_vmax[w]);
        q8_values<G>(pv, kvh, tab, npages, sc, q8_vs, vmax, red[warp], warp, lane, q8_first);
    } else {
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
        const uint4 *vr = pool + ((size_t)page * 2 * H_kv + H_kv + kvh) * kBlk + lane_off;
        uint4 vv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            vv[i] = vr[row_at(i)];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int tl = pg * kPageTokens + 2 * i + half;   // probabilities are 0 past nt
            float2 w[4];
            bf16x8(vv[i], w);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pr = sc[tl][h];
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
        decode_split_kernel<G, false, true, false><<<grid, kWarps * 32, 0, st>>>(
            pv, a.seqs, a.items, a.item_start, a.chunk, a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
    else if (pv.rope && pv.keys_pre)
        decode_split_kernel<G, true, false, true><<<grid, kWarps * 32, 0, st>>>(
            pv, a.seqs, a.items, a.item_start, a.chunk, a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
    else if (pv.rope)
        decode_split_kernel<G, true, false, false><<<grid, kWarps * 32, 0, st>>>(
            pv, a.seqs, a.items, a.item_start, a.chunk, a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
    else
        decode_split_kernel<G, false, false, false><<<grid, kWarps * 32, 0, st>>>(
            pv, a.seqs, a.items, a.item_start, a.chunk, a.H_q, q, a.ws_o, a.ws_ml, a.counters, out);
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
