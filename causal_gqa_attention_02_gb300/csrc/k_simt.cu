// k_simt.cu -- generic causal GQA attention over the paged cache on the
// CUDA cores, for fp32 caches and head sizes the tensor-core kernels do not
// take.  It is the precise path (fp32 arithmetic, expf), not the fast one.
//
// What it computes: "第二章 Prefill：整层状态演化与 KV 建立", section 2.3:
// query head h reads KV head g(h) = floor(h*H_kv/H_q); scores are
// <q, k_j>/sqrt(d_h) over the visible keys; a stable softmax over the finite
// scores weights V.  Visibility: a row at absolute position p sees cached
// positions 0..p ("KV Cache 与 Prefill/Decode 推理路径", incremental prefill:
// the old prefix is a fully visible rectangle, the new block a triangle).
//
// Shape of the work: one warp per query row.  Keys are taken 32 at a time,
// one key per lane (each lane forms its own dot product against the row's q
// held in shared memory), so a block of 32 scores costs one warp max and one
// warp sum; the running max / sum / output are rescaled once per block
// (online softmax, the FlashAttention recurrence).  The value pass keeps the
// output row spread over the lanes (lane owns elements lane, lane+32, ...).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace gqa {

namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 256;

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

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

// T: element type of q and out (and of the pool unless Q8); Q8: the pool
// holds FP8 E4M3 codes with a scale per row, read as fp32(decode(code) * s);
// KPRE: the pool holds keys before the rotation, and each key is rotated by
// its position as it is read (pairs (e, e + d/2), fp32).
template <typename T, bool Q8, bool KPRE>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_kernel(PoolView pv, const SeqDesc *__restrict__ seqs, int n, int H_q,
                 const T *__restrict__ q, T *__restrict__ out)
{
    __shared__ float sq[kWarps][kMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int i = blockIdx.x * kWarps + warp;
    if (i >= n)
        return;                                   // no block-wide barrier follows
    const SeqDesc sd = seqs[b];
    const int d = pv.d, H_kv = pv.H_kv;
    T *o = out + (((size_t)b * n + i) * H_q + h) * d;
    if (i >= sd.count) {                          // padding row: discarded, written as 0
        for (int e = lane; e < d; e += 32)
            stf(o + e, 0.0f);
        return;
    }
    const int g = (int)(((long long)h * H_kv) / H_q);
    const T *qi = q + (((size_t)b * n + i) * H_q + h) * d;
    float *qs = sq[warp];
    for (int e = lane; e < d; e += 32)
        qs[e] = ldf(qi + e);
    __syncwarp();
    if (pv.rope) {                                // rotate q by its position, pairs (e, e + d/2)
        const float2 *cs = pv.rope + (size_t)(sd.past + i) * (d / 2);
        for (int e = lane; e < d / 2; e += 32) {
            const float x = qs[e], y = qs[e + d / 2];
            const float2 t = cs[e];
            qs[e] = x * t.x - y * t.y;
            qs[e + d / 2] = x * t.y + y * t.x;
        }
        __syncwarp();
    }

    const float root_d = sqrtf((float)d);
    const int pos = sd.past + i;                  // visible keys 0..pos
    const int32_t *tab = pv.tables + (size_t)sd.row * pv.stride;
    const char *pool = (const char *)pv.pool;
    const int es = Q8 ? 1 : (int)sizeof(T);
    const int chunks = pool_chunks(d * es);
    const size_t blk_bytes = pool_block_bytes(d * es);
    const size_t k_off = (size_t)g * blk_bytes;
    const size_t v_off = (size_t)(H_kv + g) * blk_bytes;
    // Element e of the row of `slot` in block `bi` (page * 2 H_kv + kv * H_kv + g),
    // whose bytes start at `blk`.
    auto elem = [&](const char *blk, size_t bi, int slot, int e) -> float {
        if (Q8) {
            const __nv_fp8_storage_t c = *(const __nv_fp8_storage_t *)(blk + pool_in_block(chunks, slot, e));
            const float x = __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
            return __fmul_rn(x, pv.scales[bi * kPageTokens + slot]);
        }
        return ldf((const T *)(blk + pool_in_block(chunks, slot, e * es)));
    };

    float m = -INFINITY, l = 0.0f;
    float acc[kMaxD / 32];
#pragma unroll
    for (int j = 0; j < kMaxD / 32; ++j)
        acc[j] = 0.0f;

    for (int kb = window_start(pos, pv.window); kb <= pos; kb += 32) {   // keys qlo..pos
        const int t = kb + lane;
        float s = -INFINITY;
        if (t <= pos) {
            const int page = tab[t / kPageTokens];
            if ((unsigned)page < (unsigned)pv.num_pages) {
                const char *kb_ = pool + (size_t)page * 2 * H_kv * blk_bytes + k_off;
                const size_t kbi = (size_t)page * 2 * H_kv + g;
                float dot = 0.0f;
                if (KPRE) {
                    const float2 *cs = pv.rope + (size_t)t * (d / 2);
                    for (int e = 0; e < d / 2; ++e) {
                        const float x = elem(kb_, kbi, t % kPageTokens, e);
                        const float y = elem(kb_, kbi, t % kPageTokens, e + d / 2);
                        const float2 r = cs[e];
                        dot = fmaf(qs[e], x * r.x - y * r.y, dot);
                        dot = fmaf(qs[e + d / 2], x * r.y + y * r.x, dot);
                    }
                } else {
                    for (int e = 0; e < d; ++e)
                        dot = fmaf(qs[e], elem(kb_, kbi, t % kPageTokens, e), dot);
                }
                s = dot / root_d;
            } else {
                atomicOr(pv.err, kErrPageId);
            }
        }
        const float m_new = fmaxf(m, warp_max(s));
        const float corr = (m == -INFINITY) ? 0.0f : expf(m - m_new);
        const float p = (s == -INFINITY) ? 0.0f : expf(s - m_new);
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int j = 0; j < kMaxD / 32; ++j)
            acc[j] *= corr;
        const int nk = min(32, pos - kb + 1);
        for (int u = 0; u < nk; ++u) {
            const float pu = __shfl_sync(0xffffffffu, p, u);
            const int tu = kb + u;
            const int page = tab[tu / kPageTokens];
            if ((unsigned)page >= (unsigned)pv.num_pages)
                continue;
            const char *vb_ = pool + (size_t)page * 2 * H_kv * blk_bytes + v_off;
            const size_t vbi = (size_t)page * 2 * H_kv + H_kv + g;
#pragma unroll
            for (int j = 0; j < kMaxD / 32; ++j) {
                const int e = lane + 32 * j;
                if (e < d)
                    acc[j] = fmaf(pu, elem(vb_, vbi, tu % kPageTokens, e), acc[j]);
            }
        }
        m = m_new;
    }
    const float inv = 1.0f / l;
#pragma unroll
    for (int j = 0; j < kMaxD / 32; ++j) {
        const int e = lane + 32 * j;
        if (e < d)
            stf(o + e, acc[j] * inv);
    }
}

}  // namespace

cudaError_t launch_attn_simt(const PoolView &pv, int dtype, const SeqDesc *d_seqs, int B, int n,
                             int H_q, const void *q, void *out, cudaStream_t st)
{
    if (pv.d > kMaxD || pv.d < 1)
        return cudaErrorInvalidValue;
    if (B <= 0 || n <= 0)
        return cudaSuccess;
    dim3 grid((unsigned)((n + kWarps - 1) / kWarps), (unsigned)H_q, (unsigned)B);
    const bool kpre = pv.keys_pre && pv.rope;
    if (dtype == kDtypeF32 && kpre)
        attn_simt_kernel<float, false, true><<<grid, kWarps * 32, 0, st>>>(pv, d_seqs, n, H_q, (const float *)q,
                                                                         (float *)out);
    else if (dtype == kDtypeF32)
        attn_simt_kernel<float, false, false><<<grid, kWarps * 32, 0, st>>>(pv, d_seqs, n, H_q, (const float *)q,
                                                                          (float *)out);
    else if (dtype == kDtypeFp8)
        attn_simt_kernel<__nv_bfloat16, true, false><<<grid, kWarps * 32, 0, st>>>(
            pv, d_seqs, n, H_q, (const __nv_bfloat16 *)q, (__nv_bfloat16 *)out);
    else if (kpre)
        attn_simt_kernel<__nv_bfloat16, false, true><<<grid, kWarps * 32, 0, st>>>(
            pv, d_seqs, n, H_q, (const __nv_bfloat16 *)q, (__nv_bfloat16 *)out);
    else
        attn_simt_kernel<__nv_bfloat16, false, false><<<grid, kWarps * 32, 0, st>>>(
            pv, d_seqs, n, H_q, (const __nv_bfloat16 *)q, (__nv_bfloat16 *)out);
    return cudaGetLastError();
}

}  // namespace gqa
