// k_cache.cu -- cache writes: new K/V rows into their pages, and the
// copy-on-write of a shared tail page.
//
// "第二章 Prefill：整层状态演化与 KV 建立", section 2.6: each valid position's
// key (post position transform) and value are written at its logical
// position; padding is never written (invariant 2.2, item 4).
// "KV Cache 与 Prefill/Decode 推理路径", PagedAttention section: token t goes
// to logical page t/16, slot t%16, through the sequence's block table.
//
// Both kernels are pure copies, bound by HBM bandwidth: rows are moved in the
// widest unit (up to 16 bytes) that the row size and base addresses allow,
// consecutive threads taking consecutive units of one row so that both the
// read and the write are coalesced.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace gqa {

int copy_unit_bytes(size_t row_bytes, const void *a, const void *b, const void *c)
{
    const uintptr_t any = (uintptr_t)a | (uintptr_t)b | (uintptr_t)c;
    for (int u = 16; u >= 2; u >>= 1)
        if (row_bytes % u == 0 && any % u == 0)
            return u;
    return 1;
}

template <int U>
struct Unit;
template <> struct Unit<16> { using T = uint4; };
template <> struct Unit<8>  { using T = uint2; };
template <> struct Unit<4>  { using T = uint32_t; };
template <> struct Unit<2>  { using T = uint16_t; };
template <> struct Unit<1>  { using T = uint8_t; };

// Rotary position mechanism on one unit of a key row: `own` holds elements
// of one half of the row, `oth` the same elements of the other half; `first`
// says which half `own` is.  Pair (x, y) = (first half, second half) becomes
// (x*c - y*s, x*s + y*c), each product, difference and sum rounded to fp32
// (no fused multiply-add), then to the element type.
template <int U>
__device__ __forceinline__ typename Unit<U>::T rope_unit(typename Unit<U>::T own, typename Unit<U>::T oth, bool first,
                                                         const float2 *__restrict__ cs, int esize)
{
    typename Unit<U>::T res = own;
    if (esize == 2 && U >= 2) {
        const __nv_bfloat16 *a = reinterpret_cast<const __nv_bfloat16 *>(&own);
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&oth);
        __nv_bfloat16 *r = reinterpret_cast<__nv_bfloat16 *>(&res);
#pragma unroll
        for (int j = 0; j < U / 2; ++j) {
            const float x = __bfloat162float(first ? a[j] : b[j]), y = __bfloat162float(first ? b[j] : a[j]);
            const float2 t = cs[j];
            const float o = first ? __fsub_rn(__fmul_rn(x, t.x), __fmul_rn(y, t.y))
                                  : __fadd_rn(__fmul_rn(x, t.y), __fmul_rn(y, t.x));
            r[j] = __float2bfloat16_rn(o);
        }
    } else if (esize == 4 && U >= 4) {
        const float *a = reinterpret_cast<const float *>(&own);
        const float *b = reinterpret_cast<const float *>(&oth);
        float *r = reinterpret_cast<float *>(&res);
#pragma unroll
        for (int j = 0; j < U / 4; ++j) {
            const float x = first ? a[j] : b[j], y = first ? b[j] : a[j];
            const float2 t = cs[j];
            r[j] = first ? __fsub_rn(__fmul_rn(x, t.x), __fmul_rn(y, t.y)) : __fadd_rn(__fmul_rn(x, t.y), __fmul_rn(y, t.x));
        }
    }
    return res;
}

// grid: (x = token blocks, y = batch entry); one warp per token.  A token's
// K rows for all KV heads are contiguous in k (H_kv * d * esize bytes), so a
// warp reads them with consecutive lanes on consecutive units and writes each
// head's row to its (page, slot), whose 128-byte chunks are contiguous runs:
// both sides coalesced.  Every unit of the
// token is loaded before any is stored, to keep the loads in flight.
// With zero_out != nullptr the same grid also writes zeros over the padding
// rows count..n-1 of zero_out ([B, n, zero_row_bytes]).
template <int U, bool ROPE>
__global__ void __launch_bounds__(256)
cache_write_kernel(PoolView pv, int esize, const SeqDesc *__restrict__ seqs, int n, const char *__restrict__ k,
                   const char *__restrict__ v, char *__restrict__ zero_out, int zero_row_bytes)
{
    using T = typename Unit<U>::T;
    constexpr int kMaxPerLane = ROPE ? 4 : 8;           // units per lane held in registers per pass
    // A dependent attention grid may be scheduled once every block of this
    // one has started; it waits for this grid's writes before reading pages.
    asm volatile("griddepcontrol.launch_dependents;");
    const int b = blockIdx.y;
    const SeqDesc sd = seqs[b];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    const int row_bytes = pv.d * esize;
    const int cpr = row_bytes / U;                      // units per (token, head) row
    const int units = pv.H_kv * cpr;                    // units of one token's K (or V)
    const int chunks = pool_chunks(row_bytes);
    const size_t blk_bytes = pool_block_bytes(row_bytes);
    const int32_t *tab = pv.tables + (size_t)sd.row * pv.stride;
    // Rotation: the token's row of the cos/sin table, shared by all its KV
    // heads, staged once per token in this warp's slice of shared memory.
    __shared__ float2 s_cs[ROPE ? 8 : 1][ROPE ? 128 : 1];
    for (int t = blockIdx.x * wpb + warp; t < sd.count; t += gridDim.x * wpb) {
        const int pos = sd.past + t;
        if (ROPE) {
            __syncwarp();
            for (int e = lane; e < pv.d / 2; e += 32)
                s_cs[warp][e] = pv.rope[(size_t)pos * (pv.d / 2) + e];
            __syncwarp();
        }
        const int page = tab[pos / kPageTokens];
        if ((unsigned)page >= (unsigned)pv.num_pages) {
            if (lane == 0)
                atomicOr(pv.err, kErrPageId);
            continue;
        }
        const size_t src_off = ((size_t)b * n + t) * (size_t)units * U;
        const int slot = pos % kPageTokens;
        char *kd = (char *)pv.pool + (size_t)page * 2 * pv.H_kv * blk_bytes;
        char *vd = kd + (size_t)pv.H_kv * blk_bytes;
        const int half_units = cpr / 2;                   // with rotation: units of half a row
        for (int u0 = 0; u0 < units; u0 += 32 * kMaxPerLane) {
            T kr[kMaxPerLane], vr[kMaxPerLane], kp[kMaxPerLane];
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i) {
                const int u = u0 + 32 * i + lane;
                if (u < units) {
                    kr[i] = *(const T *)(k + src_off + (size_t)u * U);
                    vr[i] = *(const T *)(v + src_off + (size_t)u * U);
                    if (ROPE) {                           // the same unit of the other half
                        const int c = u % cpr;
                        const int pu = u + (c < half_units ? half_units : -half_units);
                        kp[i] = *(const T *)(k + src_off + (size_t)pu * U);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i) {
                const int u = u0 + 32 * i + lane;
                if (u < units) {
                    const int hh = u / cpr, c = u - hh * cpr;
                    const size_t off = (size_t)hh * blk_bytes + pool_in_block(chunks, slot, c * U);
                    T kw = kr[i];
                    if (ROPE) {
                        const bool first = c < half_units;
                        const int pair0 = (first ? c : c - half_units) * (U / esize);
                        kw = rope_unit<U>(kr[i], kp[i], first, &s_cs[warp][pair0], esize);
                    }
                    *(T *)(kd + off) = kw;
                    *(T *)(vd + off) = vr[i];
                }
            }
        }
    }
    if (zero_out) {
        const int zunits = zero_row_bytes / 16;
        for (int t = sd.count + blockIdx.x * wpb + warp; t < n; t += gridDim.x * wpb) {
            uint4 *dst = (uint4 *)(zero_out + ((size_t)b * n + t) * zero_row_bytes);
            for (int u = lane; u < zunits; u += 32)
                dst[u] = make_uint4(0, 0, 0, 0);
        }
    }
}

// Quantised cache ("第二章 Prefill：整层状态演化与 KV 建立" section 2.5: the
// physical cache may be quantised; the logical order is kept): a warp per
// (token, K|V, head) row of d_h bf16 values; lane l holds elements
// l*P .. l*P + P - 1 (P = d_h / 32).  s = amax / 448 (fp32 division), each
// code = E4M3(x / s) with the quotient in fp32 and the conversion rounding
// to nearest-even and saturating; a row of zeros gets s = 0 and zero codes.
// The codes go to the row's place in the block layout, s to the scale array.
// With zero_out, rows count..n-1 of zero_out ([B, n, zero_row_bytes]) are
// set to zero in the same grid, as in cache_write_kernel.
template <int P>
__global__ void __launch_bounds__(256)
cache_write_q8_kernel(PoolView pv, const SeqDesc *__restrict__ seqs, int n, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ v, char *__restrict__ zero_out, int zero_row_bytes)
{
    asm volatile("griddepcontrol.launch_dependents;");   // as in cache_write_kernel
    const int b = blockIdx.y;
    const SeqDesc sd = seqs[b];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    const int H_kv = pv.H_kv, d = pv.d;
    const int chunks = pool_chunks(d);
    const size_t blk_bytes = pool_block_bytes(d);
    const int32_t *tab = pv.tables + (size_t)sd.row * pv.stride;
    const int rows = sd.count * 2 * H_kv;
    for (int task = blockIdx.x * wpb + warp; task < rows; task += gridDim.x * wpb) {
        const int t = task / (2 * H_kv), kv = (task / H_kv) & 1, h = task % H_kv;
        const int pos = sd.past + t;
        const int page = tab[pos / kPageTokens];
        if ((unsigned)page >= (unsigned)pv.num_pages) {
            if (lane == 0)
                atomicOr(pv.err, kErrPageId);
            continue;
        }
        const __nv_bfloat16 *src = (kv ? v : k) + (((size_t)b * n + t) * H_kv + h) * d + lane * P;
        float x[P];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            x[i] = __bfloat162float(src[i]);
            amax = fmaxf(amax, fabsf(x[i]));
        }
        for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = __fdiv_rn(amax, kE4m3Max);
        unsigned char code[P];
#pragma unroll
        for (int i = 0; i < P; ++i)
            code[i] = sc > 0.0f ? (unsigned char)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], sc), __NV_SATFINITE, __NV_E4M3)
                                : (unsigned char)0;
        const int slot = pos % kPageTokens;
        const size_t blk = ((size_t)page * 2 + kv) * H_kv + h;
        unsigned char *dst = (unsigned char *)pv.pool + blk * blk_bytes;
#pragma unroll
        for (int i = 0; i < P; ++i)                    // (a lane's bytes may straddle a 128-byte chunk)
            dst[pool_in_block(chunks, slot, lane * P + i)] = code[i];
        if (lane == 0)
            pv.scales[blk * kPageTokens + slot] = sc;
    }
    if (zero_out) {
        const int zunits = zero_row_bytes / 16;
        for (int t = sd.count + blockIdx.x * wpb + warp; t < n; t += gridDim.x * wpb) {
            uint4 *dst = (uint4 *)(zero_out + ((size_t)b * n + t) * zero_row_bytes);
            for (int u = lane; u < zunits; u += 32)
                dst[u] = make_uint4(0, 0, 0, 0);
        }
    }
}

template <int U>
__global__ void cow_copy_kernel(PoolView pv, int esize, const CowDesc *__restrict__ cows)
{
    using T = typename Unit<U>::T;
    const CowDesc cd = cows[blockIdx.y];
    const int row_bytes = pv.d * esize;
    const int cpr = row_bytes / U;
    const int chunks = pool_chunks(row_bytes);
    const size_t blk_bytes = pool_block_bytes(row_bytes);
    const size_t page_bytes = 2 * (size_t)pv.H_kv * blk_bytes;
    if ((unsigned)cd.src >= (unsigned)pv.num_pages || (unsigned)cd.dst >= (unsigned)pv.num_pages) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            atomicOr(pv.err, kErrPageId);
        return;
    }
    const long long units = (long long)2 * pv.H_kv * cd.slots * cpr;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(u % cpr);
        long long r = u / cpr;
        const int slot = (int)(r % cd.slots);
        const int blk = (int)(r / cd.slots);           // kv * H_kv + head
        const size_t off = (size_t)blk * blk_bytes + pool_in_block(chunks, slot, c * U);
        *(T *)((char *)pv.pool + (size_t)cd.dst * page_bytes + off) =
            *(const T *)((const char *)pv.pool + (size_t)cd.src * page_bytes + off);
    }
    if (pv.scales && blockIdx.x == 0) {                // a quantised cache: the rows' scales too
        const int n_sc = 2 * pv.H_kv * cd.slots;
        for (int i = threadIdx.x; i < n_sc; i += blockDim.x) {
            const int blk = i / cd.slots, slot = i % cd.slots;
            pv.scales[((size_t)cd.dst * 2 * pv.H_kv + blk) * kPageTokens + slot] =
                pv.scales[((size_t)cd.src * 2 * pv.H_kv + blk) * kPageTokens + slot];
        }
    }
}

cudaError_t launch_cache_write(const PoolView &pv, int esize, const SeqDesc *d_seqs, int B, int n,
                               int max_count, const void *k, const void *v, cudaStream_t st, void *zero_out,
                               int zero_row_bytes)
{
    const int rows = zero_out ? n : max_count;          // padding rows are zeroed too
    if (B <= 0 || rows <= 0)
        return cudaSuccess;
    if (pv.dtype == kDtypeFp8) {                        // quantising write
        if (pv.d % 32 != 0 || pv.d > 256 || !pv.scales ||
            (zero_out && (zero_row_bytes % 16 != 0 || (uintptr_t)zero_out % 16 != 0)))
            return cudaErrorInvalidValue;
        int blocks = (max(max_count * 2 * pv.H_kv, rows) + 7) / 8;
        if (blocks > 1024)
            blocks = 1024;
        dim3 grid((unsigned)blocks, (unsigned)B);
        const __nv_bfloat16 *kb = (const __nv_bfloat16 *)k, *vb = (const __nv_bfloat16 *)v;
        char *z = (char *)zero_out;
        switch (pv.d / 32) {
        case 1: cache_write_q8_kernel<1><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        case 2: cache_write_q8_kernel<2><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        case 3: cache_write_q8_kernel<3><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        case 4: cache_write_q8_kernel<4><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        case 5: cache_write_q8_kernel<5><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        case 6: cache_write_q8_kernel<6><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        case 7: cache_write_q8_kernel<7><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        default: cache_write_q8_kernel<8><<<grid, 256, 0, st>>>(pv, d_seqs, n, kb, vb, z, zero_row_bytes); break;
        }
        return cudaGetLastError();
    }
    const size_t row_bytes = (size_t)pv.d * esize;
    // With rotation a unit must lie within one half of the row and hold
    // whole elements.
    // Keys are rotated when written unless the cache stores them before the
    // rotation (then the write is a plain copy and the readers rotate).
    const bool rot = pv.rope && !pv.keys_pre;
    const int U = copy_unit_bytes(rot ? row_bytes / 2 : row_bytes, k, v, pv.pool);
    if (zero_out && (zero_row_bytes % 16 != 0 || (uintptr_t)zero_out % 16 != 0))
        return cudaErrorInvalidValue;
    if (rot && U < esize)
        return cudaErrorInvalidValue;
    const int wpb = 8;                                  // at most 8: the rotation's table rows
    int blocks = (rows + wpb - 1) / wpb;
    if (blocks > 1024)
        blocks = 1024;
    dim3 grid((unsigned)blocks, (unsigned)B);
    const char *kc = (const char *)k, *vc = (const char *)v;
    char *z = (char *)zero_out;
    // The rotating kernel is a separate instantiation, so that a cache without
    // the position mechanism runs the plain copy.
#define GQA_CACHE_WRITE(UU)                                                                                    \
    (rot ? (cache_write_kernel<UU, true><<<grid, 32 * wpb, 0, st>>>(pv, esize, d_seqs, n, kc, vc, z,           \
                                                                       zero_row_bytes), 0)                    \
         : (cache_write_kernel<UU, false><<<grid, 32 * wpb, 0, st>>>(pv, esize, d_seqs, n, kc, vc, z,          \
                                                                    zero_row_bytes), 0))
    switch (U) {
    case 16: GQA_CACHE_WRITE(16); break;
    case 8:  GQA_CACHE_WRITE(8); break;
    case 4:  GQA_CACHE_WRITE(4); break;
    case 2:  GQA_CACHE_WRITE(2); break;
    default: GQA_CACHE_WRITE(1); break;
    }
#undef GQA_CACHE_WRITE
    return cudaGetLastError();
}

// Pre-position cache read by the tensor-core prefill: page u of the list
// (pool page pages[u].x at logical page pages[u].y of its sequences) is
// copied to page u of `dst` (a pool of the same block layout), its keys
// rotated by their positions 16 * pages[u].y + slot with the cache-write
// rule (fp32 cos/sin of the table, each product, sum and difference rounded
// to fp32, then to bf16), its values as they are.  bf16, d = 128: a block
// is 4 KB; thread (slot, unit) of a K block rotates the 16-byte unit of
// column half 0 with the same unit of column half 1 (columns e and e + 64
// sit at the same offset of the two 128-byte chunks of a row).
__global__ void __launch_bounds__(128)
rotate_pages_kernel(PoolView pv, const int2 *__restrict__ pages, char *__restrict__ dst)
{
    const int2 pg = pages[blockIdx.x];
    const int head = blockIdx.y, kv = blockIdx.z;
    constexpr size_t kBlk = 4096;
    if ((unsigned)pg.x >= (unsigned)pv.num_pages) {
        if (threadIdx.x == 0)
            atomicOr(pv.err, kErrPageId);
        return;
    }
    const size_t blk_src = ((size_t)pg.x * 2 + kv) * pv.H_kv + head;
    const size_t blk_dst = ((size_t)blockIdx.x * 2 + kv) * pv.H_kv + head;
    const uint4 *src = reinterpret_cast<const uint4 *>((const char *)pv.pool + blk_src * kBlk);
    uint4 *out = reinterpret_cast<uint4 *>(dst + blk_dst * kBlk);
    if (kv) {                                            // values: a plain copy
        out[threadIdx.x] = src[threadIdx.x];
        out[threadIdx.x + 128] = src[threadIdx.x + 128];
        return;
    }
    const int slot = threadIdx.x >> 3, u = threadIdx.x & 7;   // unit u of the slot's column half 0
    // uint4 index of (slot, chunk c, unit u): ((slot / 8) * 2 + c) * 64 + (slot % 8) * 8 + u
    const int i0 = ((slot >> 3) * 2) * 64 + (slot & 7) * 8 + u, i1 = i0 + 64;
    const uint4 a = src[i0], b = src[i1];
    const float2 *cs = pv.rope + (size_t)(kPageTokens * pg.y + slot) * 64 + 8 * u;
    const __nv_bfloat16 *xa = reinterpret_cast<const __nv_bfloat16 *>(&a);
    const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(&b);
    uint4 ra, rb;
    __nv_bfloat16 *ya = reinterpret_cast<__nv_bfloat16 *>(&ra), *yb = reinterpret_cast<__nv_bfloat16 *>(&rb);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float x = __bfloat162float(xa[j]), y = __bfloat162float(xb[j]);
        const float2 t = cs[j];
        ya[j] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(x, t.x), __fmul_rn(y, t.y)));
        yb[j] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(x, t.y), __fmul_rn(y, t.x)));
    }
    out[i0] = ra;
    out[i1] = rb;
}

cudaError_t launch_rotate_pages(const PoolView &pv, const int2 *d_pages, int npages, void *dst, cudaStream_t st)
{
    if (pv.d != 128 || pv.dtype != kDtypeBf16 || !pv.rope)
        return cudaErrorInvalidValue;
    if (npages <= 0)
        return cudaSuccess;
    rotate_pages_kernel<<<dim3((unsigned)npages, (unsigned)pv.H_kv, 2), 128, 0, st>>>(pv, d_pages, (char *)dst);
    return cudaGetLastError();
}

cudaError_t launch_cow_copy(const PoolView &pv, int esize, const CowDesc *d_cows, int ncows,
                            cudaStream_t st)
{
    if (ncows <= 0)
        return cudaSuccess;
    const size_t row_bytes = (size_t)pv.d * esize;
    const int U = copy_unit_bytes(row_bytes, pv.pool, pv.pool, pv.pool);
    dim3 grid(8, (unsigned)ncows);
    switch (U) {
    case 16: cow_copy_kernel<16><<<grid, 256, 0, st>>>(pv, esize, d_cows); break;
    case 8:  cow_copy_kernel<8><<<grid, 256, 0, st>>>(pv, esize, d_cows); break;
    case 4:  cow_copy_kernel<4><<<grid, 256, 0, st>>>(pv, esize, d_cows); break;
    case 2:  cow_copy_kernel<2><<<grid, 256, 0, st>>>(pv, esize, d_cows); break;
    default: cow_copy_kernel<1><<<grid, 256, 0, st>>>(pv, esize, d_cows); break;
    }
    return cudaGetLastError();
}

}  // namespace gqa
