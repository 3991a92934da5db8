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

// grid: (x = blocks over units, y = batch entry).  Unit u of entry b:
//   chunk c of row (token t, kv, head hh).
template <int U>
__global__ void cache_write_kernel(PoolView pv, int esize, const SeqDesc *__restrict__ seqs, int n,
                                   const char *__restrict__ k, const char *__restrict__ v)
{
    using T = typename Unit<U>::T;
    const int b = blockIdx.y;
    const SeqDesc sd = seqs[b];
    const size_t row_bytes = (size_t)pv.d * esize;
    const int cpr = (int)(row_bytes / U);                 // units per row
    const long long units = (long long)sd.count * pv.H_kv * 2 * cpr;
    const int32_t *tab = pv.tables + (size_t)sd.row * pv.stride;
    const size_t page_bytes = (size_t)2 * pv.H_kv * kPageTokens * row_bytes;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(u % cpr);
        long long r = u / cpr;
        const int hh = (int)(r % pv.H_kv);
        r /= pv.H_kv;
        const int kv = (int)(r % 2);
        const int t = (int)(r / 2);
        const int pos = sd.past + t;
        const int page = tab[pos / kPageTokens];
        if ((unsigned)page >= (unsigned)pv.num_pages) {
            atomicOr(pv.err, kErrPageId);
            continue;
        }
        const char *src = (kv ? v : k) + (((size_t)b * n + t) * pv.H_kv + hh) * row_bytes + (size_t)c * U;
        char *dst = (char *)pv.pool + (size_t)page * page_bytes +
                    ((size_t)(kv * pv.H_kv + hh) * kPageTokens + pos % kPageTokens) * row_bytes +
                    (size_t)c * U;
        *(T *)dst = *(const T *)src;
    }
}

template <int U>
__global__ void cow_copy_kernel(PoolView pv, int esize, const CowDesc *__restrict__ cows)
{
    using T = typename Unit<U>::T;
    const CowDesc cd = cows[blockIdx.y];
    const size_t row_bytes = (size_t)pv.d * esize;
    const int cpr = (int)(row_bytes / U);
    const size_t page_bytes = (size_t)2 * pv.H_kv * kPageTokens * row_bytes;
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
        const size_t off = ((size_t)blk * kPageTokens + slot) * row_bytes + (size_t)c * U;
        *(T *)((char *)pv.pool + (size_t)cd.dst * page_bytes + off) =
            *(const T *)((const char *)pv.pool + (size_t)cd.src * page_bytes + off);
    }
}

cudaError_t launch_cache_write(const PoolView &pv, int esize, const SeqDesc *d_seqs, int B, int n,
                               int max_count, const void *k, const void *v, cudaStream_t st)
{
    if (B <= 0 || max_count <= 0)
        return cudaSuccess;
    const size_t row_bytes = (size_t)pv.d * esize;
    const int U = copy_unit_bytes(row_bytes, k, v, pv.pool);
    const long long units = (long long)max_count * pv.H_kv * 2 * (long long)(row_bytes / U);
    const int threads = 256;
    long long blocks = (units + threads - 1) / threads;
    if (blocks > 4096)
        blocks = 4096;
    dim3 grid((unsigned)blocks, (unsigned)B);
    const char *kc = (const char *)k, *vc = (const char *)v;
    switch (U) {
    case 16: cache_write_kernel<16><<<grid, threads, 0, st>>>(pv, esize, d_seqs, n, kc, vc); break;
    case 8:  cache_write_kernel<8><<<grid, threads, 0, st>>>(pv, esize, d_seqs, n, kc, vc); break;
    case 4:  cache_write_kernel<4><<<grid, threads, 0, st>>>(pv, esize, d_seqs, n, kc, vc); break;
    case 2:  cache_write_kernel<2><<<grid, threads, 0, st>>>(pv, esize, d_seqs, n, kc, vc); break;
    default: cache_write_kernel<1><<<grid, threads, 0, st>>>(pv, esize, d_seqs, n, kc, vc); break;
    }
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
