// kernels.cuh -- descriptors and launchers shared by the host library
// (gqa_lib.cu) and the device kernels (k_*.cu).  Internal; the public
// boundary is include/gqa.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gqa {

constexpr int kPageTokens = 16;

// Page pool layout (version 2).  Block (page, kv, head), kv 0 = K, 1 = V,
// is number (page * 2 + kv) * H_kv + head and holds the 16 token rows of that
// page for that head.  A row (d * esize bytes) is cut into C = ceil(row / 128)
// chunks of 128 bytes; the 16 slots form two groups of 8, and within a group
// the rows are stored chunk-major: chunk 0 of slots 0..7, then chunk 1 of
// slots 0..7, ...  Byte b of the row of slot s is at
//     block * pool_block_bytes + ((s / 8) * C + b / 128) * 1024 + (s % 8) * 128 + b % 128.
// With 256-byte rows (bf16, d = 128) a block is 4 KB whose 8-line groups are
// exactly the 1 KB swizzle atoms of a tensor-core operand, so one TMA box
// moves a page of one head.
__host__ __device__ constexpr int pool_chunks(int row_bytes) { return (row_bytes + 127) >> 7; }

// Cache element types (mirror include/gqa.h) and the bytes of a stored element.
constexpr int32_t kDtypeBf16 = 1, kDtypeF32 = 2, kDtypeFp8 = 3;
__host__ __device__ constexpr int pool_esize(int32_t dtype)
{
    return dtype == kDtypeFp8 ? 1 : dtype == kDtypeBf16 ? 2 : 4;
}
// Largest finite FP8 E4M3 value: a quantised row's scale is amax / 448.
constexpr float kE4m3Max = 448.0f;
__host__ __device__ constexpr size_t pool_block_bytes(int row_bytes) { return (size_t)pool_chunks(row_bytes) << 11; }
__host__ __device__ constexpr size_t pool_in_block(int chunks, int slot, int b)
{
    return ((size_t)((slot >> 3) * chunks + (b >> 7)) << 10) + (size_t)((slot & 7) << 7) + (size_t)(b & 127);
}

// A view of the paged pool and the block tables as the kernels see them.
struct PoolView {
    void *pool;              // device, element type = cache dtype
    const int32_t *tables;   // device [max_seqs][stride]: logical page -> physical page
    int32_t stride;          // max_pages_per_seq
    int32_t num_pages;
    int32_t H_kv;
    int32_t d;
    int32_t *err;            // device error word (GQA_DEVERR_* bits)
    const float2 *rope;      // rotary table (cos, sin) [position][d / 2], or null: no rotation
    int32_t window;          // sliding window W (0 = none): position p sees keys max(0, p-W+1)..p
    int32_t dtype;           // kDtype*: the stored element type
    float *scales;           // FP8 E4M3: scale of (block, slot) at block * 16 + slot; else null
    int32_t keys_pre;        // 1: keys are stored before the rotation (rope != null) and rotated
                             // when read; 0: keys are stored as attention uses them
};

// First key position visible to a query at absolute position p.
__host__ __device__ inline int window_start(int p, int window)
{
    return (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
}

// Decode of a sequence of length L reads pages from this token on (the page
// holding its window's first key).
__host__ __device__ inline int decode_first_token(int L, int window)
{
    return window_start(L - 1, window) / kPageTokens * kPageTokens;
}

// One batch entry of a launching call.
struct SeqDesc {
    int32_t row;    // sequence id == block-table row
    int32_t past;   // tokens already cached before this call's rows (decode: L - 1)
    int32_t count;  // rows of this call that are valid (decode: 1)
    int32_t zero_from;  // fused prefill: rows zero_from .. n-1 of out are zeroed by the kernel (no item stores them)
};

// Copy-on-write of slots [0, slots) of page src into page dst (K and V, all heads).
struct CowDesc {
    int32_t src, dst, slots, pad_;
};

// One split-K decode work item: batch entry b, token chunk `split`.
struct DecodeItem {
    int32_t b, split;
};

// One tensor-core prefill work item: two 128-row query tiles of batch entry
// b and KV head kvh, starting at row i0 of the entry; key tiles j0 .. nt-1
// of 128.  tiles = 1 when the second query tile holds no valid row (short
// calls such as decode and multi-token decode): it is then skipped, and its
// rows are padding.  A split item (part >= 0; one tile holding every row of
// the entry) covers one range of the entry's key tiles: its unnormalised
// O, m and l go to workspace slot `part`, the group's nsplit slots are
// part - split .. part - split + nsplit - 1, and the CTA that finishes the
// group's last split merges them into out.
struct TcItem {
    int32_t b, kvh, i0, nt, j0;
    int32_t part;
    int16_t split, nsplit;    // nsplit is at most a few hundred (pieces sized for the SM count)
    int8_t tiles, pad_[3];
};
static_assert(sizeof(TcItem) == 32, "TcItem layout");

// Workspace of split items: slot s holds rows 0 .. slot_rows-1 of one query
// tile (o[(s * slot_rows + row) * 128 + column]) and (m, l) per row
// (ml[s * slot_rows + row]).  counters[first slot of a group] must
// be zero on entry; the kernel leaves them zero.
struct TcSplitWs {
    float *o = nullptr;
    float2 *ml = nullptr;
    int32_t *counters = nullptr;
    int32_t slot_rows = 0;
    bool ranged = false;      // some item starts past key tile 0 (window or split)
};

// Error-word bits (mirror include/gqa.h).
constexpr int32_t kErrPageId = 1;
constexpr int32_t kErrTimeout = 2;
constexpr int32_t kErrShape = 4;

// ---- launchers (each returns the launch's cudaError_t) --------------------

// Element-wise copy unit in bytes (16, 8, 4 or 2) usable for rows of
// `row_bytes` with the given base pointers.
int copy_unit_bytes(size_t row_bytes, const void *a, const void *b, const void *c);

cudaError_t launch_cow_copy(const PoolView &pv, int esize, const CowDesc *d_cows, int ncows,
                            cudaStream_t st);

// Pre-position cache (bf16, d = 128, rope): page u of dst = pool page
// d_pages[u].x (logical page d_pages[u].y of its sequences) with its keys
// rotated by their positions (the cache-write rounding rule) and its values
// copied; dst has npages pages in the pool's block layout.
cudaError_t launch_rotate_pages(const PoolView &pv, const int2 *d_pages, int npages, void *dst, cudaStream_t st);

// Write rows c < seqs[b].count of k/v [B, n, H_kv, d] to positions past+c.
// If zero_out is given ([B, n, zero_row_bytes], 16-byte aligned rows), its
// rows count..n-1 of every entry are set to zero in the same launch.
cudaError_t launch_cache_write(const PoolView &pv, int esize, const SeqDesc *d_seqs, int B, int n,
                               int max_count, const void *k, const void *v, cudaStream_t st,
                               void *zero_out = nullptr, int zero_row_bytes = 0);

// Generic causal attention over the pool (any d <= 256, fp32 or bf16):
// rows i < n of q [B, n, H_q, d]; row i is valid when i < count and sits at
// position past + i; invalid rows are written as zeros.
cudaError_t launch_attn_simt(const PoolView &pv, int dtype, const SeqDesc *d_seqs, int B, int n,
                             int H_q, const void *q, void *out, cudaStream_t st);

// bf16, d = 128 split-K decode with the merge done by the last CTA of each
// (entry, KV head).  counters[B * H_kv] must be zero on entry; the kernel
// leaves them zero.
struct DecodeLaunch {
    const SeqDesc *seqs;
    const DecodeItem *items;
    const int32_t *item_start;   // [B + 1]: items of entry b are item_start[b] .. item_start[b+1]-1
    int n_items;
    int chunk;
    int H_q;
    const void *q;
    float *ws_o;
    float *ws_ml;
    int32_t *counters;
    void *out;
};
bool decode_split_supported(int group);

// Tiled tensor map over `base` (bf16 elements, 128-byte swizzle; bytes:
// uint8 elements, no swizzle unless bytes_swizzled) with the driver's
// encoder.  False if the encoder is unavailable or refuses the shape.
bool encode_tmap(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
                 const cuuint32_t *box, bool bytes = false, bool bytes_swizzled = false);

// bf16, d = 128 single-token decode with each (entry, KV head) served by a
// cluster of `cluster` CTAs that split its pages and merge their partials
// through distributed shared memory.  No workspace.  app_k / app_v
// ([B, H_kv, 128], optional) fuse the append: the row of each entry is
// written at position past (its page already in the block table) by the CTA
// that reads that page.  ev_start, if given, is recorded right before the
// launch.
struct ClusterDecodeLaunch {
    const SeqDesc *seqs = nullptr;       // device descriptors [B], or
    const SeqDesc *host_seqs = nullptr;  // host descriptors, passed in the parameters (B <= decode_cluster_inline())
    int B;
    int H_q;
    int cluster;
    const void *q;
    void *out;
    const void *app_k = nullptr;
    const void *app_v = nullptr;
};
bool decode_cluster_supported(int group);
int decode_cluster_inline();   // largest B whose descriptors travel in the launch parameters
// Largest number of clusters of `cluster` CTAs the device holds at once (0:
// that size cannot be launched).  The device must be current.
int decode_cluster_capacity(int cluster);
cudaError_t launch_decode_cluster(const PoolView &pv, const ClusterDecodeLaunch &a, cudaStream_t st,
                                  cudaEvent_t ev_start = nullptr);
cudaError_t launch_decode_split(const PoolView &pv, const DecodeLaunch &a, cudaStream_t st);

// bf16, d = 128 tensor-core prefill (tcgen05 + TMEM + TMA).  Rows of the
// batch entries must already be in the cache (launch_cache_write first),
// unless fused_k / fused_v are given (see launch_prefill_tc).
bool prefill_tc_supported(int group, int H_kv);
// One block waiting, with the kernels' bounded wait, on a barrier phase that
// never completes; sets kErrTimeout in *err after limit_ns.
cudaError_t launch_wait_probe(int32_t *err, uint64_t limit_ns, cudaStream_t st);
int prefill_tc_rows_per_tile(int group);   // positions per 128-row query tile
// Persistent grid of `grid` CTAs; CTA c takes items[item_start[c] ..
// item_start[c + 1]) in order (grid + 1 offsets, every run non-empty).  Rows
// of the items' query tiles past the valid length are written as zeros;
// padding rows that no item covers must be zeroed by the caller.  ev_start,
// if given, is recorded on st right before the kernel, after the tensor maps
// are encoded on the host.  app_k / app_v (decode only: count = 1 for every
// entry, [B, H_kv, 128]) fuse the append: the row of each entry is written
// at position past by the CTA that reads that page, before it reads it.
// fused_k / fused_v (the call's k and v, [B, n, H_kv, 128], n a multiple of
// 8, every entry's past a multiple of 16, bf16 cache without rotation) fuse
// the cache write: the kernel reads the call's rows from them, writes each
// new page to the pool once, and zeroes rows zero_from .. n-1 of out for
// every entry; no cache-write launch precedes it.  Those rows, counted in
// 16-byte units entry after entry, are cleared by CTA c from unit
// d_zero_start[c] to d_zero_start[c + 1] (grid + 1 offsets).  `host`, if
// given and it fits, supplies the descriptors in the launch parameters.
// Host copies of a launch's descriptors.  When they fit kTcInlineBytes
// (prefill_tc_inline_fits) and the pool is bf16 without rotation, the launch
// can carry them in its parameters: the device copies passed to
// launch_prefill_tc are then not read, so no upload has to precede the
// kernel (a `host` that cannot be carried makes the launch fail).  `tables`
// replaces pv.tables (row stride pv.stride) when given.
struct TcHostDesc {
    const SeqDesc *seqs = nullptr;
    int n_seqs = 0;
    const TcItem *items = nullptr;
    int n_items = 0;
    const int32_t *item_start = nullptr;
    int n_start = 0;
    const int64_t *zero_start = nullptr;
    int n_zero = 0;
    const int32_t *tables = nullptr;
    size_t n_tables = 0;
};
constexpr size_t kTcInlineBytes = 28 * 1024;
bool prefill_tc_inline_fits(const TcHostDesc &h);
cudaError_t launch_prefill_tc(const PoolView &pv, const SeqDesc *d_seqs, const TcItem *d_items,
                              const int32_t *d_item_start, int grid, int B, int n, int H_q, const void *q, void *out,
                              const TcSplitWs &ws, cudaStream_t st, cudaEvent_t ev_start = nullptr,
                              const void *app_k = nullptr, const void *app_v = nullptr,
                              const void *fused_k = nullptr, const void *fused_v = nullptr,
                              const int64_t *d_zero_start = nullptr, const TcHostDesc *host = nullptr);

}  // namespace gqa
