// gqa_lib.cu -- the C ABI of include/gqa.h: the host-side cache manager
// (page pool, block tables, reference counts, copy-on-write, truncation),
// every precondition check, and the launch sequences of the hot path.
//
// Sources: "第二章 Prefill：整层状态演化与 KV 建立" (preconditions 2.1, mask
// and invalid rows 2.2, attention 2.3, cache contract and invariants 2.2 in
// 2.5, pseudocode 2.6, prefix reuse 2.9, failure table 2.11);
// "KV Cache 与 Prefill/Decode 推理路径" (edit at token m; PagedAttention block
// table and free pool; prefix sharing with reference counts).
//
// Host/device split.  All bookkeeping lives here, on the host: a call first
// validates every argument against the current metadata (so a rejected call
// changes nothing and queues nothing, as preconditions 2.1 demand), then
// commits the metadata change, uploads the block-table entries it changed
// and a small per-call descriptor block with stream-ordered copies, and
// finally queues its kernels.  Nothing here waits for the GPU.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "gqa.h"
#include "kernels.cuh"

using namespace gqa;

namespace {

thread_local std::string t_err;

// Largest per-call copy of the call's block-table rows sent with a prefill's
// descriptors (larger calls read the pool's tables, uploaded first).
constexpr size_t kCompactTableBytes = 1u << 20;

// Fixed cost of one prefill work item (Q load, pipeline refill, epilogue)
// in quarters of a key tile, for balancing items over the persistent grid.
constexpr int64_t kItemCostQuarters = 2;
#ifndef GQA_SPLIT_ITEMS_PER_SM
#define GQA_SPLIT_ITEMS_PER_SM 1
#endif
#ifndef GQA_SPLIT_MIN_TILES
#define GQA_SPLIT_MIN_TILES 4
#endif
constexpr int kSplitItemsPerSm = GQA_SPLIT_ITEMS_PER_SM;   // tensor-core split items: target per SM
constexpr int kSplitMinTiles = GQA_SPLIT_MIN_TILES;         // and the shortest piece, in key tiles
// attn_decode_static: descriptors at most 1 MiB, block-table entries at most
// 1 MiB; each of the two page-locked staging slots holds both.
constexpr size_t kStaticDescBytes = 1u << 20;
constexpr size_t kStaticStageBytes = 2u << 20;

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(GQA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct SeqState {
    bool live = false;
    int32_t len = 0;
    std::vector<int32_t> pages;
    int32_t dirty_lo = INT_MAX, dirty_hi = 0;   // block-table entries changed since upload
};

struct WriteReq {
    int32_t seq, count;
};

}  // namespace

struct gqa_cache {
    gqa_cache_desc desc{};
    int esize = 0;                       // bytes of a stored element (1 for FP8 E4M3)
    int io_esize = 0;                    // bytes of a q/k/v/out element
    bool meta_only = false;
    void *pool = nullptr;
    std::vector<int32_t> order, rank, ref;
    std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_ranks;
    std::vector<SeqState> seqs;
    std::vector<int32_t> dirty_list;
    std::vector<int32_t> h_tab;          // host mirror [max_seqs][max_pages_per_seq]
    int32_t *d_tab = nullptr;            // device block tables
    int32_t *d_err = nullptr;            // device error word
    char *d_stage = nullptr;             // per-call descriptors
    size_t stage_cap = 0;
    float *d_ws = nullptr;               // decode split partials
    size_t ws_cap = 0;
    // attn_decode_static: page-locked staging for its descriptors and block
    // tables, reserved at creation (two slots used in turn; a slot's event
    // marks the end of the copies that last read it).
    char *h_pin = nullptr;
    cudaEvent_t pin_done[2] = {nullptr, nullptr};
    int pin_next = 0;
    char *d_rot = nullptr;               // pre-position prefill: the call's pages with rotated keys
    size_t rot_cap = 0;
    std::vector<int32_t> rot_slot;       // scratch slot of a pool page during one call (-1 = none)
    int32_t *d_cnt = nullptr;            // decode merge counters [B * H_kv], kept at zero
    size_t cnt_cap = 0;
    float2 *d_rope = nullptr;            // rope = 1: (cos, sin) [max positions][d_h / 2]
    // attn_prefill_host: packed device copies of a call's valid q, k, v and
    // out rows, an upload and a download stream, and per-entry events.
    char *d_io = nullptr;
    size_t io_cap = 0;
    cudaStream_t io_up = nullptr, io_down = nullptr;
    std::vector<cudaEvent_t> io_events;
    std::vector<char> h_stage;
    int device = -1;
    int num_sms = 0;
    int cc = 0;                          // compute capability major*10+minor

    // Profiling: launch counts always; event pairs while `prof` is on.
    bool prof = false;
    int32_t decode_kernel = GQA_DECODE_AUTO;
    int32_t launches[GQA_KERNEL_COUNT] = {};
    struct ProfRec {
        int kernel;
        cudaEvent_t start, end;
    };
    std::vector<ProfRec> prof_recs;
    std::vector<cudaEvent_t> spare_events;

    size_t stride() const { return (size_t)desc.max_pages_per_seq; }

    int32_t take_page()
    {
        const int32_t r = free_ranks.top();
        free_ranks.pop();
        const int32_t p = order[r];
        ref[p] = 1;
        return p;
    }

    void drop_page(int32_t p)
    {
        if (--ref[p] == 0)
            free_ranks.push(rank[p]);
    }

    void set_entry(int32_t s, int32_t idx, int32_t page)
    {
        h_tab[(size_t)s * stride() + idx] = page;
        SeqState &S = seqs[s];
        if (S.dirty_hi <= S.dirty_lo)
            dirty_list.push_back(s);
        S.dirty_lo = std::min(S.dirty_lo, idx);
        S.dirty_hi = std::max(S.dirty_hi, idx + 1);
    }

    PoolView view() const
    {
        PoolView pv;
        pv.pool = pool;
        pv.tables = d_tab;
        pv.stride = desc.max_pages_per_seq;
        pv.num_pages = desc.num_pages;
        pv.H_kv = desc.num_kv_heads;
        pv.d = desc.head_dim;
        pv.err = d_err;
        pv.rope = d_rope;
        pv.window = desc.window;
        pv.dtype = desc.dtype;
        pv.scales = nullptr;
        pv.keys_pre = desc.keys_post_position == 0 ? 1 : 0;
        if (pool && desc.dtype == GQA_DTYPE_FP8_E4M3)   // the scales follow the blocks
            pv.scales = reinterpret_cast<float *>(
                static_cast<char *>(pool) +
                (size_t)desc.num_pages * 2 * desc.num_kv_heads * pool_block_bytes(desc.head_dim));
        return pv;
    }
};

namespace {

bool live(const gqa_cache *c, int32_t s)
{
    return s >= 0 && s < c->desc.max_seqs && c->seqs[s].live;
}

int32_t pages_for(int64_t tokens) { return (int32_t)((tokens + kPageTokens - 1) / kPageTokens); }

// Sliding window: positions m - W .. m - 1 still held (released pages are a
// prefix of the table), so queries from position m - 1 on find their keys.
bool window_holds(const gqa_cache *c, const SeqState &S, int32_t m)
{
    if (c->desc.window <= 0 || m == 0)
        return true;
    int64_t released = 0;
    while (released < (int64_t)S.pages.size() && S.pages[released] < 0)
        ++released;
    return released * kPageTokens <= (int64_t)m - c->desc.window;
}

// After a write that brought the sequences to their new lengths L: pages
// whose positions all lie before L - W go back to the pool (no query from
// position L - 1 on reads them) and their table entries become -1.  Called
// once the call's kernels are queued; later writes that reuse the pages are
// ordered after them on the stream.
void release_windows(gqa_cache *c, int32_t B, const int32_t *seq_ids)
{
    if (c->desc.window <= 0)
        return;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t s = seq_ids[b];
        SeqState &S = c->seqs[s];
        for (size_t j = 0; j < S.pages.size(); ++j) {
            if ((int64_t)kPageTokens * (int64_t)(j + 1) > (int64_t)S.len - c->desc.window)
                break;
            if (S.pages[j] >= 0) {
                c->drop_page(S.pages[j]);
                S.pages[j] = -1;
                c->set_entry(s, (int32_t)j, -1);
            }
        }
    }
}

// Validate a batched write: live and distinct sequences, capacity, pages.
int check_write(const gqa_cache *c, const WriteReq *r, int B)
{
    std::vector<char> seen((size_t)c->desc.max_seqs, 0);
    int64_t need_total = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t s = r[b].seq;
        if (!live(c, s))
            return fail(GQA_EINVAL, "batch entry %d: sequence %d is not live", b, s);
        if (seen[s])
            return fail(GQA_EINVAL, "sequence %d appears twice in one write", s);
        seen[s] = 1;
        const SeqState &S = c->seqs[s];
        const int64_t new_len = (int64_t)S.len + r[b].count;
        if (pages_for(new_len) > c->desc.max_pages_per_seq)
            return fail(GQA_ERANGE, "sequence %d: %lld tokens exceed its capacity of %d pages", s,
                        (long long)new_len, c->desc.max_pages_per_seq);
        need_total += pages_for(new_len) - (int64_t)S.pages.size();
        if (r[b].count > 0 && S.len % kPageTokens != 0 && c->ref[S.pages.back()] > 1)
            need_total += 1;                          // copy-on-write of the shared tail page
    }
    if (need_total > (int64_t)c->free_ranks.size())
        return fail(GQA_ENOMEM, "page pool exhausted: %lld pages needed, %zu free",
                    (long long)need_total, c->free_ranks.size());
    return GQA_OK;
}

// Apply a validated write to the metadata.  Pages are taken sequence by
// sequence in batch order: the copy-on-write page first, then new pages.
void commit_write(gqa_cache *c, const WriteReq *r, int B, std::vector<SeqDesc> &sds,
                  std::vector<CowDesc> &cows)
{
    sds.resize(B);
    for (int b = 0; b < B; ++b) {
        const int32_t s = r[b].seq;
        SeqState &S = c->seqs[s];
        const int32_t past = S.len, count = r[b].count;
        if (count > 0 && past % kPageTokens != 0 && c->ref[S.pages.back()] > 1) {
            const int32_t old = S.pages.back();
            const int32_t np = c->take_page();
            cows.push_back(CowDesc{old, np, past % kPageTokens, 0});
            c->drop_page(old);
            S.pages.back() = np;
            c->set_entry(s, (int32_t)S.pages.size() - 1, np);
        }
        while ((int64_t)S.pages.size() * kPageTokens < (int64_t)past + count) {
            const int32_t np = c->take_page();
            S.pages.push_back(np);
            c->set_entry(s, (int32_t)S.pages.size() - 1, np);
        }
        S.len = past + count;
        sds[b] = SeqDesc{s, past, count, 0};
    }
}

int check_device(const gqa_cache *c)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev != c->device)
        return fail(GQA_EINVAL, "current device %d is not the cache's device %d", dev, c->device);
    return GQA_OK;
}

// Copy `bytes` from host memory to device `dst` on `st` through the cache's
// page-locked staging slots (taken in turn, at most kStaticStageBytes a
// piece); before reusing a slot it waits for the copies that last read it.
// Allocates nothing.
int staged_copy(gqa_cache *c, void *dst, const void *src, size_t bytes, cudaStream_t st)
{
    for (size_t off = 0; off < bytes;) {
        const size_t piece = std::min(bytes - off, kStaticStageBytes);
        const int slot = c->pin_next;
        c->pin_next ^= 1;
        cudaError_t e = cudaEventSynchronize(c->pin_done[slot]);
        if (e != cudaSuccess)
            return cuda_fail(e, "staging slot wait");
        char *h = c->h_pin + (size_t)slot * kStaticStageBytes;
        memcpy(h, (const char *)src + off, piece);
        if ((e = cudaMemcpyAsync((char *)dst + off, h, piece, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
            (e = cudaEventRecord(c->pin_done[slot], st)) != cudaSuccess)
            return cuda_fail(e, "staged upload");
        off += piece;
    }
    return GQA_OK;
}

// Upload the block-table entries changed since the last upload: one copy of
// the span of the flat table that covers every dirty entry (rows are
// contiguous, and clean entries in between equal the device's), so a call
// pays one copy however many sequences it touched.  staged: through the
// page-locked staging slots (attn_decode_static).
int upload_tables(gqa_cache *c, cudaStream_t st, bool staged = false)
{
    size_t lo = SIZE_MAX, hi = 0;
    for (int32_t s : c->dirty_list) {
        SeqState &S = c->seqs[s];
        if (S.dirty_hi > S.dirty_lo) {
            lo = std::min(lo, (size_t)s * c->stride() + S.dirty_lo);
            hi = std::max(hi, (size_t)s * c->stride() + S.dirty_hi);
        }
        S.dirty_lo = INT_MAX;
        S.dirty_hi = 0;
    }
    c->dirty_list.clear();
    if (hi > lo && staged)
        return staged_copy(c, c->d_tab + lo, c->h_tab.data() + lo, (hi - lo) * sizeof(int32_t), st);
    if (hi > lo) {
        cudaError_t e = cudaMemcpyAsync(c->d_tab + lo, c->h_tab.data() + lo, (hi - lo) * sizeof(int32_t),
                                        cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess)
            return cuda_fail(e, "block-table upload");
    }
    return GQA_OK;
}

// Per-call descriptor block: appended pieces are 16-byte aligned.
struct Stage {
    std::vector<char> &buf;
    explicit Stage(std::vector<char> &b) : buf(b) { buf.clear(); }
    template <typename T>
    size_t add(const T *p, size_t count)
    {
        const size_t off = (buf.size() + 15) & ~(size_t)15;
        buf.resize(off + count * sizeof(T));
        if (count)
            memcpy(buf.data() + off, p, count * sizeof(T));
        return off;
    }
};

int upload_stage(gqa_cache *c, cudaStream_t st)
{
    const size_t bytes = c->h_stage.size();
    if (bytes > c->stage_cap) {
        if (c->d_stage) {
            cudaError_t e = cudaFree(c->d_stage);     // synchronises the device
            c->d_stage = nullptr;
            c->stage_cap = 0;
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaFree(stage)");
        }
        const size_t cap = std::max<size_t>((bytes + 65535) & ~(size_t)65535, 65536);
        cudaError_t e = cudaMalloc((void **)&c->d_stage, cap);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(stage)");
        c->stage_cap = cap;
    }
    if (bytes) {
        cudaError_t e = cudaMemcpyAsync(c->d_stage, c->h_stage.data(), bytes, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess)
            return cuda_fail(e, "descriptor upload");
    }
    return GQA_OK;
}

int ensure_ws(gqa_cache *c, size_t floats)
{
    const size_t bytes = floats * sizeof(float);
    if (bytes <= c->ws_cap)
        return GQA_OK;
    if (c->d_ws) {
        cudaError_t e = cudaFree(c->d_ws);
        c->d_ws = nullptr;
        c->ws_cap = 0;
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFree(workspace)");
    }
    const size_t cap = (bytes + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
    cudaError_t e = cudaMalloc((void **)&c->d_ws, cap);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(workspace)");
    c->ws_cap = cap;
    return GQA_OK;
}

// Device pages for a pre-position prefill's rotated copy, grown on demand.
int ensure_rot(gqa_cache *c, size_t bytes)
{
    if (bytes <= c->rot_cap)
        return GQA_OK;
    if (c->d_rot) {
        cudaError_t e = cudaFree(c->d_rot);
        c->d_rot = nullptr;
        c->rot_cap = 0;
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFree(rotated pages)");
    }
    const size_t cap = (bytes + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
    cudaError_t e = cudaMalloc((void **)&c->d_rot, cap);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(rotated pages)");
    c->rot_cap = cap;
    return GQA_OK;
}

// Counters the decode kernel's merge uses; zero when allocated, and the
// kernel leaves them zero.
int ensure_cnt(gqa_cache *c, size_t n)
{
    if (n <= c->cnt_cap)
        return GQA_OK;
    if (c->d_cnt) {
        cudaError_t e = cudaFree(c->d_cnt);
        c->d_cnt = nullptr;
        c->cnt_cap = 0;
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFree(counters)");
    }
    const size_t cap = std::max<size_t>(n, 4096);
    cudaError_t e = cudaMalloc((void **)&c->d_cnt, cap * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMemset(c->d_cnt, 0, cap * sizeof(int32_t));
    if (e != cudaSuccess)
        return cuda_fail(e, "counters");
    c->cnt_cap = cap;
    return GQA_OK;
}

cudaEvent_t get_event(gqa_cache *c)
{
    if (!c->spare_events.empty()) {
        cudaEvent_t e = c->spare_events.back();
        c->spare_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess)
        return nullptr;
    return e;
}

// Record the start event of a profiled launch (no-op when not profiling).
inline void rec(cudaEvent_t ev, cudaStream_t st)
{
    if (ev)
        cudaEventRecord(ev, st);
}

// Queue one kernel via `launch` (given the start event or null, returning
// cudaError_t), counting it and, when profiling is on, bracketing it with
// events on its stream.
template <typename F>
int run_kernel(gqa_cache *c, int kernel, cudaStream_t st, const char *what, F &&launch)
{
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (c->prof) {
        e0 = get_event(c);
        e1 = get_event(c);
        if (!e0 || !e1)
            e0 = e1 = nullptr;
    }
    // The launcher records e0 right before its kernel, after its host-side
    // preparation, so a GPU that waits for the host does not count that wait.
    const cudaError_t e = launch(e0);
    if (e != cudaSuccess)
        return cuda_fail(e, what);
    c->launches[kernel] += 1;
    if (e0 && e1) {
        cudaEventRecord(e1, st);
        c->prof_recs.push_back(gqa_cache::ProfRec{kernel, e0, e1});
    }
    return GQA_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char *gqa_last_error(void) { return t_err.c_str(); }

const char *gqa_version(void) { return "libgqa 0.1.0 (sm_103a)"; }

size_t gqa_pool_bytes(const gqa_cache_desc *d)
{
    if (!d || d->num_pages < 1 || d->num_kv_heads < 1 || d->head_dim < 1 ||
        (d->dtype != GQA_DTYPE_BF16 && d->dtype != GQA_DTYPE_F32 && d->dtype != GQA_DTYPE_FP8_E4M3))
        return 0;
    const int es = pool_esize(d->dtype);
    const size_t blocks = (size_t)d->num_pages * 2 * (size_t)d->num_kv_heads;
    return blocks * pool_block_bytes(d->head_dim * es) +
           (d->dtype == GQA_DTYPE_FP8_E4M3 ? blocks * kPageTokens * sizeof(float) : 0);
}

int gqa_cache_create(const gqa_cache_desc *desc, void *pool_dev, size_t pool_bytes, gqa_cache **out)
{
    if (!desc || !out)
        return fail(GQA_EINVAL, "NULL argument");
    *out = nullptr;
    const gqa_cache_desc &d = *desc;
    if (d.dtype != GQA_DTYPE_BF16 && d.dtype != GQA_DTYPE_F32 && d.dtype != GQA_DTYPE_FP8_E4M3)
        return fail(GQA_EINVAL, "unknown dtype %d", d.dtype);
    if (d.dtype == GQA_DTYPE_FP8_E4M3 && (d.head_dim % 32 != 0 || d.rope != 0))
        return fail(GQA_EINVAL, "an FP8 E4M3 cache needs d_h a multiple of 32 and no rotary mechanism");
    if (d.num_kv_heads < 1 || d.head_dim < 1 || d.head_dim > 256)
        return fail(GQA_EINVAL, "H_kv must be >= 1 and d_h in 1..256");
    if (d.page_tokens != GQA_PAGE_TOKENS)
        return fail(GQA_EINVAL, "page_tokens must be %d", GQA_PAGE_TOKENS);
    if (d.num_pages < 1 || d.max_seqs < 1 || d.max_pages_per_seq < 1)
        return fail(GQA_EINVAL, "num_pages, max_seqs and max_pages_per_seq must be >= 1");
    if ((int64_t)d.max_pages_per_seq * kPageTokens > INT_MAX)
        return fail(GQA_EINVAL, "max_pages_per_seq too large");
    if (d.keys_post_position != 1 && !(d.keys_post_position == 0 && d.rope == 1))
        return fail(GQA_ELAYOUT, "keys_post_position must be 1, or 0 with rope = 1 (keys stored before the "
                                 "library's rotation and rotated when read)");
    if (d.layout_version != GQA_LAYOUT_VERSION)
        return fail(GQA_ELAYOUT, "layout_version %d, this library writes %d", d.layout_version,
                    GQA_LAYOUT_VERSION);
    if (d.rope != 0 && d.rope != 1)
        return fail(GQA_EINVAL, "rope must be 0 (none) or 1 (rotary)");
    if (d.rope == 1 && (d.head_dim % 2 != 0 || !(d.rope_base > 1.0f) || !std::isfinite(d.rope_base)))
        return fail(GQA_EINVAL, "rope = 1 needs an even d_h and a finite rope_base > 1");
    if (d.window < 0)
        return fail(GQA_EINVAL, "window must be 0 (none) or a positive number of tokens");
    const size_t need = gqa_pool_bytes(desc);
    if (pool_dev) {
        if (pool_bytes < need)
            return fail(GQA_EINVAL, "pool has %zu bytes, the description needs %zu", pool_bytes, need);
        if ((uintptr_t)pool_dev % 256 != 0)
            return fail(GQA_EINVAL, "pool must be 256-byte aligned");
    }

    gqa_cache *c = new gqa_cache();
    c->desc = d;
    c->desc.page_order = nullptr;
    c->esize = pool_esize(d.dtype);
    c->io_esize = d.dtype == GQA_DTYPE_F32 ? 4 : 2;
    c->meta_only = pool_dev == nullptr;
    c->pool = pool_dev;
    c->order.resize(d.num_pages);
    c->rank.assign(d.num_pages, -1);
    for (int32_t r = 0; r < d.num_pages; ++r) {
        const int32_t p = d.page_order ? d.page_order[r] : r;
        if (p < 0 || p >= d.num_pages || c->rank[p] != -1) {
            delete c;
            return fail(GQA_EINVAL, "page_order is not a permutation of 0..num_pages-1");
        }
        c->order[r] = p;
        c->rank[p] = r;
    }
    c->ref.assign(d.num_pages, 0);
    {
        std::vector<int32_t> ranks(d.num_pages);
        for (int32_t r = 0; r < d.num_pages; ++r)
            ranks[r] = r;
        c->free_ranks = std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>>(
            std::greater<int32_t>(), std::move(ranks));
    }
    c->seqs.resize(d.max_seqs);
    c->h_tab.assign((size_t)d.max_seqs * d.max_pages_per_seq, 0);

    if (!c->meta_only) {
        cudaError_t e = cudaGetDevice(&c->device);
        int major = 0, minor = 0;
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, c->device);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, c->device);
        c->cc = major * 10 + minor;
        if (e == cudaSuccess)
            e = cudaMalloc((void **)&c->d_tab, c->h_tab.size() * sizeof(int32_t));
        if (e == cudaSuccess)
            e = cudaMemset(c->d_tab, 0, c->h_tab.size() * sizeof(int32_t));
        if (e == cudaSuccess)
            e = cudaMalloc((void **)&c->d_err, sizeof(int32_t));
        if (e == cudaSuccess)
            e = cudaHostAlloc((void **)&c->h_pin, 2 * kStaticStageBytes, cudaHostAllocDefault);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i)
            e = cudaEventCreateWithFlags(&c->pin_done[i], cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaMemset(c->d_err, 0, sizeof(int32_t));
        if (e == cudaSuccess)
            e = cudaMemset(pool_dev, 0, need);         // every slot starts as a finite +0
        if (e == cudaSuccess && d.rope == 1) {
            // cos/sin of pos * base^(-2e/d_h) for every position a sequence
            // can reach, in fp64, rounded to fp32 once.
            const int half = d.head_dim / 2;
            const size_t npos = (size_t)d.max_pages_per_seq * kPageTokens;
            std::vector<float2> tab(npos * half);
            std::vector<double> theta(half);
            for (int i = 0; i < half; ++i)
                theta[i] = std::pow((double)d.rope_base, -2.0 * i / d.head_dim);
            for (size_t p = 0; p < npos; ++p)
                for (int i = 0; i < half; ++i) {
                    const double a = (double)p * theta[i];
                    tab[p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
                }
            e = cudaMalloc((void **)&c->d_rope, tab.size() * sizeof(float2));
            if (e == cudaSuccess)
                e = cudaMemcpy(c->d_rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
        }
        if (e == cudaSuccess)
            e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            gqa_cache_destroy(c);
            return cuda_fail(e, "cache device set-up");
        }
    }
    *out = c;
    return GQA_OK;
}

int gqa_cache_destroy(gqa_cache *c)
{
    if (!c)
        return GQA_OK;
    cudaError_t e = cudaSuccess;
    if (!c->meta_only) {
        e = cudaDeviceSynchronize();
        if (c->d_tab) cudaFree(c->d_tab);
        if (c->d_err) cudaFree(c->d_err);
        if (c->d_stage) cudaFree(c->d_stage);
        if (c->d_ws) cudaFree(c->d_ws);
        if (c->d_rot) cudaFree(c->d_rot);
        if (c->h_pin) cudaFreeHost(c->h_pin);
        for (cudaEvent_t ev : c->pin_done)
            if (ev) cudaEventDestroy(ev);
        if (c->d_cnt) cudaFree(c->d_cnt);
        if (c->d_rope) cudaFree(c->d_rope);
        if (c->d_io) cudaFree(c->d_io);
        if (c->io_up) cudaStreamDestroy(c->io_up);
        if (c->io_down) cudaStreamDestroy(c->io_down);
        for (cudaEvent_t ev : c->io_events)
            cudaEventDestroy(ev);
        for (const auto &r : c->prof_recs) {
            cudaEventDestroy(r.start);
            cudaEventDestroy(r.end);
        }
        for (cudaEvent_t ev : c->spare_events)
            cudaEventDestroy(ev);
    }
    delete c;
    return e == cudaSuccess ? GQA_OK : cuda_fail(e, "cache destroy");
}

int gqa_cache_layout(const gqa_cache *c, gqa_layout_metadata *out)
{
    if (!c || !out)
        return fail(GQA_EINVAL, "NULL argument");
    out->keys_post_position = c->desc.keys_post_position;
    out->dtype = c->desc.dtype;
    out->page_tokens = c->desc.page_tokens;
    out->layout_version = c->desc.layout_version;
    out->num_kv_heads = c->desc.num_kv_heads;
    out->head_dim = c->desc.head_dim;
    out->rope = c->desc.rope;
    out->rope_base = c->desc.rope == 1 ? c->desc.rope_base : 0.0f;
    out->window = c->desc.window;
    return GQA_OK;
}

int gqa_layout_compatible(const gqa_layout_metadata *a, const gqa_layout_metadata *b)
{
    if (!a || !b)
        return fail(GQA_EINVAL, "NULL argument");
    if (a->keys_post_position != b->keys_post_position)
        return fail(GQA_ELAYOUT, "position convention differs (post- vs pre-position keys)");
    if (a->dtype != b->dtype || a->page_tokens != b->page_tokens || a->layout_version != b->layout_version ||
        a->num_kv_heads != b->num_kv_heads || a->head_dim != b->head_dim)
        return fail(GQA_ELAYOUT, "precision, page size, layout version or KV shape differs");
    if (a->rope != b->rope || (a->rope == 1 && a->rope_base != b->rope_base))
        return fail(GQA_ELAYOUT, "the keys were rotated with a different position mechanism");
    if (a->window != b->window)
        return fail(GQA_ELAYOUT, "sliding windows differ (pages outside the window were released)");
    return GQA_OK;
}

int gqa_seq_create(gqa_cache *c, int32_t *seq_out)
{
    if (!c || !seq_out)
        return fail(GQA_EINVAL, "NULL argument");
    for (int32_t s = 0; s < c->desc.max_seqs; ++s) {
        if (!c->seqs[s].live) {
            SeqState &S = c->seqs[s];
            S.live = true;
            S.len = 0;
            S.pages.clear();
            *seq_out = s;
            return GQA_OK;
        }
    }
    return fail(GQA_ENOMEM, "all %d sequence ids are in use", c->desc.max_seqs);
}

int gqa_seq_fork(gqa_cache *c, int32_t src, int32_t prefix_len, int32_t *seq_out)
{
    if (!c || !seq_out)
        return fail(GQA_EINVAL, "NULL argument");
    if (!live(c, src))
        return fail(GQA_EINVAL, "sequence %d is not live", src);
    if (prefix_len < 0 || prefix_len > c->seqs[src].len)
        return fail(GQA_ERANGE, "prefix %d outside 0..%d", prefix_len, c->seqs[src].len);
    if (!window_holds(c, c->seqs[src], prefix_len))
        return fail(GQA_ERANGE, "prefix %d reaches back past the sliding window", prefix_len);
    int32_t s = -1;
    int rc = gqa_seq_create(c, &s);
    if (rc != GQA_OK)
        return rc;
    const int32_t keep = pages_for(prefix_len);
    SeqState &S = c->seqs[s];
    for (int32_t i = 0; i < keep; ++i) {
        const int32_t p = c->seqs[src].pages[i];
        if (p >= 0)
            c->ref[p] += 1;
        S.pages.push_back(p);
        c->set_entry(s, i, p);
    }
    S.len = prefix_len;
    *seq_out = s;
    return GQA_OK;
}

int kv_truncate(gqa_cache *c, int32_t seq, int32_t m)
{
    if (!c)
        return fail(GQA_EINVAL, "NULL cache");
    if (!live(c, seq))
        return fail(GQA_EINVAL, "sequence %d is not live", seq);
    SeqState &S = c->seqs[seq];
    if (m < 0 || m > S.len)
        return fail(GQA_ERANGE, "truncate to %d outside 0..%d", m, S.len);
    if (!window_holds(c, S, m))
        return fail(GQA_ERANGE, "truncate to %d reaches back past the sliding window", m);
    const int32_t keep = pages_for(m);
    for (size_t i = keep; i < S.pages.size(); ++i)
        if (S.pages[i] >= 0)
            c->drop_page(S.pages[i]);
    S.pages.resize(keep);
    S.len = m;
    return GQA_OK;
}

int gqa_seq_free(gqa_cache *c, int32_t seq)
{
    int rc = kv_truncate(c, seq, 0);
    if (rc != GQA_OK)
        return rc;
    c->seqs[seq].live = false;
    return GQA_OK;
}

int gqa_seq_length(const gqa_cache *c, int32_t seq, int32_t *len_out)
{
    if (!c || !len_out)
        return fail(GQA_EINVAL, "NULL argument");
    if (!live(c, seq))
        return fail(GQA_EINVAL, "sequence %d is not live", seq);
    *len_out = c->seqs[seq].len;
    return GQA_OK;
}

int gqa_seq_block_table(const gqa_cache *c, int32_t seq, int32_t *out, int32_t cap, int32_t *count_out)
{
    if (!c || !count_out)
        return fail(GQA_EINVAL, "NULL argument");
    if (!live(c, seq))
        return fail(GQA_EINVAL, "sequence %d is not live", seq);
    const SeqState &S = c->seqs[seq];
    *count_out = (int32_t)S.pages.size();
    if ((size_t)cap < S.pages.size() || (!out && !S.pages.empty()))
        return fail(GQA_ERANGE, "block table has %zu entries, capacity %d", S.pages.size(), cap);
    std::copy(S.pages.begin(), S.pages.end(), out);
    return GQA_OK;
}

int gqa_free_pages(const gqa_cache *c, int32_t *out)
{
    if (!c || !out)
        return fail(GQA_EINVAL, "NULL argument");
    *out = (int32_t)c->free_ranks.size();
    return GQA_OK;
}

int gqa_page_refcount(const gqa_cache *c, int32_t page, int32_t *out)
{
    if (!c || !out)
        return fail(GQA_EINVAL, "NULL argument");
    if (page < 0 || page >= c->desc.num_pages)
        return fail(GQA_ERANGE, "page %d outside 0..%d", page, c->desc.num_pages - 1);
    *out = c->ref[page];
    return GQA_OK;
}

// ---------------------------------------------------------------------------
// Work plan of the tensor-core kernel.
// ---------------------------------------------------------------------------

struct TcPlan {
    std::vector<TcItem> items;        // grouped by CTA
    std::vector<int32_t> item_start;  // grid + 1 offsets
    int grid = 1;
    int32_t slots = 0;                // split workspace slots
    int32_t slot_rows = 0;
    bool ranged = false;              // an item starts past key tile 0
    std::vector<int64_t> load;        // per CTA: cost of its items (quarter key tiles)
};

// Items: two query tiles of 128 / G positions of one (entry, KV head) each;
// the second tile is skipped when it has no valid row.  An entry whose rows
// all fit the first tile (decode, multi-token decode) may be split along its
// key tiles into pieces of about `piece` tiles so that there are several
// items per SM; the pieces' partial results are merged by the kernel.
// Items are then placed longest-first on the least-loaded CTA (LPT); a CTA
// runs its items in that order.  Cost of an item, in quarter key tiles:
// 4 per tile with two query tiles, 3 with one, plus a fixed share for the
// Q load, the pipeline refill and the epilogue.
void plan_tc(const gqa_cache *c, const std::vector<SeqDesc> &sds, int G, TcPlan &pl)
{
    const int rows_pos = prefill_tc_rows_per_tile(G), span = 2 * rows_pos;
    const int B = (int)sds.size();
    std::vector<TcItem> items;
    int64_t split_tiles = 0;
    for (int b = 0; b < B; ++b)
        for (int32_t i0 = 0; i0 < sds[b].count; i0 += span) {
            const int32_t last = std::min<int32_t>(i0 + span, sds[b].count) - 1;
            const int32_t nt = (sds[b].past + last) / 128 + 1;
            // Under a sliding window the item's first row sees the oldest key.
            const int32_t j0 = window_start(sds[b].past + i0, c->desc.window) / 128;
            const int32_t tiles = i0 + rows_pos < sds[b].count ? 2 : 1;
            for (int32_t h = 0; h < c->desc.num_kv_heads; ++h)
            {
                TcItem x{};
                x.b = b;
                x.kvh = h;
                x.i0 = i0;
                x.nt = nt;
                x.j0 = j0;
                x.tiles = (int8_t)tiles;
                x.part = -1;
                x.split = 0;
                x.nsplit = 1;
                items.push_back(x);
            }
            split_tiles += (int64_t)(nt - j0) * c->desc.num_kv_heads;
        }
    // Pieces of at least kSplitMinTiles key tiles, sized for about
    // kSplitItemsPerSm items per SM.
    const int64_t per = (int64_t)kSplitItemsPerSm * c->num_sms;
    const int64_t piece = std::max<int64_t>(kSplitMinTiles, (split_tiles + per - 1) / per);
    std::vector<TcItem> all;
    all.reserve(items.size());
    for (const TcItem &it : items) {
        const int32_t K = it.nt - it.j0;
        if (it.i0 != 0 || it.tiles != 1 || sds[it.b].count > rows_pos || K <= piece) {
            all.push_back(it);
            continue;
        }
        const int32_t S = (int32_t)((K + piece - 1) / piece);
        for (int32_t q = 0; q < S; ++q) {
            TcItem x = it;
            x.j0 = it.j0 + (int32_t)((int64_t)q * K / S);
            x.nt = it.j0 + (int32_t)((int64_t)(q + 1) * K / S);
            x.part = pl.slots + q;
            x.split = (int16_t)q;
            x.nsplit = (int16_t)S;
            all.push_back(x);
        }
        pl.slots += S;
        pl.slot_rows = std::max<int32_t>(pl.slot_rows, sds[it.b].count * G);
    }
    auto cost = [](const TcItem &x) { return (int64_t)(x.tiles > 1 ? 4 : 3) * (x.nt - x.j0) + kItemCostQuarters; };
    std::stable_sort(all.begin(), all.end(), [&](const TcItem &x, const TcItem &y) { return cost(x) > cost(y); });
    pl.grid = std::max(1, std::min<int>(c->num_sms, (int)all.size()));
    std::vector<std::vector<int>> runs(pl.grid);
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int i = 0; i < pl.grid; ++i)
        heap.push({0, i});
    for (size_t i = 0; i < all.size(); ++i) {
        Load top = heap.top();
        heap.pop();
        runs[top.second].push_back((int)i);
        top.first += cost(all[i]);
        heap.push(top);
    }
    pl.load.assign(pl.grid, 0);
    while (!heap.empty()) {
        pl.load[heap.top().second] = heap.top().first;
        heap.pop();
    }
    pl.items.clear();
    pl.items.reserve(all.size());
    pl.item_start.assign(1, 0);
    for (const auto &run : runs) {
        for (int i : run) {
            pl.items.push_back(all[i]);
            pl.ranged |= all[i].j0 > 0;
        }
        pl.item_start.push_back((int32_t)pl.items.size());
    }
}

// Host descriptors of a tensor-core launch (no zero shares, the cache's own
// tables), and whether the launch can carry them in its parameters.
static TcHostDesc tc_host(const std::vector<SeqDesc> &sds, const TcPlan &plan)
{
    TcHostDesc h;
    h.seqs = sds.data();
    h.n_seqs = (int)sds.size();
    h.items = plan.items.data();
    h.n_items = (int)plan.items.size();
    h.item_start = plan.item_start.data();
    h.n_start = (int)plan.item_start.size();
    return h;
}

static bool tc_inline_ok(const gqa_cache *c, const TcHostDesc &h)
{
    return c->desc.dtype == GQA_DTYPE_BF16 && c->desc.rope == 0 && prefill_tc_inline_fits(h);
}

// Fused prefill: the padding rows of out that no item stores (`units`
// 16-byte units in all) are cleared by the CTAs after their items, the
// least-loaded CTAs taking the most (water-filling their loads up to a
// common level, about 16 KB per quarter key tile of spare time).  Returns
// grid + 1 offsets into the units.
std::vector<int64_t> zero_shares(const TcPlan &pl, int64_t units)
{
    constexpr double kUnitsPerQuarter = 1024.0;
    const int g = pl.grid;
    std::vector<int64_t> start(g + 1, 0);
    if (units <= 0 || g < 1)
        return start;
    std::vector<int64_t> L = pl.load;
    std::sort(L.begin(), L.end());
    const double need = (double)units / kUnitsPerQuarter;
    double level = (double)L[g - 1], below = 0.0;
    for (int k = 1; k <= g; ++k) {
        below += (double)L[k - 1];                    // sum of the k smallest loads
        const double t = (need + below) / k;          // level filling exactly the k smallest
        if (k == g || t <= (double)L[k]) {
            level = t;
            break;
        }
    }
    int64_t given = 0;
    for (int c = 0; c < g; ++c) {
        const int64_t share = (int64_t)std::max(0.0, (level - (double)pl.load[c]) * kUnitsPerQuarter);
        start[c + 1] = start[c] + std::min(share, units - given);
        given = start[c + 1];
    }
    start[g] = units;                                 // rounding: the last CTA takes the rest
    return start;
}

// Split workspace of a plan in the cache's growable buffers.
int tc_workspace(gqa_cache *c, const TcPlan &pl, TcSplitWs &ws)
{
    ws.ranged = pl.ranged;
    ws.slot_rows = pl.slot_rows;
    if (pl.slots == 0)
        return GQA_OK;
    const size_t rows = (size_t)pl.slots * pl.slot_rows;
    int rc = ensure_ws(c, rows * 128 + rows * 2);
    if (rc == GQA_OK)
        rc = ensure_cnt(c, (size_t)pl.slots);
    if (rc != GQA_OK)
        return rc;
    ws.o = c->d_ws;
    ws.ml = reinterpret_cast<float2 *>(c->d_ws + rows * 128);
    ws.counters = c->d_cnt;
    return GQA_OK;
}

// Which decode kernel a call runs: 1 = tensor-core, 0 = CUDA-core, -1 = the
// tensor-core kernel was asked for but cannot serve this cache or group.
int decode_uses_tc(const gqa_cache *c, int G)
{
    // Pre-position keys are rotated as they are read, on the CUDA cores.
    const bool ok = (c->desc.dtype == GQA_DTYPE_BF16 || c->desc.dtype == GQA_DTYPE_FP8_E4M3) &&
                    c->desc.head_dim == 128 && c->cc >= 100 && c->desc.keys_post_position == 1 &&
                    prefill_tc_supported(G, c->desc.num_kv_heads);
    if (c->decode_kernel == GQA_DECODE_CUDA_CORE)
        return 0;
    if (c->decode_kernel == GQA_DECODE_TENSOR_CORE)
        return ok ? 1 : -1;
    // Automatic: the tensor-core kernel for bf16.  A quantised cache decodes
    // faster on the CUDA-core kernel, which reads the codes directly; on the
    // tensor-core kernel each stage's codes are converted in place to bf16
    // operands before use, so a stage's next load waits for its landing,
    // conversion and use, and the load latency is no longer hidden.
    return ok && c->desc.dtype == GQA_DTYPE_BF16 ? 1 : 0;
}

// Cluster size of the clustered decode kernel for a call of B single-token
// queries whose longest sequence holds max_len tokens (the query's own
// included), with query rows q and, for a fused append, new rows k_new and
// v_new (bf16 caches only: an FP8 cache's write quantises in its own
// kernel); 0 when another kernel serves the call; -1 when the clustered
// kernel was asked for but cannot serve it.  Automatic choice: when there
// are at most half as many (entry, KV head) pairs as SMs, so every pair
// gets two or more SMs (larger batches run the tensor-core kernel, or for
// an FP8 cache the split-K CUDA-core one: one CTA per pair walking a whole
// sequence leaves an SM too few warps to hide HBM latency behind the
// conversions of the codes).  The cluster is the largest size (at most 16,
// and at most the pages of the longest sequence) such that the pairs'
// clusters fit the SMs and are resident together.
int decode_cluster_for(const gqa_cache *c, int G, int B, int32_t max_len, const void *q,
                       const void *k_new = nullptr, const void *v_new = nullptr)
{
    const int32_t H_kv = c->desc.num_kv_heads;
    const bool q8 = c->desc.dtype == GQA_DTYPE_FP8_E4M3;
    const bool ok = (c->desc.dtype == GQA_DTYPE_BF16 || q8) && c->desc.head_dim == 128 && c->cc >= 100 &&
                    c->desc.rope == 0 && decode_cluster_supported(G) && B >= 1 && B <= 65535 && H_kv <= 65535 &&
                    !(q8 && k_new) && ((uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new) % 16 == 0;
    if (c->decode_kernel == GQA_DECODE_CLUSTER) {
        if (!ok)
            return -1;
    } else if (c->decode_kernel != GQA_DECODE_AUTO || !ok) {
        return 0;
    }
    const int64_t pairs = (int64_t)B * H_kv;
    if (c->decode_kernel == GQA_DECODE_AUTO && pairs * 2 > c->num_sms)
        return 0;
    const int32_t pages = (max_len - decode_first_token(max_len, c->desc.window) + kPageTokens - 1) / kPageTokens;
    for (int cs = 16; cs >= 2; --cs)
        if (cs <= pages && pairs * cs <= c->num_sms && decode_cluster_capacity(cs) >= pairs)
            return cs;
    return 1;
}

static const char *kClusterNeeds = "the clustered decode kernel needs a bf16 or FP8 E4M3 cache with d_h = 128, "
                                   "no rotary, H_q/H_kv <= 16 and 16-byte aligned q (and k_new, v_new)";

// ---------------------------------------------------------------------------
// The hot path.
// ---------------------------------------------------------------------------

// Every precondition of a prefill call, checked before anything changes
// (req: one write request per entry; max_nb: the longest valid length).
static int validate_prefill(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t n, int32_t H_q, bool have_io,
                            const int32_t *valid_lengths, const int32_t *positions, std::vector<WriteReq> &req,
                            int32_t &max_nb)
{
    if (!c || !seq_ids || !valid_lengths)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || n < 1 || H_q < 1)
        return fail(GQA_EINVAL, "B, n and H_q must be >= 1");
    if (H_q % c->desc.num_kv_heads != 0)
        return fail(GQA_EINVAL, "H_kv = %d does not divide H_q = %d", c->desc.num_kv_heads, H_q);
    if (!c->meta_only && !have_io)
        return fail(GQA_EINVAL, "NULL tensor pointer");
    req.assign(B, WriteReq{});
    max_nb = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t nb = valid_lengths[b];
        if (nb < 1 || nb > n)
            return fail(GQA_EMASK, "batch entry %d: valid length %d outside 1..%d leaves a query row "
                                   "without a finite score", b, nb, n);
        req[b] = WriteReq{seq_ids[b], nb};
        max_nb = std::max(max_nb, nb);
    }
    int rc = check_write(c, req.data(), B);
    if (rc != GQA_OK)
        return rc;
    if (positions) {
        for (int b = 0; b < B; ++b) {
            const int32_t P = c->seqs[seq_ids[b]].len;
            for (int32_t i = 0; i < req[b].count; ++i)
                if (positions[(size_t)b * n + i] != P + i)
                    return fail(GQA_ERANGE, "batch entry %d row %d: position %d, the cache continues at %d",
                                b, i, positions[(size_t)b * n + i], P + i);
        }
    }
    if (!c->meta_only && (rc = check_device(c)) != GQA_OK)
        return rc;
    return GQA_OK;
}

static int attn_prefill_impl(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t n, int32_t H_q, const void *q,
                 const void *k, const void *v, const int32_t *valid_lengths, const int32_t *positions,
                 void *out, void *stream)
{
    std::vector<WriteReq> req;
    int32_t max_nb = 0;
    int rc = validate_prefill(c, B, seq_ids, n, H_q, q && k && v && out, valid_lengths, positions, req, max_nb);
    if (rc != GQA_OK)
        return rc;

    std::vector<SeqDesc> sds;
    std::vector<CowDesc> cows;
    commit_write(c, req.data(), B, sds, cows);
    if (c->meta_only)
        return GQA_OK;

    cudaStream_t st = (cudaStream_t)stream;
    const int G = H_q / c->desc.num_kv_heads;
    const bool use_tc = (c->desc.dtype == GQA_DTYPE_BF16 || c->desc.dtype == GQA_DTYPE_FP8_E4M3) &&
                        c->desc.head_dim == 128 && c->cc >= 100 && prefill_tc_supported(G, c->desc.num_kv_heads);
    // The call's own block-table rows (row b = entry b, every page of the
    // sequence after this write) travel with its descriptors in one upload;
    // the device's table array is brought up to date by the next call that
    // reads it (its entries stay marked dirty).  One copy queued before the
    // kernels instead of two.  Pre-position calls rotate the pool's pages
    // by the pool's tables and keep them current.
    const bool pre = use_tc && c->desc.keys_post_position == 0;
    std::vector<int32_t> ctab;
    int32_t cstride = 1;
    if (!pre) {
        for (int b = 0; b < B; ++b)
            cstride = std::max<int32_t>(cstride, (int32_t)c->seqs[sds[b].row].pages.size());
        if ((size_t)B * cstride * sizeof(int32_t) > kCompactTableBytes)
            cstride = 0;                                 // too large: the kernels read the pool's tables
    }
    if (!pre && cstride > 0) {
        ctab.assign((size_t)B * cstride, -1);
        for (int b = 0; b < B; ++b) {
            const int32_t row = sds[b].row;
            const size_t np = c->seqs[row].pages.size();
            std::copy(c->h_tab.begin() + (size_t)row * c->stride(), c->h_tab.begin() + (size_t)row * c->stride() + np,
                      ctab.begin() + (size_t)b * cstride);
            sds[b].row = b;
        }
    } else if ((rc = upload_tables(c, st)) != GQA_OK) {
        return rc;
    }
    // Pre-position keys on the tensor-core path: the kernel reads keys as
    // stored, so every distinct page the call reads is first copied, keys
    // rotated by their positions, to a compact scratch pool, and the kernel
    // reads that copy through block tables remapped to it (row b = entry b).
    // Each page is rotated once per call however many items read it.
    const bool pre_tc = use_tc && c->desc.keys_post_position == 0;
    std::vector<int2> rot_pages;
    std::vector<int32_t> rot_tab;
    std::vector<SeqDesc> rot_sds;
    int32_t rot_stride = 1;
    if (pre_tc) {
        for (int b = 0; b < B; ++b)
            rot_stride = std::max<int32_t>(rot_stride, (int32_t)c->seqs[sds[b].row].pages.size());
        rot_tab.assign((size_t)B * rot_stride, -1);
        c->rot_slot.resize(c->desc.num_pages, -1);
        for (int b = 0; b < B; ++b) {
            const std::vector<int32_t> &pg = c->seqs[sds[b].row].pages;
            for (size_t lp = 0; lp < pg.size(); ++lp) {
                const int32_t ph = pg[lp];
                if (ph < 0)
                    continue;                             // released by the sliding window
                if (c->rot_slot[ph] < 0) {
                    c->rot_slot[ph] = (int32_t)rot_pages.size();
                    rot_pages.push_back(make_int2(ph, (int)lp));   // shared pages sit at one logical index
                }
                rot_tab[(size_t)b * rot_stride + lp] = c->rot_slot[ph];
            }
        }
        for (const int2 &x : rot_pages)
            c->rot_slot[x.x] = -1;
        rot_sds = sds;
        for (int b = 0; b < B; ++b)
            rot_sds[b].row = b;
    }
    TcPlan plan;
    if (use_tc)
        plan_tc(c, sds, G, plan);
    // Fused cache write: the tensor-core kernel reads this call's rows from
    // k and v and writes their pages itself when every entry starts on a
    // page boundary (each page then holds old rows only or new rows only;
    // no copy-on-write), for a bf16 cache without rotation; k and v are
    // read as groups of 8 rows, so n must be a multiple of 8.
    bool fused = use_tc && c->desc.dtype == GQA_DTYPE_BF16 && c->desc.rope == 0 && cows.empty() && n % 8 == 0 &&
                 ((uintptr_t)k | (uintptr_t)v) % 16 == 0;
    for (int b = 0; fused && b < B; ++b)
        fused = sds[b].past % kPageTokens == 0;
    if (fused) {
        // Rows an item's epilogue stores: its query tiles' rows (a split
        // item's merge stores the valid rows only); out rows from zero_from
        // on are zeroed by the kernel.
        const int rows_pos = prefill_tc_rows_per_tile(G);
        std::vector<int32_t> cover(B, 0);
        for (const TcItem &it : plan.items)
            cover[it.b] = std::max(cover[it.b], it.part >= 0 ? sds[it.b].count : it.i0 + it.tiles * rows_pos);
        for (int b = 0; b < B; ++b)
            sds[b].zero_from = std::min(n, cover[b]);
    }
    std::vector<int64_t> zstart;
    if (fused) {
        int64_t units = 0;
        for (int b = 0; b < B; ++b)
            units += (int64_t)(n - sds[b].zero_from) * H_q * (c->desc.head_dim * c->io_esize / 16);
        zstart = zero_shares(plan, units);
    }
    Stage stg(c->h_stage);
    const size_t o_sds = stg.add(sds.data(), sds.size());
    const size_t o_cow = stg.add(cows.data(), cows.size());
    const size_t o_items = stg.add(plan.items.data(), plan.items.size());
    const size_t o_start = stg.add(plan.item_start.data(), plan.item_start.size());
    const size_t o_zero = stg.add(zstart.data(), zstart.size());
    const size_t o_rpages = stg.add(rot_pages.data(), rot_pages.size());
    const size_t o_rtab = stg.add(rot_tab.data(), rot_tab.size());
    const size_t o_rsds = stg.add(rot_sds.data(), rot_sds.size());
    const size_t o_ctab = stg.add(ctab.data(), ctab.size());
    if (pre_tc && (rc = ensure_rot(c, rot_pages.size() * 2 * (size_t)c->desc.num_kv_heads * 4096)) != GQA_OK)
        return rc;
    TcSplitWs ws;
    if (use_tc && (rc = tc_workspace(c, plan, ws)) != GQA_OK)
        return rc;
    // A fused tensor-core call with nothing else to launch can carry its
    // descriptors in the kernel parameters: then no copy precedes the kernel.
    TcHostDesc hd;
    if (use_tc && fused && cows.empty() && !pre_tc) {
        hd.seqs = sds.data();
        hd.n_seqs = B;
        hd.items = plan.items.data();
        hd.n_items = (int)plan.items.size();
        hd.item_start = plan.item_start.data();
        hd.n_start = (int)plan.item_start.size();
        hd.zero_start = zstart.data();
        hd.n_zero = (int)zstart.size();
        hd.tables = ctab.empty() ? nullptr : ctab.data();
        hd.n_tables = ctab.size();
    }
    const bool inl = use_tc && fused && cows.empty() && !pre_tc && tc_inline_ok(c, hd);
    if (!inl && (rc = upload_stage(c, st)) != GQA_OK)
        return rc;
    PoolView pv = c->view();
    if (!ctab.empty()) {
        pv.tables = (const int32_t *)(c->d_stage + o_ctab);
        pv.stride = cstride;
    }
    const SeqDesc *d_sds = (const SeqDesc *)(c->d_stage + o_sds);
    if (!cows.empty() &&
        (rc = run_kernel(c, GQA_KERNEL_COW_COPY, st, "copy-on-write kernel", [&](cudaEvent_t ev) {
             rec(ev, st);
             return launch_cow_copy(pv, c->esize, (const CowDesc *)(c->d_stage + o_cow), (int)cows.size(), st);
         })) != GQA_OK)
        return rc;
    // Unfused, on the tensor-core path the write kernel also zeroes the
    // padding rows of out (discarded rows are written as zeros); the
    // prefill kernel then writes the valid rows only.
    const int out_row_bytes = H_q * c->desc.head_dim * c->io_esize;
    if (!fused && (rc = run_kernel(c, GQA_KERNEL_CACHE_WRITE, st, "cache write kernel", [&](cudaEvent_t ev) {
                       rec(ev, st);
                       return launch_cache_write(pv, c->esize, d_sds, B, n, max_nb, k, v, st, use_tc ? out : nullptr,
                                                 out_row_bytes);
                   })) != GQA_OK)
        return rc;
    if (pre_tc) {
        if ((rc = run_kernel(c, GQA_KERNEL_ROTATE_PAGES, st, "page rotation kernel", [&](cudaEvent_t ev) {
                 rec(ev, st);
                 return launch_rotate_pages(pv, (const int2 *)(c->d_stage + o_rpages), (int)rot_pages.size(),
                                            c->d_rot, st);
             })) != GQA_OK)
            return rc;
        PoolView rv = pv;
        rv.pool = c->d_rot;
        rv.tables = (const int32_t *)(c->d_stage + o_rtab);
        rv.stride = rot_stride;
        rv.num_pages = (int32_t)rot_pages.size();
        rv.keys_pre = 0;                                  // the copy holds the keys as attention uses them
        return run_kernel(c, GQA_KERNEL_PREFILL_TC, st, "tensor-core prefill kernel", [&](cudaEvent_t ev) {
            return launch_prefill_tc(rv, (const SeqDesc *)(c->d_stage + o_rsds), (const TcItem *)(c->d_stage + o_items),
                                     (const int32_t *)(c->d_stage + o_start), plan.grid, B, n, H_q, q, out, ws, st, ev);
        });
    }
    if (use_tc) {
        return run_kernel(c, GQA_KERNEL_PREFILL_TC, st, "tensor-core prefill kernel", [&](cudaEvent_t ev) {
            return launch_prefill_tc(pv, d_sds, (const TcItem *)(c->d_stage + o_items),
                                     (const int32_t *)(c->d_stage + o_start), plan.grid, B, n, H_q, q, out, ws, st, ev,
                                     nullptr, nullptr, fused ? k : nullptr, fused ? v : nullptr,
                                     fused ? (const int64_t *)(c->d_stage + o_zero) : nullptr, inl ? &hd : nullptr);
        });
    }
    return run_kernel(c, GQA_KERNEL_ATTN_SIMT, st, "attention kernel", [&](cudaEvent_t ev) {
        rec(ev, st);
        return launch_attn_simt(pv, c->desc.dtype, d_sds, B, n, H_q, q, out, st);
    });
}

static int kv_append_impl(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t n, const int32_t *counts,
              const void *k_new, const void *v_new, void *stream)
{
    if (!c || !seq_ids)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || n < 1)
        return fail(GQA_EINVAL, "B and n must be >= 1");
    if (!c->meta_only && (!k_new || !v_new))
        return fail(GQA_EINVAL, "NULL tensor pointer");
    std::vector<WriteReq> req(B);
    int32_t max_c = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t cnt = counts ? counts[b] : n;
        if (cnt < 0 || cnt > n)
            return fail(GQA_EINVAL, "batch entry %d: count %d outside 0..%d", b, cnt, n);
        req[b] = WriteReq{seq_ids[b], cnt};
        max_c = std::max(max_c, cnt);
    }
    int rc = check_write(c, req.data(), B);
    if (rc != GQA_OK)
        return rc;
    if (!c->meta_only && (rc = check_device(c)) != GQA_OK)
        return rc;
    std::vector<SeqDesc> sds;
    std::vector<CowDesc> cows;
    commit_write(c, req.data(), B, sds, cows);
    if (c->meta_only)
        return GQA_OK;

    cudaStream_t st = (cudaStream_t)stream;
    if ((rc = upload_tables(c, st)) != GQA_OK)
        return rc;
    Stage stg(c->h_stage);
    const size_t o_sds = stg.add(sds.data(), sds.size());
    const size_t o_cow = stg.add(cows.data(), cows.size());
    if ((rc = upload_stage(c, st)) != GQA_OK)
        return rc;
    const PoolView pv = c->view();
    if (!cows.empty() &&
        (rc = run_kernel(c, GQA_KERNEL_COW_COPY, st, "copy-on-write kernel", [&](cudaEvent_t ev) {
             rec(ev, st);
             return launch_cow_copy(pv, c->esize, (const CowDesc *)(c->d_stage + o_cow), (int)cows.size(), st);
         })) != GQA_OK)
        return rc;
    return run_kernel(c, GQA_KERNEL_CACHE_WRITE, st, "cache write kernel", [&](cudaEvent_t ev) {
        rec(ev, st);
        return launch_cache_write(pv, c->esize, (const SeqDesc *)(c->d_stage + o_sds), B, n, max_c, k_new, v_new,
                                  st);
    });
}

int attn_prefill(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t n, int32_t H_q, const void *q,
                 const void *k, const void *v, const int32_t *valid_lengths, const int32_t *positions, void *out,
                 void *stream)
{
    const int rc = attn_prefill_impl(c, B, seq_ids, n, H_q, q, k, v, valid_lengths, positions, out, stream);
    if (rc == GQA_OK)
        release_windows(c, B, seq_ids);
    return rc;
}

// The packed device rows, copy streams and events of attn_prefill_host,
// grown on demand (a growth frees the old rows, which waits for the device).
static int ensure_io(gqa_cache *c, size_t bytes, size_t events)
{
    cudaError_t e = cudaSuccess;
    if (bytes > c->io_cap) {
        if (c->d_io) {
            e = cudaFree(c->d_io);
            c->d_io = nullptr;
            c->io_cap = 0;
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaFree(host-call rows)");
        }
        const size_t cap = (bytes + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
        if ((e = cudaMalloc((void **)&c->d_io, cap)) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(host-call rows)");
        c->io_cap = cap;
    }
    if (!c->io_up && (e = cudaStreamCreateWithFlags(&c->io_up, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e, "upload stream");
    if (!c->io_down && (e = cudaStreamCreateWithFlags(&c->io_down, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e, "download stream");
    while (c->io_events.size() < events) {
        cudaEvent_t ev;
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "event");
        c->io_events.push_back(ev);
    }
    return GQA_OK;
}

int attn_prefill_host(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t n, int32_t H_q, const void *q,
                      const void *k, const void *v, const int32_t *valid_lengths, const int32_t *positions,
                      void *out, void *stream)
{
    // The whole batch is checked first, so a rejected call queues and
    // changes nothing; each entry then runs as a one-entry prefill whose
    // checks repeat what was checked here.
    std::vector<WriteReq> req;
    int32_t max_nb = 0;
    int rc = validate_prefill(c, B, seq_ids, n, H_q, q && k && v && out, valid_lengths, positions, req, max_nb);
    if (rc != GQA_OK)
        return rc;
    // Largest entries first: the last entry's prefill and download are the
    // part of the call that nothing overlaps.
    std::vector<int> order(B);
    for (int b = 0; b < B; ++b)
        order[b] = b;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return valid_lengths[x] > valid_lengths[y]; });
    if (c->meta_only) {
        for (int b : order) {
            if ((rc = attn_prefill_impl(c, 1, seq_ids + b, valid_lengths[b], H_q, nullptr, nullptr, nullptr,
                                        valid_lengths + b, positions ? positions + (size_t)b * n : nullptr, nullptr,
                                        nullptr)) != GQA_OK)
                return rc;
            release_windows(c, 1, seq_ids + b);
        }
        return GQA_OK;
    }
    const size_t d = (size_t)c->desc.head_dim, es = (size_t)c->io_esize;
    const size_t row_q = (size_t)H_q * d * es, row_kv = (size_t)c->desc.num_kv_heads * d * es;
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    // Each entry's packed rows are padded to a multiple of 8 (the one-entry
    // prefill runs with n = that, so the tensor-core kernel can read its k
    // and v rows in groups of 8; the padding rows are never valid).
    auto rows8 = [&](int b) { return ((size_t)valid_lengths[b] + 7) & ~(size_t)7; };
    std::vector<size_t> off(B);                      // entry b's packed q, k, v, out rows, in call order
    size_t bytes = 0;
    for (int b : order) {
        off[b] = bytes;
        bytes += al(rows8(b) * row_q) * 2 + al(rows8(b) * row_kv) * 2;
    }
    if ((rc = ensure_io(c, bytes, 2 * (size_t)B + 2)) != GQA_OK)
        return rc;
    cudaStream_t st = (cudaStream_t)stream;
    cudaEvent_t *ev = c->io_events.data();            // [0] call start, [1] downloads done, then in/out per entry
    cudaError_t e = cudaEventRecord(ev[0], st);      // the previous call's users of the rows are done
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(c->io_up, ev[0], 0);
    for (int i = 0; e == cudaSuccess && i < B; ++i) {
        const int b = order[i];
        const size_t nb = (size_t)valid_lengths[b], n8 = rows8(b);
        char *base = c->d_io + off[b];
        const char *qh = (const char *)q + (size_t)b * n * row_q, *kh = (const char *)k + (size_t)b * n * row_kv,
                   *vh = (const char *)v + (size_t)b * n * row_kv;
        if ((e = cudaMemcpyAsync(base, qh, nb * row_q, cudaMemcpyHostToDevice, c->io_up)) == cudaSuccess &&
            (e = cudaMemcpyAsync(base + al(n8 * row_q), kh, nb * row_kv, cudaMemcpyHostToDevice, c->io_up)) ==
                cudaSuccess &&
            (e = cudaMemcpyAsync(base + al(n8 * row_q) + al(n8 * row_kv), vh, nb * row_kv, cudaMemcpyHostToDevice,
                                 c->io_up)) == cudaSuccess)
            e = cudaEventRecord(ev[2 + 2 * i], c->io_up);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "host-call upload");
    for (int i = 0; i < B; ++i) {
        const int b = order[i];
        const size_t nb = (size_t)valid_lengths[b], n8 = rows8(b);
        char *dq = c->d_io + off[b], *dk = dq + al(n8 * row_q), *dv = dk + al(n8 * row_kv),
             *dout = dv + al(n8 * row_kv);
        if ((e = cudaStreamWaitEvent(st, ev[2 + 2 * i], 0)) != cudaSuccess)
            return cuda_fail(e, "host-call wait for upload");
        if ((rc = attn_prefill_impl(c, 1, seq_ids + b, (int32_t)n8, H_q, dq, dk, dv, valid_lengths + b,
                                    positions ? positions + (size_t)b * n : nullptr, dout, st)) != GQA_OK)
            return rc;
        release_windows(c, 1, seq_ids + b);
        if ((e = cudaEventRecord(ev[3 + 2 * i], st)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(c->io_down, ev[3 + 2 * i], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync((char *)out + (size_t)b * n * row_q, dout, nb * row_q, cudaMemcpyDeviceToHost,
                                 c->io_down)) != cudaSuccess)
            return cuda_fail(e, "host-call download");
    }
    if ((e = cudaEventRecord(ev[1], c->io_down)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, ev[1], 0)) != cudaSuccess)
        return cuda_fail(e, "host-call completion");
    return GQA_OK;
}

int kv_append(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t n, const int32_t *counts,
              const void *k_new, const void *v_new, void *stream)
{
    const int rc = kv_append_impl(c, B, seq_ids, n, counts, k_new, v_new, stream);
    if (rc == GQA_OK)
        release_windows(c, B, seq_ids);
    return rc;
}

// Decode of B queries described by sds (row = block-table row, past = L - 1)
// through the tables and stride of pv: the kernel choice, its work plan and
// its launch.  The caller has validated everything and uploaded the tables.
static int decode_launch(gqa_cache *c, const PoolView &pv, const std::vector<SeqDesc> &sds, int32_t H_q,
                         const void *q, void *out, cudaStream_t st)
{
    const int B = (int)sds.size();
    const int32_t H_kv = c->desc.num_kv_heads;
    const int G = H_q / H_kv;
    int64_t total = 0;
    for (int b = 0; b < B; ++b)
        total += sds[b].past + 1 - decode_first_token(sds[b].past + 1, c->desc.window);
    int32_t max_len = 1;
    for (int b = 0; b < B; ++b)
        max_len = std::max(max_len, sds[b].past + 1);
    Stage stg(c->h_stage);
    const size_t o_sds = stg.add(sds.data(), sds.size());
    int rc;
    const int cs = decode_cluster_for(c, G, B, max_len, q);
    if (cs < 0)
        return fail(GQA_EINVAL, "%s", kClusterNeeds);
    if (cs > 0) {
        // Small batches pass their descriptors in the launch parameters: no
        // upload precedes the kernel.
        ClusterDecodeLaunch a;
        if (B <= decode_cluster_inline()) {
            a.host_seqs = sds.data();
        } else {
            if ((rc = upload_stage(c, st)) != GQA_OK)
                return rc;
            a.seqs = (const SeqDesc *)(c->d_stage + o_sds);
        }
        a.B = B;
        a.H_q = H_q;
        a.cluster = cs;
        a.q = q;
        a.out = out;
        return run_kernel(c, GQA_KERNEL_DECODE_CLUSTER, st, "clustered decode kernel",
                          [&](cudaEvent_t ev) { return launch_decode_cluster(pv, a, st, ev); });
    }
    if ((rc = decode_uses_tc(c, G)) < 0)
        return fail(GQA_EINVAL, "the tensor-core decode kernel needs a bf16 cache with d_h = 128, post-position keys and H_q/H_kv <= 128");
    if (rc == 1) {
        // The prefill kernel at one query row per sequence, each sequence's
        // key tiles split across SMs and merged in the kernel.
        TcPlan plan;
        plan_tc(c, sds, G, plan);
        const size_t o_items = stg.add(plan.items.data(), plan.items.size());
        const size_t o_start = stg.add(plan.item_start.data(), plan.item_start.size());
        TcSplitWs ws;
        if ((rc = tc_workspace(c, plan, ws)) != GQA_OK)
            return rc;
        const TcHostDesc hd = tc_host(sds, plan);
        const bool inl = tc_inline_ok(c, hd);      // descriptors in the launch parameters: no copy
        if (!inl && (rc = upload_stage(c, st)) != GQA_OK)
            return rc;
        return run_kernel(c, GQA_KERNEL_PREFILL_TC, st, "tensor-core decode kernel", [&](cudaEvent_t ev) {
            return launch_prefill_tc(pv, (const SeqDesc *)(c->d_stage + o_sds),
                                     (const TcItem *)(c->d_stage + o_items),
                                     (const int32_t *)(c->d_stage + o_start), plan.grid, B, 1, H_q, q, out, ws, st, ev,
                                     nullptr, nullptr, nullptr, nullptr, nullptr, inl ? &hd : nullptr);
        });
    }
    if ((c->desc.dtype == GQA_DTYPE_BF16 || c->desc.dtype == GQA_DTYPE_FP8_E4M3) && c->desc.head_dim == 128 &&
        decode_split_supported(G)) {
        // Chunk: a multiple of the page size, large enough to amortise the
        // partials, small enough for several CTAs per SM.
        int64_t target = total * H_kv / (int64_t)std::max(1, c->num_sms * 4);
        int chunk = (int)std::min<int64_t>(512, std::max<int64_t>(128, (target + 127) / 128 * 128));
        std::vector<DecodeItem> items;
        std::vector<int32_t> start(B + 1, 0);
        for (int b = 0; b < B; ++b) {
            const int32_t L = sds[b].past + 1;
            const int32_t ns = (L - decode_first_token(L, c->desc.window) + chunk - 1) / chunk;
            start[b] = (int32_t)items.size();
            for (int32_t s = 0; s < ns; ++s)
                items.push_back(DecodeItem{b, s});
        }
        start[B] = (int32_t)items.size();
        const size_t o_items = stg.add(items.data(), items.size());
        const size_t o_start = stg.add(start.data(), start.size());
        const size_t n_part = items.size() * (size_t)H_kv * G;
        if ((rc = ensure_ws(c, n_part * 128 + n_part * 2)) != GQA_OK)
            return rc;
        if ((rc = ensure_cnt(c, (size_t)B * H_kv)) != GQA_OK)
            return rc;
        if ((rc = upload_stage(c, st)) != GQA_OK)
            return rc;
        DecodeLaunch a;
        a.seqs = (const SeqDesc *)(c->d_stage + o_sds);
        a.items = (const DecodeItem *)(c->d_stage + o_items);
        a.item_start = (const int32_t *)(c->d_stage + o_start);
        a.n_items = (int)items.size();
        a.chunk = chunk;
        a.H_q = H_q;
        a.q = q;
        a.ws_o = c->d_ws;
        a.ws_ml = c->d_ws + n_part * 128;
        a.counters = c->d_cnt;
        a.out = out;
        return run_kernel(c, GQA_KERNEL_DECODE_SPLIT, st, "decode kernel",
                          [&](cudaEvent_t ev) {
                              rec(ev, st);
                              return launch_decode_split(pv, a, st);
                          });
    }
    if ((rc = upload_stage(c, st)) != GQA_OK)
        return rc;
    return run_kernel(c, GQA_KERNEL_ATTN_SIMT, st, "attention kernel", [&](cudaEvent_t ev) {
        rec(ev, st);
        return launch_attn_simt(pv, c->desc.dtype, (const SeqDesc *)(c->d_stage + o_sds), B, 1, H_q, q, out, st);
    });
}

int attn_decode(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t H_q, const void *q, void *out,
                void *stream)
{
    if (!c || !seq_ids)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || H_q < 1)
        return fail(GQA_EINVAL, "B and H_q must be >= 1");
    const int32_t H_kv = c->desc.num_kv_heads;
    if (H_q % H_kv != 0)
        return fail(GQA_EINVAL, "H_kv = %d does not divide H_q = %d", H_kv, H_q);
    if (!c->meta_only && (!q || !out))
        return fail(GQA_EINVAL, "NULL tensor pointer");
    std::vector<SeqDesc> sds(B);
    for (int b = 0; b < B; ++b) {
        const int32_t s = seq_ids[b];
        if (!live(c, s))
            return fail(GQA_EINVAL, "batch entry %d: sequence %d is not live", b, s);
        const int32_t L = c->seqs[s].len;
        if (L < 1)
            return fail(GQA_EMASK, "sequence %d is empty: the decode query has no visible key", s);
        sds[b] = SeqDesc{s, L - 1, 1, 0};
    }
    int rc;
    if (c->meta_only)
        return GQA_OK;
    if ((rc = check_device(c)) != GQA_OK)
        return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if ((rc = upload_tables(c, st)) != GQA_OK)
        return rc;
    return decode_launch(c, c->view(), sds, H_q, q, out, st);
}

int attn_decode_tables(gqa_cache *c, int32_t B, const int32_t *block_table_dev, int32_t stride,
                       const int32_t *lengths, int32_t H_q, const void *q, void *out, void *stream)
{
    if (!c || !lengths)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || H_q < 1 || stride < 1)
        return fail(GQA_EINVAL, "B, H_q and stride must be >= 1");
    const int32_t H_kv = c->desc.num_kv_heads;
    if (H_q % H_kv != 0)
        return fail(GQA_EINVAL, "H_kv = %d does not divide H_q = %d", H_kv, H_q);
    if (c->meta_only)
        return fail(GQA_EINVAL, "attn_decode_tables needs a cache with a device pool");
    if (!block_table_dev || !q || !out)
        return fail(GQA_EINVAL, "NULL tensor pointer");
    if (c->desc.rope == 1 && (int64_t)stride > c->desc.max_pages_per_seq)
        return fail(GQA_ERANGE, "stride %d exceeds the rotary table's %d pages", stride, c->desc.max_pages_per_seq);
    std::vector<SeqDesc> sds(B);
    for (int b = 0; b < B; ++b) {
        const int32_t L = lengths[b];
        if (L < 1)
            return fail(GQA_EMASK, "batch entry %d: length %d leaves the decode query without a visible key", b, L);
        if ((int64_t)L > (int64_t)stride * kPageTokens)
            return fail(GQA_ERANGE, "batch entry %d: length %d exceeds the table row's %d pages", b, L, stride);
        sds[b] = SeqDesc{b, L - 1, 1, 0};
    }
    int rc = check_device(c);
    if (rc != GQA_OK)
        return rc;
    PoolView pv = c->view();
    pv.tables = block_table_dev;
    pv.stride = stride;
    return decode_launch(c, pv, sds, H_q, q, out, (cudaStream_t)stream);
}

int attn_decode_append(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t H_q, const void *q,
                       const void *k_new, const void *v_new, void *out, void *stream)
{
    if (!c || !seq_ids)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || H_q < 1)
        return fail(GQA_EINVAL, "B and H_q must be >= 1");
    const int32_t H_kv = c->desc.num_kv_heads;
    if (H_q % H_kv != 0)
        return fail(GQA_EINVAL, "H_kv = %d does not divide H_q = %d", H_kv, H_q);
    if (!c->meta_only && (!q || !k_new || !v_new || !out))
        return fail(GQA_EINVAL, "NULL tensor pointer");
    const int G = H_q / H_kv;
    const int use_tc = c->meta_only ? 0 : decode_uses_tc(c, G);
    if (use_tc < 0)
        return fail(GQA_EINVAL, "the tensor-core decode kernel needs a bf16 cache with d_h = 128, post-position keys and H_q/H_kv <= 128");
    int cs = 0;
    if (!c->meta_only) {
        // The clustered kernel's choice needs the lengths: unknown sequences
        // are reported by the write checks below.
        int32_t max_len = 1;
        bool known = true;
        for (int b = 0; b < B && known; ++b) {
            known = live(c, seq_ids[b]);
            if (known)
                max_len = std::max(max_len, c->seqs[seq_ids[b]].len + 1);
        }
        // An FP8 cache's write quantises in its own kernel: write, then decode.
        if (known && c->desc.dtype != GQA_DTYPE_FP8_E4M3 &&
            (cs = decode_cluster_for(c, G, B, max_len, q, k_new, v_new)) < 0)
            return fail(GQA_EINVAL, "%s", kClusterNeeds);
    }
    if (cs == 0 && (!use_tc || c->desc.dtype == GQA_DTYPE_FP8_E4M3)) {
        // CUDA-core kernels (and the quantised cache, whose write rounds in
        // its own kernel): the write, then the decode.
        int rc = kv_append(c, B, seq_ids, 1, nullptr, k_new, v_new, stream);
        return rc != GQA_OK ? rc : attn_decode(c, B, seq_ids, H_q, q, out, stream);
    }
    std::vector<WriteReq> req(B);
    for (int b = 0; b < B; ++b)
        req[b] = WriteReq{seq_ids[b], 1};
    int rc = check_write(c, req.data(), B);
    if (rc != GQA_OK)
        return rc;
    if ((rc = check_device(c)) != GQA_OK)
        return rc;
    std::vector<SeqDesc> sds;                 // past = the length before this call, count = 1
    std::vector<CowDesc> cows;
    commit_write(c, req.data(), B, sds, cows);
    cudaStream_t st = (cudaStream_t)stream;
    if ((rc = upload_tables(c, st)) != GQA_OK)
        return rc;
    const PoolView pv = c->view();
    if (cs > 0) {
        // Clustered decode: the CTA that reads the new position's page
        // writes the row.
        Stage stg(c->h_stage);
        const size_t o_sds = stg.add(sds.data(), sds.size());
        const size_t o_cow = stg.add(cows.data(), cows.size());
        const bool inl = B <= decode_cluster_inline();
        if ((!inl || !cows.empty()) && (rc = upload_stage(c, st)) != GQA_OK)
            return rc;
        if (!cows.empty() &&
            (rc = run_kernel(c, GQA_KERNEL_COW_COPY, st, "copy-on-write kernel", [&](cudaEvent_t ev) {
                 rec(ev, st);
                 return launch_cow_copy(pv, c->esize, (const CowDesc *)(c->d_stage + o_cow), (int)cows.size(), st);
             })) != GQA_OK)
            return rc;
        ClusterDecodeLaunch a;
        if (inl)
            a.host_seqs = sds.data();
        else
            a.seqs = (const SeqDesc *)(c->d_stage + o_sds);
        a.B = B;
        a.H_q = H_q;
        a.cluster = cs;
        a.q = q;
        a.out = out;
        a.app_k = k_new;
        a.app_v = v_new;
        rc = run_kernel(c, GQA_KERNEL_DECODE_CLUSTER, st, "clustered decode kernel",
                        [&](cudaEvent_t ev) { return launch_decode_cluster(pv, a, st, ev); });
        if (rc == GQA_OK)
            release_windows(c, B, seq_ids);
        return rc;
    }
    TcPlan plan;
    plan_tc(c, sds, G, plan);
    Stage stg(c->h_stage);
    const size_t o_sds = stg.add(sds.data(), sds.size());
    const size_t o_cow = stg.add(cows.data(), cows.size());
    const size_t o_items = stg.add(plan.items.data(), plan.items.size());
    const size_t o_start = stg.add(plan.item_start.data(), plan.item_start.size());
    TcSplitWs ws;
    if ((rc = tc_workspace(c, plan, ws)) != GQA_OK)
        return rc;
    const TcHostDesc hd = tc_host(sds, plan);
    const bool inl = cows.empty() && tc_inline_ok(c, hd);   // descriptors in the launch parameters: no copy
    if (!inl && (rc = upload_stage(c, st)) != GQA_OK)
        return rc;
    if (!cows.empty() &&
        (rc = run_kernel(c, GQA_KERNEL_COW_COPY, st, "copy-on-write kernel", [&](cudaEvent_t ev) {
             rec(ev, st);
             return launch_cow_copy(pv, c->esize, (const CowDesc *)(c->d_stage + o_cow), (int)cows.size(), st);
         })) != GQA_OK)
        return rc;
    rc = run_kernel(c, GQA_KERNEL_PREFILL_TC, st, "tensor-core decode kernel", [&](cudaEvent_t ev) {
        return launch_prefill_tc(pv, (const SeqDesc *)(c->d_stage + o_sds), (const TcItem *)(c->d_stage + o_items),
                                 (const int32_t *)(c->d_stage + o_start), plan.grid, B, 1, H_q, q, out, ws, st, ev,
                                 k_new, v_new, nullptr, nullptr, nullptr, inl ? &hd : nullptr);
    });
    if (rc == GQA_OK)
        release_windows(c, B, seq_ids);
    return rc;
}

int attn_decode_append_host(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t H_q, const void *q,
                            const void *k_new, const void *v_new, void *out, void *stream)
{
    // The checks of attn_decode_append first, so a rejected call queues and
    // changes nothing.
    if (!c || !seq_ids)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || H_q < 1)
        return fail(GQA_EINVAL, "B and H_q must be >= 1");
    const int32_t H_kv = c->desc.num_kv_heads;
    if (H_q % H_kv != 0)
        return fail(GQA_EINVAL, "H_kv = %d does not divide H_q = %d", H_kv, H_q);
    if (c->meta_only)
        return attn_decode_append(c, B, seq_ids, H_q, nullptr, nullptr, nullptr, nullptr, stream);
    if (!q || !k_new || !v_new || !out)
        return fail(GQA_EINVAL, "NULL buffer");
    if (decode_uses_tc(c, H_q / H_kv) < 0)
        return fail(GQA_EINVAL, "the tensor-core decode kernel needs a bf16 cache with d_h = 128, post-position keys "
                                "and H_q/H_kv <= 128");
    std::vector<WriteReq> req(B);
    for (int b = 0; b < B; ++b)
        req[b] = WriteReq{seq_ids[b], 1};
    int rc = check_write(c, req.data(), B);
    if (rc != GQA_OK || (rc = check_device(c)) != GQA_OK)
        return rc;
    const size_t es = (size_t)c->io_esize, d = (size_t)c->desc.head_dim;
    const size_t bq = (size_t)B * H_q * d * es, bkv = (size_t)B * H_kv * d * es;
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    if ((rc = ensure_io(c, 2 * al(bq) + 2 * al(bkv), 2)) != GQA_OK)
        return rc;
    cudaStream_t st = (cudaStream_t)stream;
    char *dq = c->d_io, *dk = dq + al(bq), *dv = dk + al(bkv), *dout = dv + al(bkv);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(dq, q, bq, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk, k_new, bkv, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv, v_new, bkv, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return cuda_fail(e, "host-call upload");
    if ((rc = attn_decode_append(c, B, seq_ids, H_q, dq, dk, dv, dout, stream)) != GQA_OK)
        return rc;
    if ((e = cudaMemcpyAsync(out, dout, bq, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e, "host-call download");
    return GQA_OK;
}

int gqa_selftest_bounded_wait(gqa_cache *c, int64_t limit_ns, void *stream)
{
    if (!c)
        return fail(GQA_EINVAL, "NULL cache");
    if (limit_ns < 1 || limit_ns > 10000000000ll)
        return fail(GQA_ERANGE, "limit_ns %lld outside 1..10^10", (long long)limit_ns);
    if (c->meta_only)
        return fail(GQA_EINVAL, "the self-test needs a cache with a device pool");
    int rc = check_device(c);
    if (rc != GQA_OK)
        return rc;
    const cudaError_t e = launch_wait_probe(c->d_err, (uint64_t)limit_ns, (cudaStream_t)stream);
    return e == cudaSuccess ? GQA_OK : cuda_fail(e, "wait probe");
}

int gqa_set_decode_kernel(gqa_cache *c, int32_t kernel)
{
    if (!c)
        return fail(GQA_EINVAL, "NULL cache");
    if (kernel != GQA_DECODE_AUTO && kernel != GQA_DECODE_TENSOR_CORE && kernel != GQA_DECODE_CUDA_CORE &&
        kernel != GQA_DECODE_CLUSTER)
        return fail(GQA_EINVAL, "decode kernel %d is not GQA_DECODE_AUTO, _TENSOR_CORE, _CUDA_CORE or _CLUSTER",
                    kernel);
    if (kernel == GQA_DECODE_CLUSTER &&
        ((c->desc.dtype != GQA_DTYPE_BF16 && c->desc.dtype != GQA_DTYPE_FP8_E4M3) || c->desc.head_dim != 128 ||
         c->desc.rope != 0))
        return fail(GQA_EINVAL, "the clustered decode kernel needs a bf16 or FP8 E4M3 cache with d_h = 128 and "
                                "no rotary");
    if (kernel == GQA_DECODE_TENSOR_CORE &&
        ((c->desc.dtype != GQA_DTYPE_BF16 && c->desc.dtype != GQA_DTYPE_FP8_E4M3) || c->desc.head_dim != 128 ||
         c->desc.keys_post_position != 1))
        return fail(GQA_EINVAL, "the tensor-core decode kernel needs a bf16 or FP8 E4M3 cache with d_h = 128 and "
                                "post-position keys");
    c->decode_kernel = kernel;
    return GQA_OK;
}

int gqa_profile_enable(gqa_cache *c, int on)
{
    if (!c)
        return fail(GQA_EINVAL, "NULL cache");
    c->prof = on != 0 && !c->meta_only;
    return GQA_OK;
}

int gqa_profile_read(gqa_cache *c, int32_t kernel, int32_t *launches, double *total_ms)
{
    if (!c || !launches || !total_ms)
        return fail(GQA_EINVAL, "NULL argument");
    if (kernel < 0 || kernel >= GQA_KERNEL_COUNT)
        return fail(GQA_ERANGE, "kernel id %d outside 0..%d", kernel, GQA_KERNEL_COUNT - 1);
    *launches = c->launches[kernel];
    c->launches[kernel] = 0;
    double sum = 0.0;
    std::vector<gqa_cache::ProfRec> keep;
    for (const auto &r : c->prof_recs) {
        if (r.kernel != kernel) {
            keep.push_back(r);
            continue;
        }
        float ms = 0.0f;
        cudaError_t e = cudaEventSynchronize(r.end);
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms, r.start, r.end);
        if (e != cudaSuccess)
            return cuda_fail(e, "profile event");
        sum += ms;
        c->spare_events.push_back(r.start);
        c->spare_events.push_back(r.end);
    }
    c->prof_recs.swap(keep);
    *total_ms = sum;
    return GQA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode: the split-K partials and the per-call descriptors
// live in one file-scope device array instead of library-allocated memory.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GQA_STATIC_SCRATCH_BYTES];

constexpr size_t kStaticCntBytes = 64u << 10;       // merge counters; the rest holds partials
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
char *g_static_addr[kMaxDevices] = {};

// Device address of g_static_scratch on `dev` (which must be current).  In
// host code the array's name only stands for the symbol, so its address is
// looked up once per device and cached.
int static_scratch(int dev, char **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GQA_EINVAL, "device %d outside 0..%d", dev, kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(static decode scratch)");
        g_static_addr[dev] = (char *)p;
    }
    *out = g_static_addr[dev];
    return GQA_OK;
}

}  // namespace

extern "C" int attn_decode_static(gqa_cache *c, int32_t B, const int32_t *seq_ids, int32_t H_q, const void *q,
                                  void *out, void *stream)
{
    if (!c || !seq_ids)
        return fail(GQA_EINVAL, "NULL argument");
    if (B < 1 || H_q < 1)
        return fail(GQA_EINVAL, "B and H_q must be >= 1");
    const int32_t H_kv = c->desc.num_kv_heads;
    if (H_q % H_kv != 0)
        return fail(GQA_EINVAL, "H_kv = %d does not divide H_q = %d", H_kv, H_q);
    const int G = H_q / H_kv;
    const int use_tc = decode_uses_tc(c, G);
    if (use_tc < 0)
        return fail(GQA_EINVAL, "the tensor-core decode kernel needs a bf16 cache with d_h = 128, post-position keys "
                                "and H_q/H_kv <= 128");
    if (c->meta_only)
        return fail(GQA_EINVAL, "attn_decode_static needs a cache with a device pool");
    if (!q || !out)
        return fail(GQA_EINVAL, "NULL tensor pointer");
    std::vector<SeqDesc> sds(B);
    int64_t total = 0;
    int32_t max_len = 1;
    for (int b = 0; b < B; ++b) {
        const int32_t s = seq_ids[b];
        if (!live(c, s))
            return fail(GQA_EINVAL, "batch entry %d: sequence %d is not live", b, s);
        const int32_t L = c->seqs[s].len;
        if (L < 1)
            return fail(GQA_EMASK, "sequence %d is empty: the decode query has no visible key", s);
        sds[b] = SeqDesc{s, L - 1, 1, 0};
        total += L - decode_first_token(L, c->desc.window);
        max_len = std::max(max_len, L);
    }
    int rc = check_device(c);
    if (rc != GQA_OK)
        return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t part_bytes = GQA_STATIC_SCRATCH_BYTES - kStaticDescBytes - kStaticCntBytes;

    const int cs = decode_cluster_for(c, G, B, max_len, q);
    if (cs < 0)
        return fail(GQA_EINVAL, "%s", kClusterNeeds);
    if (cs > 0) {
        // The clustered kernel of attn_decode: no partials leave the
        // cluster, so at most the descriptors go to the static array (small
        // batches pass them in the launch parameters).
        std::vector<char> desc;
        Stage stg(desc);
        const size_t o_sds = stg.add(sds.data(), sds.size());
        if (desc.size() > kStaticDescBytes)
            return fail(GQA_ERANGE, "decode descriptors need %zu bytes; the static scratch reserves %zu",
                        desc.size(), kStaticDescBytes);
        const bool inl = B <= decode_cluster_inline();
        char *scratch = nullptr;
        if (!inl && (rc = static_scratch(c->device, &scratch)) != GQA_OK)
            return rc;
        if ((rc = upload_tables(c, st, true)) != GQA_OK ||
            (!inl && (rc = staged_copy(c, scratch, desc.data(), desc.size(), st)) != GQA_OK))
            return rc;
        ClusterDecodeLaunch a;
        if (inl)
            a.host_seqs = sds.data();
        else
            a.seqs = (const SeqDesc *)(scratch + o_sds);
        a.B = B;
        a.H_q = H_q;
        a.cluster = cs;
        a.q = q;
        a.out = out;
        const PoolView pv = c->view();
        return run_kernel(c, GQA_KERNEL_DECODE_CLUSTER, st, "clustered decode kernel (static scratch)",
                          [&](cudaEvent_t ev) { return launch_decode_cluster(pv, a, st, ev); });
    }
    if (!use_tc && ((c->desc.dtype != GQA_DTYPE_BF16 && c->desc.dtype != GQA_DTYPE_FP8_E4M3) ||
                    c->desc.head_dim != 128 || !decode_split_supported(G)))
        return fail(GQA_EINVAL, "attn_decode_static needs a bf16 or FP8 E4M3 cache with d_h = 128 (and H_q/H_kv <= "
                                "8 on the CUDA-core kernel)");

    if (use_tc) {
        // The plan of attn_decode (so the results are the same bits), with
        // its descriptors, merge counters and partials in the static array.
        TcPlan plan;
        plan_tc(c, sds, G, plan);
        std::vector<char> desc;
        Stage stg(desc);
        const size_t o_sds = stg.add(sds.data(), sds.size());
        const size_t o_items = stg.add(plan.items.data(), plan.items.size());
        const size_t o_start = stg.add(plan.item_start.data(), plan.item_start.size());
        const size_t rows = (size_t)plan.slots * plan.slot_rows;
        if (desc.size() > kStaticDescBytes)
            return fail(GQA_ERANGE, "decode descriptors need %zu bytes; the static scratch reserves %zu",
                        desc.size(), kStaticDescBytes);
        if ((size_t)plan.slots * sizeof(int32_t) > kStaticCntBytes)
            return fail(GQA_ERANGE, "%d merge counters exceed the static scratch's %zu", plan.slots,
                        kStaticCntBytes / sizeof(int32_t));
        if (rows * 130 * sizeof(float) > part_bytes)
            return fail(GQA_ERANGE, "decode partials need %zu bytes; the static scratch holds %zu",
                        rows * 130 * sizeof(float), part_bytes);
        char *scratch = nullptr;
        if ((rc = static_scratch(c->device, &scratch)) != GQA_OK)
            return rc;
        if ((rc = upload_tables(c, st, true)) != GQA_OK || (rc = staged_copy(c, scratch, desc.data(), desc.size(), st)) != GQA_OK)
            return rc;
        int32_t *counters = (int32_t *)(scratch + kStaticDescBytes);
        cudaError_t e;
        if (plan.slots > 0 && (e = cudaMemsetAsync(counters, 0, (size_t)plan.slots * sizeof(int32_t), st)) !=
                                  cudaSuccess)
            return cuda_fail(e, "counter clear (static scratch)");
        TcSplitWs ws;
        ws.o = (float *)(scratch + kStaticDescBytes + kStaticCntBytes);
        ws.ml = reinterpret_cast<float2 *>(ws.o + rows * 128);
        ws.counters = counters;
        ws.slot_rows = plan.slot_rows;
        ws.ranged = plan.ranged;
        const PoolView pv = c->view();
        return run_kernel(c, GQA_KERNEL_PREFILL_TC, st, "tensor-core decode kernel (static scratch)",
                          [&](cudaEvent_t ev) {
                              return launch_prefill_tc(pv, (const SeqDesc *)(scratch + o_sds),
                                                       (const TcItem *)(scratch + o_items),
                                                       (const int32_t *)(scratch + o_start), plan.grid, B, 1, H_q, q,
                                                       out, ws, st, ev);
                          });
    }

    // The chunk rule of attn_decode (the same work split, so the same bits);
    // a call whose partials do not fit the array is refused.
    if ((size_t)B * H_kv * sizeof(int32_t) > kStaticCntBytes)
        return fail(GQA_ERANGE, "B * H_kv = %lld merge counters exceed the static scratch's %zu",
                    (long long)B * H_kv, kStaticCntBytes / sizeof(int32_t));
    const int64_t target = total * H_kv / (int64_t)std::max(1, c->num_sms * 4);
    const int chunk = (int)std::min<int64_t>(512, std::max<int64_t>(128, (target + 127) / 128 * 128));
    std::vector<DecodeItem> items;
    std::vector<int32_t> start(B + 1, 0);
    for (int b = 0; b < B; ++b) {
        const int32_t ns =
            (sds[b].past + 1 - decode_first_token(sds[b].past + 1, c->desc.window) + chunk - 1) / chunk;
        start[b] = (int32_t)items.size();
        for (int32_t s = 0; s < ns; ++s)
            items.push_back(DecodeItem{b, s});
    }
    start[B] = (int32_t)items.size();
    const size_t n_part = items.size() * (size_t)H_kv * G;
    if (n_part * 130 * sizeof(float) > part_bytes)
        return fail(GQA_ERANGE, "decode partials need %zu bytes; the static scratch holds %zu",
                    n_part * 130 * sizeof(float), part_bytes);
    std::vector<char> desc;
    Stage stg(desc);
    const size_t o_sds = stg.add(sds.data(), sds.size());
    const size_t o_items = stg.add(items.data(), items.size());
    const size_t o_start = stg.add(start.data(), start.size());
    if (desc.size() > kStaticDescBytes)
        return fail(GQA_ERANGE, "decode descriptors need %zu bytes; the static scratch reserves %zu",
                    desc.size(), kStaticDescBytes);

    char *scratch = nullptr;
    if ((rc = static_scratch(c->device, &scratch)) != GQA_OK)
        return rc;
    if ((rc = upload_tables(c, st, true)) != GQA_OK || (rc = staged_copy(c, scratch, desc.data(), desc.size(), st)) != GQA_OK)
        return rc;
    // The merge counters must start at zero: clear the ones this call uses.
    int32_t *counters = (int32_t *)(scratch + kStaticDescBytes);
    cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)B * H_kv * sizeof(int32_t), st);
    if (e != cudaSuccess)
        return cuda_fail(e, "counter clear (static scratch)");
    DecodeLaunch a;
    a.seqs = (const SeqDesc *)(scratch + o_sds);
    a.items = (const DecodeItem *)(scratch + o_items);
    a.item_start = (const int32_t *)(scratch + o_start);
    a.n_items = (int)items.size();
    a.chunk = chunk;
    a.H_q = H_q;
    a.q = q;
    a.ws_o = (float *)(scratch + kStaticDescBytes + kStaticCntBytes);
    a.ws_ml = a.ws_o + n_part * 128;
    a.counters = counters;
    a.out = out;
    const PoolView pv = c->view();
    return run_kernel(c, GQA_KERNEL_DECODE_SPLIT, st, "decode kernel (static scratch)", [&](cudaEvent_t ev) {
        rec(ev, st);
        return launch_decode_split(pv, a, st);
    });
}

extern "C" {

int gqa_cache_check(gqa_cache *c, void *stream, int32_t *flags_out)
{
    if (!c || !flags_out)
        return fail(GQA_EINVAL, "NULL argument");
    *flags_out = 0;
    if (c->meta_only)
        return GQA_OK;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(st);
    int32_t h = 0;
    if (e == cudaSuccess)
        e = cudaMemcpy(&h, c->d_err, sizeof(h), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && h != 0)
        e = cudaMemset(c->d_err, 0, sizeof(int32_t));
    if (e != cudaSuccess)
        return cuda_fail(e, "error-word read");
    *flags_out = h;
    if (h)
        return fail(GQA_EDEVICE, "device error word 0x%x", h);
    return GQA_OK;
}

}  // extern "C"
