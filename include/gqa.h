/*
 * gqa.h -- C ABI of libgqa: causal grouped-query attention, prefill and
 * decode, over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *  [P1] "第二章 Prefill：整层状态演化与 KV 建立" (glenzli.com, vol. 2, ch. 2):
 *       2.1 prefill interface and preconditions 2.1; 2.2 mask M and the rule
 *       for invalid query rows; 2.3 attention equations (g(h), S, A, O);
 *       2.5 cache contract, layout_metadata and cache invariants 2.2;
 *       2.6 prefill pseudocode (write valid positions, then attend);
 *       2.9 prefix reuse conditions; 2.11 failure table.
 *  [P2] "模型执行：从 token 到 Prefill 与 Decode" (blog.mlxb.cc): prefill vs
 *       decode shapes; decode reads the old cache plus its own new entry.
 *  [P3] "KV Cache 与 Prefill/Decode 推理路径" (wiki.maxwellmou.com, unit 10):
 *       edit at token m (keep the KV before m, truncate, re-prefill the
 *       suffix); GQA head axis; causal tile skipping; PagedAttention block
 *       tables and the free pool; incremental prefill mask; prefix sharing
 *       with reference counts.
 *
 * Conventions for every call
 *  - Every function returns GQA_OK (0) or a negative GQA_E* status.  The
 *    message of the last failure on the calling thread is gqa_last_error().
 *  - Preconditions are checked on the host before anything is queued on the
 *    GPU.  A call that fails a check changes neither the cache nor any output
 *    ([P1] preconditions 2.1: fail before the first layer runs).
 *  - "device" pointers are CUDA device addresses on the current device;
 *    "host" pointers are ordinary host memory, read before the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Launching calls are asynchronous and stream-ordered; they do
 *    not synchronise except to report a CUDA error.  All calls on one cache
 *    must be issued on one stream, or ordered by the caller.
 *  - Tensors are dense, row-major, in the cache's element type (bf16 or
 *    fp32; bf16 for a GQA_DTYPE_FP8_E4M3 cache, whose pages hold quantised
 *    K/V).  Shapes below list the outermost dimension first.
 *  - Token-major layouts: q is [B, n, H_q, d_h] and k, v are
 *    [B, n, H_kv, d_h] -- a permuted view of [P1] 2.3's [B, H, n, d_h].
 *
 * Page pool layout, version 2 (device memory owned by the caller, described
 * by the cache): num_pages pages of page_tokens = 16 token slots.  A row of
 * R = d_h * element-size bytes is cut into C = ceil(R / 128) chunks of 128
 * bytes (the last one zero-padded when 128 does not divide R).  Page p holds,
 * for kv = 0 (K) and 1 (V) and each KV head h, a block of 16 * C * 128 bytes,
 * block number (p*2 + kv)*H_kv + h; within it, byte b of the row of slot s is
 * at byte
 *      ((s/8)*C + b/128)*1024 + (s%8)*128 + b%128,
 * i.e. the 16 slots form two groups of 8 and each group stores chunk 0 of its
 * 8 rows, then chunk 1, ...  (for bf16, d_h = 128 this puts each group of 8
 * tokens in the layout the tensor-core operands read, so one 4 KB copy moves
 * a page of one head).  Token t of a sequence lives in logical page t/16 at
 * slot t%16; a per-sequence block table maps logical pages to physical pages
 * ([P3] PagedAttention).
 *
 * Quantised cache (dtype GQA_DTYPE_FP8_E4M3; [P1] 2.5: the physical cache
 * may be quantised as long as the logical order is kept).  A row is d_h
 * bytes of FP8 E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; largest finite value 448) in the block layout above, plus one fp32
 * scale per row.  The scales follow the blocks in the same buffer: after
 * the num_pages * 2 * H_kv blocks, scale of (block, slot s) at float index
 * block*16 + s.  A row x (the bf16 values given) is stored as s = amax|x| /
 * 448 (fp32) and codes E4M3(x_i / s) (the quotient in fp32, rounded to
 * nearest-even, saturating at +-448); a row of zeros has s = 0 and zero
 * codes.  Attention reads the value fp32(decode(code) * s) (the tensor-core
 * kernel rounds it to bf16 for its operands).
 *
 * Allocation rules (deterministic; the tests restate them independently):
 *  - a free page is taken in the order `page_order` gives (identity when
 *    NULL): always the free page that comes first in that order;
 *  - pages carry reference counts; a page returns to the pool when its count
 *    reaches zero ([P3] prefix tree: shared blocks are reclaimed only after
 *    every request that uses them is done);
 *  - writing into a tail page that another sequence shares first copies its
 *    occupied slots to a fresh page (copy-on-write);
 *  - within one batched call, pages are taken sequence by sequence in batch
 *    order, and per sequence the copy-on-write page first, then new pages in
 *    logical order;
 *  - a new sequence gets the smallest unused id in [0, max_seqs).
 */
#ifndef GQA_H_
#define GQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define GQA_OK        0
#define GQA_EINVAL   -1  /* bad argument: NULL pointer, bad shape, unknown or duplicated sequence */
#define GQA_ERANGE   -2  /* a length, position, page id or capacity is out of range */
#define GQA_EMASK    -3  /* a valid query row would have no finite score ([P1] 2.3: reject at mask construction) */
#define GQA_ENOMEM   -4  /* the page pool or the sequence-id space is exhausted */
#define GQA_ELAYOUT  -5  /* layout_metadata incompatible ([P1] invariant 2.2 item 5; 2.9 item 4) */
#define GQA_ECUDA    -6  /* a CUDA runtime call failed */
#define GQA_EDEVICE  -7  /* a kernel reported an error word (see gqa_cache_check) */

/* Device error-word bits reported by gqa_cache_check. */
#define GQA_DEVERR_PAGE_ID   1  /* a block-table entry was >= num_pages (access skipped) */
#define GQA_DEVERR_TIMEOUT   2  /* a bounded wait inside a kernel gave up */
#define GQA_DEVERR_SHAPE     4  /* a kernel saw a shape it does not support (work skipped) */

#define GQA_DTYPE_BF16     1
#define GQA_DTYPE_F32      2
#define GQA_DTYPE_FP8_E4M3 3  /* quantised pages; q, k, v and out in bf16 (layout above) */

#define GQA_PAGE_TOKENS    16
#define GQA_LAYOUT_VERSION 2

/* Cache description ([P1] 2.5: cache_config fixes the KV layout and the
 * position convention). */
typedef struct {
    int32_t dtype;               /* GQA_DTYPE_BF16, GQA_DTYPE_F32 or GQA_DTYPE_FP8_E4M3     */
    int32_t num_kv_heads;        /* H_kv >= 1                                              */
    int32_t head_dim;            /* d_h, 1..256 (bf16 d_h = 128 takes the tensor-core path;
                                    FP8_E4M3 needs a multiple of 32)                        */
    int32_t page_tokens;         /* must be GQA_PAGE_TOKENS                                 */
    int32_t num_pages;           /* pages in the pool, >= 1                                 */
    int32_t max_seqs;            /* sequence ids are 0..max_seqs-1                          */
    int32_t max_pages_per_seq;   /* block-table capacity of one sequence                    */
    int32_t keys_post_position;  /* [P1] 2.5: whether the cached keys were taken after (1) or
                                    before (0) the position transform.  1: keys are stored as
                                    attention uses them (rotated when written if rope = 1).
                                    0 (only with rope = 1): keys are stored exactly as given
                                    and every attention kernel rotates each key by its
                                    position as it reads it, so the stored keys do not depend
                                    on where they sit ([P3] prefix caching).  A bf16 prefill
                                    with d_h = 128 on such a cache first copies every page the
                                    call reads, keys rotated, to library-owned scratch (one
                                    rotation per page per call) and runs the tensor-core kernel
                                    on the copy; decode runs on the split-K CUDA-core kernel,
                                    which rotates each key in registers as it reads it.       */
    int32_t layout_version;      /* must be GQA_LAYOUT_VERSION                              */
    const int32_t *page_order;   /* host, optional: permutation of 0..num_pages-1 giving the
                                    order in which free pages are handed out (NULL = identity).
                                    Copied; the caller keeps ownership.                      */
    int32_t rope;                /* position mechanism applied by the library ([P1] 2.3: Q~, K~
                                    are Q, K after it; [P3]: RoPE rotates Q/K by the position
                                    ID): 0 = none, q/k arrive already transformed; 1 = rotary:
                                    dimension pairs (e, e + d_h/2), e < d_h/2, rotated
                                    counter-clockwise by pos * rope_base^(-2e/d_h).  Keys are
                                    rotated when written (keys_post_position = 1) or when read
                                    (keys_post_position = 0), queries inside the attention
                                    kernels.                                                  */
    float rope_base;             /* rope = 1: the frequency base, > 1 (e.g. 10000)           */
    int32_t window;              /* sliding window W ([P3] sliding window and ring cache): 0 =
                                    none; W >= 1: the query at position p sees keys
                                    max(0, p - W + 1) .. p (its own position included).  K/V
                                    outside every future window is released: a write that
                                    brings a sequence to length L returns to the pool each page
                                    whose 16 positions all lie before L - W, and its block-table
                                    entry becomes -1.  A sequence then holds at most
                                    ceil(W / 16) + 1 pages.                                    */
} gqa_cache_desc;

/* layout_metadata of [P1] 2.5 / invariant 2.2 item 5. */
typedef struct {
    int32_t keys_post_position;
    int32_t dtype;
    int32_t page_tokens;
    int32_t layout_version;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t rope;                /* the cache's position mechanism (keys were rotated with it) */
    float rope_base;
    int32_t window;              /* sliding window (pages outside it were released)           */
} gqa_layout_metadata;

typedef struct gqa_cache gqa_cache;

/* Bytes the page pool of `desc` occupies: num_pages * 2 * H_kv * 16 * C *
 * 128 with C = ceil(d_h * element size / 128) (layout version 2 above;
 * element size 1 for FP8_E4M3, whose pool adds num_pages * 2 * H_kv * 16
 * fp32 scales).  Returns 0 for an invalid description. */
size_t gqa_pool_bytes(const gqa_cache_desc *desc);

/* Create a cache over a caller-owned device pool (`pool_dev`, at least
 * gqa_pool_bytes(desc) bytes, 256-byte aligned).  The library allocates its
 * own small device metadata (block tables, lengths, per-call descriptors, an
 * error word) with cudaMalloc on the current device and clears the pool
 * (cudaMemset, synchronous) so that every slot holds a finite value.
 *
 * pool_dev == NULL makes a metadata-only cache: no device memory is touched
 * or allocated; launching calls validate their arguments and update block
 * tables and lengths exactly as they would on a device cache, but queue no
 * GPU work and write no outputs.  It exists so the host-side allocator can be
 * exercised without a GPU.
 * With rope = 1 the library also allocates a cos/sin table of
 * max_pages_per_seq * 16 positions x d_h/2 frequencies (fp32, computed in
 * fp64 on the host).  It also reserves 4 MiB of page-locked host memory
 * (cudaHostAlloc) through which attn_decode_static uploads its descriptors
 * and block tables.
 * Errors: GQA_EINVAL (bad description, pool too small, misaligned; rope not
 *         0/1, or rope = 1 with an odd d_h or rope_base <= 1; FP8_E4M3 with
 *         d_h not a multiple of 32 or with rope = 1),
 *         GQA_ELAYOUT (keys_post_position not 1, or 0 without rope = 1; unknown
 *         layout_version),
 *         GQA_ECUDA. */
int gqa_cache_create(const gqa_cache_desc *desc, void *pool_dev, size_t pool_bytes,
                     gqa_cache **out);

/* Release the cache's host and device metadata (synchronises the device).
 * The pool stays the caller's.  NULL is accepted. */
int gqa_cache_destroy(gqa_cache *cache);

/* The cache's layout_metadata ([P1] 2.5). */
int gqa_cache_layout(const gqa_cache *cache, gqa_layout_metadata *out);

/* GQA_OK if a cache written under `a` may be read under `b` (every field
 * equal), else GQA_ELAYOUT ([P1] 2.9 item 4; invariant 2.2 item 5). */
int gqa_layout_compatible(const gqa_layout_metadata *a, const gqa_layout_metadata *b);

/* ---- sequences (host metadata only; no GPU work) ------------------------ */

/* New empty sequence; smallest unused id.  GQA_ENOMEM if none is free. */
int gqa_seq_create(gqa_cache *cache, int32_t *seq_out);

/* New sequence that shares the first `prefix_len` positions of `src`
 * ([P1] 2.9 prefix reuse; [P3] prefix sharing): it references src's first
 * ceil(prefix_len/16) pages (reference counts + 1) and has length
 * prefix_len.  GQA_ERANGE unless 0 <= prefix_len <= length(src), and, with
 * a sliding window W, unless prefix_len = 0 or positions prefix_len - W ..
 * prefix_len - 1 are still held (released entries are shared as -1). */
int gqa_seq_fork(gqa_cache *cache, int32_t src, int32_t prefix_len, int32_t *seq_out);

/* Drop every page reference of `seq` and release its id. */
int gqa_seq_free(gqa_cache *cache, int32_t seq);

/* Current logical length of `seq`. */
int gqa_seq_length(const gqa_cache *cache, int32_t seq, int32_t *len_out);

/* Copy `seq`'s block table (physical page of each logical page) into host
 * `out` (capacity `cap` entries); *count_out = number of pages in the table.
 * Entries released by a sliding window are -1.
 * GQA_ERANGE if cap is too small (nothing copied). */
int gqa_seq_block_table(const gqa_cache *cache, int32_t seq, int32_t *out, int32_t cap,
                        int32_t *count_out);

/* Number of free pages and the reference count of page `page`. */
int gqa_free_pages(const gqa_cache *cache, int32_t *out);
int gqa_page_refcount(const gqa_cache *cache, int32_t page, int32_t *out);

/* ---- the hot path --------------------------------------------------------- */

/* Causal GQA prefill, incremental when the sequences already hold tokens
 * ([P1] 2.2-2.3, 2.6; [P3] incremental prefill).
 *
 * For each batch entry b, with sequence s = seq_ids[b] of current length P_b
 * and n_b = valid_lengths[b] valid (right-aligned padding) rows:
 *  1. the K/V rows i < n_b are written to the cache at positions P_b + i,
 *     bit for bit (with rope = 1 and post-position keys, K is rotated by
 *     position P_b + i first: each pair (x, y) becomes (x*c - y*s, x*s + y*c),
 *     every product, sum and difference rounded to fp32, then rounded to the
 *     cache type; c, s are the fp32 cos/sin of the table; pre-position keys
 *     are stored as given); padding rows are never written ([P1] 2.6;
 *     invariant 2.2 item 4);
 *  2. for every query head h and valid row i, with g(h) = floor(h*H_kv/H_q)
 *     ([P1] 2.3), the output is softmax over the finite scores
 *     <q[b,i,h], K[s, j, g(h)]> / sqrt(d_h), j = 0 .. P_b + i, applied to V
 *     (with rope = 1, q rotated by its position P_b + i, and pre-position
 *     keys rotated by theirs, in fp32, as they are read): the old prefix is
 *     fully visible and the new block is lower-triangular ([P3] incremental
 *     prefill);
 *  3. padding rows i >= n_b of `out` are written as zeros (they are
 *     discarded, [P1] 2.2);
 *  4. the sequence's length becomes P_b + n_b.
 *
 * Arguments
 *  seq_ids        host int32[B], distinct live sequences.
 *  n              padded rows per batch entry (>= 1).
 *  H_q            query heads; H_kv must divide it ([P1] 2.3).
 *  q              device [B, n, H_q, d_h]      (read)
 *  k, v           device [B, n, H_kv, d_h]     (read; post-position keys when
 *                 rope = 0, keys before the rotation when rope = 1)
 * With every entry starting on a page boundary (P_b a multiple of 16), n a
 * multiple of 8, a bf16 cache without rotation and d_h = 128, the cache
 * write is part of the attention kernel (one launch); otherwise a write
 * launch precedes it.  The results are the same bits either way.
 *  valid_lengths  host int32[B], 1 <= n_b <= n.
 *  positions      host int32[B, n] or NULL.  When given, positions[b, i]
 *                 must equal P_b + i for every valid row: positions continue
 *                 the cached sequence and never restart ([P1] 2.11, position
 *                 IDs restarting after reuse).  NULL means exactly that.
 *  out            device [B, n, H_q, d_h]      (written)
 * Errors: GQA_EINVAL (NULL pointer, shapes, H_kv does not divide H_q,
 *         duplicate or unknown sequence), GQA_EMASK (n_b < 1 or n_b > n:
 *         a row without a finite score), GQA_ERANGE (positions, sequence
 *         capacity), GQA_ENOMEM (pool exhausted), GQA_ECUDA. */
int attn_prefill(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t n, int32_t H_q,
                 const void *q, const void *k, const void *v,
                 const int32_t *valid_lengths, const int32_t *positions,
                 void *out, void *stream);

/* attn_prefill on HOST buffers: the same computation and cache effects,
 * with the host<->device transfers inside the call.
 *
 * The whole batch is checked first (every error of attn_prefill; nothing is
 * queued or changed when a check fails).  Then, largest n_b first, entry b's
 * valid rows of q, k, v (n_b of its n rows each) are copied to library-owned
 * device memory on the cache's upload stream, the entry runs as a one-entry
 * attn_prefill on `stream` once its rows are in, and its n_b valid output
 * rows are copied back on the cache's download stream while later entries
 * compute.  `stream` waits for the last download before the call's work
 * ends, so `out` is complete once `stream` is synchronised.
 *
 * Arguments as attn_prefill, except:
 *  q              host [B, n, H_q, d_h]   (read when the call's work runs)
 *  k, v           host [B, n, H_kv, d_h]  (read when the call's work runs)
 *  out            host [B, n, H_q, d_h]   (written); rows i >= n_b of an
 *                 entry are NOT written (only valid rows cross the link)
 * The host buffers must stay valid until `stream` has passed the call.
 * Page-locked (pinned) buffers let the copies overlap the attention of other
 * entries; pageable ones work, with copies the driver may serialise.
 * Calls on one cache must be ordered on one stream (the device copies of
 * the rows are reused by the next call).  The device memory for the rows
 * grows on demand (a growth frees the old block, which waits for the device).
 * Errors: those of attn_prefill; a GQA_ECUDA after some entries were queued
 * leaves those entries written (as a sequence of one-entry calls would). */
int attn_prefill_host(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t n, int32_t H_q,
                      const void *q, const void *k, const void *v,
                      const int32_t *valid_lengths, const int32_t *positions,
                      void *out, void *stream);

/* Append new K/V rows at each sequence's tail without attention ([P3]
 * decode: append the step's k_t, v_t after the old cache; [P1] 2.6 cache
 * write).  Row c < counts[b] of entry b goes to position P_b + c (with
 * rope = 1 its key is rotated by P_b + c as in attn_prefill step 1).
 *  seq_ids  host int32[B], distinct live sequences.
 *  n        rows per entry in k_new/v_new (1 for a decode step).
 *  counts   host int32[B] with 0 <= counts[b] <= n, or NULL (= n for all).
 *  k_new, v_new  device [B, n, H_kv, d_h].
 * Errors: GQA_EINVAL, GQA_ERANGE (capacity), GQA_ENOMEM, GQA_ECUDA. */
int kv_append(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t n,
              const int32_t *counts, const void *k_new, const void *v_new, void *stream);

/* Single-token decode ([P3] decode lesson: one query reads every cached key;
 * [P2]: old cache plus this step's own entry).  Query b sits at position
 * L_b - 1 of sequence seq_ids[b] (L_b = its current length, which includes
 * the entry appended for this step) and attends over all L_b cached tokens
 * through the sequence's block table:
 *      out[b, h, :] = sum_t softmax_t(<q[b,h], K[t, g(h)]>/sqrt(d_h)) V[t, g(h)]
 * (with rope = 1, q rotated by L_b - 1).
 *  seq_ids  host int32[B], live sequences of length >= 1 (repeats allowed).
 *  q        device [B, H_q, d_h];  out  device [B, H_q, d_h].
 * The kernel is chosen by gqa_set_decode_kernel.  Split-K partials and merge
 * counters live in library-owned device memory that grows with cudaMalloc on
 * first use of a larger shape.
 * Errors: GQA_EINVAL, GQA_EMASK (empty sequence), GQA_ECUDA. */
int attn_decode(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t H_q,
                const void *q, void *out, void *stream);

/* attn_decode_tables -- attn_decode over block tables the caller owns (the
 * spec call attn_decode(q, cache, block_table, lengths)): the cache
 * supplies the pool and its layout (dtype, window, rotation), the caller the
 * page mapping and the lengths, and no sequence state of the cache is read
 * or changed.  Query b sits at position lengths[b] - 1 and attends over
 * tokens 0 .. lengths[b] - 1, token t in physical page
 * block_table[b * stride + t / 16] at slot t % 16.
 *  block_table  device int32 [B][stride], page ids of this cache's pool (-1
 *               for pages a sliding window released; such pages are never
 *               read).  Read on `stream`.
 *  lengths      host int32[B], 1 <= lengths[b] <= stride * 16.
 *  q, out       device [B, H_q, d_h].
 * Page ids outside 0..num_pages-1 where a key is read are skipped and
 * reported as GQA_DEVERR_PAGE_ID by gqa_cache_check.  The kernel is the one
 * attn_decode would choose, with the same bits for the same tables.
 * Errors: GQA_EINVAL, GQA_EMASK (a length < 1), GQA_ERANGE (a length beyond
 * the row, or with rope = 1 a stride beyond max_pages_per_seq), GQA_ECUDA. */
int attn_decode_tables(gqa_cache *cache, int32_t B, const int32_t *block_table_dev, int32_t stride,
                       const int32_t *lengths, int32_t H_q, const void *q, void *out, void *stream);

/* attn_decode_append -- one decode step: kv_append of one token per
 * sequence, then attn_decode at that token ([P3] decode: the step's own key
 * and value join the cache and the query attends to the old cache plus
 * them; [P2] toy decoder).  For each b, k_new[b] and v_new[b] are written at
 * position L_b (the length before the call; rotated as in kv_append when
 * rope = 1), the length becomes L_b + 1, and out[b] is attn_decode's result
 * for the query at position L_b.  The cache and out hold the same bits as
 * kv_append(n = 1) followed by attn_decode.  On the tensor-core decode
 * kernel the write happens inside the attention kernel: the CTA that reads
 * a sequence's last page writes the row there first, so a step is one
 * launch (two when a shared tail page must first be copied).  Otherwise
 * the two calls run in turn.
 *  seq_ids  host int32[B], distinct live sequences.
 *  q        device [B, H_q, d_h];  k_new, v_new  device [B, H_kv, d_h];
 *  out      device [B, H_q, d_h].
 * Errors: those of kv_append and attn_decode. */
int attn_decode_append(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t H_q,
                       const void *q, const void *k_new, const void *v_new, void *out, void *stream);

/* attn_decode_append on HOST buffers: one decode step with the transfers
 * inside the call.  The checks of attn_decode_append come first (nothing is
 * queued or changed when one fails); then q, k_new and v_new are copied to
 * library-owned device memory on `stream`, the step runs as
 * attn_decode_append, and out is copied back on `stream`.  out is complete
 * once `stream` is synchronised; the host buffers must stay valid until
 * then.  Page-locked buffers make the copies asynchronous.
 *  q        host [B, H_q, d_h];  k_new, v_new  host [B, H_kv, d_h];
 *  out      host [B, H_q, d_h] (written).
 * Calls on one cache must be ordered on one stream (the device copies are
 * reused by the next call); the device memory grows on demand.
 * Errors: those of attn_decode_append. */
int attn_decode_append_host(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t H_q,
                            const void *q, const void *k_new, const void *v_new, void *out, void *stream);

/* attn_decode_static -- attn_decode that allocates no device memory.
 *
 * The pages define no counterpart to this call.  It is for callers that must
 * not allocate device memory while they decode.  Examples: a serving loop
 * that reserved all of its GPU memory at start-up; a host process whose
 * allocator belongs to another framework; a latency-bound step that cannot
 * afford the device-wide synchronisation of cudaFree.  attn_decode may hit
 * that synchronisation when its workspace grows.
 *
 * Arguments, results and errors are those of attn_decode, and so are the
 * kernel and its work split: the results are the same bits.  The cache must
 * be bf16 or FP8 E4M3 with d_h = 128 (and H_q / H_kv at most 8 on the
 * CUDA-core kernel); other shapes get GQA_EINVAL.
 * The split-K partials, the per-call descriptors and the merge counters live
 * in one static device array of GQA_STATIC_SCRATCH_BYTES.  The library reserves that array
 * on every GPU that loads it, until the process exits.  A call whose partials
 * or descriptors would not fit returns GQA_ERANGE with the bytes it needed
 * and queues nothing (the work split is never changed to make it fit).
 * No cudaMalloc, cudaFree or other allocating routine is called.  The
 * descriptors and the changed block-table entries are copied into one of
 * two page-locked host slots that the cache reserved when it was created,
 * and uploaded from there on `stream`.  Before reusing a slot, the call waits
 * on the host until the copies that last read it have finished, which
 * happens only when the host is two calls ahead of the GPU.
 * On each device, the first call looks up the array's device address
 * (cudaGetSymbolAddress).  Make that first call before any stream capture.
 * On the clustered decode kernel (GQA_DECODE_CLUSTER, the automatic choice
 * for small batches) partials never leave the cluster: only the descriptors
 * of a call with more than 16 entries go to the array (up to 16 travel in
 * the launch parameters), and no counters are used.
 * Every call shares the one array, and the array keeps the last call's
 * contents.  The merge counters must start at zero, so each call clears the
 * ones it uses (an asynchronous memset on `stream`); every other part is
 * written by the call before it is read.  Calls whose GPU work overlaps race
 * on the array: calls on different streams, or on different caches of one
 * device.  Order such calls yourself. */
#define GQA_STATIC_SCRATCH_BYTES (16u << 20)
int attn_decode_static(gqa_cache *cache, int32_t B, const int32_t *seq_ids, int32_t H_q,
                       const void *q, void *out, void *stream);

/* Decode kernel of attn_decode and attn_decode_static.
 *  GQA_DECODE_AUTO         (default) for a bf16 or FP8 E4M3 cache with
 *                          d_h = 128: the clustered kernel when it can serve
 *                          the call and there are at most half as many
 *                          (entry, KV head) pairs as SMs; else tensor-core
 *                          for bf16 and CUDA-core for FP8 (which decodes a
 *                          large batch faster there); CUDA-core for other
 *                          caches.
 *  GQA_DECODE_TENSOR_CORE  the prefill kernel with one query row per
 *                          sequence: every KV head's key tiles are read once
 *                          by TMA, a sequence's tiles are split into ranges
 *                          across SMs when there are too few sequences, and
 *                          the ranges' partial (m, l, O) are merged inside
 *                          the kernel by the CTA that finishes last.  Needs
 *                          bf16 or FP8 E4M3 and d_h = 128 (else GQA_EINVAL
 *                          here).  FP8 codes are dequantised into bf16
 *                          operands in shared memory (code times scale in
 *                          fp32, rounded to bf16).
 *  GQA_DECODE_CUDA_CORE    the split-K CUDA-core decode kernel (bf16 or FP8
 *                          E4M3, d_h = 128, H_q / H_kv <= 8), else the
 *                          generic CUDA-core kernel.
 *  GQA_DECODE_CLUSTER      the clustered decode kernel: each (entry, KV
 *                          head) is one thread-block cluster of up to 16
 *                          CTAs that split its pages (each page's K and V
 *                          read once by TMA, both products on mma.sync) and
 *                          merge their partial (m, l, O) through distributed
 *                          shared memory; no workspace.  FP8 E4M3 codes are
 *                          read as stored (f16 products, scales on the
 *                          scores and on P).  Needs a bf16 or FP8 E4M3 cache
 *                          with d_h = 128 and no rotary (else GQA_EINVAL
 *                          here), H_q / H_kv <= 16 and q (for the fused
 *                          append, bf16 only, also k_new and v_new) 16-byte
 *                          aligned (else GQA_EINVAL from the decode call).
 * All compute the same softmax; they differ in rounding order only.
 * Errors: GQA_EINVAL (unknown choice, or a kernel that cannot serve this
 * cache). */
#define GQA_DECODE_AUTO         0
#define GQA_DECODE_TENSOR_CORE  1
#define GQA_DECODE_CUDA_CORE    2
#define GQA_DECODE_CLUSTER      3
int gqa_set_decode_kernel(gqa_cache *cache, int32_t kernel);

/* Self-test of the failure path of the kernels' waits.  Queues one block
 * that waits, with the bounded wait the pipelines use, on a barrier phase
 * nothing completes; after limit_ns it gives up and sets GQA_DEVERR_TIMEOUT
 * in the cache's error word (read it with gqa_cache_check), as a timed-out
 * pipeline wait would.  Nothing faults or traps, and the context stays
 * usable.  Not part of the hot path.
 * Errors: GQA_EINVAL (no device pool), GQA_ERANGE (limit_ns outside
 * 1..10^10), GQA_ECUDA. */
int gqa_selftest_bounded_wait(gqa_cache *cache, int64_t limit_ns, void *stream);

/* Prefix-edit invalidation ([P3] edit at token m): keep positions < m of
 * `seq`, drop the rest.  Pages wholly beyond position m lose one reference
 * (and return to the pool at zero).  A partially kept tail page stays; if it
 * is shared, the next write copies it first.  Host metadata only.
 * Errors: GQA_EINVAL (unknown sequence), GQA_ERANGE unless 0 <= m <= length,
 * and, with a sliding window W, unless m = 0 or positions m - W .. m - 1 are
 * still held (a windowed cache cannot rewind past what it released). */
int kv_truncate(gqa_cache *cache, int32_t seq, int32_t m);

/* Synchronise `stream`, read and clear the cache's device error word.
 * *flags_out receives GQA_DEVERR_* bits (0 = clean).  Returns GQA_EDEVICE
 * if any bit was set, GQA_ECUDA on a CUDA error. */
int gqa_cache_check(gqa_cache *cache, void *stream, int32_t *flags_out);

/* ---- profiling ------------------------------------------------------------ */

/* Kernel ids for gqa_profile_read. */
#define GQA_KERNEL_CACHE_WRITE     0  /* new K/V rows into their pages           */
#define GQA_KERNEL_COW_COPY        1  /* copy-on-write of a shared tail page      */
#define GQA_KERNEL_PREFILL_TC      2  /* tensor-core attention (bf16, 128): prefill, multi-token and tensor-core decode */
#define GQA_KERNEL_ATTN_SIMT       3  /* CUDA-core attention (fp32 / other d_h)   */
#define GQA_KERNEL_DECODE_SPLIT    4  /* split-K decode (bf16, 128), merge included */
#define GQA_KERNEL_DECODE_COMBINE  5  /* reserved: the merge runs inside the split kernel */
#define GQA_KERNEL_ROTATE_PAGES    6  /* pre-position prefill: the call's pages, keys rotated */
#define GQA_KERNEL_DECODE_CLUSTER  7  /* clustered decode (bf16, 128), merge in the cluster */
#define GQA_KERNEL_COUNT           8

/* Turn per-launch timing on or off.  While on, every kernel launch of this
 * cache is bracketed by two CUDA events recorded on the launch's own stream.
 * Launches are counted whether or not timing is on. */
int gqa_profile_enable(gqa_cache *cache, int on);

/* For kernel id `kernel`: the number of launches since the last read, and the
 * summed device time (ms) of the timed ones among them (0 if timing was
 * off).  Waits for the recorded events; clears the kernel's records. */
int gqa_profile_read(gqa_cache *cache, int32_t kernel, int32_t *launches, double *total_ms);

/* Message of the last failing call on this thread ("" if none). */
const char *gqa_last_error(void);

/* Library version string. */
const char *gqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H_ */
