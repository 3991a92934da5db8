"""fp64 CPU oracle for causal grouped-query attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  It shares no code with the CUDA library
``causal_gqa_attention_02_gb300``; neither imports the other.  The only
module both sides use is ``workloads`` (seeded inputs, no arithmetic).

Sources, cited by page title and section:
  [P1] "第二章 Prefill：整层状态演化与 KV 建立" (glenzli.com, vol. 2 ch. 2):
       2.2 mask M; 2.3 attention equations; 2.5 cache contract and
       invariants 2.2; 2.6 pseudocode (write valid positions only).
  [P2] "模型执行：从 token 到 Prefill 与 Decode" (blog.mlxb.cc): the hand-
       worked attention example; the cached-vs-recompute comparison.
  [P3] "KV Cache 与 Prefill/Decode 推理路径" (wiki.maxwellmou.com, unit 10):
       edit-at-m invalidation; PagedAttention block table and free pool;
       incremental prefill; prefix sharing with reference counts.

Contents:
  attention()        the definition of [P1] 2.3, in plain fp64 C (threaded).
  attention_dense()  a second, independent form: materialise S with the -inf
                     mask M of [P1] 2.2, two-pass softmax, numpy matmuls.
  CacheModel         the logical cache plus the page-allocation rules (block
                     table, free pool taken in a fixed order, reference counts,
                     copy-on-write of a shared tail page, truncation), restated
                     from [P3] and the library's documented allocator rules.
  prefill()/decode()/append() drive CacheModel and attention() for a batch.
  rope()             the rotary position mechanism ([P1] 2.3 applies "the
                     position mechanism" to Q and K; [P3]'s prefix-caching
                     section describes RoPE as a rotation by the position ID
                     whose inner products depend only on position differences),
                     and rope_stored_bf16(), the key bytes a rotating cache holds.
  keys_at_read(), attention_pre_position()
                     a pre-position cache ([P1] 2.5's layout_metadata: keys
                     stored before the position transform): keys kept as given,
                     rotated by their positions when read.
  e4m3_encode/_decode, quantize_e4m3_rows(), dequantize_e4m3_rows()
                     the quantised cache ([P1] 2.5: the physical cache may be
                     quantised as long as the logical order is kept): FP8
                     E4M3 codes (the OCP 8-bit floating-point format, written
                     out from its definition) with one fp32 scale per token
                     row of each KV head.

Every function here is pinned by tests in tests/test_oracle_pins.py against
values the pages print, closed forms, special cases and brute force.
"""
from __future__ import annotations

import ctypes
import heapq
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liborc.so")
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_lock = threading.Lock()
_lib = None

PAGE_TOKENS = 16


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_int64)
            lib.orc_attention.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          dp, lp, ctypes.c_int, dp, dp, dp, ctypes.c_int]
            lib.orc_attention.restype = ctypes.c_int
            lib.orc_attention_window.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 dp, lp, ctypes.c_int, dp, dp, dp, ctypes.c_int, ctypes.c_int64]
            lib.orc_attention_window.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------------------
# Stored values -> fp64 (exact for bf16 and fp32).
# ---------------------------------------------------------------------------

def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bit patterns (uint16) or float32 values -> float64, exactly; a
    quantised ("fp8") cache's packed rows -> their dequantised values."""
    if dtype == "fp8":
        return dequantize_e4m3_rows(np.asarray(x, dtype=np.uint8)).astype(np.float64)
    if dtype == "bf16":
        u = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# The attention definition ([P1] 2.3).
# ---------------------------------------------------------------------------

def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, qpos, nthreads: int | None = None, window: int = 0):
    """q [n_q, H_q, d], K/V [L, H_kv, d] (float64), qpos [n_q] absolute
    positions.  Query i sees keys 0..qpos[i], or with window W > 0 keys
    max(0, qpos[i] - W + 1)..qpos[i] ([P3] sliding window: the current
    position counts in the window).  Returns O [n_q, H_q, d]."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    qpos = np.ascontiguousarray(qpos, dtype=np.int64)
    n_q, H_q, d = q.shape
    L, H_kv, d2 = K.shape
    assert d2 == d and V.shape == K.shape and qpos.shape == (n_q,)
    out = np.zeros((n_q, H_q, d), dtype=np.float64)
    if n_q == 0:
        return out
    dp = ctypes.POINTER(ctypes.c_double)
    rc = lib.orc_attention_window(n_q, H_q, H_kv, d, q.ctypes.data_as(dp),
                                  qpos.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  L, K.ctypes.data_as(dp), V.ctypes.data_as(dp),
                                  out.ctypes.data_as(dp), int(nthreads or default_threads()), int(window))
    if rc != 0:
        raise ValueError("oracle precondition failed (rc=%d)" % rc)
    return out


def attention_dense(q: np.ndarray, K: np.ndarray, V: np.ndarray, qpos, window: int = 0):
    """Second form of [P1] 2.3 for small inputs: build S = QK^T/sqrt(d) + M with
    M = -inf on invisible keys, take each row's finite max, exponentiate the
    finite entries, normalise, multiply by V."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    qpos = np.asarray(qpos, dtype=np.int64)
    n_q, H_q, d = q.shape
    L, H_kv, _ = K.shape
    out = np.zeros((n_q, H_q, d))
    j = np.arange(L)[None, :]
    visible = j <= qpos[:, None]
    if window > 0:
        visible &= j > qpos[:, None] - window
    M = np.where(visible, 0.0, -np.inf)
    for h in range(H_q):
        g = (h * H_kv) // H_q
        S = (q[:, h, :] @ K[:, g, :].T) / np.sqrt(d) + M
        finite = np.isfinite(S)
        if not finite.any(axis=1).all():
            raise ValueError("a query row has no finite score")
        m = np.where(finite, S, -np.inf).max(axis=1)
        E = np.where(finite, np.exp(np.where(finite, S, 0.0) - m[:, None]), 0.0)
        A = E / E.sum(axis=1, keepdims=True)
        out[:, h, :] = A @ V[:, g, :]
    return out


# ---------------------------------------------------------------------------
# Rotary position mechanism ([P1] 2.3: Q~, K~ are Q, K after the position
# mechanism; [P3] prefix caching: RoPE rotates Q/K at position i by a
# rotation fixed by the position ID, and the rotated inner product depends
# only on the position difference).  The pages give no formula; the reading
# here: dimension pairs (k, k + d/2), k < d/2, each rotated counter-clockwise
# by pos * base^(-2k/d).
# ---------------------------------------------------------------------------

def rope_theta(d: int, base: float) -> np.ndarray:
    """Frequencies base^(-2k/d), k = 0..d/2-1 (fp64)."""
    return np.power(float(base), -2.0 * np.arange(d // 2, dtype=np.float64) / d)


def rope(x: np.ndarray, positions, base: float) -> np.ndarray:
    """Rotate the last axis of x [n, ..., d] (fp64) at positions [n]."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    pos = np.asarray(positions, dtype=np.float64).reshape((-1,) + (1,) * (x.ndim - 1))
    ang = pos * rope_theta(d, base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def rope_stored_bf16(k_bits: np.ndarray, positions, base: float) -> np.ndarray:
    """The bytes a rotating bf16 cache stores for keys k [n, H, d] (bf16
    bits) at positions [n]: cos/sin of pos * theta_k rounded to fp32, each
    product and the sum or difference rounded to fp32 (no fused
    multiply-add), then rounded to bf16 (nearest, ties to even)."""
    x = to_f64(k_bits, "bf16").astype(np.float32)
    d = x.shape[-1]
    h = d // 2
    pos = np.asarray(positions, dtype=np.float64).reshape((-1,) + (1,) * (x.ndim - 1))
    ang = pos * rope_theta(d, base)
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    x1, x2 = x[..., :h], x[..., h:]
    y1 = (x1 * c).astype(np.float32) - (x2 * s).astype(np.float32)
    y2 = (x1 * s).astype(np.float32) + (x2 * c).astype(np.float32)
    return _f32_to_bf16_bits(np.concatenate([y1, y2], axis=-1).astype(np.float32))


# ---------------------------------------------------------------------------
# Pre-position keys ([P1] 2.5: layout_metadata records whether the cached
# keys are taken before or after the position transform; [P3] prefix
# caching: keys rotated by their position ID can only be reused at the same
# absolute positions).  A pre-position cache stores each key as given and a
# reader rotates it by its position before the score; in exact arithmetic
# that is the post-position definition, and the stored keys can be read at
# any common position offset.
# ---------------------------------------------------------------------------

def keys_at_read(K_stored: np.ndarray, positions, base: float) -> np.ndarray:
    """Keys a reader of a pre-position cache uses: each stored key K_stored
    [L, H, d] (fp64 values, as given to the cache) rotated by its position."""
    return rope(K_stored, positions, base)


def attention_pre_position(q: np.ndarray, K_stored: np.ndarray, V: np.ndarray, qpos, base: float,
                           offset: int = 0, window: int = 0, nthreads: int | None = None):
    """Attention over a pre-position cache: queries q [n, H_q, d] (before the
    rotation) at positions qpos, stored keys K_stored [L, H_kv, d] at
    positions 0..L-1; both read at absolute positions shifted by `offset`
    (0: as written) and rotated there, then the definition of [P1] 2.3
    (visibility by qpos)."""
    qpos = np.asarray(qpos, dtype=np.int64)
    L = K_stored.shape[0]
    return attention(rope(q, qpos + offset, base), keys_at_read(K_stored, np.arange(L) + offset, base), V, qpos,
                     nthreads, window)


# ---------------------------------------------------------------------------
# Logical paged cache ([P1] 2.5; [P3] PagedAttention, prefix sharing, edit).
# ---------------------------------------------------------------------------

# ---------------------------------------------------------------------------
# Quantised cache: FP8 E4M3 codes with one fp32 scale per row ([P1] 2.5
# allows a quantised physical layout; the scheme below is this library's).
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """FP8 E4M3 code bytes -> float64, from the format's definition: sign bit,
    4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
    (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN, so the largest finite
    value is 1.75 * 2^8 = 448; there are no infinities."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """float values -> E4M3 code bytes: round to nearest, ties to even
    mantissa, magnitudes beyond 448 saturate to 448 (no NaN for finite
    input).  Computed in fp64 from the definition above."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # Subnormals (and the boundary into the first normal binade): m = a / 2^-9.
    code = np.where(sub, np.rint(a / 2.0 ** -9).astype(np.int64), code)
    # Normals: a = 2^e (1 + f), m = rint(8 f); a carry moves to the next binade.
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(sub, 1.0, a))).astype(np.int64)
    frac = np.where(sub, 0.0, a / np.exp2(e.astype(np.float64)) - 1.0)
    m = np.rint(frac * 8.0).astype(np.int64)
    e = np.where(m == 8, e + 1, e)
    m = np.where(m == 8, 0, m)
    normal = ((e + 7) << 3) | m
    code = np.where(sub, code, normal)
    code = np.where(a >= E4M3_MAX, 0x7E, np.minimum(code, 0x7E))
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def quantize_e4m3_rows(x) -> tuple:
    """Rows x [..., d] (float32 values) -> (codes [..., d] uint8, scales [...]
    float32).  Per row: s = amax / 448 in fp32; code = E4M3(x / s) with x / s
    in fp32 (round to nearest); a row of zeros gets s = 0 and zero codes.
    Dequantised value: fp32(decode(code) * s)."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    y = (x / safe[..., None]).astype(np.float32)
    codes = e4m3_encode(y)
    codes = np.where((s > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes, s


def pack_e4m3_rows(codes, scales) -> np.ndarray:
    """A quantised row as the cache model stores it: d code bytes followed
    by the 4 bytes of its fp32 scale."""
    sb = np.ascontiguousarray(np.asarray(scales, dtype=np.float32)).view(np.uint8).reshape(*np.shape(scales), 4)
    return np.concatenate([np.asarray(codes, dtype=np.uint8), sb], axis=-1)


def dequantize_e4m3_rows(packed) -> np.ndarray:
    """Packed rows [..., d + 4] -> float32 values fp32(decode(code) * s)."""
    packed = np.asarray(packed, dtype=np.uint8)
    codes = packed[..., :-4]
    s = np.ascontiguousarray(packed[..., -4:]).view(np.float32)[..., 0]
    return (e4m3_decode(codes).astype(np.float32) * s[..., None]).astype(np.float32)


class CacheError(Exception):
    def __init__(self, kind: str, msg: str = ""):
        super().__init__("%s: %s" % (kind, msg))
        self.kind = kind


class CacheModel:
    """Logical KV cache with a block table per sequence.

    Rules (the pages give the mechanism; the fixed choices are the library's
    documented ones, restated here independently):
      * token t of a sequence lives in logical page t // 16 at offset t % 16,
        and the block table maps logical page -> physical page ([P3]
        PagedAttention: block size B_s, logical block and offset);
      * a new page comes from the free pool when the tail page is full, and
        the pool may hand out any free page ([P3] PagedAttention, growth of a
        request); the library fixes the choice as the free page of smallest
        rank in a page order given at creation (identity by default);
      * pages are reference counted; a page returns to the pool only when no
        sequence references it ([P3] prefix tree: a shared block is reclaimed
        once every request that uses it has finished);
      * writing into a shared tail page first copies it to a fresh page
        ([P3] prefix tree: a fork inside a block needs copy-on-write);
      * truncate(m) keeps positions < m and drops the rest ([P3] edit at m:
        keep the KV before m, truncate the suffix);
      * fork(src, k) starts a sequence on src's first k positions, sharing
        their pages ([P1] 2.9 prefix reuse);
      * with a sliding window W ([P3] sliding window and ring cache: K/V
        outside the window is never read again, so it need not be kept), a
        write that brings a sequence to length L releases every page whose
        positions all lie before L - W (no query at a position >= L - 1 sees
        them); its block-table entry becomes -1.  Truncating or forking at
        m > 0 needs the positions m - W .. m - 1 still held, else ERANGE.
    Within one batched call, pages are taken sequence by sequence in batch
    order; for each sequence the copy-on-write page comes first, then new
    pages in logical order.  A call that cannot be satisfied changes nothing.
    """

    def __init__(self, num_pages, max_seqs, max_pages_per_seq, H_kv, d, dtype,
                 page_order=None, window=0):
        self.window = int(window)
        self.num_pages = int(num_pages)
        self.max_seqs = int(max_seqs)
        self.max_pages_per_seq = int(max_pages_per_seq)
        self.H_kv, self.d, self.dtype = int(H_kv), int(d), dtype
        order = np.arange(self.num_pages) if page_order is None else np.asarray(page_order)
        assert sorted(order.tolist()) == list(range(self.num_pages))
        self.rank = np.empty(self.num_pages, dtype=np.int64)
        self.rank[order] = np.arange(self.num_pages)
        self.order = order.astype(np.int64)
        self.free = list(range(self.num_pages))   # heap of ranks
        heapq.heapify(self.free)
        self.ref = np.zeros(self.num_pages, dtype=np.int64)
        self.seqs = {}                            # id -> dict(pages, len, k, v)
        self.copies = []                          # (src_page, dst_page, slots) log

    # -- page pool ---------------------------------------------------------
    def _take(self):
        r = heapq.heappop(self.free)
        p = int(self.order[r])
        assert self.ref[p] == 0
        self.ref[p] = 1
        return p

    def _drop(self, p):
        self.ref[p] -= 1
        assert self.ref[p] >= 0
        if self.ref[p] == 0:
            heapq.heappush(self.free, int(self.rank[p]))

    def free_pages(self):
        return len(self.free)

    # -- sequences ---------------------------------------------------------
    @property
    def io_dtype(self):
        """Type of q, k, v and out at the interface (bf16 for a quantised cache)."""
        return "bf16" if self.dtype == "fp8" else self.dtype

    def _empty_rows(self):
        if self.dtype == "fp8":                   # codes + 4 scale bytes per row
            return np.zeros((0, self.H_kv, self.d + 4), dtype=np.uint8)
        dt = np.uint16 if self.dtype == "bf16" else np.float32
        return np.zeros((0, self.H_kv, self.d), dtype=dt)

    def _stored(self, rows):
        """Input rows (bf16 bits, or fp32 values) as this cache stores them."""
        if self.dtype == "fp8":
            codes, sc = quantize_e4m3_rows(to_f64(rows, "bf16").astype(np.float32))
            return pack_e4m3_rows(codes, sc)
        return np.asarray(rows, dtype=np.uint16 if self.dtype == "bf16" else np.float32)

    def create(self):
        for s in range(self.max_seqs):
            if s not in self.seqs:
                self.seqs[s] = {"pages": [], "len": 0, "k": self._empty_rows(), "v": self._empty_rows()}
                return s
        raise CacheError("ENOMEM", "no free sequence id")

    def _released(self, S):
        return sum(1 for p in S["pages"] if p < 0)

    def _window_holds(self, S, m):
        """True if positions m - W .. m - 1 are still held (or no window)."""
        return self.window <= 0 or m == 0 or PAGE_TOKENS * self._released(S) <= m - self.window

    def fork(self, src, prefix_len):
        S = self._seq(src)
        if not (0 <= prefix_len <= S["len"]):
            raise CacheError("ERANGE", "prefix beyond source length")
        if not self._window_holds(S, prefix_len):
            raise CacheError("ERANGE", "prefix reaches back past the sliding window")
        s = self.create()
        keep = -(-prefix_len // PAGE_TOKENS)
        pages = list(S["pages"][:keep])
        for p in pages:
            if p >= 0:
                self.ref[p] += 1
        self.seqs[s].update(pages=pages, len=prefix_len,
                            k=S["k"][:prefix_len].copy(), v=S["v"][:prefix_len].copy())
        return s

    def free_seq(self, s):
        self.truncate(s, 0)
        del self.seqs[s]

    def truncate(self, s, m):
        S = self._seq(s)
        if not (0 <= m <= S["len"]):
            raise CacheError("ERANGE", "truncate beyond length")
        if not self._window_holds(S, m):
            raise CacheError("ERANGE", "truncate reaches back past the sliding window")
        keep = -(-m // PAGE_TOKENS)
        for p in S["pages"][keep:]:
            if p >= 0:
                self._drop(p)
        S["pages"] = S["pages"][:keep]
        S["len"] = m
        S["k"] = S["k"][:m].copy()
        S["v"] = S["v"][:m].copy()

    def _seq(self, s):
        if s not in self.seqs:
            raise CacheError("EINVAL", "unknown sequence %r" % (s,))
        return self.seqs[s]

    def length(self, s):
        return self._seq(s)["len"]

    def block_table(self, s):
        return list(self._seq(s)["pages"])

    # -- writes --------------------------------------------------------------
    def _pages_needed(self, S, count):
        P = S["len"]
        need = -(-(P + count) // PAGE_TOKENS) - len(S["pages"])
        cow = 1 if (count > 0 and P % PAGE_TOKENS != 0 and self.ref[S["pages"][-1]] > 1) else 0
        return need, cow

    def write(self, seq_ids, k_rows, v_rows):
        """Append k_rows[b], v_rows[b] ([c_b, H_kv, d] stored values) to
        sequence seq_ids[b], for every b, as one atomic call."""
        if len(set(seq_ids)) != len(seq_ids):
            raise CacheError("EINVAL", "a sequence appears twice in one write")
        total = 0
        for s, kr in zip(seq_ids, k_rows):
            S = self._seq(s)
            c = kr.shape[0]
            if -(-(S["len"] + c) // PAGE_TOKENS) > self.max_pages_per_seq:
                raise CacheError("ERANGE", "sequence capacity exceeded")
            need, cow = self._pages_needed(S, c)
            total += need + cow
        if total > self.free_pages():
            raise CacheError("ENOMEM", "page pool exhausted")
        for s, kr, vr in zip(seq_ids, k_rows, v_rows):
            S = self._seq(s)
            c = kr.shape[0]
            need, cow = self._pages_needed(S, c)
            if cow:
                old = S["pages"][-1]
                new = self._take()
                self.copies.append((old, new, S["len"] % PAGE_TOKENS))
                self._drop(old)
                S["pages"][-1] = new
            for _ in range(need):
                S["pages"].append(self._take())
            S["k"] = np.concatenate([S["k"], self._stored(kr)], axis=0)
            S["v"] = np.concatenate([S["v"], self._stored(vr)], axis=0)
            S["len"] += c
        # Release only once every entry is written: the call's own readers (a
        # prefill over these rows) still see the keys it wrote, so no page of
        # this call goes back to the pool before the call ends.
        if self.window > 0:
            for s in seq_ids:
                S = self._seq(s)
                for j, p in enumerate(S["pages"]):
                    if p >= 0 and PAGE_TOKENS * (j + 1) <= S["len"] - self.window:
                        self._drop(p)
                        S["pages"][j] = -1

    def kv(self, s):
        """Logical K, V of sequence s as fp64 arrays [len, H_kv, d]."""
        S = self._seq(s)
        return to_f64(S["k"], self.dtype), to_f64(S["v"], self.dtype)

    def raw_kv(self, s):
        S = self._seq(s)
        return S["k"], S["v"]


# ---------------------------------------------------------------------------
# Batched drivers.
# ---------------------------------------------------------------------------

def prefill(cache: CacheModel, seq_ids, q, k, v, valid_lengths, nthreads=None, rope_base=None):
    """[P1] 2.6: write each sequence's valid K/V rows at positions P_b.. into
    the cache, then causal attention of the valid query rows over the cache.
    q [B, n, H_q, d], k/v [B, n, H_kv, d] stored values.  Padding rows
    (i >= n_b) are discarded ([P1] 2.2) and returned as zeros.  With
    rope_base, q and every key are rotated by their positions first (the
    cache model keeps the unrotated keys: the bytes a pre-position cache
    stores; a post-position cache stores rope_stored_bf16 of them)."""
    dt = cache.io_dtype
    B, n, H_q, d = q.shape
    nb = [int(x) for x in valid_lengths]
    if any(x < 1 or x > n for x in nb):
        raise CacheError("EMASK", "each sequence needs 1..n valid rows")
    past = [cache.length(s) for s in seq_ids]
    cache.write(list(seq_ids), [k[b, :nb[b]] for b in range(B)], [v[b, :nb[b]] for b in range(B)])
    out = np.zeros((B, n, H_q, d))
    for b, s in enumerate(seq_ids):
        K, V = cache.kv(s)
        qpos = past[b] + np.arange(nb[b])
        qb = to_f64(q[b, :nb[b]], dt)
        if rope_base is not None:
            qb, K = rope(qb, qpos, rope_base), rope(K, np.arange(K.shape[0]), rope_base)
        out[b, :nb[b]] = attention(qb, K, V, qpos, nthreads, window=cache.window)
    return out


def append(cache: CacheModel, seq_ids, k_new, v_new, counts=None):
    """[P3] decode: append each sequence's new k/v rows at its tail.
    k_new/v_new [B, c, H_kv, d] (or [B, H_kv, d] for one token each)."""
    if k_new.ndim == 3:
        k_new, v_new = k_new[:, None], v_new[:, None]
    B = k_new.shape[0]
    cnt = [k_new.shape[1]] * B if counts is None else [int(c) for c in counts]
    cache.write(list(seq_ids), [k_new[b, :cnt[b]] for b in range(B)], [v_new[b, :cnt[b]] for b in range(B)])


def decode(cache: CacheModel, seq_ids, q, nthreads=None, rope_base=None):
    """[P3] single-token decode: query b at position L_b - 1 reads all L_b
    cached entries (its own appended entry included).  q [B, H_q, d].  With
    rope_base, q and the keys are rotated by their positions first."""
    dt = cache.io_dtype
    B, H_q, d = q.shape
    out = np.zeros((B, H_q, d))
    for b, s in enumerate(seq_ids):
        K, V = cache.kv(s)
        L = K.shape[0]
        if L < 1:
            raise CacheError("EMASK", "decode over an empty cache")
        qb = to_f64(q[b][None], dt)
        if rope_base is not None:
            qb, K = rope(qb, [L - 1], rope_base), rope(K, np.arange(L), rope_base)
        out[b] = attention(qb, K, V, np.array([L - 1]), nthreads, window=cache.window)[0]
    return out

