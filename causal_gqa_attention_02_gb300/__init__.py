"""Python binding of libgqa (include/gqa.h): causal GQA prefill and decode
over a paged KV cache on GB300.

This module only marshals arguments: it turns torch tensors into device
pointers and CUDA streams into handles, and raises on non-zero status.  Every
step of the hot path runs in the CUDA library.  There is no fallback: if
``_lib/libgqa.so`` has not been built, importing this package fails.

PyTorch supplies device memory (the page pool, q/k/v/out) and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import work  # noqa: F401  (work counts for throughput figures)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgqa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libgqa.so is not built (%s); run __graft_entry__.build() first" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

OK, EINVAL, ERANGE, EMASK, ENOMEM, ELAYOUT, ECUDA, EDEVICE = 0, -1, -2, -3, -4, -5, -6, -7
ERRNAMES = {EINVAL: "EINVAL", ERANGE: "ERANGE", EMASK: "EMASK", ENOMEM: "ENOMEM",
            ELAYOUT: "ELAYOUT", ECUDA: "ECUDA", EDEVICE: "EDEVICE"}
DTYPE_BF16, DTYPE_F32, DTYPE_FP8_E4M3 = 1, 2, 3
PAGE_TOKENS = 16
LAYOUT_VERSION = 2
DEVERR_PAGE_ID, DEVERR_TIMEOUT, DEVERR_SHAPE = 1, 2, 4
KERNELS = {"cache_write": 0, "cow_copy": 1, "prefill_tc": 2, "attn_simt": 3,
           "decode_split": 4, "decode_combine": 5, "rotate_pages": 6, "decode_cluster": 7}
DECODE_KERNELS = {"auto": 0, "tensor_core": 1, "cuda_core": 2, "cluster": 3}

_I32P = ctypes.POINTER(ctypes.c_int32)


class CacheDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("keys_post_position", ctypes.c_int32),
                ("layout_version", ctypes.c_int32), ("page_order", _I32P),
                ("rope", ctypes.c_int32), ("rope_base", ctypes.c_float), ("window", ctypes.c_int32)]


class LayoutMetadata(ctypes.Structure):
    _fields_ = [("keys_post_position", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("layout_version", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope", ctypes.c_int32), ("rope_base", ctypes.c_float), ("window", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def _sig(name, res, *args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = list(args)
    return fn


_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_sig("gqa_pool_bytes", _sz, ctypes.POINTER(CacheDesc))
_sig("gqa_cache_create", ctypes.c_int, ctypes.POINTER(CacheDesc), _vp, _sz, ctypes.POINTER(_vp))
_sig("gqa_cache_destroy", ctypes.c_int, _vp)
_sig("gqa_cache_layout", ctypes.c_int, _vp, ctypes.POINTER(LayoutMetadata))
_sig("gqa_layout_compatible", ctypes.c_int, ctypes.POINTER(LayoutMetadata), ctypes.POINTER(LayoutMetadata))
_sig("gqa_seq_create", ctypes.c_int, _vp, _I32P)
_sig("gqa_seq_fork", ctypes.c_int, _vp, _i32, _i32, _I32P)
_sig("gqa_seq_free", ctypes.c_int, _vp, _i32)
_sig("gqa_seq_length", ctypes.c_int, _vp, _i32, _I32P)
_sig("gqa_seq_block_table", ctypes.c_int, _vp, _i32, _I32P, _i32, _I32P)
_sig("gqa_free_pages", ctypes.c_int, _vp, _I32P)
_sig("gqa_page_refcount", ctypes.c_int, _vp, _i32, _I32P)
_sig("attn_prefill", ctypes.c_int, _vp, _i32, _I32P, _i32, _i32, _vp, _vp, _vp, _I32P, _I32P, _vp, _vp)
_sig("attn_prefill_host", ctypes.c_int, _vp, _i32, _I32P, _i32, _i32, _vp, _vp, _vp, _I32P, _I32P, _vp, _vp)
_sig("kv_append", ctypes.c_int, _vp, _i32, _I32P, _i32, _I32P, _vp, _vp, _vp)
_sig("attn_decode", ctypes.c_int, _vp, _i32, _I32P, _i32, _vp, _vp, _vp)
_sig("attn_decode_static", ctypes.c_int, _vp, _i32, _I32P, _i32, _vp, _vp, _vp)
_sig("attn_decode_append", ctypes.c_int, _vp, _i32, _I32P, _i32, _vp, _vp, _vp, _vp, _vp)
_sig("attn_decode_append_host", ctypes.c_int, _vp, _i32, _I32P, _i32, _vp, _vp, _vp, _vp, _vp)
_sig("attn_decode_tables", ctypes.c_int, _vp, _i32, _vp, _i32, _I32P, _i32, _vp, _vp, _vp)
_sig("kv_truncate", ctypes.c_int, _vp, _i32, _i32)
_sig("gqa_cache_check", ctypes.c_int, _vp, _vp, _I32P)
_sig("gqa_profile_enable", ctypes.c_int, _vp, ctypes.c_int)
_sig("gqa_set_decode_kernel", ctypes.c_int, _vp, ctypes.c_int32)
_sig("gqa_selftest_bounded_wait", ctypes.c_int, _vp, ctypes.c_int64, _vp)
_sig("gqa_profile_read", ctypes.c_int, _vp, _i32, _I32P, ctypes.POINTER(ctypes.c_double))
_sig("gqa_last_error", ctypes.c_char_p)
_sig("gqa_version", ctypes.c_char_p)


class GqaError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s (%d): %s" % (ERRNAMES.get(code, "?"), code, msg))
        self.code = code
        self.name = ERRNAMES.get(code, "?")


def _check(rc):
    if rc != OK:
        raise GqaError(rc, _lib.gqa_last_error().decode(errors="replace"))


def version() -> str:
    return _lib.gqa_version().decode()


def _i32_array(values):
    if values is None:
        return None, None
    vals = [int(x) for x in (values.reshape(-1).tolist() if hasattr(values, "reshape") else values)]
    arr = (ctypes.c_int32 * max(1, len(vals)))(*vals)
    return arr, ctypes.cast(arr, _I32P)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device=None):
    """cudaStream_t of `stream` (default: the current stream of `device`)."""
    if stream is None:
        if _raw_stream is not None and device is not None:
            return _raw_stream(device)
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# Element type of q, k, v and out (a quantised cache takes and returns bf16).
_TORCH_DTYPE = {DTYPE_BF16: torch.bfloat16, DTYPE_F32: torch.float32, DTYPE_FP8_E4M3: torch.bfloat16}
_DTYPE_CODE = {"bf16": DTYPE_BF16, "f32": DTYPE_F32, "fp8": DTYPE_FP8_E4M3}


class Cache:
    """A paged KV cache: a torch-owned device page pool plus the library's
    host metadata.  ``metadata_only=True`` creates no pool (no GPU needed);
    launching calls then only validate and update block tables/lengths."""

    def __init__(self, num_kv_heads, head_dim, num_pages, max_seqs, max_pages_per_seq,
                 dtype="bf16", page_order=None, device=None, metadata_only=False,
                 keys_post_position=1, layout_version=LAYOUT_VERSION, rope=False, rope_base=10000.0, window=0):
        self.dtype_code = (DTYPE_BF16 if dtype is torch.bfloat16 else DTYPE_F32 if dtype is torch.float32
                           else _DTYPE_CODE[dtype])
        self.torch_dtype = _TORCH_DTYPE[self.dtype_code]
        self._order_keep, order_ptr = _i32_array(page_order)
        self.desc = CacheDesc(self.dtype_code, num_kv_heads, head_dim, PAGE_TOKENS, num_pages,
                              max_seqs, max_pages_per_seq, keys_post_position, layout_version,
                              order_ptr, int(rope), float(rope_base), int(window))
        self.rope, self.rope_base, self.window = int(rope), float(rope_base), int(window)
        self.num_kv_heads, self.head_dim, self.num_pages = num_kv_heads, head_dim, num_pages
        self.max_seqs, self.max_pages_per_seq = max_seqs, max_pages_per_seq
        self.pool = None
        self.device_index = None
        self._h = ctypes.c_void_p()
        nbytes = _lib.gqa_pool_bytes(ctypes.byref(self.desc))
        if metadata_only:
            _check(_lib.gqa_cache_create(ctypes.byref(self.desc), None, 0, ctypes.byref(self._h)))
        else:
            dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
            self.pool = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
            self.device_index = self.pool.device.index
            with torch.cuda.device(dev):
                _check(_lib.gqa_cache_create(ctypes.byref(self.desc), ctypes.c_void_p(self.pool.data_ptr()),
                                             nbytes, ctypes.byref(self._h)))

    @property
    def handle(self):
        return self._h

    def pool_view(self):
        """The pool as [num_pages, 2 (K, V), H_kv, 2 (slot groups), C (128-byte
        chunks of a row), 8 (slots), 128 / element size] of the cache dtype:
        slot s of a page is group s // 8, position s % 8; element e of its row
        is chunk e // (128 / element size).  Elements past d_h in the last
        chunk are padding."""
        if self.dtype_code == DTYPE_FP8_E4M3:             # code bytes; the scales follow
            chunks = -(-self.head_dim // 128)
            nb = self.num_pages * 2 * self.num_kv_heads * PAGE_TOKENS * chunks * 128
            return self.pool[:nb].view(self.num_pages, 2, self.num_kv_heads, 2, chunks, PAGE_TOKENS // 2, 128)
        es = 2 if self.torch_dtype == torch.bfloat16 else 4
        per = 128 // es
        chunks = -(-self.head_dim * es // 128)
        return self.pool.view(self.torch_dtype).view(self.num_pages, 2, self.num_kv_heads, 2, chunks,
                                                     PAGE_TOKENS // 2, per)

    def scales_view(self):
        """FP8 E4M3 cache: the fp32 scales as [num_pages, 2 (K, V), H_kv, 16 slots]."""
        chunks = -(-self.head_dim // 128)
        nb = self.num_pages * 2 * self.num_kv_heads * PAGE_TOKENS * chunks * 128
        return self.pool[nb:].view(torch.float32).view(self.num_pages, 2, self.num_kv_heads, PAGE_TOKENS)

    def close(self):
        if self._h:
            _lib.gqa_cache_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- sequences -----------------------------------------------------------
    def seq_create(self) -> int:
        s = ctypes.c_int32()
        _check(_lib.gqa_seq_create(self._h, ctypes.byref(s)))
        return s.value

    def seq_fork(self, src: int, prefix_len: int) -> int:
        s = ctypes.c_int32()
        _check(_lib.gqa_seq_fork(self._h, src, prefix_len, ctypes.byref(s)))
        return s.value

    def seq_free(self, seq: int):
        _check(_lib.gqa_seq_free(self._h, seq))

    def seq_length(self, seq: int) -> int:
        n = ctypes.c_int32()
        _check(_lib.gqa_seq_length(self._h, seq, ctypes.byref(n)))
        return n.value

    def block_table(self, seq: int):
        cnt = ctypes.c_int32()
        buf = (ctypes.c_int32 * max(1, self.max_pages_per_seq))()
        _check(_lib.gqa_seq_block_table(self._h, seq, buf, self.max_pages_per_seq, ctypes.byref(cnt)))
        return list(buf[: cnt.value])

    def free_pages(self) -> int:
        n = ctypes.c_int32()
        _check(_lib.gqa_free_pages(self._h, ctypes.byref(n)))
        return n.value

    def refcount(self, page: int) -> int:
        n = ctypes.c_int32()
        _check(_lib.gqa_page_refcount(self._h, page, ctypes.byref(n)))
        return n.value

    def layout(self) -> LayoutMetadata:
        m = LayoutMetadata()
        _check(_lib.gqa_cache_layout(self._h, ctypes.byref(m)))
        return m

    def set_decode_kernel(self, kernel: str):
        """Decode kernel of attn_decode / attn_decode_static: "auto",
        "tensor_core", "cuda_core" or "cluster"."""
        _check(_lib.gqa_set_decode_kernel(self._h, DECODE_KERNELS[kernel]))

    def selftest_bounded_wait(self, limit_ns: int, stream=None):
        """Queue a block whose bounded wait runs out after limit_ns and sets
        the timeout bit of the error word (see include/gqa.h)."""
        st = _stream_handle(stream, self.device_index) if self.pool is not None else None
        _check(_lib.gqa_selftest_bounded_wait(self._h, int(limit_ns), st))

    def profile(self, on: bool):
        """Bracket every kernel launch with CUDA events (on its stream)."""
        _check(_lib.gqa_profile_enable(self._h, 1 if on else 0))

    def profile_read(self):
        """{kernel: (launches, total_ms)} since the last read; waits for events."""
        res = {}
        for name, kid in KERNELS.items():
            n, ms = ctypes.c_int32(), ctypes.c_double()
            _check(_lib.gqa_profile_read(self._h, kid, ctypes.byref(n), ctypes.byref(ms)))
            res[name] = (n.value, ms.value)
        return res

    def check(self, stream=None) -> int:
        """Synchronise and read/clear the device error word (0 = clean)."""
        flags = ctypes.c_int32()
        st = _stream_handle(stream, self.device_index) if self.pool is not None else None
        rc = _lib.gqa_cache_check(self._h, st,
                                  ctypes.byref(flags))
        if rc not in (OK, EDEVICE):
            _check(rc)
        return flags.value


def layout_compatible(a: LayoutMetadata, b: LayoutMetadata) -> bool:
    rc = _lib.gqa_layout_compatible(ctypes.byref(a), ctypes.byref(b))
    if rc not in (OK, ELAYOUT):
        _check(rc)
    return rc == OK


def _dev_ptr(t, what, dtype, shape=None):
    if t is None:
        return None
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous()
            and (shape is None or t.shape == shape)):
        return t.data_ptr()                       # the common case, checked in one pass
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % what)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (what, tuple(t.shape), tuple(shape)))
    return ctypes.c_void_p(t.data_ptr())


def attn_prefill(cache: Cache, seq_ids, q, k, v, valid_lengths, positions=None, out=None, stream=None):
    """Causal GQA prefill (see include/gqa.h).  q [B, n, H_q, d],
    k/v [B, n, H_kv, d]; returns out [B, n, H_q, d]."""
    B, n, H_q = len(seq_ids), q.shape[1], q.shape[2]
    dt = cache.torch_dtype
    d = cache.head_dim
    if out is None:
        out = torch.empty_like(q)
    keep_s, sp = _i32_array(seq_ids)
    keep_v, vp = _i32_array(valid_lengths)
    keep_p, pp = _i32_array(positions)
    _check(_lib.attn_prefill(cache.handle, B, sp, n, H_q,
                             _dev_ptr(q, "q", dt, (B, n, H_q, d)),
                             _dev_ptr(k, "k", dt, (B, n, cache.num_kv_heads, d)),
                             _dev_ptr(v, "v", dt, (B, n, cache.num_kv_heads, d)),
                             vp, pp, _dev_ptr(out, "out", dt, (B, n, H_q, d)),
                             _stream_handle(stream, cache.device_index) if cache.pool is not None else None))
    return out


def _host_ptr(t, what, dtype, shape):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a host (CPU) tensor" % what)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (what, tuple(t.shape), tuple(shape)))
    return t.data_ptr()


def attn_prefill_host(cache: Cache, seq_ids, q, k, v, valid_lengths, positions=None, out=None, stream=None):
    """attn_prefill on host tensors (see include/gqa.h): q [B, n, H_q, d],
    k/v [B, n, H_kv, d] on the CPU, pinned for overlapped copies; returns
    out [B, n, H_q, d] on the CPU (allocated pinned like q if not given).
    Only valid rows of out are written.  The result is complete once
    `stream` (default: the current stream) is synchronised."""
    B, n, H_q = len(seq_ids), q.shape[1], q.shape[2]
    dt, d, H_kv = cache.torch_dtype, cache.head_dim, cache.num_kv_heads
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    keep_s, sp = _i32_array(seq_ids)
    keep_v, vp = _i32_array(valid_lengths)
    keep_p, pp = _i32_array(positions)
    _check(_lib.attn_prefill_host(cache.handle, B, sp, n, H_q,
                                  _host_ptr(q, "q", dt, (B, n, H_q, d)),
                                  _host_ptr(k, "k", dt, (B, n, H_kv, d)),
                                  _host_ptr(v, "v", dt, (B, n, H_kv, d)),
                                  vp, pp, _host_ptr(out, "out", dt, (B, n, H_q, d)),
                                  _stream_handle(stream, cache.device_index)))
    return out


def attn_prefill_host_meta(cache: Cache, seq_ids, n, H_q, valid_lengths, positions=None):
    """attn_prefill_host on a metadata-only cache (no buffers)."""
    keep_s, sp = _i32_array(seq_ids)
    keep_v, vp = _i32_array(valid_lengths)
    keep_p, pp = _i32_array(positions)
    _check(_lib.attn_prefill_host(cache.handle, len(seq_ids), sp, n, H_q, None, None, None, vp, pp, None, None))


def attn_prefill_meta(cache: Cache, seq_ids, n, H_q, valid_lengths, positions=None):
    """attn_prefill on a metadata-only cache (no tensors)."""
    keep_s, sp = _i32_array(seq_ids)
    keep_v, vp = _i32_array(valid_lengths)
    keep_p, pp = _i32_array(positions)
    _check(_lib.attn_prefill(cache.handle, len(seq_ids), sp, n, H_q, None, None, None, vp, pp, None, None))


def kv_append(cache: Cache, seq_ids, k_new, v_new, counts=None, stream=None):
    """Append rows at each sequence's tail.  k_new/v_new [B, n, H_kv, d] or
    [B, H_kv, d] (one row each)."""
    if k_new.dim() == 3:
        k_new, v_new = k_new.unsqueeze(1), v_new.unsqueeze(1)
    B, n = len(seq_ids), k_new.shape[1]
    shape = (B, n, cache.num_kv_heads, cache.head_dim)
    keep_s, sp = _i32_array(seq_ids)
    keep_c, cp = _i32_array(counts)
    _check(_lib.kv_append(cache.handle, B, sp, n, cp,
                          _dev_ptr(k_new, "k_new", cache.torch_dtype, shape),
                          _dev_ptr(v_new, "v_new", cache.torch_dtype, shape),
                          _stream_handle(stream, cache.device_index)))


def kv_append_meta(cache: Cache, seq_ids, n, counts=None):
    keep_s, sp = _i32_array(seq_ids)
    keep_c, cp = _i32_array(counts)
    _check(_lib.kv_append(cache.handle, len(seq_ids), sp, n, cp, None, None, None))


def attn_decode(cache: Cache, seq_ids, q, out=None, stream=None):
    """Single-token decode.  q [B, H_q, d]; returns out [B, H_q, d]."""
    B, H_q = len(seq_ids), q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    shape = (B, H_q, cache.head_dim)
    keep_s, sp = _i32_array(seq_ids)
    _check(_lib.attn_decode(cache.handle, B, sp, H_q, _dev_ptr(q, "q", cache.torch_dtype, shape),
                            _dev_ptr(out, "out", cache.torch_dtype, shape),
                            _stream_handle(stream, cache.device_index)))
    return out


def attn_decode_tables(cache: Cache, block_table, lengths, q, out=None, stream=None):
    """Decode over caller-owned block tables: block_table is a device int32
    tensor [B, stride] of page ids of this cache's pool, lengths a host
    sequence of B lengths; q [B, H_q, d]."""
    B, H_q = len(lengths), q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if (not isinstance(block_table, torch.Tensor) or not block_table.is_cuda or block_table.dtype != torch.int32
            or block_table.dim() != 2 or block_table.shape[0] != B or not block_table.is_contiguous()):
        raise ValueError("block_table must be a contiguous CUDA int32 tensor [B, stride]")
    shape = (B, H_q, cache.head_dim)
    keep_l, lp = _i32_array(lengths)
    _check(_lib.attn_decode_tables(cache.handle, B, block_table.data_ptr(), block_table.shape[1], lp, H_q,
                                   _dev_ptr(q, "q", cache.torch_dtype, shape),
                                   _dev_ptr(out, "out", cache.torch_dtype, shape),
                                   _stream_handle(stream, cache.device_index)))
    return out


def attn_decode_append(cache: Cache, seq_ids, q, k_new, v_new, out=None, stream=None):
    """One decode step: append k_new, v_new [B, H_kv, d] at each sequence's
    tail and attend q [B, H_q, d] to the cache including them."""
    B, H_q = len(seq_ids), q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    shape = (B, H_q, cache.head_dim)
    kv_shape = (B, cache.num_kv_heads, cache.head_dim)
    keep_s, sp = _i32_array(seq_ids)
    _check(_lib.attn_decode_append(cache.handle, B, sp, H_q, _dev_ptr(q, "q", cache.torch_dtype, shape),
                                   _dev_ptr(k_new, "k_new", cache.torch_dtype, kv_shape),
                                   _dev_ptr(v_new, "v_new", cache.torch_dtype, kv_shape),
                                   _dev_ptr(out, "out", cache.torch_dtype, shape),
                            _stream_handle(stream, cache.device_index)))
    return out


def attn_decode_append_host(cache: Cache, seq_ids, q, k_new, v_new, out=None, stream=None):
    """attn_decode_append on host tensors (see include/gqa.h): q [B, H_q, d],
    k_new/v_new [B, H_kv, d] on the CPU (pinned for asynchronous copies);
    returns out [B, H_q, d] on the CPU (allocated like q if not given),
    complete once `stream` (default: the current stream) is synchronised."""
    B, H_q = len(seq_ids), q.shape[1]
    dt, d, H_kv = cache.torch_dtype, cache.head_dim, cache.num_kv_heads
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    keep_s, sp = _i32_array(seq_ids)
    _check(_lib.attn_decode_append_host(cache.handle, B, sp, H_q, _host_ptr(q, "q", dt, (B, H_q, d)),
                                        _host_ptr(k_new, "k_new", dt, (B, H_kv, d)),
                                        _host_ptr(v_new, "v_new", dt, (B, H_kv, d)),
                                        _host_ptr(out, "out", dt, (B, H_q, d)),
                                        _stream_handle(stream, cache.device_index)))
    return out


def attn_decode_append_meta(cache: Cache, seq_ids, H_q):
    keep_s, sp = _i32_array(seq_ids)
    _check(_lib.attn_decode_append(cache.handle, len(seq_ids), sp, H_q, None, None, None, None, None))


def attn_decode_static(cache: Cache, seq_ids, q, out=None, stream=None):
    """attn_decode without device allocation: the split-K partials live in
    the library's fixed static device array (see include/gqa.h)."""
    B, H_q = len(seq_ids), q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    shape = (B, H_q, cache.head_dim)
    keep_s, sp = _i32_array(seq_ids)
    _check(_lib.attn_decode_static(cache.handle, B, sp, H_q, _dev_ptr(q, "q", cache.torch_dtype, shape),
                                   _dev_ptr(out, "out", cache.torch_dtype, shape),
                            _stream_handle(stream, cache.device_index)))
    return out


def attn_decode_meta(cache: Cache, seq_ids, H_q):
    keep_s, sp = _i32_array(seq_ids)
    _check(_lib.attn_decode(cache.handle, len(seq_ids), sp, H_q, None, None, None))


def kv_truncate(cache: Cache, seq: int, m: int):
    _check(_lib.kv_truncate(cache.handle, seq, m))


def exported_symbols():
    """Names the header declares; used by the tests to check the exports."""
    return ["gqa_pool_bytes", "gqa_cache_create", "gqa_cache_destroy", "gqa_cache_layout",
            "gqa_layout_compatible", "gqa_seq_create", "gqa_seq_fork", "gqa_seq_free",
            "gqa_seq_length", "gqa_seq_block_table", "gqa_free_pages", "gqa_page_refcount",
            "attn_prefill", "kv_append", "attn_decode", "attn_decode_static", "kv_truncate", "gqa_cache_check",
            "gqa_profile_enable", "gqa_profile_read", "gqa_last_error", "gqa_version", "gqa_set_decode_kernel",
            "attn_decode_append", "gqa_selftest_bounded_wait", "attn_decode_tables", "attn_prefill_host",
            "attn_decode_append_host"]
