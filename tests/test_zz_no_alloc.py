"""attn_decode_static: the decode entry point that allocates no device memory.

It exists for callers that must not allocate while decoding, such as a serving
loop that reserved its GPU memory up front, or a step that cannot pay for the
device-wide synchronisation of cudaFree.  Its split-K partials live in a fixed
static device array, not in a workspace the library grows with cudaMalloc.

The test calls it through the C ABI twice in a row, with the cache state and
the query changed in between, so the second call reuses a scratch array that
still holds the first call's contents.  Each result must be the same bits as
attn_decode, the allocating entry point, on the same state (same kernel, same
work split), on every decode kernel, and match the fp64 oracle within the
bf16 decode tolerance used elsewhere (max abs 2e-2, mean abs 2e-3).  A call
whose partials would not fit the array is refused with GQA_ERANGE and leaves
the output untouched.  The file name sorts last, so a run that stops at the
first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _call_static(cache, ids, q, out, expect=0):
    """Call attn_decode_static directly through ctypes (the C ABI)."""
    lib = ctypes.CDLL(gqa.LIB_PATH)
    fn = lib.attn_decode_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.gqa_last_error.restype = ctypes.c_char_p
    arr = (ctypes.c_int32 * len(ids))(*ids)
    rc = fn(cache.handle, len(ids), arr, q.shape[1], ctypes.c_void_p(q.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == expect, (rc, lib.gqa_last_error())
    return lib.gqa_last_error().decode()


def _compare(got, ref):
    g = got.float().cpu().numpy()
    r = ref.float().cpu().numpy()
    diff = np.abs(g - r)
    assert np.all(np.isfinite(g))
    assert diff.max() <= 2e-2 and diff.mean() <= 2e-3, (diff.max(), diff.mean())


@pytest.mark.parametrize("kernel", ["tensor_core", "cuda_core", "cluster"])
def test_static_decode_matches_allocating_decode_on_two_calls(kernel):
    H_kv, G, d = 4, 4, 128
    H_q = H_kv * G
    lengths = [1, 16, 17, 300, 2049]
    B = len(lengths)
    rng = np.random.default_rng(4242)
    pages = sum(workloads.pages_for(L + 2) for L in lengths) + 8
    order = rng.permutation(pages)
    cache = gqa.Cache(H_kv, d, pages, B, 256, dtype="bf16", page_order=order)
    cache.set_decode_kernel(kernel)
    model = oracle.CacheModel(pages, B, 256, H_kv, d, "bf16", page_order=order)
    ids = [cache.seq_create() for _ in range(B)]
    mids = [model.create() for _ in range(B)]
    n = max(lengths)
    k = np.zeros((B, n, H_kv, d), np.uint16)
    v = np.zeros((B, n, H_kv, d), np.uint16)
    for b, L in enumerate(lengths):
        k[b, :L] = workloads.normal_bf16(rng, (L, H_kv, d))
        v[b, :L] = workloads.normal_bf16(rng, (L, H_kv, d))
    gqa.kv_append(cache, ids, _dev(k), _dev(v), counts=lengths)
    oracle.append(model, mids, k, v, counts=lengths)

    for call in range(2):
        qh = workloads.normal_bf16(rng, (B, H_q, d))
        q = _dev(qh)
        ref = gqa.attn_decode(cache, ids, q)
        got = torch.full_like(q, float("nan"))
        _call_static(cache, ids, q, got)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), "not the same bits as attn_decode"
        _compare(got, torch.from_numpy(oracle.decode(model, mids, qh)).float())
        # Change the cache between the calls: one more token per sequence.
        knh, vnh = workloads.normal_bf16(rng, (B, H_kv, d)), workloads.normal_bf16(rng, (B, H_kv, d))
        gqa.kv_append(cache, ids, _dev(knh), _dev(vnh))
        oracle.append(model, mids, knh, vnh)
    assert cache.check() == 0


def test_static_decode_refuses_partials_beyond_the_array():
    # 1024 one-page sequences with H_kv = 8, g = 8 on the CUDA-core kernel:
    # 1024 chunks x 64 heads of partials (about 34 MB) exceed the 16 MiB
    # array.  The call is refused before anything is queued: the output keeps
    # its contents.
    H_kv, G, d, B = 8, 8, 128, 1024
    cache = gqa.Cache(H_kv, d, B + 8, B, 2, dtype="bf16")
    cache.set_decode_kernel("cuda_core")
    ids = [cache.seq_create() for _ in range(B)]
    zeros = _dev(np.zeros((B, 1, H_kv, d), np.uint16))
    gqa.kv_append(cache, ids, zeros, zeros)
    q = _dev(np.zeros((B, H_kv * G, d), np.uint16))
    out = torch.full_like(q, 3.0)
    msg = _call_static(cache, ids, q, out, expect=gqa.ERANGE)
    assert "partials" in msg
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    # attn_decode itself (a workspace that grows) serves the same call
    gqa.attn_decode(cache, ids, q, out=out)
    torch.cuda.synchronize()
    assert cache.check() == 0


def test_static_decode_rejects_unsupported_shapes():
    cache = gqa.Cache(1, 64, 8, 1, 4, dtype="bf16")
    s = cache.seq_create()
    gqa.kv_append(cache, [s], _dev(np.zeros((1, 1, 1, 64), np.uint16)), _dev(np.zeros((1, 1, 1, 64), np.uint16)))
    with pytest.raises(gqa.GqaError) as e:
        gqa.attn_decode_static(cache, [s], _dev(np.zeros((1, 2, 64), np.uint16)))
    assert e.value.name == "EINVAL"
