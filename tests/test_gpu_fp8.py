"""GPU parity of the quantised (FP8 E4M3) cache against the fp64 oracle:
the stored codes and per-row scales bit for bit (the cache write's rounding
decides integers, so both sides decide them in fp32 as the header states),
block tables and lengths exact, and attention outputs -- over the
dequantised values -- within the bf16 tolerance, on the CUDA-core kernels
and on the tensor-core kernel (which dequantises each tile into bf16
operands in shared memory)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _raw_rows(cache):
    """Codes [pages, 2, H_kv, 16, d] and scales [pages, 2, H_kv, 16] read back
    from the pool bytes with the documented layout (row bytes = d_h)."""
    d, H = cache.head_dim, cache.num_kv_heads
    C = -(-d // 128)
    raw = cache.pool.detach().cpu().numpy().view(np.uint8)
    nb = cache.num_pages * 2 * H * 16 * C * 128
    blocks = raw[:nb].reshape(cache.num_pages, 2, H, 16 * C * 128)
    s = np.arange(16)[:, None]
    b = np.arange(d)[None, :]
    off = ((s // 8) * C + b // 128) * 1024 + (s % 8) * 128 + b % 128
    codes = blocks[..., off]                                                # [P, 2, H, 16, d]
    scales = raw[nb: nb + cache.num_pages * 2 * H * 16 * 4].view(np.float32).reshape(cache.num_pages, 2, H, 16)
    return codes, scales


def _check_stored(c, m, pairs):
    codes, scales = _raw_rows(c)
    d = c.head_dim
    for s, ms in pairs:
        L = m.length(ms)
        table = c.block_table(s)
        assert c.seq_length(s) == L and table == m.block_table(ms)
        t = np.arange(L)
        pg = np.asarray(table)[t // 16]
        rk, rv = m.raw_kv(ms)
        for kv, raw in ((0, rk), (1, rv)):
            got_c = codes[pg, kv, :, t % 16, :]                              # [L, H, d]
            got_s = scales[pg, kv, :, t % 16]
            assert np.array_equal(got_c, raw[..., :d]), "stored codes differ"
            want_s = np.ascontiguousarray(raw[..., d:]).view(np.float32)[..., 0]
            assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), "stored scales differ"


def _caches(B, H_kv, d, pages, per_seq, max_seqs=None):
    c = gqa.Cache(H_kv, d, pages, max_seqs or B, per_seq, dtype="fp8")
    m = oracle.CacheModel(pages, max_seqs or B, per_seq, H_kv, d, "fp8")
    return c, m, [c.seq_create() for _ in range(B)], [m.create() for _ in range(B)]


@pytest.mark.parametrize("H_q,H_kv,d,n,nb", [
    (8, 2, 128, 70, [70, 33, 1]),
    (6, 3, 64, 40, [40, 17, 29]),
    (4, 2, 160, 37, [37, 20, 5]),        # a lane's bytes straddle the first 128-byte chunk
    (8, 8, 256, 24, [24, 9, 16]),
])
def test_fp8_prefill_codes_scales_and_outputs(H_q, H_kv, d, n, nb):
    rng = np.random.default_rng(110 + d)
    B = len(nb)
    q = workloads.normal_bf16(rng, (B, n, H_q, d))
    k = workloads.normal_bf16(rng, (B, n, H_kv, d))
    v = workloads.normal_bf16(rng, (B, n, H_kv, d))
    k[0, 3, 0] = 0                                           # a row of zeros: scale 0, zero codes
    c, m, ids, mids = _caches(B, H_kv, d, 32, 8)
    out = host_f64(gqa.attn_prefill(c, ids, dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), nb), "bf16")
    ref = oracle.prefill(m, mids, q, k, v, nb)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], "bf16", "fp8 prefill")
    assert np.all(out[~mask] == 0)
    _check_stored(c, m, list(zip(ids, mids)))
    assert c.check() == 0


def test_fp8_decode_steps_fork_and_fused_call():
    rng = np.random.default_rng(120)
    H_q, H_kv, d = 8, 2, 128
    c, m, ids, mids = _caches(2, H_kv, d, 40, 16, max_seqs=3)
    k = workloads.normal_bf16(rng, (2, 45, H_kv, d))
    v = workloads.normal_bf16(rng, (2, 45, H_kv, d))
    gqa.kv_append(c, ids, dev(k, "bf16"), dev(v, "bf16"), counts=[45, 30])
    oracle.append(m, mids, k, v, counts=[45, 30])
    f = c.seq_fork(ids[0], 37)                                # shares a partly filled page
    fm = m.fork(mids[0], 37)
    allids, allm = ids + [f], mids + [fm]
    for t in range(20):
        qt = workloads.normal_bf16(rng, (3, H_q, d))
        kt = workloads.normal_bf16(rng, (3, H_kv, d))
        vt = workloads.normal_bf16(rng, (3, H_kv, d))
        if t % 2:
            o = gqa.attn_decode_append(c, allids, dev(qt, "bf16"), dev(kt, "bf16"), dev(vt, "bf16"))
        else:
            gqa.kv_append(c, allids, dev(kt, "bf16"), dev(vt, "bf16"))
            o = gqa.attn_decode(c, allids, dev(qt, "bf16"))
        oracle.append(m, allm, kt, vt)
        assert_close(host_f64(o, "bf16"), oracle.decode(m, allm, qt), "bf16", "fp8 decode %d" % t)
    assert len(m.copies) >= 1
    _check_stored(c, m, list(zip(allids, allm)))
    assert c.check() == 0


@pytest.mark.parametrize("H_q,H_kv,lengths", [(32, 8, [1, 17, 300, 2049, 5000]), (8, 8, [4097, 33]), (64, 8, [700])])
def test_fp8_split_decode_kernel(H_q, H_kv, lengths):
    # bf16, d_h = 128, H_q/H_kv <= 8: the split-K CUDA-core decode kernel reads
    # the codes and scales directly (half the bytes of a bf16 cache).
    rng = np.random.default_rng(130 + H_q)
    B, d = len(lengths), 128
    pages = sum(workloads.pages_for(L) for L in lengths) + 4
    c, m, ids, mids = _caches(B, H_kv, d, pages, workloads.pages_for(max(lengths)) + 1)
    c.set_decode_kernel("cuda_core")
    for b, L in enumerate(lengths):
        k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        gqa.kv_append(c, [ids[b]], dev(k, "bf16"), dev(v, "bf16"))
        oracle.append(m, [mids[b]], k, v)
    q = workloads.normal_bf16(rng, (B, H_q, d))
    c.profile_read()
    o = gqa.attn_decode(c, ids, dev(q, "bf16"))
    launched = c.profile_read()
    assert launched["decode_split" if H_q // H_kv <= 8 else "attn_simt"][0] == 1, launched
    assert_close(host_f64(o, "bf16"), oracle.decode(m, mids, q), "bf16", "fp8 split decode")
    if H_q // H_kv <= 8:
        s = gqa.attn_decode_static(c, ids, dev(q, "bf16"))
        assert torch.equal(o.view(torch.int16), s.view(torch.int16))
    assert c.check() == 0


@pytest.mark.parametrize("H_q,H_kv,lengths,window", [
    (32, 8, [1, 17, 300, 2049, 5000], 0),
    (48, 8, [8300], 0),                  # one long sequence: key ranges split across SMs and merged
    (128, 8, [700, 3000], 0),            # g = 16
    (32, 8, [6000, 250, 1800], 500),
])
def test_fp8_tensor_core_decode(H_q, H_kv, lengths, window):
    rng = np.random.default_rng(140 + H_q + window)
    B, d = len(lengths), 128
    pages = sum(workloads.pages_for(L) for L in lengths) + 4
    per_seq = workloads.pages_for(max(lengths)) + 1
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype="fp8", window=window)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, "fp8", window=window)
    ids, mids = [c.seq_create() for _ in range(B)], [m.create() for _ in range(B)]
    c.set_decode_kernel("tensor_core")
    for b, L in enumerate(lengths):
        k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        gqa.kv_append(c, [ids[b]], dev(k, "bf16"), dev(v, "bf16"))
        oracle.append(m, [mids[b]], k, v)
    for t in range(3):
        q = workloads.normal_bf16(rng, (B, H_q, d))
        kt = workloads.normal_bf16(rng, (B, H_kv, d))
        vt = workloads.normal_bf16(rng, (B, H_kv, d))
        c.profile_read()
        o = gqa.attn_decode_append(c, ids, dev(q, "bf16"), dev(kt, "bf16"), dev(vt, "bf16"))
        launched = c.profile_read()
        assert launched["prefill_tc"][0] == 1 and launched["cache_write"][0] == 1, launched
        oracle.append(m, mids, kt, vt)
        assert_close(host_f64(o, "bf16"), oracle.decode(m, mids, q), "bf16", "fp8 tensor-core decode %d" % t)
        s = gqa.attn_decode_static(c, ids, dev(q, "bf16"))
        assert torch.equal(o.view(torch.int16), s.view(torch.int16))
    if window == 0:
        _check_stored(c, m, list(zip(ids, mids)))
    assert c.check() == 0


@pytest.mark.parametrize("B,H_q,H_kv,n,lo,hi", [
    (3, 32, 8, 300, 100, 300),
    (2, 16, 2, 520, 300, 520),
])
def test_fp8_tensor_core_prefill(B, H_q, H_kv, n, lo, hi):
    w = workloads.ragged_prefill(seed=150 + H_q, B=B, H_q=H_q, H_kv=H_kv, n=n, lo=lo, hi=hi)
    nb = w["valid_lengths"]
    pages = sum(workloads.pages_for(x) for x in nb) + 8
    c, m, ids, mids = _caches(B, H_kv, 128, pages, workloads.pages_for(n) + 1)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"), nb),
                   "bf16")
    assert c.profile_read()["prefill_tc"][0] == 1
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], nb)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], "bf16", "fp8 tensor-core prefill")
    assert np.all(out[~mask] == 0)
    _check_stored(c, m, list(zip(ids, mids)))
    # A second, incremental call reads the first call's codes.
    q2 = workloads.normal_bf16(np.random.default_rng(1), (B, 40, H_q, 128))
    k2 = workloads.normal_bf16(np.random.default_rng(2), (B, 40, H_kv, 128))
    v2 = workloads.normal_bf16(np.random.default_rng(3), (B, 40, H_kv, 128))
    o2 = host_f64(gqa.attn_prefill(c, ids, dev(q2, "bf16"), dev(k2, "bf16"), dev(v2, "bf16"), [40] * B), "bf16")
    assert_close(o2, oracle.prefill(m, mids, q2, k2, v2, [40] * B), "bf16", "fp8 incremental prefill")
    assert c.check() == 0
