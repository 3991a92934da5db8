"""GPU parity of the sliding window (window = W > 0 caches) against the fp64
oracle: a query at position p attends to keys max(0, p - W + 1)..p, and pages
whose positions all lie before the window are released after each write.
Outputs within the bf16 / fp32 tolerances; block tables (with their -1
entries), lengths, free-page counts and every held K/V value exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _caches(B, H_kv, d, dt, pages, per_seq, window, rope=False, max_seqs=None):
    c = gqa.Cache(H_kv, d, pages, max_seqs or B, per_seq, dtype=dt, window=window, rope=rope)
    m = oracle.CacheModel(pages, max_seqs or B, per_seq, H_kv, d, dt, window=window)
    return c, m, [c.seq_create() for _ in range(B)], [m.create() for _ in range(B)]


def _same_state(c, m, ids, mids):
    assert_cache_matches(c, m, list(zip(ids, mids)))
    assert c.free_pages() == m.free_pages()


@pytest.mark.parametrize("B,H_q,H_kv,n,lo,hi,W", [
    (3, 8, 2, 300, 100, 300, 100),    # g = 4 (32 positions per tile): window spans several tiles
    (2, 16, 2, 520, 300, 520, 129),   # g = 8: the window edge crosses a key tile inside an item
    (2, 8, 8, 400, 250, 400, 1),      # g = 1, W = 1: each position sees only itself
    (2, 12, 2, 200, 150, 200, 4096),  # g = 6, W beyond every length: plain causal
])
def test_window_bf16_prefill_tensor_core(B, H_q, H_kv, n, lo, hi, W):
    w = workloads.ragged_prefill(seed=500 + W, B=B, H_q=H_q, H_kv=H_kv, n=n, lo=lo, hi=hi)
    nb = w["valid_lengths"]
    pages = sum(workloads.pages_for(x) for x in nb) + 4
    c, m, ids, mids = _caches(B, H_kv, 128, "bf16", pages, workloads.pages_for(n) + 1, W)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"), nb),
                   "bf16")
    assert c.profile_read()["prefill_tc"][0] == 1
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], nb)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], "bf16", "window prefill W=%d" % W)
    assert np.all(out[~mask] == 0)
    _same_state(c, m, ids, mids)
    if W < 150:
        assert any(-1 in c.block_table(s) for s in ids)   # pages went back to the pool
    assert c.check() == 0


@pytest.mark.parametrize("rope", [False, True])
def test_window_incremental_prefill_then_decode(rope):
    # Prefill 400, then 77 more rows, then decode steps that cross page
    # boundaries, each releasing the page that leaves the window.
    rng = np.random.default_rng(61 + rope)
    H_q, H_kv, d, W = 16, 2, 128, 150
    P0, n1, steps = 400, 77, 20
    q0 = workloads.normal_bf16(rng, (2, P0, H_q, d))
    k0 = workloads.normal_bf16(rng, (2, P0, H_kv, d))
    v0 = workloads.normal_bf16(rng, (2, P0, H_kv, d))
    q1 = workloads.normal_bf16(rng, (2, n1, H_q, d))
    k1 = workloads.normal_bf16(rng, (2, n1, H_kv, d))
    v1 = workloads.normal_bf16(rng, (2, n1, H_kv, d))
    per_seq = workloads.pages_for(P0 + n1 + steps) + 1
    c, m, ids, mids = _caches(2, H_kv, d, "bf16", 2 * per_seq, per_seq, W, rope=rope)
    base = 10000.0 if rope else None
    nb0, nb1 = [P0, 333], [n1, 40]
    gqa.attn_prefill(c, ids, dev(q0, "bf16"), dev(k0, "bf16"), dev(v0, "bf16"), nb0)
    oracle.prefill(m, mids, q0, k0, v0, nb0, rope_base=base)
    if not rope:
        _same_state(c, m, ids, mids)
    out = host_f64(gqa.attn_prefill(c, ids, dev(q1, "bf16"), dev(k1, "bf16"), dev(v1, "bf16"), nb1), "bf16")
    ref = oracle.prefill(m, mids, q1, k1, v1, nb1, rope_base=base)
    mask = np.arange(n1)[None, :] < np.asarray(nb1)[:, None]
    assert_close(out[mask], ref[mask], "bf16", "incremental window prefill")
    for t in range(steps):
        kt = workloads.normal_bf16(rng, (2, H_kv, d))
        vt = workloads.normal_bf16(rng, (2, H_kv, d))
        qt = workloads.normal_bf16(rng, (2, H_q, d))
        gqa.kv_append(c, ids, dev(kt, "bf16"), dev(vt, "bf16"))
        oracle.append(m, mids, kt, vt)
        o = host_f64(gqa.attn_decode(c, ids, dev(qt, "bf16")), "bf16")
        assert_close(o, oracle.decode(m, mids, qt, rope_base=base), "bf16", "window decode %d" % t)
        s = gqa.attn_decode_static(c, ids, dev(qt, "bf16"))
        assert np.array_equal(host_f64(s, "bf16"), o)
    for s, ms in zip(ids, mids):
        assert c.block_table(s) == m.block_table(ms)
    assert c.free_pages() == m.free_pages()
    if not rope:
        _same_state(c, m, ids, mids)
    assert c.check() == 0


def test_window_decode_long_context_reads_only_the_window():
    # L = 3000 per sequence with W = 64: all but the last five pages are
    # released, so a decode that read outside the window would hit -1 pages.
    rng = np.random.default_rng(62)
    B, H_q, H_kv, d, L, W = 4, 32, 8, 128, 3000, 64
    per_seq = workloads.pages_for(L + 4) + 1
    c, m, ids, mids = _caches(B, H_kv, d, "bf16", B * 16, per_seq, W)
    for start in range(0, L, 100):                       # appends of 100 keep the pool small
        k = workloads.normal_bf16(rng, (B, 100, H_kv, d))
        v = workloads.normal_bf16(rng, (B, 100, H_kv, d))
        gqa.kv_append(c, ids, dev(k, "bf16"), dev(v, "bf16"))
        oracle.append(m, mids, k, v)
    _same_state(c, m, ids, mids)
    assert all(sum(p >= 0 for p in c.block_table(s)) <= 6 for s in ids)
    q = workloads.normal_bf16(rng, (B, H_q, d))
    o = host_f64(gqa.attn_decode(c, ids, dev(q, "bf16")), "bf16")
    assert_close(o, oracle.decode(m, mids, q), "bf16", "long-context window decode")
    assert c.check() == 0


def test_window_fp32_cuda_core_path():
    rng = np.random.default_rng(63)
    B, n, H_q, H_kv, d, W = 2, 70, 4, 2, 16, 19
    q = rng.uniform(-1, 1, (B, n, H_q, d)).astype(np.float32)
    k = rng.uniform(-1, 1, (B, n, H_kv, d)).astype(np.float32)
    v = rng.uniform(-1, 1, (B, n, H_kv, d)).astype(np.float32)
    nb = [70, 45]
    c, m, ids, mids = _caches(B, H_kv, d, "f32", 16, 8, W)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(q, "f32"), dev(k, "f32"), dev(v, "f32"), nb), "f32")
    assert c.profile_read()["attn_simt"][0] == 1
    ref = oracle.prefill(m, mids, q, k, v, nb)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], "f32", "window fp32 prefill")
    for t in range(20):
        qd = rng.uniform(-1, 1, (B, H_q, d)).astype(np.float32)
        kd = rng.uniform(-1, 1, (B, H_kv, d)).astype(np.float32)
        vd = rng.uniform(-1, 1, (B, H_kv, d)).astype(np.float32)
        gqa.kv_append(c, ids, dev(kd, "f32"), dev(vd, "f32"))
        oracle.append(m, mids, kd, vd)
        o = host_f64(gqa.attn_decode(c, ids, dev(qd, "f32")), "f32")
        assert_close(o, oracle.decode(m, mids, qd), "f32", "window fp32 decode %d" % t)
    _same_state(c, m, ids, mids)
    assert c.check() == 0


def test_window_fork_and_truncate_keep_what_the_window_needs():
    rng = np.random.default_rng(64)
    H_q, H_kv, d, W, L = 8, 2, 128, 40, 215     # pages 0..9 released: rewinds to m >= 200 allowed
    c, m, ids, mids = _caches(1, H_kv, d, "bf16", 40, 16, W, max_seqs=2)
    k = workloads.normal_bf16(rng, (1, L, H_kv, d))
    v = workloads.normal_bf16(rng, (1, L, H_kv, d))
    gqa.kv_append(c, ids, dev(k, "bf16"), dev(v, "bf16"))
    oracle.append(m, mids, k, v)
    held = next(j for j, p in enumerate(c.block_table(ids[0])) if p >= 0) * 16
    with pytest.raises(gqa.GqaError) as e:              # would need positions before `held`
        c.seq_fork(ids[0], held + W - 1)
    assert e.value.name == "ERANGE"
    with pytest.raises(gqa.GqaError) as e:
        gqa.kv_truncate(c, ids[0], held + W - 1)
    assert e.value.name == "ERANGE"
    f = c.seq_fork(ids[0], held + W + 5)
    fm = m.fork(mids[0], held + W + 5)
    gqa.kv_truncate(c, ids[0], held + W)
    m.truncate(mids[0], held + W)
    for s, ms in ((ids[0], mids[0]), (f, fm)):
        kt = workloads.normal_bf16(rng, (1, H_kv, d))
        vt = workloads.normal_bf16(rng, (1, H_kv, d))
        qt = workloads.normal_bf16(rng, (1, H_q, d))
        gqa.kv_append(c, [s], dev(kt, "bf16"), dev(vt, "bf16"))
        oracle.append(m, [ms], kt, vt)
        o = host_f64(gqa.attn_decode(c, [s], dev(qt, "bf16")), "bf16")
        assert_close(o, oracle.decode(m, [ms], qt), "bf16", "decode after rewind")
    _same_state(c, m, [ids[0], f], [mids[0], fm])
    assert c.check() == 0
