"""GPU parity of the rotary position mechanism (rope = 1 caches) against the
fp64 oracle: queries rotated inside the attention kernels, keys rotated when
written.  Outputs within the bf16 / fp32 tolerances; cached keys within one
bf16 step of the documented fp32 rounding rule (oracle.rope_stored_bf16);
values, lengths and block tables exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_close, dev, gather_seq, host_f64, raw_pool

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu

BASE = 10000.0


def _caches(B, H_kv, d, dt, pages, per_seq):
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype=dt, rope=True, rope_base=BASE)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, dt)
    return c, m, [c.seq_create() for _ in range(B)], [m.create() for _ in range(B)]


def _check_cache(c, m, ids, mids, dt):
    pool = raw_pool(c)
    for s, ms in zip(ids, mids):
        L = m.length(ms)
        assert c.seq_length(s) == L and c.block_table(s) == m.block_table(ms)
        K, V = gather_seq(pool, c.block_table(s), L)
        rk, rv = m.raw_kv(ms)
        assert np.array_equal(V, rv), "cached V differs"
        if dt == "bf16":
            want = oracle.to_f64(oracle.rope_stored_bf16(rk, np.arange(L), BASE), "bf16")
            got = oracle.to_f64(K, "bf16")
            step = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
            assert np.all(np.abs(got - want) <= step), "cached K further than one bf16 step from the rule"
        else:
            want = oracle.rope(oracle.to_f64(rk, "f32"), np.arange(L), BASE)
            assert np.max(np.abs(oracle.to_f64(K, "f32") - want)) <= 1e-5


@pytest.mark.parametrize("B,H_q,H_kv,n,lo,hi", [
    (3, 8, 2, 300, 100, 300),     # g = 4, several key tiles, ragged tails
    (2, 12, 2, 200, 150, 200),    # g = 6
])
def test_rope_bf16_prefill_tensor_core(B, H_q, H_kv, n, lo, hi):
    w = workloads.ragged_prefill(seed=300 + H_q, B=B, H_q=H_q, H_kv=H_kv, n=n, lo=lo, hi=hi)
    nb = w["valid_lengths"]
    pages = sum(workloads.pages_for(x) for x in nb) + 4
    c, m, ids, mids = _caches(B, H_kv, 128, "bf16", pages, workloads.pages_for(n) + 1)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"), nb),
                   "bf16")
    launched = c.profile_read()
    assert launched["prefill_tc"][0] == 1, launched
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], nb, rope_base=BASE)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], "bf16", "rope prefill")
    assert np.all(out[~mask] == 0)
    _check_cache(c, m, ids, mids, "bf16")
    assert c.check() == 0


def test_rope_bf16_incremental_prefill_then_decode():
    rng = np.random.default_rng(41)
    H_q, H_kv, d = 8, 2, 128
    P0, n1, steps = 200, 77, 5
    q0 = workloads.normal_bf16(rng, (1, P0, H_q, d))
    k0 = workloads.normal_bf16(rng, (1, P0, H_kv, d))
    v0 = workloads.normal_bf16(rng, (1, P0, H_kv, d))
    q1 = workloads.normal_bf16(rng, (1, n1, H_q, d))
    k1 = workloads.normal_bf16(rng, (1, n1, H_kv, d))
    v1 = workloads.normal_bf16(rng, (1, n1, H_kv, d))
    per_seq = workloads.pages_for(P0 + n1 + steps) + 1
    c, m, ids, mids = _caches(1, H_kv, d, "bf16", per_seq + 2, per_seq)
    gqa.attn_prefill(c, ids, dev(q0, "bf16"), dev(k0, "bf16"), dev(v0, "bf16"), [P0])
    oracle.prefill(m, mids, q0, k0, v0, [P0], rope_base=BASE)
    out = host_f64(gqa.attn_prefill(c, ids, dev(q1, "bf16"), dev(k1, "bf16"), dev(v1, "bf16"), [n1]), "bf16")
    ref = oracle.prefill(m, mids, q1, k1, v1, [n1], rope_base=BASE)
    assert_close(out, ref, "bf16", "incremental rope prefill")
    for t in range(steps):
        kt = workloads.normal_bf16(rng, (1, H_kv, d))
        vt = workloads.normal_bf16(rng, (1, H_kv, d))
        qt = workloads.normal_bf16(rng, (1, H_q, d))
        gqa.kv_append(c, ids, dev(kt, "bf16"), dev(vt, "bf16"))
        oracle.append(m, mids, kt, vt)
        o = host_f64(gqa.attn_decode(c, ids, dev(qt, "bf16")), "bf16")
        assert_close(o, oracle.decode(m, mids, qt, rope_base=BASE), "bf16", "rope decode %d" % t)
    _check_cache(c, m, ids, mids, "bf16")
    assert c.check() == 0


def test_rope_fp32_cuda_core_path():
    rng = np.random.default_rng(42)
    B, n, H_q, H_kv, d = 2, 37, 4, 2, 16
    q = rng.uniform(-1, 1, (B, n, H_q, d)).astype(np.float32)
    k = rng.uniform(-1, 1, (B, n, H_kv, d)).astype(np.float32)
    v = rng.uniform(-1, 1, (B, n, H_kv, d)).astype(np.float32)
    nb = [37, 20]
    c, m, ids, mids = _caches(B, H_kv, d, "f32", 16, 6)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(q, "f32"), dev(k, "f32"), dev(v, "f32"), nb), "f32")
    assert c.profile_read()["attn_simt"][0] == 1
    ref = oracle.prefill(m, mids, q, k, v, nb, rope_base=BASE)
    assert_close(out, ref, "f32", "rope fp32 prefill")
    qd = rng.uniform(-1, 1, (B, H_q, d)).astype(np.float32)
    kd = rng.uniform(-1, 1, (B, H_kv, d)).astype(np.float32)
    vd = rng.uniform(-1, 1, (B, H_kv, d)).astype(np.float32)
    gqa.kv_append(c, ids, dev(kd, "f32"), dev(vd, "f32"))
    oracle.append(m, mids, kd, vd)
    o = host_f64(gqa.attn_decode(c, ids, dev(qd, "f32")), "f32")
    assert_close(o, oracle.decode(m, mids, qd, rope_base=BASE), "f32", "rope fp32 decode")
    _check_cache(c, m, ids, mids, "f32")
    assert c.check() == 0


def test_rope_static_decode_matches_allocating_decode():
    rng = np.random.default_rng(43)
    B, H_q, H_kv, d, L = 3, 16, 4, 128, 600
    per_seq = workloads.pages_for(L + 1) + 1
    c = gqa.Cache(H_kv, d, B * per_seq, B, per_seq, dtype="bf16", rope=True, rope_base=BASE)
    ids = [c.seq_create() for _ in range(B)]
    k = workloads.normal_bf16(rng, (B, L, H_kv, d))
    v = workloads.normal_bf16(rng, (B, L, H_kv, d))
    gqa.kv_append(c, ids, dev(k, "bf16"), dev(v, "bf16"))
    q = dev(workloads.normal_bf16(rng, (B, H_q, d)), "bf16")
    a = gqa.attn_decode(c, ids, q)
    b = gqa.attn_decode_static(c, ids, q)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
