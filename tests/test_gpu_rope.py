"""GPU parity of the rotary position mechanism (rope = 1 caches) against the
fp64 oracle: queries rotated inside the attention kernels; keys rotated when
written (post-position caches) or stored as given and rotated when read
(pre-position caches).  Outputs within the bf16 / fp32 tolerances; cached
post-position keys within one bf16 step of the documented fp32 rounding
rule (oracle.rope_stored_bf16), pre-position keys equal to the input bytes;
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


def test_rope_bf16_multi_token_chunks():
    # Draft chunks of up to 4 rows over a rotary cache whose lengths are not
    # on a page boundary: the new keys are rotated by their positions as
    # written, and cache and outputs follow the oracle.
    rng = np.random.default_rng(43)
    B, H_q, H_kv, d, n = 2, 8, 2, 128, 4
    P0 = [203, 90]
    per_seq = workloads.pages_for(max(P0) + 3 * n) + 1
    c, m, ids, mids = _caches(B, H_kv, d, "bf16", B * per_seq + 2, per_seq)
    for b in range(B):
        q0 = workloads.normal_bf16(rng, (1, P0[b], H_q, d))
        k0 = workloads.normal_bf16(rng, (1, P0[b], H_kv, d))
        v0 = workloads.normal_bf16(rng, (1, P0[b], H_kv, d))
        gqa.attn_prefill(c, [ids[b]], dev(q0, "bf16"), dev(k0, "bf16"), dev(v0, "bf16"), [P0[b]])
        oracle.prefill(m, [mids[b]], q0, k0, v0, [P0[b]], rope_base=BASE)
    for T in ([3, 4], [4, 1], [2, 4]):
        q = workloads.normal_bf16(rng, (B, n, H_q, d))
        k = workloads.normal_bf16(rng, (B, n, H_kv, d))
        v = workloads.normal_bf16(rng, (B, n, H_kv, d))
        c.profile_read()
        got = host_f64(gqa.attn_prefill(c, ids, dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), T), "bf16")
        launched = c.profile_read()
        assert launched["prefill_tc"][0] == 1, launched
        ref = oracle.prefill(m, mids, q, k, v, T, rope_base=BASE)
        mask = np.arange(n)[None, :] < np.asarray(T)[:, None]
        assert np.all(got[~mask] == 0)
        assert_close(got[mask], ref[mask], "bf16", "rope multi-token chunk %s" % T)
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


# ---- pre-position caches: keys stored as given, rotated when read ----------
# ([P1] 2.5: layout_metadata records keys taken before the position
# transform.)  Prefill of a bf16, d_h = 128 cache rotates every page the call
# reads into a scratch copy that the tensor-core kernel reads; other shapes
# run the CUDA-core prefill, and decode the split-K kernel, both rotating
# each key as they load it.  The cached keys and values must be the input
# bytes exactly.

def _pre_caches(B, H_kv, d, dt, pages, per_seq, window=0, max_seqs=None):
    ms = max_seqs or B
    c = gqa.Cache(H_kv, d, pages, ms, per_seq, dtype=dt, rope=True, rope_base=BASE, keys_post_position=0,
                  window=window)
    m = oracle.CacheModel(pages, ms, per_seq, H_kv, d, dt, window=window)
    return c, m, [c.seq_create() for _ in range(B)], [m.create() for _ in range(B)]


@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (16, 2)])
def test_pre_position_prefill_and_decode_kernels(H_q, H_kv):
    from _helpers import assert_cache_matches
    B, n, d = 3, 150, 128
    w = workloads.ragged_prefill(seed=330 + H_q, B=B, H_q=H_q, H_kv=H_kv, n=n, lo=60, hi=n)
    nb = w["valid_lengths"]
    per_seq = workloads.pages_for(n + 8) + 1
    c, m, ids, mids = _pre_caches(B, H_kv, d, "bf16", B * per_seq, per_seq)
    assert c.layout().keys_post_position == 0
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"), nb),
                   "bf16")
    launched = c.profile_read()
    assert launched["rotate_pages"][0] == 1 and launched["prefill_tc"][0] == 1, launched
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], nb, rope_base=BASE)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], "bf16", "pre-position prefill")
    assert np.all(out[~mask] == 0)
    assert_cache_matches(c, m, zip(ids, mids))            # stored keys are the input bytes
    with pytest.raises(gqa.GqaError) as e:
        c.set_decode_kernel("tensor_core")
    assert e.value.name == "EINVAL"
    rng = np.random.default_rng(331)
    for t, kernel in enumerate(["auto", "cuda_core", "auto"]):
        c.set_decode_kernel(kernel)
        kt, vt = workloads.normal_bf16(rng, (B, H_kv, d)), workloads.normal_bf16(rng, (B, H_kv, d))
        qt = workloads.normal_bf16(rng, (B, H_q, d))
        c.profile_read()
        o = host_f64(gqa.attn_decode_append(c, ids, dev(qt, "bf16"), dev(kt, "bf16"), dev(vt, "bf16")), "bf16")
        launched = c.profile_read()
        assert launched["prefill_tc"][0] == 0, launched
        assert launched["decode_split" if H_q // H_kv <= 8 else "attn_simt"][0] == 1, launched
        oracle.append(m, mids, kt, vt)
        assert_close(o, oracle.decode(m, mids, qt, rope_base=BASE), "bf16", "pre-position decode %d" % t)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_pre_position_incremental_prefill_window_and_static_decode():
    from _helpers import assert_cache_matches
    rng = np.random.default_rng(340)
    H_q, H_kv, d, W = 8, 2, 128, 100
    P0, n1 = 230, 45
    per_seq = workloads.pages_for(P0 + n1 + 4) + 1
    for window in (0, W):
        c, m, ids, mids = _pre_caches(1, H_kv, d, "bf16", per_seq + 2, per_seq, window=window)
        q0, k0, v0 = (workloads.normal_bf16(rng, (1, P0, H, d)) for H in (H_q, H_kv, H_kv))
        q1, k1, v1 = (workloads.normal_bf16(rng, (1, n1, H, d)) for H in (H_q, H_kv, H_kv))
        gqa.attn_prefill(c, ids, dev(q0, "bf16"), dev(k0, "bf16"), dev(v0, "bf16"), [P0])
        oracle.prefill(m, mids, q0, k0, v0, [P0], rope_base=BASE)
        out = host_f64(gqa.attn_prefill(c, ids, dev(q1, "bf16"), dev(k1, "bf16"), dev(v1, "bf16"), [n1]), "bf16")
        ref = oracle.prefill(m, mids, q1, k1, v1, [n1], rope_base=BASE)
        assert_close(out, ref, "bf16", "pre-position incremental prefill, window %d" % window)
        assert_cache_matches(c, m, zip(ids, mids))
        qt = dev(workloads.normal_bf16(rng, (1, H_q, d)), "bf16")
        a = gqa.attn_decode(c, ids, qt)
        b = gqa.attn_decode_static(c, ids, qt)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        ref = oracle.decode(m, mids, qt.view(torch.int16).cpu().numpy().view(np.uint16), rope_base=BASE)
        assert_close(host_f64(a, "bf16"), ref, "bf16", "pre-position decode, window %d" % window)
        assert c.check() == 0


@pytest.mark.parametrize("dt,d", [("f32", 16), ("bf16", 64)])
def test_pre_position_cuda_core_prefill(dt, d):
    from _helpers import assert_cache_matches
    rng = np.random.default_rng(350 + d)
    B, n, H_q, H_kv = 2, 41, 4, 2
    q, k, v = (workloads.draw(rng, dt, (B, n, H, d)) for H in (H_q, H_kv, H_kv))
    nb = [41, 19]
    c, m, ids, mids = _pre_caches(B, H_kv, d, dt, 16, 6)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(q, dt), dev(k, dt), dev(v, dt), nb), dt)
    assert c.profile_read()["attn_simt"][0] == 1
    ref = oracle.prefill(m, mids, q, k, v, nb, rope_base=BASE)
    mask = np.arange(n)[None, :] < np.asarray(nb)[:, None]
    assert_close(out[mask], ref[mask], dt, "pre-position CUDA-core prefill")
    qd, kd, vd = (workloads.draw(rng, dt, (B, H, d)) for H in (H_q, H_kv, H_kv))
    gqa.kv_append(c, ids, dev(kd, dt), dev(vd, dt))
    oracle.append(m, mids, kd, vd)
    o = host_f64(gqa.attn_decode(c, ids, dev(qd, dt)), dt)
    assert_close(o, oracle.decode(m, mids, qd, rope_base=BASE), dt, "pre-position CUDA-core decode")
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_pre_position_forks_share_rotated_prefix():
    # A 300-token prefix shared by three forks (tail page shared and partly
    # full); each fork prefills its own rows: the prefix pages are rotated
    # once per call and read by every fork's items.
    from _helpers import assert_cache_matches
    rng = np.random.default_rng(360)
    H_q, H_kv, d, P0 = 16, 4, 128, 300
    per_seq = workloads.pages_for(P0 + 80) + 1
    c, m, ids, mids = _pre_caches(1, H_kv, d, "bf16", 4 * per_seq, per_seq, max_seqs=4)
    pre = workloads.ragged_prefill(seed=361, B=1, H_q=H_q, H_kv=H_kv, n=P0, lo=P0, hi=P0)
    gqa.attn_prefill(c, ids, dev(pre["q"], "bf16"), dev(pre["k"], "bf16"), dev(pre["v"], "bf16"), [P0])
    oracle.prefill(m, mids, pre["q"], pre["k"], pre["v"], [P0], rope_base=BASE)
    forks = [c.seq_fork(ids[0], P0) for _ in range(3)]
    mforks = [m.fork(mids[0], P0) for _ in range(3)]
    new = workloads.ragged_prefill(seed=362, B=3, H_q=H_q, H_kv=H_kv, n=80, lo=20, hi=80)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, forks, dev(new["q"], "bf16"), dev(new["k"], "bf16"), dev(new["v"], "bf16"),
                                    new["valid_lengths"]), "bf16")
    assert c.profile_read()["rotate_pages"][0] == 1
    ref = oracle.prefill(m, mforks, new["q"], new["k"], new["v"], new["valid_lengths"], rope_base=BASE)
    mask = np.arange(80)[None, :] < np.asarray(new["valid_lengths"])[:, None]
    assert_close(out[mask], ref[mask], "bf16", "pre-position forks")
    assert_cache_matches(c, m, list(zip(forks, mforks)) + [(ids[0], mids[0])])
    assert c.check() == 0
