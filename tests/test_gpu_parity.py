"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Every case runs the same seeded inputs through the library and through the
oracle and compares: cache contents, lengths and block tables exactly;
outputs within max abs 1e-5 (fp32) or max abs 2e-2 / mean abs 2e-3 (bf16).
Sizes span several tiles and leave ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, host_f64, valid_mask

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _prefill_case(w, pages=None, per_seq=None, past=None):
    dt = w["dtype"]
    B, n, H_q, H_kv, d = w["B"], w["n"], w["H_q"], w["H_kv"], w["d"]
    nb = w["valid_lengths"]
    P = past if past is not None else [0] * B
    need = sum(workloads.pages_for(p + x) for p, x in zip(P, nb))
    pages = pages or need + 4
    per_seq = per_seq or max(workloads.pages_for(p + n) for p in P) + 1
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype=dt)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, dt)
    ids = [c.seq_create() for _ in range(B)]
    mids = [m.create() for _ in range(B)]
    return c, m, ids, mids


def test_worked_example_2d(golden):
    g = golden("worked_example_2d.txt")
    w = workloads.worked_example_2d()
    c, m, ids, mids = _prefill_case(w)
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "f32"), dev(w["k"], "f32"), dev(w["v"], "f32"),
                                    w["valid_lengths"]), "f32")[0, :, 0, :]
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], w["valid_lengths"])[0, :, 0, :]
    assert_close(out, ref, "f32", "worked example")
    assert np.all(np.abs(out[1] - np.array(g["out_pos2"])) <= 0.5e-5 + 1e-5)
    assert np.all(np.abs(out[0] - np.array(g["out_pos1"])) <= 1e-5)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_tiny_fp32_prefill_then_three_decode_steps():
    w = workloads.tiny_fp32()
    c, m, ids, mids = _prefill_case(w, pages=8, per_seq=4)
    out = gqa.attn_prefill(c, ids, dev(w["q"], "f32"), dev(w["k"], "f32"), dev(w["v"], "f32"), w["valid_lengths"])
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], w["valid_lengths"])
    assert_close(host_f64(out, "f32"), ref, "f32", "prefill")
    for t in range(3):
        gqa.kv_append(c, ids, dev(w["dec_k"][t], "f32"), dev(w["dec_v"][t], "f32"))
        oracle.append(m, mids, w["dec_k"][t], w["dec_v"][t])
        o = gqa.attn_decode(c, ids, dev(w["dec_q"][t], "f32"))
        assert c.seq_length(ids[0]) == 5 + t
        assert_close(host_f64(o, "f32"), oracle.decode(m, mids, w["dec_q"][t]), "f32", "decode %d" % t)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


@pytest.mark.parametrize("B,H_q,H_kv,n,lo,hi", [
    (3, 8, 2, 300, 100, 300),     # g = 4, several 128-key tiles, ragged tails
    (2, 6, 6, 129, 1, 129),       # MHA, one-row sequence allowed
    (2, 12, 2, 200, 150, 200),    # g = 6
    (1, 16, 2, 257, 257, 257),    # g = 8, all valid
])
def test_bf16_ragged_prefill(B, H_q, H_kv, n, lo, hi):
    w = workloads.ragged_prefill(seed=100 + H_q, B=B, H_q=H_q, H_kv=H_kv, n=n, lo=lo, hi=hi)
    c, m, ids, mids = _prefill_case(w)
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"),
                                    w["valid_lengths"]), "bf16")
    launched = c.profile_read()
    assert launched["prefill_tc"][0] == 1 and launched["attn_simt"][0] == 0, launched
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], w["valid_lengths"])
    mask = valid_mask(w["valid_lengths"], n)
    assert_close(out[mask], ref[mask], "bf16", "ragged prefill")
    assert np.all(out[~mask] == 0), "padding rows must be written as zeros"
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_fp32_head_dim_128_prefill():
    w = workloads.ragged_prefill(seed=5, B=2, H_q=4, H_kv=2, n=70, lo=20, hi=70, dtype="f32")
    c, m, ids, mids = _prefill_case(w)
    out = host_f64(gqa.attn_prefill(c, ids, dev(w["q"], "f32"), dev(w["k"], "f32"), dev(w["v"], "f32"),
                                    w["valid_lengths"]), "f32")
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], w["valid_lengths"])
    mask = valid_mask(w["valid_lengths"], 70)
    assert_close(out[mask], ref[mask], "f32", "fp32 prefill")
    assert_cache_matches(c, m, zip(ids, mids))


@pytest.mark.parametrize("G", [1, 2, 3, 4, 6, 8])
def test_bf16_decode_split_k(G):
    H_kv, d = 2, 128
    H_q = G * H_kv
    lengths = [1, 15, 16, 17, 700, 1601]
    B = len(lengths)
    rng = np.random.default_rng(200 + G)
    pages = sum(workloads.pages_for(L) for L in lengths) + 8
    order = rng.permutation(pages)
    c = gqa.Cache(H_kv, d, pages, B, 128, dtype="bf16", page_order=order)
    m = oracle.CacheModel(pages, B, 128, H_kv, d, "bf16", page_order=order)
    ids = [c.seq_create() for _ in range(B)]
    mids = [m.create() for _ in range(B)]
    hist = [workloads.normal_bf16(rng, (L - 1, H_kv, d)) for L in lengths]
    hv = [workloads.normal_bf16(rng, (L - 1, H_kv, d)) for L in lengths]
    n = max(lengths) - 1
    kpad = np.zeros((B, n, H_kv, d), np.uint16)
    vpad = np.zeros((B, n, H_kv, d), np.uint16)
    for b in range(B):
        kpad[b, : lengths[b] - 1] = hist[b]
        vpad[b, : lengths[b] - 1] = hv[b]
    counts = [L - 1 for L in lengths]
    gqa.kv_append(c, ids, dev(kpad, "bf16"), dev(vpad, "bf16"), counts=counts)
    oracle.append(m, mids, kpad, vpad, counts=counts)
    kn, vn = workloads.normal_bf16(rng, (B, H_kv, d)), workloads.normal_bf16(rng, (B, H_kv, d))
    q = workloads.normal_bf16(rng, (B, H_q, d))
    gqa.kv_append(c, ids, dev(kn, "bf16"), dev(vn, "bf16"))
    oracle.append(m, mids, kn, vn)
    out = host_f64(gqa.attn_decode(c, ids, dev(q, "bf16")), "bf16")
    assert_close(out, oracle.decode(m, mids, q), "bf16", "decode G=%d" % G)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_incremental_prefill_over_shared_unaligned_prefix():
    # A 37-token prefix (tail page shared and partly full) forked twice; each
    # fork runs an incremental prefill, which must copy the shared tail page
    # before writing into it, and attend to the whole prefix plus its own
    # lower triangle.
    rng = np.random.default_rng(31)
    H_q, H_kv, d, dt = 8, 2, 128, "bf16"
    c = gqa.Cache(H_kv, d, 64, 4, 16, dtype=dt)
    m = oracle.CacheModel(64, 4, 16, H_kv, d, dt)
    a, ma = c.seq_create(), m.create()
    pre = workloads.ragged_prefill(seed=32, B=1, H_q=H_q, H_kv=H_kv, n=37, lo=37, hi=37)
    gqa.attn_prefill(c, [a], dev(pre["q"], dt), dev(pre["k"], dt), dev(pre["v"], dt), [37])
    oracle.prefill(m, [ma], pre["q"], pre["k"], pre["v"], [37])
    kids = [(c.seq_fork(a, 37), m.fork(ma, 37)), (c.seq_fork(a, 30), m.fork(ma, 30))]
    new = workloads.ragged_prefill(seed=33, B=2, H_q=H_q, H_kv=H_kv, n=45, lo=20, hi=45)
    ids, mids = [x for x, _ in kids], [y for _, y in kids]
    positions = np.zeros((2, 45), np.int32)
    for b, (s, _) in enumerate(kids):
        positions[b] = c.seq_length(s) + np.arange(45)
    out = host_f64(gqa.attn_prefill(c, ids, dev(new["q"], dt), dev(new["k"], dt), dev(new["v"], dt),
                                    new["valid_lengths"], positions=positions), dt)
    ref = oracle.prefill(m, mids, new["q"], new["k"], new["v"], new["valid_lengths"])
    mask = valid_mask(new["valid_lengths"], 45)
    assert_close(out[mask], ref[mask], dt, "incremental prefill")
    assert len(m.copies) == 2
    assert_cache_matches(c, m, [(a, ma)] + kids)
    # One decode step on all three.
    allids, allm = [a] + ids, [ma] + mids
    kn, vn = workloads.normal_bf16(rng, (3, H_kv, d)), workloads.normal_bf16(rng, (3, H_kv, d))
    q = workloads.normal_bf16(rng, (3, H_q, d))
    gqa.kv_append(c, allids, dev(kn, dt), dev(vn, dt))
    oracle.append(m, allm, kn, vn)
    assert_close(host_f64(gqa.attn_decode(c, allids, dev(q, dt)), dt), oracle.decode(m, allm, q), dt, "decode")
    assert_cache_matches(c, m, zip(allids, allm))
    assert c.check() == 0


def test_padding_contents_are_bitwise_irrelevant():
    w = workloads.ragged_prefill(seed=41, B=3, H_q=8, H_kv=2, n=200, lo=50, hi=180)
    outs, pools = [], []
    for poison in (False, True):
        q, k, v = w["q"].copy(), w["k"].copy(), w["v"].copy()
        if poison:
            for b, nb in enumerate(w["valid_lengths"]):
                q[b, nb:] = 0x7FC0       # bf16 NaN
                k[b, nb:] = 0x7F80       # +inf
                v[b, nb:] = 0xFFC0       # NaN
        c = gqa.Cache(2, 128, 64, 3, 16, dtype="bf16")
        ids = [c.seq_create() for _ in range(3)]
        o = gqa.attn_prefill(c, ids, dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), w["valid_lengths"])
        outs.append(o.view(torch.int16).cpu().numpy())
        pools.append([c.block_table(s) for s in ids])
        assert c.check() == 0
    assert np.array_equal(outs[0], outs[1])
    assert pools[0] == pools[1]


def test_decode_equals_last_row_of_prefill():
    # The cached decode step reproduces the last row of recomputing the whole
    # context (the check the toy decoder runs after every step).
    L, H_q, H_kv, d, dt = 333, 16, 4, 128, "bf16"
    w = workloads.ragged_prefill(seed=51, B=1, H_q=H_q, H_kv=H_kv, n=L, lo=L, hi=L)
    c1 = gqa.Cache(H_kv, d, 32, 1, 32, dtype=dt)
    s1 = c1.seq_create()
    full = host_f64(gqa.attn_prefill(c1, [s1], dev(w["q"], dt), dev(w["k"], dt), dev(w["v"], dt), [L]), dt)
    c2 = gqa.Cache(H_kv, d, 32, 1, 32, dtype=dt)
    s2 = c2.seq_create()
    gqa.kv_append(c2, [s2], dev(w["k"], dt), dev(w["v"], dt))
    dec = host_f64(gqa.attn_decode(c2, [s2], dev(np.ascontiguousarray(w["q"][:, -1]), dt)), dt)
    m = oracle.CacheModel(32, 1, 32, H_kv, d, dt)
    ms = m.create()
    ref = oracle.prefill(m, [ms], w["q"], w["k"], w["v"], [L])
    assert_close(dec[0], ref[0, -1], dt, "decode")
    assert_close(full[0, -1], ref[0, -1], dt, "prefill last row")
    assert np.abs(dec[0] - full[0, -1]).max() <= 2 * 2e-2


@pytest.mark.parametrize("m_edit", [96, 100])
def test_edit_at_m_keeps_rows_and_cache_before_m(m_edit):
    # Edit at token m: a full re-prefill of the edited sequence gives output
    # rows < m bit-identical to the original run; truncating at m and
    # re-prefilling the suffix keeps the cached K/V < m bit-identical and
    # matches the oracle.
    n, H_q, H_kv, d, dt = 260, 8, 2, 128, "bf16"
    w = workloads.ragged_prefill(seed=61, B=1, H_q=H_q, H_kv=H_kv, n=n, lo=n, hi=n)
    rng = np.random.default_rng(62)
    e = {x: w[x].copy() for x in ("q", "k", "v")}
    for x, H in (("q", H_q), ("k", H_kv), ("v", H_kv)):
        e[x][0, m_edit:] = workloads.normal_bf16(rng, (n - m_edit, H, d))

    def full(q, k, v):
        c = gqa.Cache(H_kv, d, 32, 1, 32, dtype=dt)
        s = c.seq_create()
        o = gqa.attn_prefill(c, [s], dev(q, dt), dev(k, dt), dev(v, dt), [n])
        return c, s, o.view(torch.int16).cpu().numpy()

    c0, s0, o0 = full(w["q"], w["k"], w["v"])
    _, _, o1 = full(e["q"], e["k"], e["v"])
    assert np.array_equal(o0[0, :m_edit], o1[0, :m_edit])
    assert not np.array_equal(o0[0, m_edit:], o1[0, m_edit:])

    from _helpers import gather_seq, raw_pool
    before = gather_seq(raw_pool(c0), c0.block_table(s0), m_edit)
    gqa.kv_truncate(c0, s0, m_edit)
    assert c0.seq_length(s0) == m_edit
    suffix = {x: np.ascontiguousarray(e[x][:, m_edit:]) for x in e}
    o2 = host_f64(gqa.attn_prefill(c0, [s0], dev(suffix["q"], dt), dev(suffix["k"], dt), dev(suffix["v"], dt),
                                   [n - m_edit]), dt)
    after = gather_seq(raw_pool(c0), c0.block_table(s0), m_edit)
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    mm = oracle.CacheModel(32, 1, 32, H_kv, d, dt)
    ms = mm.create()
    ref = oracle.prefill(mm, [ms], e["q"], e["k"], e["v"], [n])
    assert_close(o2[0], ref[0, m_edit:], dt, "re-prefill")
    assert_cache_matches(c0, mm, [(s0, ms)])
    assert c0.check() == 0
