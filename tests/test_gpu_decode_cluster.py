"""GPU parity of the clustered decode kernel against the fp64 oracle.

The kernel serves single-token decode of small batches ("KV Cache 与
Prefill/Decode 推理路径", decode lesson: the new query reads every cached key,
its own included; PagedAttention: keys through the block table): each
(entry, KV head) is one thread-block cluster whose CTAs split its pages and
merge their partial (m, l, O) in distributed shared memory.  Cases: every
group size it serves (g = 1 .. 16), cluster sizes from 3 to 16 (powers of
two and not), descriptors in the launch parameters (up to 16 entries) and
in device memory (20 entries), ragged lengths from one token (so some
CTAs of a cluster hold no page) to past 8K, page-boundary lengths, the
wide-GQA decode at full size (every output element), sliding windows,
scores whose maximum grows by far more than 2^8 from page range to page
range (the cluster merge weighs ranges whose maxima are far apart), the
fused append (same bits as append then decode, cache bytes exact, with
copy-on-write after a fork), attn_decode_static (same bits), the automatic
choice (small batches only) and the rejections.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu

DT = "bf16"


def _filled(rng, H_kv, lengths, window=0, key_scale=None, spare=4, max_seqs=None):
    B, d = len(lengths), 128
    per_seq = workloads.pages_for(max(lengths) + spare) + 1
    pages = 2 * sum(workloads.pages_for(L + spare) for L in lengths) + 8
    c = gqa.Cache(H_kv, d, pages, max_seqs or B, per_seq, dtype=DT, window=window)
    m = oracle.CacheModel(pages, max_seqs or B, per_seq, H_kv, d, DT, window=window)
    ids = [c.seq_create() for _ in range(B)]
    mids = [m.create() for _ in range(B)]
    for b, L in enumerate(lengths):
        if key_scale is None:
            k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        else:
            k = workloads.bf16_bits(rng.standard_normal(size=(1, L, H_kv, d), dtype=np.float32) *
                                    key_scale(L)[None])
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        gqa.kv_append(c, [ids[b]], dev(k, DT), dev(v, DT))
        oracle.append(m, [mids[b]], k, v)
    return c, m, ids, mids


def _decode(c, ids, q, kernel="decode_cluster"):
    c.profile_read()
    o = gqa.attn_decode(c, ids, q)
    launched = c.profile_read()
    assert launched[kernel][0] == 1, launched
    return o


CASES = [
    (8, 8, [4097, 33, 1]),                # g = 1; a one-token sequence: 15 of 16 CTAs hold no page
    (16, 8, [15, 16, 17, 31, 32, 33]),    # g = 2; lengths around page boundaries
    (32, 8, [1, 17, 129, 2000, 5003]),    # g = 4, ragged
    (48, 8, [8300, 700]),                 # g = 6, long
    (64, 8, [3000]),                      # g = 8
    (12, 1, [9000, 257]),                 # g = 12, one KV head
    (128, 8, [700, 3000]),                # g = 16: every MMA row a head
    (8, 2, [40 * i + 3 for i in range(20)]),   # 20 entries: descriptors from device memory, clusters of 3
]


@pytest.mark.parametrize("H_q,H_kv,lengths", CASES)
def test_cluster_decode_matches_oracle(H_q, H_kv, lengths):
    rng = np.random.default_rng(300 + H_q + len(lengths))
    c, m, ids, mids = _filled(rng, H_kv, lengths)
    c.set_decode_kernel("cluster")
    q = workloads.normal_bf16(rng, (len(lengths), H_q, 128))
    o = _decode(c, ids, dev(q, DT))
    assert_close(host_f64(o, DT), oracle.decode(m, mids, q), DT, "cluster decode")
    s = gqa.attn_decode_static(c, ids, dev(q, DT))
    assert torch.equal(o.view(torch.int16), s.view(torch.int16)), "static decode differs"
    assert c.check() == 0


def test_wide_gqa_decode_full_size_every_element():
    # B = 1, H_q = 48, H_kv = 8 (g = 6), a 8192-token prefix and 16 decode
    # steps with the append fused: every output element of every step.
    H_q, H_kv, d, T = 48, 8, 128, 8192
    rng = np.random.default_rng(320)
    c, m, ids, mids = _filled(rng, H_kv, [T], spare=32)
    for step in range(16):
        q = workloads.normal_bf16(rng, (1, H_q, d))
        kn, vn = workloads.normal_bf16(rng, (1, H_kv, d)), workloads.normal_bf16(rng, (1, H_kv, d))
        c.profile_read()
        o = gqa.attn_decode_append(c, ids, dev(q, DT), dev(kn, DT), dev(vn, DT))
        launched = c.profile_read()
        assert launched["decode_cluster"][0] == 1 and launched["cache_write"][0] == 0, launched
        oracle.append(m, mids, kn, vn)
        assert_close(host_f64(o, DT), oracle.decode(m, mids, q), DT, "wide decode step %d" % step)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


@pytest.mark.parametrize("window", [1, 100, 1000])
def test_cluster_decode_with_window(window):
    rng = np.random.default_rng(330 + window)
    H_q, H_kv = 32, 8
    c, m, ids, mids = _filled(rng, H_kv, [6000, 250, 1800], window=window)
    c.set_decode_kernel("cluster")
    q = workloads.normal_bf16(rng, (3, H_q, 128))
    o = _decode(c, ids, dev(q, DT))
    assert_close(host_f64(o, DT), oracle.decode(m, mids, q), DT, "windowed cluster decode")
    assert c.check() == 0


@pytest.mark.parametrize("growing", [True, False])
def test_cluster_merge_with_far_apart_maxima(growing):
    # Keys grow (or shrink) in scale along the sequence, and q is scaled up:
    # the CTAs' maxima differ by far more than 2^8, and within a CTA the
    # running maximum jumps from page to page (or stays stale).
    H_q, H_kv, L = 16, 2, 6000
    rng = np.random.default_rng(340 + growing)

    def scale(n):
        t = np.arange(n) // 128
        s = 1.0 + 0.1 * (t if growing else t.max() - t)
        return s.astype(np.float32)[:, None, None]

    c, m, ids, mids = _filled(rng, H_kv, [L], key_scale=scale)
    c.set_decode_kernel("cluster")
    q = workloads.bf16_bits(rng.standard_normal(size=(1, H_q, 128), dtype=np.float32) * np.float32(6.0))
    o = _decode(c, ids, dev(q, DT))
    assert_close(host_f64(o, DT), oracle.decode(m, mids, q), DT, "cluster merge, far-apart maxima")
    assert c.check() == 0


def test_cluster_append_matches_append_then_decode_with_fork():
    # The fused append writes the same bits into the pool as kv_append and
    # gives the same output as kv_append + attn_decode on the same kernel;
    # a fork shares the tail page, so the first step copies it first.
    H_q, H_kv, d = 32, 4, 128
    rng = np.random.default_rng(350)
    lengths = [37, 1000, 16]
    res = []
    for fused in (True, False):
        r = np.random.default_rng(351)
        c, m, ids, mids = _filled(r, H_kv, lengths, spare=40, max_seqs=4)
        c.set_decode_kernel("cluster")
        f = c.seq_fork(ids[0], lengths[0])
        fm = m.fork(mids[0], lengths[0])
        ids2, mids2 = ids + [f], mids + [fm]
        outs = []
        for step in range(4):
            q = workloads.normal_bf16(r, (4, H_q, d))
            kn, vn = workloads.normal_bf16(r, (4, H_kv, d)), workloads.normal_bf16(r, (4, H_kv, d))
            if fused:
                o = gqa.attn_decode_append(c, ids2, dev(q, DT), dev(kn, DT), dev(vn, DT))
            else:
                gqa.kv_append(c, ids2, dev(kn[:, None], DT), dev(vn[:, None], DT))
                o = gqa.attn_decode(c, ids2, dev(q, DT))
            oracle.append(m, mids2, kn, vn)
            assert_close(host_f64(o, DT), oracle.decode(m, mids2, q), DT, "append step %d" % step)
            outs.append(o.view(torch.int16).cpu().numpy())
        assert_cache_matches(c, m, zip(ids2, mids2))
        assert c.check() == 0
        res.append(outs)
    for a, b in zip(*res):
        assert np.array_equal(a, b), "fused append differs from append + decode"


def test_automatic_choice_small_batches_only():
    rng = np.random.default_rng(360)
    H_q, H_kv = 32, 8
    c, m, ids, mids = _filled(rng, H_kv, [600] * 9)
    q = workloads.normal_bf16(rng, (9, H_q, 128))
    # 9 entries x 8 heads = 72 pairs <= half the SMs of a GB300: clustered.
    o = _decode(c, ids[:9], dev(q, DT), "decode_cluster")
    assert_close(host_f64(o, DT), oracle.decode(m, mids, q), DT, "auto, small batch")
    # The same call on the tensor-core kernel: same values within tolerance.
    c.set_decode_kernel("tensor_core")
    o2 = _decode(c, ids[:9], dev(q, DT), "prefill_tc")
    assert_close(host_f64(o2, DT), oracle.decode(m, mids, q), DT, "tensor-core")
    c.set_decode_kernel("auto")
    big = workloads.pages_for(40) * 100 + 8
    c2 = gqa.Cache(H_kv, 128, big, 100, 4, dtype=DT)
    s2 = [c2.seq_create() for _ in range(100)]
    z = dev(workloads.normal_bf16(rng, (100, 40, H_kv, 128)), DT)
    gqa.kv_append(c2, s2, z, z)
    # 100 x 8 = 800 pairs: the tensor-core kernel.
    _decode(c2, s2, dev(workloads.normal_bf16(rng, (100, H_q, 128)), DT), "prefill_tc")
    assert c.check() == 0 and c2.check() == 0


def test_cluster_rejections():
    rng = np.random.default_rng(370)
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 128, 8, 1, 4, dtype="bf16", rope=True).set_decode_kernel("cluster")
    assert e.value.name == "EINVAL"
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 64, 8, 1, 4, dtype="bf16").set_decode_kernel("cluster")
    assert e.value.name == "EINVAL"
    c, m, ids, mids = _filled(rng, 2, [100])
    c.set_decode_kernel("cluster")
    q = torch.zeros(1, 17 * 2 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gqa.GqaError) as e:                     # g = 17 > 16
        gqa.attn_decode(c, ids, q[:, : 17 * 2 * 128].view(1, 34, 128))
    assert e.value.name == "EINVAL"
    with pytest.raises(gqa.GqaError) as e:                     # q 2 bytes off a 16-byte boundary
        gqa.attn_decode(c, ids, q[:, 1: 1 + 4 * 2 * 128].view(1, 8, 128))
    assert e.value.name == "EINVAL"
    assert c.check() == 0


def _filled_fp8(rng, H_kv, lengths, window=0, zero_rows=False):
    B, d = len(lengths), 128
    per_seq = workloads.pages_for(max(lengths) + 4) + 1
    pages = 2 * sum(workloads.pages_for(L + 4) for L in lengths) + 8
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype="fp8", window=window)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, "fp8", window=window)
    ids, mids = [c.seq_create() for _ in range(B)], [m.create() for _ in range(B)]
    for b, L in enumerate(lengths):
        k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        if zero_rows:
            # rows of zeros: scale 0 and zero codes, in K and in V, including
            # every V row of the first pages (the value-scale maximum stays 0)
            k[0, ::7] = 0
            v[0, : min(L, 40)] = 0
            v[0, ::5] = 0
        gqa.kv_append(c, [ids[b]], dev(k, DT), dev(v, DT))
        oracle.append(m, [mids[b]], k, v)
    return c, m, ids, mids


FP8_CASES = [
    (32, 8, [1, 17, 300, 2049, 5000], 0, False),
    (48, 8, [8300], 0, False),             # the wide-GQA shape: clusters of 12
    (128, 8, [700, 3000], 0, False),       # g = 16
    (8, 8, [4097, 33], 0, True),           # g = 1, zero rows
    (32, 8, [6000, 250, 1800], 500, False),
    (24, 2, [40 * i + 9 for i in range(20)], 0, True),   # 20 entries: descriptors in device memory
]


@pytest.mark.parametrize("H_q,H_kv,lengths,window,zero_rows", FP8_CASES)
def test_cluster_decode_fp8_cache(H_q, H_kv, lengths, window, zero_rows):
    # The codes stream through the page ring as they are stored (half the
    # bytes of bf16); both products run on f16 mma.sync with the scales
    # applied to the scores and folded into P.  The automatic choice for an
    # FP8 cache with few (entry, KV head) pairs.
    rng = np.random.default_rng(380 + H_q + len(lengths) + window)
    c, m, ids, mids = _filled_fp8(rng, H_kv, lengths, window, zero_rows)
    q = workloads.normal_bf16(rng, (len(lengths), H_q, 128))
    o = _decode(c, ids, dev(q, DT))
    assert_close(host_f64(o, DT), oracle.decode(m, mids, q), DT, "fp8 cluster decode")
    s = gqa.attn_decode_static(c, ids, dev(q, DT))
    assert torch.equal(o.view(torch.int16), s.view(torch.int16)), "static decode differs"
    c.set_decode_kernel("cluster")
    o2 = _decode(c, ids, dev(q, DT))
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert c.check() == 0


def test_cluster_decode_fp8_large_scores():
    # q scaled by 40 and keys growing along the sequence: scores far from
    # N(0,1), the per-head power-of-two scaling of q and the key scales
    # carry the range.
    H_q, H_kv, L = 16, 2, 3000
    rng = np.random.default_rng(395)
    c = gqa.Cache(H_kv, 128, workloads.pages_for(L) + 8, 1, workloads.pages_for(L) + 1, dtype="fp8")
    m = oracle.CacheModel(workloads.pages_for(L) + 8, 1, workloads.pages_for(L) + 1, H_kv, 128, "fp8")
    s, ms = c.seq_create(), m.create()
    scale = (1.0 + 0.02 * (np.arange(L) // 16)).astype(np.float32)[:, None, None]
    k = workloads.bf16_bits(rng.standard_normal(size=(L, H_kv, 128), dtype=np.float32) * scale)
    v = workloads.normal_bf16(rng, (L, H_kv, 128))
    gqa.kv_append(c, [s], dev(k[None], DT), dev(v[None], DT))
    oracle.append(m, [ms], k[None], v[None])
    q = workloads.bf16_bits(rng.standard_normal(size=(1, H_q, 128), dtype=np.float32) * np.float32(40.0))
    o = _decode(c, [s], dev(q, DT))
    assert_close(host_f64(o, DT), oracle.decode(m, [ms], q), DT, "fp8 cluster decode, large scores")
    assert c.check() == 0
