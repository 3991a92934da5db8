"""The cache write fused into the tensor-core prefill.

"第二章 Prefill：整层状态演化与 KV 建立", section 2.6: a prefill writes each
valid position's K/V into the cache and attends over it; a fused kernel may
do both as long as the results are those of the plain sequence.  When every
batch entry starts on a page boundary (and n is a multiple of 8) the
tensor-core kernel reads the call's rows straight from k and v and stores
each new page itself; otherwise a cache-write launch precedes it.  Both
paths run the same attention arithmetic over the same values, so they must
give the same bits, and both must match the fp64 oracle and its cache model
exactly (cache bytes) or within the bf16 tolerance (outputs).

Cases: a fresh ragged batch with every query-tile shape (g = 1, 4, 6, 16,
32); incremental prefills over prefixes of 16, 48, 128 and 2000 tokens (a
key tile split between old pages and new rows); entries with different
prefixes in one call; a window; split items (few rows over a long prefix);
NaN/Inf in the padding rows; and the host-buffer entry point.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, gather_seq, host_f64, raw_pool, valid_mask

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu

DT = "bf16"


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _run(w, n, past_rows=None, window=0):
    """Prefill w's rows (padded to n) into a fresh cache after optional
    prefixes past_rows[b] = (k, v) bits [P_b, H_kv, d]; returns the cache,
    its sequence ids, out bits and the launch counts of the prefill."""
    B, H_q, H_kv, d = w["B"], w["H_q"], w["H_kv"], w["d"]
    nb = [int(x) for x in w["valid_lengths"]]
    P = [0 if past_rows is None else past_rows[b][0].shape[0] for b in range(B)]
    per_seq = max(workloads.pages_for(p + n) for p in P) + 1
    pages = sum(workloads.pages_for(p + n) for p in P) + 8
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype=DT, window=window)
    ids = [c.seq_create() for _ in range(B)]
    for b in range(B):
        if P[b]:
            gqa.kv_append(c, [ids[b]], dev(past_rows[b][0][None], DT), dev(past_rows[b][1][None], DT))
    q = np.zeros((B, n, H_q, d), np.uint16)
    k = np.zeros((B, n, H_kv, d), np.uint16)
    v = np.zeros((B, n, H_kv, d), np.uint16)
    m = min(n, w["n"])
    q[:, :m], k[:, :m], v[:, :m] = w["q"][:, :m], w["k"][:, :m], w["v"][:, :m]
    torch.cuda.synchronize()
    c.profile_read()
    out = gqa.attn_prefill(c, ids, dev(q, DT), dev(k, DT), dev(v, DT), nb)
    launched = c.profile_read()
    assert c.check() == 0
    return c, ids, out, launched


def _oracle(w, past_rows=None, window=0, pages=4096):
    B, H_q, H_kv, d = w["B"], w["H_q"], w["H_kv"], w["d"]
    m = oracle.CacheModel(pages, B, 512, H_kv, d, DT, window=window)
    mids = [m.create() for _ in range(B)]
    for b in range(B):
        if past_rows is not None and past_rows[b][0].shape[0]:
            m.write([mids[b]], [past_rows[b][0]], [past_rows[b][1]])
    ref = oracle.prefill(m, mids, w["q"], w["k"], w["v"], w["valid_lengths"])
    return m, mids, ref


@pytest.mark.parametrize("H_q,H_kv,n,lo,hi", [
    (8, 8, 264, 1, 264),      # g = 1: an item spans two key tiles
    (8, 2, 392, 100, 392),    # g = 4
    (12, 2, 208, 150, 208),   # g = 6: 21 positions per query tile
    (32, 2, 136, 40, 136),    # g = 16: an item covers one page
    (64, 2, 96, 33, 96),      # g = 32: a page spans two items
])
def test_fused_fresh_prefill_matches_unfused_and_oracle(H_q, H_kv, n, lo, hi):
    w = workloads.ragged_prefill(seed=700 + H_q, B=3, H_q=H_q, H_kv=H_kv, n=n, lo=lo, hi=hi)
    c1, ids1, o1, l1 = _run(w, n)                 # n % 8 == 0: fused
    c2, ids2, o2, l2 = _run(w, n + 1)             # n % 8 != 0: cache write, then attention
    assert l1["cache_write"][0] == 0 and l1["prefill_tc"][0] == 1, l1
    assert l2["cache_write"][0] == 1 and l2["prefill_tc"][0] == 1, l2
    b1, b2 = _bits(o1), _bits(o2)
    assert np.array_equal(b1, b2[:, :n]), "fused and unfused prefill differ"
    m, mids, ref = _oracle(w)
    mask = valid_mask(w["valid_lengths"], n)
    out = host_f64(o1, DT)
    assert_close(out[mask], ref[mask], DT, "fused prefill")
    assert np.all(b1[~mask] == 0), "padding rows must be written as zeros"
    assert_cache_matches(c1, m, zip(ids1, mids))
    assert_cache_matches(c2, m, zip(ids2, mids))


@pytest.mark.parametrize("prefix", [16, 48, 128, 2000])
def test_fused_incremental_prefill_over_page_aligned_prefix(prefix):
    # prefix 48 and 2000: the first new key tile holds old pages (from the
    # pool) and new pages (from k and v).
    H_q, H_kv, d, n = 16, 4, 128, 200
    rng = np.random.default_rng(710 + prefix)
    w = workloads.ragged_prefill(seed=720 + prefix, B=2, H_q=H_q, H_kv=H_kv, n=n, lo=60, hi=n)
    past = [(workloads.normal_bf16(rng, (prefix, H_kv, d)), workloads.normal_bf16(rng, (prefix, H_kv, d)))
            for _ in range(2)]
    c1, ids1, o1, l1 = _run(w, n, past)
    c2, ids2, o2, l2 = _run(w, n + 3, past)
    assert l1["cache_write"][0] == 0 and l2["cache_write"][0] == 1
    assert np.array_equal(_bits(o1), _bits(o2)[:, :n])
    m, mids, ref = _oracle(w, past)
    mask = valid_mask(w["valid_lengths"], n)
    assert_close(host_f64(o1, DT)[mask], ref[mask], DT, "incremental fused prefill")
    assert_cache_matches(c1, m, zip(ids1, mids))
    assert_cache_matches(c2, m, zip(ids2, mids))


def test_fused_entries_with_different_prefixes_and_window():
    H_q, H_kv, d, n = 8, 2, 128, 320
    rng = np.random.default_rng(731)
    w = workloads.ragged_prefill(seed=732, B=3, H_q=H_q, H_kv=H_kv, n=n, lo=90, hi=n)
    past = [(workloads.normal_bf16(rng, (P, H_kv, d)), workloads.normal_bf16(rng, (P, H_kv, d)))
            for P in (0, 32, 400)]
    for window in (0, 100):
        c1, ids1, o1, l1 = _run(w, n, past, window=window)
        c2, ids2, o2, l2 = _run(w, n + 5, past, window=window)
        assert l1["cache_write"][0] == 0 and l2["cache_write"][0] == 1
        assert np.array_equal(_bits(o1), _bits(o2)[:, :n])
        m, mids, ref = _oracle(w, past, window=window)
        mask = valid_mask(w["valid_lengths"], n)
        assert_close(host_f64(o1, DT)[mask], ref[mask], DT, "window %d" % window)
        assert_cache_matches(c1, m, zip(ids1, mids))


def test_fused_split_items_few_rows_over_long_prefix():
    # Five new rows over a 4096-token prefix, one entry: the items are split
    # along the key tiles and merged in the kernel; rows 5..15 of out are
    # zeroed by the kernel.
    H_q, H_kv, d, n = 32, 8, 128, 16
    rng = np.random.default_rng(741)
    w = workloads.ragged_prefill(seed=742, B=1, H_q=H_q, H_kv=H_kv, n=n, lo=5, hi=5)
    past = [(workloads.normal_bf16(rng, (4096, H_kv, d)), workloads.normal_bf16(rng, (4096, H_kv, d)))]
    c1, ids1, o1, l1 = _run(w, n, past)
    c2, ids2, o2, l2 = _run(w, n + 1, past)
    assert l1["cache_write"][0] == 0 and l2["cache_write"][0] == 1
    b1 = _bits(o1)
    assert np.array_equal(b1, _bits(o2)[:, :n])
    assert np.all(b1[0, 5:] == 0)
    m, mids, ref = _oracle(w, past)
    assert_close(host_f64(o1, DT)[0, :5], ref[0, :5], DT, "split fused prefill")
    assert_cache_matches(c1, m, zip(ids1, mids))


def test_fused_padding_rows_never_reach_cache_or_outputs():
    # NaN / Inf in every padding row: outputs, cache contents and the unused
    # slots of each sequence's last page are what they are with zeros there.
    w = workloads.ragged_prefill(seed=751, B=3, H_q=8, H_kv=2, n=264, lo=17, hi=250)
    nb = [int(x) for x in w["valid_lengths"]]
    res = []
    for poison in (False, True):
        q, k, v = w["q"].copy(), w["k"].copy(), w["v"].copy()
        if poison:
            for b, x in enumerate(nb):
                q[b, x:] = 0x7FC0
                k[b, x:] = 0x7F80
                v[b, x:] = 0xFFC0
        c = gqa.Cache(2, 128, 64, 3, 20, dtype=DT)
        ids = [c.seq_create() for _ in range(3)]
        c.profile_read()
        o = gqa.attn_prefill(c, ids, dev(q, DT), dev(k, DT), dev(v, DT), nb)
        assert c.profile_read()["cache_write"][0] == 0
        assert c.check() == 0
        pool = raw_pool(c)
        tails = []
        for b, s in enumerate(ids):
            tab = c.block_table(s)
            full_k, full_v = gather_seq(pool, tab, 16 * len(tab))
            assert np.all(np.isfinite(oracle.to_f64(full_k, DT))) and np.all(np.isfinite(oracle.to_f64(full_v, DT)))
            tails.append((full_k[nb[b]:], full_v[nb[b]:]))
        res.append((_bits(o), [c.block_table(s) for s in ids], tails))
    assert np.array_equal(res[0][0], res[1][0])
    assert res[0][1] == res[1][1]
    for (k0, v0), (k1, v1) in zip(res[0][2], res[1][2]):
        assert np.array_equal(k0, k1) and np.array_equal(v0, v1)


def test_fused_then_decode_reads_the_written_pages():
    # The pages the fused prefill stored are what later decode steps read.
    H_q, H_kv, d, n = 16, 2, 128, 520
    w = workloads.ragged_prefill(seed=761, B=2, H_q=H_q, H_kv=H_kv, n=n, lo=300, hi=n)
    c, ids, o, l = _run(w, n)
    assert l["cache_write"][0] == 0
    m, mids, _ = _oracle(w)
    rng = np.random.default_rng(762)
    for t in range(3):
        kn, vn = workloads.normal_bf16(rng, (2, H_kv, d)), workloads.normal_bf16(rng, (2, H_kv, d))
        q = workloads.normal_bf16(rng, (2, H_q, d))
        got = host_f64(gqa.attn_decode_append(c, ids, dev(q, DT), dev(kn, DT), dev(vn, DT)), DT)
        oracle.append(m, mids, kn, vn)
        assert_close(got, oracle.decode(m, mids, q), DT, "decode step %d" % t)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0
