"""attn_decode_append: one decode step (append one token per sequence, then
attend at it) in a single call.  Checked against the two calls it replaces
-- kv_append then attn_decode -- for the same bits in the output and in the
raw page pool, on both decode kernels, across page boundaries, after a fork
that shares a partly filled tail page (copy-on-write first), and with the
rotary mechanism and a sliding window; and against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_close, assert_cache_matches, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _pair(rng, H_kv, lengths, extra, kernel, window=0, rope=False, max_seqs=None):
    B, d = len(lengths), 128
    per_seq = workloads.pages_for(max(lengths) + extra) + 1
    pages = 2 * sum(workloads.pages_for(L + extra) for L in lengths) + 8
    caches = []
    for _ in range(2):
        c = gqa.Cache(H_kv, d, pages, max_seqs or B, per_seq, dtype="bf16", window=window, rope=rope)
        c.set_decode_kernel(kernel)
        caches.append(c)
    m = oracle.CacheModel(pages, max_seqs or B, per_seq, H_kv, d, "bf16", window=window)
    ids = [[c.seq_create() for _ in range(B)] for c in caches]
    mids = [m.create() for _ in range(B)]
    for b, L in enumerate(lengths):
        k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        for c, i in zip(caches, ids):
            gqa.kv_append(c, [i[b]], dev(k, "bf16"), dev(v, "bf16"))
        oracle.append(m, [mids[b]], k, v)
    return caches, ids, m, mids


def _step(rng, caches, ids, m, mids, H_q, H_kv, base=None):
    B = len(mids)
    q = workloads.normal_bf16(rng, (B, H_q, 128))
    k = workloads.normal_bf16(rng, (B, H_kv, 128))
    v = workloads.normal_bf16(rng, (B, H_kv, 128))
    gqa.kv_append(caches[0], ids[0], dev(k, "bf16"), dev(v, "bf16"))
    a = gqa.attn_decode(caches[0], ids[0], dev(q, "bf16"))
    caches[1].profile_read()
    b = gqa.attn_decode_append(caches[1], ids[1], dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"))
    launched = caches[1].profile_read()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "fused step differs from append + decode"
    assert torch.equal(caches[0].pool, caches[1].pool), "fused step wrote different cache bytes"
    oracle.append(m, mids, k, v)
    assert_close(host_f64(b, "bf16"), oracle.decode(m, mids, q, rope_base=base), "bf16", "fused decode step")
    return launched


@pytest.mark.parametrize("kernel", ["tensor_core", "cuda_core", "cluster"])
def test_fused_step_equals_append_then_decode(kernel):
    rng = np.random.default_rng(100)
    H_q, H_kv = 32, 8
    lengths = [14, 1000, 2047, 3000, 1]             # tails at slots 14, 8, 15, 8, 1
    caches, ids, m, mids = _pair(rng, H_kv, lengths, 40, kernel)
    for t in range(20):                              # crosses page and key-tile boundaries
        launched = _step(rng, caches, ids, m, mids, H_q, H_kv)
        if kernel == "tensor_core":
            assert launched["prefill_tc"][0] == 1 and launched["cache_write"][0] == 0, launched
        elif kernel == "cluster":
            assert launched["decode_cluster"][0] == 1 and launched["cache_write"][0] == 0, launched
        else:
            assert launched["cache_write"][0] == 1, launched
    for c, i in zip(caches, ids):
        assert_cache_matches(c, m, list(zip(i, mids)))
        assert c.check() == 0


def test_fused_step_after_fork_copies_the_shared_tail_first():
    rng = np.random.default_rng(101)
    H_q, H_kv = 16, 8
    caches, ids, m, mids = _pair(rng, H_kv, [1000], 40, "tensor_core", max_seqs=3)
    forks = [c.seq_fork(i[0], 997) for c, i in zip(caches, ids)]     # shares a page filled to slot 4
    fm = m.fork(mids[0], 997)
    for t in range(3):
        _step(rng, caches, [[f] for f in forks], m, [fm], H_q, H_kv)
        _step(rng, caches, [[i[0]] for i in ids], m, [mids[0]], H_q, H_kv)
    assert len(m.copies) >= 1
    for c, i, f in zip(caches, ids, forks):
        assert_cache_matches(c, m, [(i[0], mids[0]), (f, fm)])
        assert c.check() == 0


@pytest.mark.parametrize("window,rope", [(0, True), (200, False), (150, True)])
def test_fused_step_with_rope_and_window(window, rope):
    rng = np.random.default_rng(102 + window)
    H_q, H_kv = 32, 8
    caches, ids, m, mids = _pair(rng, H_kv, [700, 2500, 33], 40, "tensor_core", window=window, rope=rope)
    for t in range(18):
        _step(rng, caches, ids, m, mids, H_q, H_kv, base=10000.0 if rope else None)
    for c, i in zip(caches, ids):
        for s, ms in zip(i, mids):
            assert c.block_table(s) == m.block_table(ms)
        assert c.free_pages() == m.free_pages()
        assert c.check() == 0


def test_small_batch_long_context_fused_steps():
    # One long sequence: the key tiles are split across SMs and the last
    # split writes the token.
    rng = np.random.default_rng(103)
    H_q, H_kv = 48, 8
    caches, ids, m, mids = _pair(rng, H_kv, [8192], 24, "tensor_core")
    for t in range(12):
        _step(rng, caches, ids, m, mids, H_q, H_kv)
    for c in caches:
        assert c.check() == 0
