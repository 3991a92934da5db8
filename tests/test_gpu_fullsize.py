"""Parity at the full sizes the benchmark runs, in the launch configuration it
times.  Every valid output element is compared with the fp64 oracle (max abs
and mean abs over all of them, at the bf16 tolerances); padding rows must be
exact zeros; cache contents, lengths, block tables and reference counts are
compared exactly.

Workloads (seeded, synthetic):
  ragged prefill  B=4, H_q=32, H_kv=8, d_h=128, n=2048, valid ~U{512..2048}
  paged decode    B=64, H_q=32, H_kv=8, cache lengths ~U{1024..8192}, pages
                  placed by a seeded permutation
  wide GQA        B=1, H_q=48, H_kv=8, prefill T=8192, then 256 append+decode
  prefix reuse    4096-token prefix, 8 forks x 512-token incremental prefill,
                  then an edit at m=2000 (truncate + re-prefill)
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import TOL, dev, gather_seq, host_f64, raw_pool

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


class _Errors:
    """Max and mean abs error accumulated over every compared element."""

    def __init__(self, what):
        self.what, self.max, self.sum, self.count = what, 0.0, 0.0, 0

    def add(self, got, ref):
        assert np.all(np.isfinite(got)), self.what + ": non-finite output"
        diff = np.abs(got - ref)
        self.max = max(self.max, float(diff.max()))
        self.sum += float(diff.sum())
        self.count += diff.size

    def check(self):
        mean = self.sum / max(1, self.count)
        print("%s: %d elements, max abs %.3g, mean abs %.3g" % (self.what, self.count, self.max, mean))
        assert self.max <= TOL["bf16"]["max"], "%s: max abs %g" % (self.what, self.max)
        assert mean <= TOL["bf16"]["mean"], "%s: mean abs %g" % (self.what, mean)


def _compare_all_rows(err, got, q_bits, K, V, qpos0, chunk=1024):
    """Every row of got [rows, H_q, d] against the oracle, in chunks of rows
    (query row i at absolute position qpos0 + i)."""
    rows = got.shape[0]
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        ref = oracle.attention(oracle.to_f64(q_bits[r0:r1], "bf16"), K, V, qpos0 + np.arange(r0, r1))
        err.add(got[r0:r1], ref)


def test_ragged_prefill_full_size():
    w = workloads.ragged_prefill(workloads.seed_for(2))
    B, n, H_q, H_kv, d = w["B"], w["n"], w["H_q"], w["H_kv"], w["d"]
    nb = [int(x) for x in w["valid_lengths"]]
    pages = sum(workloads.pages_for(x) for x in nb) + 16
    c = gqa.Cache(H_kv, d, pages, B, workloads.pages_for(n) + 1, dtype="bf16")
    ids = [c.seq_create() for _ in range(B)]
    out = gqa.attn_prefill(c, ids, dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"), nb)
    got = host_f64(out, "bf16")
    assert c.check() == 0
    pool = raw_pool(c)
    model = oracle.CacheModel(pages, B, workloads.pages_for(n) + 1, H_kv, d, "bf16")
    mids = [model.create() for _ in range(B)]
    model.write(mids, [w["k"][b, :nb[b]] for b in range(B)], [w["v"][b, :nb[b]] for b in range(B)])
    err = _Errors("ragged prefill")
    for b in range(B):
        assert c.block_table(ids[b]) == model.block_table(mids[b])
        Kraw, Vraw = gather_seq(pool, c.block_table(ids[b]), nb[b])
        assert np.array_equal(Kraw, w["k"][b, :nb[b]]) and np.array_equal(Vraw, w["v"][b, :nb[b]])
        assert np.all(got[b, nb[b]:] == 0)
        K, V = model.kv(mids[b])
        _compare_all_rows(err, got[b, :nb[b]], w["q"][b, :nb[b]], K, V, 0)
    err.check()


def test_paged_decode_full_size():
    w = workloads.paged_decode(workloads.seed_for(3))
    B, H_q, H_kv, d = w["B"], w["H_q"], w["H_kv"], w["d"]
    L = [int(x) for x in w["lengths"]]
    per_seq = workloads.pages_for(max(L)) + 1
    c = gqa.Cache(H_kv, d, w["num_pages"], B, per_seq, dtype="bf16", page_order=w["page_order"])
    ids = [c.seq_create() for _ in range(B)]
    for b in range(B):
        gqa.kv_append(c, [ids[b]], dev(w["hist_k"][b][None], "bf16"), dev(w["hist_v"][b][None], "bf16"))
    # The step the benchmark times: the new token appended and attended in one call.
    got = host_f64(gqa.attn_decode_append(c, ids, dev(w["q"], "bf16"), dev(w["new_k"], "bf16"),
                                          dev(w["new_v"], "bf16")), "bf16")
    assert c.check() == 0
    model = oracle.CacheModel(w["num_pages"], B, per_seq, H_kv, d, "bf16", page_order=w["page_order"])
    mids = [model.create() for _ in range(B)]
    for b in range(B):
        model.write([mids[b]], [w["hist_k"][b]], [w["hist_v"][b]])
    oracle.append(model, mids, w["new_k"], w["new_v"])
    for b in range(B):
        assert c.seq_length(ids[b]) == L[b]
        assert c.block_table(ids[b]) == model.block_table(mids[b])
    ref = oracle.decode(model, mids, w["q"])
    err = _Errors("paged decode")
    err.add(got, ref)
    err.check()
    pool = raw_pool(c)
    for b in range(B):
        Kraw, Vraw = gather_seq(pool, c.block_table(ids[b]), L[b])
        mk, mv = model.raw_kv(mids[b])
        assert np.array_equal(Kraw, mk) and np.array_equal(Vraw, mv)


def test_wide_gqa_long_context_full_size():
    w = workloads.wide_gqa(workloads.seed_for(4))
    T, H_q, H_kv, d, steps = w["n"], w["H_q"], w["H_kv"], w["d"], w["steps"]
    per_seq = workloads.pages_for(T + steps) + 1
    c = gqa.Cache(H_kv, d, per_seq + 4, 1, per_seq, dtype="bf16")
    s = c.seq_create()
    out = host_f64(gqa.attn_prefill(c, [s], dev(w["q"], "bf16"), dev(w["k"], "bf16"), dev(w["v"], "bf16"), [T]),
                   "bf16")
    K = oracle.to_f64(w["k"][0], "bf16")
    V = oracle.to_f64(w["v"][0], "bf16")
    err = _Errors("wide-GQA prefill")
    _compare_all_rows(err, out[0], w["q"][0], K, V, 0)
    err.check()
    check_steps = set(range(0, steps, 16)) | {1, 2, steps - 1}
    derr = _Errors("wide-GQA decode steps")
    dq = dev(w["dec_q"], "bf16")
    dk, dv = dev(w["dec_k"], "bf16"), dev(w["dec_v"], "bf16")
    Kl, Vl = [K], [V]
    for t in range(steps):
        o = gqa.attn_decode_append(c, [s], dq[t], dk[t], dv[t])
        Kl.append(oracle.to_f64(w["dec_k"][t], "bf16"))
        Vl.append(oracle.to_f64(w["dec_v"][t], "bf16"))
        if t in check_steps:
            Kc, Vc = np.concatenate(Kl), np.concatenate(Vl)
            ref = oracle.attention(oracle.to_f64(w["dec_q"][t], "bf16"), Kc, Vc, [T + t])
            derr.add(host_f64(o, "bf16"), ref)
    derr.check()
    assert c.seq_length(s) == T + steps
    assert c.check() == 0
    Kraw, Vraw = gather_seq(raw_pool(c), c.block_table(s), T + steps)
    assert np.array_equal(Kraw, np.concatenate([w["k"][0], w["dec_k"][:, 0]]))
    assert np.array_equal(Vraw, np.concatenate([w["v"][0], w["dec_v"][:, 0]]))


def test_prefix_reuse_and_edit_full_size():
    w = workloads.prefix_edit(workloads.seed_for(5))
    P0, B, n_new, m = w["prefix"], w["B"], w["n_new"], w["m"]
    H_q, H_kv, d = w["H_q"], w["H_kv"], w["d"]
    per_seq = workloads.pages_for(P0 + n_new) + 1
    # prefix + every fork's own pages + the edited fork's re-prefill (its
    # pages past m stay referenced by the other forks)
    pages = workloads.pages_for(P0) + B * workloads.pages_for(n_new) + workloads.pages_for(P0 + n_new) + 16
    c = gqa.Cache(H_kv, d, pages, B + 2, per_seq, dtype="bf16")
    model = oracle.CacheModel(pages, B + 2, per_seq, H_kv, d, "bf16")
    root, mroot = c.seq_create(), model.create()
    gqa.attn_prefill(c, [root], dev(w["pre_q"], "bf16"), dev(w["pre_k"], "bf16"), dev(w["pre_v"], "bf16"), [P0])
    model.write([mroot], [w["pre_k"][0]], [w["pre_v"][0]])
    forks = [c.seq_fork(root, P0) for _ in range(B)]
    mforks = [model.fork(mroot, P0) for _ in range(B)]
    for p in range(workloads.pages_for(P0)):
        assert c.refcount(c.block_table(root)[p]) == B + 1
    out = host_f64(gqa.attn_prefill(c, forks, dev(w["new_q"], "bf16"), dev(w["new_k"], "bf16"),
                                    dev(w["new_v"], "bf16"), [n_new] * B), "bf16")
    model.write(mforks, [w["new_k"][b] for b in range(B)], [w["new_v"][b] for b in range(B)])
    err = _Errors("prefix-reuse incremental prefill")
    for b in range(B):
        assert c.block_table(forks[b]) == model.block_table(mforks[b])
        K, V = model.kv(mforks[b])
        _compare_all_rows(err, out[b], w["new_q"][b], K, V, P0)
    err.check()
    pool = raw_pool(c)
    for b in range(B):
        Kraw, Vraw = gather_seq(pool, c.block_table(forks[b]), P0 + n_new)
        mk, mv = model.raw_kv(mforks[b])
        assert np.array_equal(Kraw, mk) and np.array_equal(Vraw, mv)

    # Edit token m of fork 0: truncate at m, re-prefill the suffix.
    s0, ms0 = forks[0], mforks[0]
    before = gather_seq(pool, c.block_table(s0), m)
    gqa.kv_truncate(c, s0, m)
    model.truncate(ms0, m)
    n_re = P0 + n_new - m
    re = host_f64(gqa.attn_prefill(c, [s0], dev(w["edit_q"], "bf16"), dev(w["edit_k"], "bf16"),
                                   dev(w["edit_v"], "bf16"), [n_re]), "bf16")
    model.write([ms0], [w["edit_k"][0]], [w["edit_v"][0]])
    assert c.block_table(s0) == model.block_table(ms0)
    after = gather_seq(raw_pool(c), c.block_table(s0), m)
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    K, V = model.kv(ms0)
    err = _Errors("re-prefill after the edit")
    _compare_all_rows(err, re[0], w["edit_q"][0], K, V, m)
    err.check()
    assert c.check() == 0

    # Rows < m are bit-identical between a full prefill of the original
    # sequence and of the edited one.
    full_q = np.concatenate([w["pre_q"][0], w["new_q"][0]])[None]
    full_k = np.concatenate([w["pre_k"][0], w["new_k"][0]])[None]
    full_v = np.concatenate([w["pre_v"][0], w["new_v"][0]])[None]
    edit_q = np.concatenate([full_q[0, :m], w["edit_q"][0]])[None]
    edit_k = np.concatenate([full_k[0, :m], w["edit_k"][0]])[None]
    edit_v = np.concatenate([full_v[0, :m], w["edit_v"][0]])[None]
    outs = []
    for q, k, v in ((full_q, full_k, full_v), (edit_q, edit_k, edit_v)):
        cc = gqa.Cache(H_kv, d, per_seq + 2, 1, per_seq, dtype="bf16")
        ss = cc.seq_create()
        o = gqa.attn_prefill(cc, [ss], dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), [P0 + n_new])
        outs.append(o.view(torch.int16).cpu().numpy())
        assert cc.check() == 0
    assert np.array_equal(outs[0][0, :m], outs[1][0, :m])
    assert not np.array_equal(outs[0][0, m:], outs[1][0, m:])
