"""GPU parity of the host-buffer entry points.  attn_prefill_host: the prefill
on host buffers, its copies inside the call.  The batch is checked as a whole, then each entry runs as a
one-entry prefill, longest valid length first (ties in batch order), so the
oracle's cache model takes its pages in that order.  Outputs within the
declared tolerance of the oracle, cache bytes and tables exact, output rows
past an entry's valid length left untouched.  attn_decode_append_host: one
decode step on host buffers, the same bits as the device-buffer step."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, valid_mask

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _host(a, dt, pinned=True):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
    return t.pin_memory() if pinned else t.clone()


def _f64(t, dt):
    if dt == "bf16":
        return oracle.to_f64(t.view(torch.int16).numpy().view(np.uint16), "bf16")
    return t.numpy().astype(np.float64)


def _run(w, pinned=True, past=None, window=0):
    dt = w["dtype"]
    B, n, H_q, H_kv, d = w["B"], w["n"], w["H_q"], w["H_kv"], w["d"]
    nb = [int(x) for x in w["valid_lengths"]]
    P = past or [0] * B
    pages = sum(workloads.pages_for(p + x) for p, x in zip(P, nb)) + 8
    per_seq = max(workloads.pages_for(p + n) for p in P) + 1
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype=dt, window=window)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, dt, window=window)
    ids = [c.seq_create() for _ in range(B)]
    mids = [m.create() for _ in range(B)]
    rng = np.random.default_rng(5)
    for b in range(B):                                    # an existing prefix, if asked for
        if P[b]:
            k0 = workloads.draw(rng, dt, (1, P[b], H_kv, d))
            v0 = workloads.draw(rng, dt, (1, P[b], H_kv, d))
            gqa.kv_append(c, [ids[b]], dev(k0, dt), dev(v0, dt))
            oracle.append(m, [mids[b]], k0, v0)
    out = _host(np.full((B, n, H_q, d), 7 if dt == "f32" else 0x40e0, dtype=np.float32 if dt == "f32"
                        else np.uint16), dt, pinned)      # sentinel 7.0 in every row
    c.profile_read()
    gqa.attn_prefill_host(c, ids, _host(w["q"], dt, pinned), _host(w["k"], dt, pinned), _host(w["v"], dt, pinned),
                          nb, out=out)
    torch.cuda.synchronize()
    launched = c.profile_read()
    ref = np.zeros((B, n, H_q, d))
    for b in sorted(range(B), key=lambda b: -nb[b]):
        ref[b:b + 1] = oracle.prefill(m, [mids[b]], w["q"][b:b + 1], w["k"][b:b + 1], w["v"][b:b + 1], [nb[b]])
    got = _f64(out, dt)
    mask = valid_mask(nb, n)
    return c, m, ids, mids, got, ref, mask, launched


@pytest.mark.parametrize("B,H_q,H_kv,n,lo,hi", [
    (4, 8, 2, 300, 100, 300),     # g = 4, ragged tails, several key tiles
    (3, 12, 2, 200, 1, 200),      # g = 6, a one-row entry possible
    (2, 16, 2, 257, 257, 257),    # g = 8, equal lengths (ties keep batch order)
])
def test_host_buffer_prefill_matches_oracle(B, H_q, H_kv, n, lo, hi):
    w = workloads.ragged_prefill(seed=300 + H_q, B=B, H_q=H_q, H_kv=H_kv, n=n, lo=lo, hi=hi)
    c, m, ids, mids, got, ref, mask, launched = _run(w)
    assert launched["prefill_tc"][0] == B, launched        # one one-entry prefill per entry
    assert_close(got[mask], ref[mask], "bf16", "host-buffer prefill")
    assert np.all(got[~mask] == 7.0), "rows past the valid length must be left as they were"
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_host_buffer_prefill_equals_device_prefill_per_entry():
    # The device entry point on the same one-entry calls gives the same bits.
    w = workloads.ragged_prefill(seed=41, B=3, H_q=8, H_kv=2, n=260, lo=60, hi=260)
    c, m, ids, mids, got, ref, mask, _ = _run(w)
    nb = [int(x) for x in w["valid_lengths"]]
    c2 = gqa.Cache(2, 128, c.num_pages, 3, 20, dtype="bf16")
    ids2 = [c2.seq_create() for _ in range(3)]
    for b in sorted(range(3), key=lambda b: -nb[b]):
        o = gqa.attn_prefill(c2, [ids2[b]], dev(w["q"][b:b + 1, :nb[b]], "bf16"),
                             dev(w["k"][b:b + 1, :nb[b]], "bf16"), dev(w["v"][b:b + 1, :nb[b]], "bf16"), [nb[b]])
        assert np.array_equal(_f64(o.cpu(), "bf16")[0], got[b, :nb[b]])
    for s, s2 in zip(ids, ids2):
        assert c.block_table(s) == c2.block_table(s2)


def test_host_buffer_prefill_fp32_pageable_incremental_windowed():
    # fp32 (CUDA-core kernel), pageable buffers, an existing prefix and a
    # sliding window: the same contract.
    w = workloads.ragged_prefill(seed=42, B=3, H_q=4, H_kv=2, n=90, lo=10, hi=90, dtype="f32")
    c, m, ids, mids, got, ref, mask, _ = _run(w, pinned=False, past=[37, 0, 150], window=64)
    assert_close(got[mask], ref[mask], "f32", "fp32 host-buffer prefill")
    assert np.all(got[~mask] == 7.0)
    assert_cache_matches(c, m, zip(ids, mids))
    assert c.check() == 0


def test_host_buffer_prefill_rejection_queues_nothing():
    w = workloads.ragged_prefill(seed=43, B=2, H_q=8, H_kv=2, n=64, lo=64, hi=64)
    c = gqa.Cache(2, 128, 5, 2, 4, dtype="bf16")          # room for 80 tokens in all
    ids = [c.seq_create(), c.seq_create()]
    out = _host(np.zeros((2, 64, 8, 128), dtype=np.uint16), "bf16")
    with pytest.raises(gqa.GqaError) as e:
        gqa.attn_prefill_host(c, ids, _host(w["q"], "bf16"), _host(w["k"], "bf16"), _host(w["v"], "bf16"),
                              [64, 64], out=out)
    torch.cuda.synchronize()
    assert e.value.name == "ENOMEM"
    assert [c.seq_length(s) for s in ids] == [0, 0] and c.free_pages() == 5
    assert np.all(out.view(torch.int16).numpy() == 0)
    with pytest.raises(TypeError):
        gqa.attn_prefill_host(c, ids, dev(w["q"], "bf16"), _host(w["k"], "bf16"), _host(w["v"], "bf16"), [1, 1])


# ---- attn_decode_append_host: one decode step on host buffers --------------

@pytest.mark.parametrize("dt,d,pinned", [("bf16", 128, True), ("bf16", 128, False), ("f32", 64, True)])
def test_host_buffer_decode_step_equals_device_step(dt, d, pinned):
    # The same step through device buffers and through host buffers gives
    # the same bits in out and in the pool, and matches the oracle.
    rng = np.random.default_rng(900 + d)
    B, H_q, H_kv = 5, 16, 4
    lengths = [1, 15, 16, 200, 1030]
    per_seq = workloads.pages_for(max(lengths) + 4) + 1
    pages = B * per_seq
    caches = [gqa.Cache(H_kv, d, pages, B, per_seq, dtype=dt) for _ in range(2)]
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, dt)
    ids = [[c.seq_create() for _ in range(B)] for c in caches]
    mids = [m.create() for _ in range(B)]
    n = max(lengths)
    k = np.zeros((B, n, H_kv, d), np.uint16 if dt == "bf16" else np.float32)
    v = np.zeros_like(k)
    for b, L in enumerate(lengths):
        k[b, :L] = workloads.draw(rng, dt, (L, H_kv, d))
        v[b, :L] = workloads.draw(rng, dt, (L, H_kv, d))
    for c, s in zip(caches, ids):
        gqa.kv_append(c, s, dev(k, dt), dev(v, dt), counts=lengths)
    oracle.append(m, mids, k, v, counts=lengths)
    for step in range(2):
        q, kn, vn = (workloads.draw(rng, dt, (B, H, d)) for H in (H_q, H_kv, H_kv))
        a = gqa.attn_decode_append(caches[0], ids[0], dev(q, dt), dev(kn, dt), dev(vn, dt))
        b = gqa.attn_decode_append_host(caches[1], ids[1], _host(q, dt, pinned), _host(kn, dt, pinned),
                                        _host(vn, dt, pinned))
        torch.cuda.synchronize()
        av = a.cpu().view(torch.int32 if dt == "f32" else torch.int16)
        bv = b.view(torch.int32 if dt == "f32" else torch.int16)
        assert torch.equal(av, bv), "host-buffer step differs from the device step"
        oracle.append(m, mids, kn, vn)
        assert_close(_f64(b, dt), oracle.decode(m, mids, q), dt, "host-buffer decode step %d" % step)
    for c, s in zip(caches, ids):
        assert_cache_matches(c, m, zip(s, mids))
        assert c.check() == 0


def test_host_buffer_decode_step_rejection_changes_nothing():
    c = gqa.Cache(2, 128, 8, 2, 4, dtype="bf16")
    s = c.seq_create()
    q = torch.zeros((2, 8, 128), dtype=torch.bfloat16)
    kv = torch.zeros((2, 2, 128), dtype=torch.bfloat16)
    out = torch.full((2, 8, 128), 5.0, dtype=torch.bfloat16)
    with pytest.raises(gqa.GqaError) as e:
        gqa.attn_decode_append_host(c, [s, 7], q, kv, kv, out=out)    # sequence 7 is not live
    assert e.value.name == "EINVAL"
    torch.cuda.synchronize()
    assert c.seq_length(s) == 0 and bool((out == 5.0).all())
