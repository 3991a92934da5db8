"""GPU parity of multi-token decode: a short causal block of T new tokens per
sequence over a long cached prefix (the incremental-prefill mask at small M:
new row i at position P_b + i sees cached keys 0..P_b + i).  This is
attn_prefill with a small n; on the tensor-core path an item whose second
query tile holds no valid row runs one tile.  Outputs within the bf16
tolerance, cache bytes and tables exact."""
import numpy as np
import pytest

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _filled(rng, B, H_q, H_kv, d, lengths, extra, window=0):
    per_seq = workloads.pages_for(max(lengths) + extra) + 1
    pages = sum(workloads.pages_for(L + extra) for L in lengths) + 8
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype="bf16", window=window)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, "bf16", window=window)
    ids = [c.seq_create() for _ in range(B)]
    mids = [m.create() for _ in range(B)]
    for b, L in enumerate(lengths):
        k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        gqa.kv_append(c, [ids[b]], dev(k, "bf16"), dev(v, "bf16"))
        oracle.append(m, [mids[b]], k, v)
    return c, m, ids, mids


def _chunk(c, m, ids, mids, rng, H_q, H_kv, d, T, n):
    B = len(ids)
    q = workloads.normal_bf16(rng, (B, n, H_q, d))
    k = workloads.normal_bf16(rng, (B, n, H_kv, d))
    v = workloads.normal_bf16(rng, (B, n, H_kv, d))
    c.profile_read()
    out = host_f64(gqa.attn_prefill(c, ids, dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), T), "bf16")
    launched = c.profile_read()
    ref = oracle.prefill(m, mids, q, k, v, T)
    mask = np.arange(n)[None, :] < np.asarray(T)[:, None]
    assert np.all(out[~mask] == 0)
    return out[mask], ref[mask], launched


@pytest.mark.parametrize("H_q,H_kv,T,n", [
    (32, 8, [1, 2, 3, 4, 5, 8], 8),          # g = 4: one 32-position tile covers every chunk
    (64, 8, [16, 17, 20, 9, 1, 31], 32),     # g = 8: 16 positions per tile, some chunks need both tiles
    (8, 8, [1, 64, 65, 100, 7, 128], 128),   # g = 1: the second tile starts at row 128
])
def test_multi_token_decode_matches_oracle(H_q, H_kv, T, n):
    rng = np.random.default_rng(70 + H_q)
    B, d = len(T), 128
    lengths = [int(x) for x in rng.integers(500, 3000, B)]
    c, m, ids, mids = _filled(rng, B, H_q, H_kv, d, lengths, n)
    got, ref, launched = _chunk(c, m, ids, mids, rng, H_q, H_kv, d, T, n)
    assert launched["prefill_tc"][0] == 1, launched
    assert_close(got, ref, "bf16", "multi-token decode")
    assert_cache_matches(c, m, list(zip(ids, mids)))
    assert c.check() == 0


def test_speculative_chunks_accept_reject_and_continue():
    # Draft 4 tokens, keep a per-sequence prefix of them (truncate the rest),
    # then draft again from there: every round agrees with the oracle.
    rng = np.random.default_rng(71)
    B, H_q, H_kv, d = 4, 32, 8, 128
    lengths = [700, 1500, 2100, 129]
    c, m, ids, mids = _filled(rng, B, H_q, H_kv, d, lengths, 64)
    for rnd in range(5):
        T = [4] * B
        got, ref, _ = _chunk(c, m, ids, mids, rng, H_q, H_kv, d, T, 4)
        assert_close(got, ref, "bf16", "draft round %d" % rnd)
        for b in range(B):
            keep = int(rng.integers(0, 5))
            L = m.length(mids[b]) - 4 + keep
            gqa.kv_truncate(c, ids[b], L)
            m.truncate(mids[b], L)
    assert_cache_matches(c, m, list(zip(ids, mids)))
    assert c.check() == 0


def test_multi_token_decode_with_sliding_window():
    rng = np.random.default_rng(72)
    B, H_q, H_kv, d, W = 4, 32, 8, 128, 300
    lengths = [1000, 2000, 450, 3000]
    c, m, ids, mids = _filled(rng, B, H_q, H_kv, d, lengths, 16, window=W)
    got, ref, launched = _chunk(c, m, ids, mids, rng, H_q, H_kv, d, [3, 8, 1, 6], 8)
    assert launched["prefill_tc"][0] == 1
    assert_close(got, ref, "bf16", "windowed multi-token decode")
    assert_cache_matches(c, m, list(zip(ids, mids)))
    assert c.check() == 0
