"""Shared helpers for the GPU parity tests: host <-> device marshalling of the
seeded inputs, reading the page pool back through a block table, and the
comparison protocol (exact for cache bytes, lengths and tables; declared
tolerances for attention outputs)."""
import numpy as np
import torch

import oracle

TOL = {"f32": {"max": 1e-5}, "bf16": {"max": 2e-2, "mean": 2e-3}}


def dev(a, dt, device="cuda"):
    a = np.ascontiguousarray(a)
    if dt == "bf16":
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def host_f64(t, dt):
    t = t.detach().cpu()
    if dt == "bf16":
        return oracle.to_f64(t.view(torch.int16).numpy().view(np.uint16), "bf16")
    return t.numpy().astype(np.float64)


def raw_pool(cache):
    """Pool as host raw values [pages, 2, H_kv, 16, d] (uint16 bits or f32),
    decoded from the byte layout the header documents: the block of (page,
    K|V, head) holds two groups of 8 slots; a group stores its rows' 128-byte
    chunk 0, then chunk 1, ...; byte b of slot s's row is at
    ((s // 8) * C + b // 128) * 1024 + (s % 8) * 128 + b % 128."""
    bf16 = cache.torch_dtype == torch.bfloat16
    es = 2 if bf16 else 4
    d, H = cache.head_dim, cache.num_kv_heads
    C = -(-d * es // 128)
    raw = cache.pool.detach().cpu().numpy().view(np.uint8)
    blocks = raw[: cache.num_pages * 2 * H * 16 * C * 128].reshape(cache.num_pages, 2, H, 16 * C * 128)
    s = np.arange(16)[:, None]
    b = (np.arange(d) * es)[None, :]
    off = ((s // 8) * C + b // 128) * 1024 + (s % 8) * 128 + b % 128          # [16, d] byte offsets
    idx = off[..., None] + np.arange(es)                                       # [16, d, es]
    vals = np.ascontiguousarray(blocks[..., idx])                              # [P, 2, H, 16, d, es]
    return vals.view(np.uint16 if bf16 else np.float32)[..., 0]


def held_from(table):
    """First position whose page is still held: under a sliding window the
    released pages (entry -1) lead the table."""
    r = 0
    while r < len(table) and table[r] < 0:
        r += 1
    return 16 * r


def gather_seq(pool, table, length, start=0):
    """Logical K, V [start:length, H_kv, d] of one sequence, read through its table."""
    t = np.arange(start, length)
    pages = np.asarray(table, dtype=np.int64)[t // 16]
    slots = t % 16
    return pool[pages, 0, :, slots, :], pool[pages, 1, :, slots, :]


def assert_cache_matches(cache, model, seq_pairs):
    """Lengths and block tables equal; every cached K/V value bit-identical."""
    pool = raw_pool(cache)
    for s_lib, s_ref in seq_pairs:
        L = model.length(s_ref)
        assert cache.seq_length(s_lib) == L
        assert cache.block_table(s_lib) == model.block_table(s_ref)
        t0 = min(held_from(cache.block_table(s_lib)), L)
        K, V = gather_seq(pool, cache.block_table(s_lib), L, t0)
        rk, rv = model.raw_kv(s_ref)
        assert np.array_equal(K, rk[t0:]), "cached K differs"
        assert np.array_equal(V, rv[t0:]), "cached V differs"


def assert_close(got, ref, dt, what=""):
    diff = np.abs(got - ref)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    assert diff.max() <= TOL[dt]["max"], "%s max abs %g" % (what, diff.max())
    if "mean" in TOL[dt]:
        assert diff.mean() <= TOL[dt]["mean"], "%s mean abs %g" % (what, diff.mean())
    return diff.max(), diff.mean()


def valid_mask(valid_lengths, n):
    return np.arange(n)[None, :] < np.asarray(valid_lengths)[:, None]
