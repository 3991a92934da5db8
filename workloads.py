"""Seeded synthetic inputs for the causal GQA prefill / paged decode workloads.

Both sides of every comparison draw their inputs from here: the fp64 oracle
under ``oracle/`` and the CUDA library under ``causal_gqa_attention_02_gb300``.
This module holds none of the attention arithmetic -- only shapes, random
draws, length mixes and page orders -- so that it can serve both sides
without coupling them.

Values are returned as host numpy arrays.  Half-precision tensors are
returned as their raw bf16 bit patterns (``uint16``), rounded to nearest-even
from a float32 draw; fp32 tensors are returned as ``float32``.

Workload shapes follow the five configurations the path is specified on:
  1. fp32 tiny prefill + 3 decode steps (and the 2-D worked example),
  2. bf16 ragged prefill, right padded,
  3. bf16 paged decode with a randomly permuted page placement,
  4. wide-GQA long context: 8192-token prefill then 256 decode steps,
  5. prefix reuse: one shared 4096-token prefix, 8 forks, then an edit,
  6. multi-token decode: T-token draft chunks over configuration 3's cache.
"""
from __future__ import annotations

import numpy as np

PAGE_TOKENS = 16        # tokens per cache page (the library's fixed page size)
BASE_SEED = 20261202    # seed of configuration k is BASE_SEED + k


def seed_for(config_index: int) -> int:
    return BASE_SEED + int(config_index)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def uniform_f32(rng: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def draw(rng: np.random.Generator, dtype: str, shape) -> np.ndarray:
    """N(0,1) for bf16 workloads, U(-1,1) for fp32 workloads."""
    if dtype == "bf16":
        return normal_bf16(rng, shape)
    if dtype == "f32":
        return uniform_f32(rng, shape)
    raise ValueError(dtype)


def pages_for(tokens: int) -> int:
    return (int(tokens) + PAGE_TOKENS - 1) // PAGE_TOKENS


# --------------------------------------------------------------------------
# Configuration 1: fp32 tiny, and the 2-D worked example.
# --------------------------------------------------------------------------

def worked_example_2d():
    """The hand-worked attention example of "模型执行：从 token 到 Prefill 与
    Decode" (section "手算一次 Attention"): one head, d = 2, two positions.

    q is the query at the second position; row 0 of ``q`` is a query at the
    first position chosen equal to it (the page evaluates the first position
    with the same q)."""
    q = np.array([[[1.0, 0.0]], [[1.0, 0.0]]], dtype=np.float32)   # [n=2, H_q=1, d=2]
    k = np.array([[[1.0, 0.0]], [[0.0, 1.0]]], dtype=np.float32)   # [n=2, H_kv=1, d=2]
    v = np.array([[[10.0, 0.0]], [[0.0, 20.0]]], dtype=np.float32)
    return {"dtype": "f32", "B": 1, "n": 2, "H_q": 1, "H_kv": 1, "d": 2,
            "q": q[None], "k": k[None], "v": v[None],
            "valid_lengths": np.array([2], dtype=np.int32)}


def tiny_fp32(seed: int = seed_for(1)):
    """B=1, H_q=2, H_kv=1, d_h=4: prefill n=4 (all valid), then 3 single-token
    decode steps (cache lengths 5, 6, 7); U(-1,1) values."""
    rng = np.random.default_rng(seed)
    B, H_q, H_kv, d, n, steps = 1, 2, 1, 4, 4, 3
    return {"dtype": "f32", "B": B, "n": n, "H_q": H_q, "H_kv": H_kv, "d": d,
            "q": draw(rng, "f32", (B, n, H_q, d)),
            "k": draw(rng, "f32", (B, n, H_kv, d)),
            "v": draw(rng, "f32", (B, n, H_kv, d)),
            "valid_lengths": np.full(B, n, dtype=np.int32),
            "dec_q": draw(rng, "f32", (steps, B, H_q, d)),
            "dec_k": draw(rng, "f32", (steps, B, H_kv, d)),
            "dec_v": draw(rng, "f32", (steps, B, H_kv, d))}


# --------------------------------------------------------------------------
# Configuration 2: ragged, right-padded prefill.
# --------------------------------------------------------------------------

def ragged_prefill(seed: int = seed_for(2), B=4, H_q=32, H_kv=8, d=128, n=2048,
                   lo=512, hi=2048, dtype="bf16", past=None):
    """Right-padded prefill batch; valid_lengths ~ U{lo..hi}.  Padding rows of
    q/k/v hold ordinary random values (they must never matter).  ``past`` (an
    optional list of per-sequence cache lengths) adds, per sequence, the
    already-cached K/V rows ``past_k``/``past_v`` [P_b, H_kv, d]."""
    rng = np.random.default_rng(seed)
    valid = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    out = {"dtype": dtype, "B": B, "n": n, "H_q": H_q, "H_kv": H_kv, "d": d,
           "valid_lengths": valid,
           "q": draw(rng, dtype, (B, n, H_q, d)),
           "k": draw(rng, dtype, (B, n, H_kv, d)),
           "v": draw(rng, dtype, (B, n, H_kv, d))}
    if past is not None:
        out["past"] = np.asarray(past, dtype=np.int64)
        out["past_k"] = [draw(rng, dtype, (int(P), H_kv, d)) for P in past]
        out["past_v"] = [draw(rng, dtype, (int(P), H_kv, d)) for P in past]
    return out


# --------------------------------------------------------------------------
# Configuration 3: paged decode over a permuted page placement.
# --------------------------------------------------------------------------

def paged_decode(seed: int = seed_for(3), B=64, H_q=32, H_kv=8, d=128,
                 lo=1024, hi=8192, dtype="bf16", spare_pages=64):
    """One query per sequence against a cache of L_b ~ U{lo..hi} tokens
    (the last of which is the token appended in this step).

    ``page_order`` is a seeded random permutation of the physical pages; the
    cache hands out free pages in this order, so logical pages land on
    scattered physical pages."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    num_pages = int(sum(pages_for(L) for L in lengths)) + spare_pages
    page_order = rng.permutation(num_pages).astype(np.int32)
    kv_k = [draw(rng, dtype, (int(L) - 1, H_kv, d)) for L in lengths]
    kv_v = [draw(rng, dtype, (int(L) - 1, H_kv, d)) for L in lengths]
    return {"dtype": dtype, "B": B, "H_q": H_q, "H_kv": H_kv, "d": d,
            "lengths": lengths, "num_pages": num_pages, "page_order": page_order,
            "hist_k": kv_k, "hist_v": kv_v,
            "new_k": draw(rng, dtype, (B, H_kv, d)),
            "new_v": draw(rng, dtype, (B, H_kv, d)),
            "q": draw(rng, dtype, (B, H_q, d))}


def draft_chunk(seed: int = seed_for(6), B=64, T=4, H_q=32, H_kv=8, d=128, dtype="bf16"):
    """T new tokens per sequence (a multi-token decode / speculative draft
    block) to run over an existing cache: q [B, T, H_q, d], k and v
    [B, T, H_kv, d]."""
    rng = np.random.default_rng(seed)
    return {"dtype": dtype, "B": B, "T": T, "H_q": H_q, "H_kv": H_kv, "d": d,
            "q": draw(rng, dtype, (B, T, H_q, d)),
            "k": draw(rng, dtype, (B, T, H_kv, d)),
            "v": draw(rng, dtype, (B, T, H_kv, d))}


# --------------------------------------------------------------------------
# Configuration 4: wide GQA, long context, one layer.
# --------------------------------------------------------------------------

def wide_gqa(seed: int = seed_for(4), T=8192, steps=256, H_q=48, H_kv=8, d=128,
             dtype="bf16"):
    rng = np.random.default_rng(seed)
    return {"dtype": dtype, "B": 1, "n": T, "H_q": H_q, "H_kv": H_kv, "d": d,
            "valid_lengths": np.array([T], dtype=np.int32),
            "q": draw(rng, dtype, (1, T, H_q, d)),
            "k": draw(rng, dtype, (1, T, H_kv, d)),
            "v": draw(rng, dtype, (1, T, H_kv, d)),
            "steps": steps,
            "dec_q": draw(rng, dtype, (steps, 1, H_q, d)),
            "dec_k": draw(rng, dtype, (steps, 1, H_kv, d)),
            "dec_v": draw(rng, dtype, (steps, 1, H_kv, d))}


# --------------------------------------------------------------------------
# Configuration 5: prefix reuse and an edit at position m.
# --------------------------------------------------------------------------

def prefix_edit(seed: int = seed_for(5), prefix=4096, B=8, n_new=512, m=2000,
                H_q=32, H_kv=8, d=128, dtype="bf16"):
    """One shared ``prefix``-token prefix, B forks that each append ``n_new``
    tokens by incremental prefill, then sequence 0 is edited at token m.

    An edit at token m changes every row at positions >= m of every layer
    above the embedding, so the edited sequence's q/k/v rows at positions
    >= m are fresh draws while rows < m are unchanged."""
    rng = np.random.default_rng(seed)
    total0 = prefix + n_new
    out = {"dtype": dtype, "B": B, "H_q": H_q, "H_kv": H_kv, "d": d,
           "prefix": prefix, "n_new": n_new, "m": m,
           "pre_q": draw(rng, dtype, (1, prefix, H_q, d)),
           "pre_k": draw(rng, dtype, (1, prefix, H_kv, d)),
           "pre_v": draw(rng, dtype, (1, prefix, H_kv, d)),
           "new_q": draw(rng, dtype, (B, n_new, H_q, d)),
           "new_k": draw(rng, dtype, (B, n_new, H_kv, d)),
           "new_v": draw(rng, dtype, (B, n_new, H_kv, d)),
           "edit_q": draw(rng, dtype, (1, total0 - m, H_q, d)),
           "edit_k": draw(rng, dtype, (1, total0 - m, H_kv, d)),
           "edit_v": draw(rng, dtype, (1, total0 - m, H_kv, d))}
    return out
