"""Algorithmic work counts used to turn times into throughput.

Prefill: the number of (query, key) pairs with a finite score, times
4 * d_h flops per pair (2 for the QK^T product, 2 for the PV product) and
H_q heads -- the causal count, excluding padding rows and keys above the
diagonal even where a kernel touches them.  "模型执行：从 token 到 Prefill 与
Decode" counts attention work the same way (its "score pairs" table, and
4 B H_q S^2 d for the full, unmasked matrix products).

A sliding window W caps each position's keys at W, in both counts.

Decode: the K/V bytes the method must read, each KV head counted once (the
query heads of a group share it: "KV Cache 与 Prefill/Decode 推理路径", GQA
lesson), 2 (K and V) * H_kv * d_h * element size per cached token.
"""
from __future__ import annotations


def causal_pairs(past: int, new: int, window: int = 0) -> int:
    """Pairs (i, j) with j <= past + i for new query rows i = 0..new-1 at
    positions past..past+new-1; with a sliding window W > 0 also
    j >= past + i - W + 1, so a position p counts min(p + 1, W) keys."""
    past, new, window = int(past), int(new), int(window)
    full = new * past + new * (new + 1) // 2
    if window <= 0 or past + new <= window:
        return full
    # Positions p >= W see exactly W keys instead of p + 1.
    first = max(past, window)                  # first capped position
    last = past + new - 1
    cnt = last - first + 1
    over = cnt * (first + last) // 2 + cnt - cnt * window   # sum over capped p of (p + 1 - W)
    return full - over


def prefill_flops(pasts, news, H_q: int, d: int, window: int = 0) -> int:
    return 4 * int(d) * int(H_q) * sum(causal_pairs(p, n, window) for p, n in zip(pasts, news))


def window_tokens(L: int, window: int = 0) -> int:
    """Cached tokens a decode of a length-L sequence must read."""
    return min(int(L), int(window)) if window > 0 else int(L)


def decode_kv_bytes(lengths, H_kv: int, d: int, esize: int = 2, window: int = 0, row_extra: int = 0) -> int:
    """K and V bytes a decode reads: per visible token and KV head, d * esize
    bytes of each, plus row_extra (a quantised cache's per-row scale)."""
    return sum(window_tokens(L, window) for L in lengths) * 2 * int(H_kv) * (int(d) * int(esize) + int(row_extra))


def decode_flops(lengths, H_q: int, d: int, window: int = 0) -> int:
    return 4 * int(d) * int(H_q) * sum(window_tokens(L, window) for L in lengths)
