"""Pins of the oracle's logical paged-cache model (block tables, free pool,
reference counts, copy-on-write, truncation) against the pages' block
arithmetic and the allocation rules' special cases."""
import numpy as np
import pytest

import oracle


def _cm(pages=32, seqs=8, per_seq=16, order=None, H_kv=1, d=2):
    return oracle.CacheModel(pages, seqs, per_seq, H_kv, d, "f32", page_order=order)


def _rows(c, H_kv=1, d=2, base=0.0):
    return (np.arange(c * H_kv * d, dtype=np.float32).reshape(c, H_kv, d) + base)


def test_eighteen_tokens_take_two_pages_with_fourteen_free(golden):
    g = golden("page_arithmetic.txt")
    cm = _cm()
    s = cm.create()
    cm.write([s], [_rows(int(g["tokens"]))], [_rows(int(g["tokens"]))])
    assert len(cm.block_table(s)) == g["blocks"]
    assert len(cm.block_table(s)) * g["block_tokens"] - cm.length(s) == g["free_slots_in_tail"]


def test_tail_waste_is_below_one_page(golden):
    g = golden("page_arithmetic.txt")
    rng = np.random.default_rng(0)
    cm = _cm(pages=400, seqs=20, per_seq=64)
    for _ in range(20):
        s = cm.create()
        L = int(rng.integers(1, 1000))
        cm.write([s], [_rows(L)], [_rows(L)])
        waste = len(cm.block_table(s)) * 16 - L
        assert 0 <= waste <= g["max_tail_waste"]
        cm.free_seq(s)


def test_shape_ledger_cache_scalars(golden):
    g = golden("shape_ledger.txt")
    n, H_kv, d, layers = int(g["n"]), int(g["H_kv"]), int(g["d_h"]), int(g["layers"])
    total = 0
    for _ in range(layers):          # one cache per layer
        cm = oracle.CacheModel(8, 1, 8, H_kv, d, "f32")
        s = cm.create()
        cm.write([s], [_rows(n, H_kv, d)], [_rows(n, H_kv, d)])
        K, V = cm.kv(s)
        total += K.size + V.size
    assert total == g["cache_scalars"]


def test_identity_order_hands_out_lowest_pages_first():
    cm = _cm()
    a, b = cm.create(), cm.create()
    cm.write([a, b], [_rows(20), _rows(33)], [_rows(20), _rows(33)])
    assert cm.block_table(a) == [0, 1]
    assert cm.block_table(b) == [2, 3, 4]


def test_permuted_order_is_followed():
    order = [5, 3, 7, 0, 1, 2, 4, 6]
    cm = _cm(pages=8, order=order)
    a = cm.create()
    cm.write([a], [_rows(40)], [_rows(40)])
    assert cm.block_table(a) == [5, 3, 7]
    cm.truncate(a, 17)                 # releases page 7
    b = cm.create()
    cm.write([b], [_rows(16)], [_rows(16)])
    assert cm.block_table(b) == [7]    # smallest free rank again


def test_fork_shares_pages_and_copy_on_write_on_shared_tail():
    cm = _cm()
    a = cm.create()
    cm.write([a], [_rows(20)], [_rows(20)])
    b = cm.fork(a, 20)
    assert cm.block_table(b) == cm.block_table(a) == [0, 1]
    assert cm.ref[0] == 2 and cm.ref[1] == 2
    cm.write([b], [_rows(1, base=100)], [_rows(1, base=100)])
    assert cm.block_table(b) == [0, 2]          # tail page copied to page 2
    assert cm.copies[-1] == (1, 2, 4)           # slots 0..3 copied
    assert cm.ref[1] == 1 and cm.ref[2] == 1
    Ka, _ = cm.kv(a)
    Kb, _ = cm.kv(b)
    assert Ka.shape[0] == 20 and Kb.shape[0] == 21
    assert np.array_equal(Ka, Kb[:20])


def test_page_aligned_fork_needs_no_copy():
    cm = _cm()
    a = cm.create()
    cm.write([a], [_rows(32)], [_rows(32)])
    b = cm.fork(a, 32)
    cm.write([b], [_rows(3)], [_rows(3)])
    assert cm.block_table(b) == [0, 1, 2]
    assert cm.copies == []


def test_truncate_releases_and_frees_at_zero_references():
    cm = _cm()
    a = cm.create()
    cm.write([a], [_rows(64)], [_rows(64)])
    b = cm.fork(a, 64)
    cm.truncate(a, 0)
    assert cm.free_pages() == 32 - 4           # b still holds all four
    cm.truncate(b, 17)
    assert cm.free_pages() == 32 - 2
    assert cm.block_table(b) == [0, 1]
    cm.free_seq(b)
    assert cm.free_pages() == 32


def test_truncate_bounds():
    cm = _cm()
    a = cm.create()
    cm.write([a], [_rows(5)], [_rows(5)])
    with pytest.raises(oracle.CacheError) as e:
        cm.truncate(a, 6)
    assert e.value.kind == "ERANGE"
    cm.truncate(a, 5)
    assert cm.length(a) == 5


def test_pool_exhaustion_changes_nothing():
    cm = _cm(pages=4)
    a, b = cm.create(), cm.create()
    cm.write([a], [_rows(40)], [_rows(40)])       # 3 pages
    before = (cm.block_table(a), cm.free_pages())
    with pytest.raises(oracle.CacheError) as e:
        cm.write([a, b], [_rows(8), _rows(17)], [_rows(8), _rows(17)])
    assert e.value.kind == "ENOMEM"
    assert (cm.block_table(a), cm.free_pages()) == before
    assert cm.length(a) == 40 and cm.length(b) == 0


def test_sequence_capacity_is_enforced():
    cm = _cm(per_seq=2)
    a = cm.create()
    with pytest.raises(oracle.CacheError) as e:
        cm.write([a], [_rows(33)], [_rows(33)])
    assert e.value.kind == "ERANGE"


def test_duplicate_sequence_in_one_write_is_rejected():
    cm = _cm()
    a = cm.create()
    with pytest.raises(oracle.CacheError):
        cm.write([a, a], [_rows(1), _rows(1)], [_rows(1), _rows(1)])


def test_gather_through_permuted_table_restores_logical_order():
    # Physical placement differs, logical content does not: scatter every
    # token into a pool image through the block table and gather it back.
    order = np.random.default_rng(1).permutation(16)
    cm = _cm(pages=16, order=order)
    a = cm.create()
    K = _rows(70)
    cm.write([a], [K], [K])
    pool = np.full((16, 16, 1, 2), np.nan, dtype=np.float32)
    bt = cm.block_table(a)
    for t in range(70):
        pool[bt[t // 16], t % 16] = K[t]
    back = np.stack([pool[bt[t // 16], t % 16] for t in range(70)])
    assert np.array_equal(back, K)
    assert bt != sorted(bt)
