"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
header declares, and its host-side logic (validation, allocator, reference
counts, copy-on-write planning, truncation) agrees with the oracle's cache
model.  Metadata-only caches need no GPU and queue no device work."""
import copy
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gqa.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    body = text[text.index('extern "C" {'):]
    names = re.findall(r"^(?:const\s+)?(?:int|size_t|char|void)\s*\*?\s*(\w+)\s*\(", body, re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "attn_prefill" in names and "attn_decode" in names and "kv_truncate" in names
    lib = ctypes.CDLL(gqa.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(gqa.exported_symbols()) == names


def test_version_string():
    assert "sm_103a" in gqa.version()


def _pair(pages=64, seqs=8, per_seq=32, H_kv=2, d=8, order=None, window=0):
    lib = gqa.Cache(H_kv, d, pages, seqs, per_seq, dtype="f32", page_order=order, metadata_only=True,
                    window=window)
    model = oracle.CacheModel(pages, seqs, per_seq, H_kv, d, "f32", page_order=order, window=window)
    return lib, model


def _same_state(lib, model):
    for s in model.seqs:
        assert lib.seq_length(s) == model.length(s)
        assert lib.block_table(s) == model.block_table(s)
    assert lib.free_pages() == model.free_pages()
    for p in range(model.num_pages):
        assert lib.refcount(p) == model.ref[p]


def _rows(c, H_kv=2, d=8):
    return np.zeros((c, H_kv, d), dtype=np.float32)


@pytest.mark.parametrize("window", [0, 1, 16, 37])
def test_allocator_matches_oracle_model_under_random_operations(window):
    # With a sliding window the model releases pages wholly before the window
    # after every write and refuses rewinds past it; the library must agree.
    rng = np.random.default_rng(7 + window)
    order = rng.permutation(96)
    lib, model = _pair(pages=96, seqs=6, per_seq=40, order=order, window=window)
    live = []
    released_seen, refusals = False, 0
    for step in range(400):
        op = rng.integers(0, 6)
        try:
            if op == 0 or not live:
                s_m = model.create()
                s_l = lib.seq_create()
                assert s_l == s_m
                live.append(s_m)
            elif op == 1:                                     # batched prefill
                batch = list(rng.choice(live, size=min(len(live), int(rng.integers(1, 4))), replace=False))
                n = int(rng.integers(1, 40))
                nb = [int(rng.integers(1, n + 1)) for _ in batch]
                err_m = err_l = None
                try:
                    model.write(batch, [_rows(x) for x in nb], [_rows(x) for x in nb])
                except oracle.CacheError as e:
                    err_m = e.kind
                try:
                    gqa.attn_prefill_meta(lib, batch, n, 4, nb)
                except gqa.GqaError as e:
                    err_l = e.name
                assert err_m == err_l
            elif op == 2:                                     # append
                batch = list(rng.choice(live, size=min(len(live), int(rng.integers(1, 4))), replace=False))
                cnt = [int(rng.integers(0, 3)) for _ in batch]
                err_m = err_l = None
                try:
                    model.write(batch, [_rows(x) for x in cnt], [_rows(x) for x in cnt])
                except oracle.CacheError as e:
                    err_m = e.kind
                try:
                    gqa.kv_append_meta(lib, batch, 2, cnt)
                except gqa.GqaError as e:
                    err_l = e.name
                assert err_m == err_l
            elif op == 3:                                     # fork
                src = int(rng.choice(live))
                k = int(rng.integers(0, model.length(src) + 1))
                try:
                    s_m = model.fork(src, k)
                except oracle.CacheError as e:
                    with pytest.raises(gqa.GqaError) as el:
                        lib.seq_fork(src, k)
                    assert el.value.name == e.kind
                    assert e.kind == "ENOMEM" or (e.kind == "ERANGE" and window > 0)
                else:
                    assert lib.seq_fork(src, k) == s_m
                    live.append(s_m)
            elif op == 4:                                     # truncate
                s = int(rng.choice(live))
                m = int(rng.integers(0, model.length(s) + 1))
                try:
                    model.truncate(s, m)
                except oracle.CacheError as e:
                    assert e.kind == "ERANGE" and window > 0
                    refusals += 1
                    with pytest.raises(gqa.GqaError) as el:
                        gqa.kv_truncate(lib, s, m)
                    assert el.value.name == "ERANGE"
                else:
                    gqa.kv_truncate(lib, s, m)
            else:                                             # free
                s = int(rng.choice(live))
                model.free_seq(s)
                lib.seq_free(s)
                live.remove(s)
        except oracle.CacheError as e:
            assert e.kind == "ENOMEM"
            with pytest.raises(gqa.GqaError):
                lib.seq_create()
        _same_state(lib, model)
        released_seen |= any(-1 in model.block_table(s) for s in model.seqs)
    assert len(model.copies) > 0          # copy-on-write was exercised
    if window > 0:                        # pages were released and rewinds refused
        assert released_seen and refusals > 0


@pytest.mark.parametrize("call", ["attn_prefill_meta", "attn_prefill_host_meta"])
def test_prefill_rejections_change_nothing(call):
    prefill = getattr(gqa, call)
    lib, model = _pair(pages=7, per_seq=4)
    a, b = lib.seq_create(), lib.seq_create()
    gqa.attn_prefill_meta(lib, [a], 20, 4, [20])
    before = (lib.block_table(a), lib.seq_length(a), lib.free_pages())
    cases = [
        (dict(seq_ids=[a], n=8, H_q=4, valid_lengths=[0]), "EMASK"),          # no valid row
        (dict(seq_ids=[a], n=8, H_q=4, valid_lengths=[9]), "EMASK"),          # more valid rows than n
        (dict(seq_ids=[a], n=8, H_q=3, valid_lengths=[8]), "EINVAL"),         # H_kv does not divide H_q
        (dict(seq_ids=[a, a], n=8, H_q=4, valid_lengths=[1, 1]), "EINVAL"),   # duplicate sequence
        (dict(seq_ids=[5], n=8, H_q=4, valid_lengths=[1]), "EINVAL"),         # not live
        (dict(seq_ids=[a], n=64, H_q=4, valid_lengths=[64]), "ERANGE"),       # past 4 pages/seq
        (dict(seq_ids=[a, b], n=64, H_q=4, valid_lengths=[30, 64]), "ENOMEM"),
        (dict(seq_ids=[a], n=4, H_q=4, valid_lengths=[4],
              positions=np.arange(4, dtype=np.int32)[None]), "ERANGE"),     # positions restart at 0
    ]
    for kw, want in cases:
        with pytest.raises(gqa.GqaError) as e:
            prefill(lib, **kw)
        assert e.value.name == want, (kw, e.value)
        assert (lib.block_table(a), lib.seq_length(a), lib.free_pages()) == before
    # Correct positions are accepted.
    prefill(lib, [a], 4, 4, [3], positions=np.array([[20, 21, 22, 999]], dtype=np.int32))
    assert lib.seq_length(a) == 23


@pytest.mark.parametrize("window", [0, 48])
def test_host_buffer_prefill_bookkeeping(window):
    # attn_prefill_host checks the whole batch like attn_prefill, then runs
    # its entries as one-entry prefills, longest first (ties in batch order):
    # pages, tables and refusals must match the model doing exactly that.
    rng = np.random.default_rng(11 + window)
    lib, model = _pair(pages=30, seqs=6, per_seq=12, order=rng.permutation(30), window=window)
    ids = [lib.seq_create() for _ in range(5)]
    assert ids == [model.create() for _ in range(5)]
    refusals = 0
    for step in range(150):
        batch = [int(x) for x in rng.choice(ids, size=int(rng.integers(1, 4)), replace=False)]
        n = int(rng.integers(1, 40))
        nb = [int(rng.integers(1, n + 1)) for _ in batch]
        err_m = err_l = None
        try:
            copy.deepcopy(model).write(batch, [_rows(x) for x in nb], [_rows(x) for x in nb])
        except oracle.CacheError as e:
            err_m = e.kind
        if err_m is None:
            for i in sorted(range(len(batch)), key=lambda i: -nb[i]):
                model.write([batch[i]], [_rows(nb[i])], [_rows(nb[i])])
        try:
            gqa.attn_prefill_host_meta(lib, batch, n, 4, nb)
        except gqa.GqaError as e:
            err_l = e.name
        assert err_m == err_l
        refusals += err_m is not None
        _same_state(lib, model)
        if rng.random() < 0.15:
            s = int(rng.choice(ids))
            gqa.kv_truncate(lib, s, 0)
            model.truncate(s, 0)
            _same_state(lib, model)
    assert refusals > 0


def test_decode_rejects_an_empty_sequence():
    lib, _ = _pair()
    a = lib.seq_create()
    with pytest.raises(gqa.GqaError) as e:
        gqa.attn_decode_meta(lib, [a], 4)
    assert e.value.name == "EMASK"
    gqa.kv_append_meta(lib, [a], 1)
    gqa.attn_decode_meta(lib, [a, a], 4)       # repeats are fine for a read


def test_truncate_and_fork_bounds():
    lib, _ = _pair()
    a = lib.seq_create()
    gqa.kv_append_meta(lib, [a], 5)
    for bad in (-1, 6):
        with pytest.raises(gqa.GqaError) as e:
            gqa.kv_truncate(lib, a, bad)
        assert e.value.name == "ERANGE"
        with pytest.raises(gqa.GqaError) as e:
            lib.seq_fork(a, bad)
        assert e.value.name == "ERANGE"


def test_layout_metadata_and_compatibility():
    lib, _ = _pair()
    m = lib.layout()
    assert m.keys_post_position == 1 and m.page_tokens == 16 and m.layout_version == gqa.LAYOUT_VERSION
    assert gqa.layout_compatible(m, lib.layout())
    other = gqa.LayoutMetadata(**m.as_dict())
    other.keys_post_position = 0
    assert not gqa.layout_compatible(m, other)
    other = gqa.LayoutMetadata(**m.as_dict())
    other.dtype = gqa.DTYPE_BF16
    assert not gqa.layout_compatible(m, other)
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 8, 8, 2, 2, dtype="f32", metadata_only=True, keys_post_position=0)
    assert e.value.name == "ELAYOUT"
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 8, 8, 2, 2, dtype="f32", metadata_only=True, layout_version=99)
    assert e.value.name == "ELAYOUT"


def test_pre_position_layout_rules():
    # Keys stored before the position transform ([P1] 2.5) need the
    # library's own position mechanism to rotate them when read.
    pre = gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, rope=True, keys_post_position=0)
    m = pre.layout()
    assert m.keys_post_position == 0 and m.rope == 1
    post = gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, rope=True).layout()
    assert post.keys_post_position == 1
    # a post-position reader refuses a pre-position cache and the reverse
    import ctypes
    assert gqa._lib.gqa_layout_compatible(ctypes.byref(post), ctypes.byref(m)) == gqa.ELAYOUT
    assert gqa._lib.gqa_layout_compatible(ctypes.byref(m), ctypes.byref(post)) == gqa.ELAYOUT
    assert gqa.layout_compatible(m, pre.layout())
    # without a position mechanism there is nothing to apply at read
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, keys_post_position=0)
    assert e.value.name == "ELAYOUT"
    # prefill, append and decode bookkeeping as for any cache
    s = pre.seq_create()
    gqa.attn_prefill_meta(pre, [s], 20, 4, [20])
    assert pre.seq_length(s) == 20


def test_rope_description_checks_and_layout():
    m = gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, rope=True, rope_base=500.0).layout()
    assert m.rope == 1 and m.rope_base == 500.0
    plain = gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True).layout()
    assert plain.rope == 0
    assert not gqa.layout_compatible(m, plain)
    other = gqa.LayoutMetadata(**m.as_dict())
    other.rope_base = 10000.0
    assert not gqa.layout_compatible(m, other)
    assert gqa.layout_compatible(m, gqa.LayoutMetadata(**m.as_dict()))
    for kw in ({"head_dim": 7}, {"rope_base": 1.0}, {"rope_base": 0.5}, {"rope_base": float("inf")}):
        args = dict(num_kv_heads=2, head_dim=8, num_pages=8, max_seqs=2, max_pages_per_seq=2, dtype="bf16",
                    metadata_only=True, rope=True, rope_base=10000.0)
        args.update(kw)
        with pytest.raises(gqa.GqaError) as e:
            gqa.Cache(**args)
        assert e.value.name == "EINVAL", kw
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, rope=2)
    assert e.value.name == "EINVAL"


def test_page_order_must_be_a_permutation():
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(1, 4, 4, 2, 2, dtype="f32", metadata_only=True, page_order=[0, 1, 1, 2])
    assert e.value.name == "EINVAL"


def test_sequence_ids_run_out():
    lib, _ = _pair(seqs=2)
    lib.seq_create(); lib.seq_create()
    with pytest.raises(gqa.GqaError) as e:
        lib.seq_create()
    assert e.value.name == "ENOMEM"


def test_causal_pair_counts_match_the_toy_decoder(golden):
    # Full recompute at context lengths 4, 5, 6, 7 versus prefill of 4 then
    # three cached single-token steps, per query head and layer.
    g = golden("work_counts.txt")
    W = gqa.work
    P, steps = int(g["prompt"]), int(g["decode_steps"])
    per = int(g["layers"]) * int(g["query_heads"])
    full = sum(W.causal_pairs(0, P + t) for t in range(steps + 1))
    cached = W.causal_pairs(0, P) + sum(W.causal_pairs(P + t, 1) for t in range(steps))
    assert per * full == g["score_pairs_full_recompute"]
    assert per * cached == g["score_pairs_cached"]


def test_window_description_checks_and_layout():
    m = gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, window=100).layout()
    assert m.window == 100
    plain = gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True).layout()
    assert plain.window == 0
    assert not gqa.layout_compatible(m, plain)
    assert gqa.layout_compatible(m, gqa.LayoutMetadata(**m.as_dict()))
    with pytest.raises(gqa.GqaError) as e:
        gqa.Cache(2, 8, 8, 2, 2, dtype="bf16", metadata_only=True, window=-1)
    assert e.value.name == "EINVAL"


def test_window_rewinds_need_the_window_held():
    # W = 40, 215 tokens: pages 0..9 (positions < 160) are released, so a
    # rewind to m needs m - 40 >= 160.
    lib, model = _pair(pages=20, per_seq=16, window=40)
    a = lib.seq_create()
    model.create()
    gqa.kv_append_meta(lib, [a], 215)
    model.write([a], [_rows(215)], [_rows(215)])
    _same_state(lib, model)
    assert lib.block_table(a)[:10] == [-1] * 10
    for m in (1, 150, 199):                 # (m = 0 empties the sequence: always allowed)
        for call in (lambda: gqa.kv_truncate(lib, a, m), lambda: lib.seq_fork(a, m)):
            with pytest.raises(gqa.GqaError) as e:
                call()
            assert e.value.name == "ERANGE", m
    f = lib.seq_fork(a, 205)
    assert lib.block_table(f) == lib.block_table(a)[:13]
    gqa.kv_truncate(lib, a, 200)
    assert lib.seq_length(a) == 200 and lib.seq_length(f) == 205


def test_windowed_work_counts_match_brute_force():
    # The throughput accounting counts the pairs the oracle's dense form
    # leaves visible: keys max(0, p - W + 1)..p of each position p.
    for past in (0, 1, 15, 40, 130):
        for new in (0, 1, 17, 64):
            for W in (0, 1, 2, 16, 37, 200):
                qpos = np.arange(past, past + new)
                j = np.arange(past + new)
                vis = j[None, :] <= qpos[:, None]
                if W > 0:
                    vis &= j[None, :] > qpos[:, None] - W
                assert gqa.work.causal_pairs(past, new, W) == int(vis.sum()), (past, new, W)
    assert gqa.work.decode_kv_bytes([10, 100], 2, 8, 2, window=16) == (10 + 16) * 2 * 2 * 8 * 2


def test_decode_kernel_choice_is_checked():
    c = gqa.Cache(2, 8, 8, 2, 2, dtype="f32", metadata_only=True)
    c.set_decode_kernel("cuda_core")
    c.set_decode_kernel("auto")
    with pytest.raises(gqa.GqaError) as e:          # the tensor-core kernel is bf16, d_h = 128 only
        c.set_decode_kernel("tensor_core")
    assert e.value.name == "EINVAL"
    with pytest.raises(gqa.GqaError) as e:
        gqa._check(gqa._lib.gqa_set_decode_kernel(c.handle, 7))
    assert e.value.name == "EINVAL"
    b = gqa.Cache(2, 128, 8, 2, 2, dtype="bf16", metadata_only=True)
    b.set_decode_kernel("tensor_core")


def test_fused_decode_step_bookkeeping_matches_append():
    lib, model = _pair(pages=10, per_seq=6)
    a, b = lib.seq_create(), lib.seq_create()
    model.create(), model.create()
    gqa.kv_append_meta(lib, [a, b], 16, [15, 3])
    model.write([a, b], [_rows(15), _rows(3)], [_rows(15), _rows(3)])
    for t in range(20):
        gqa.attn_decode_append_meta(lib, [a, b], 4)
        model.write([a, b], [_rows(1), _rows(1)], [_rows(1), _rows(1)])
        _same_state(lib, model)
    with pytest.raises(gqa.GqaError) as e:                      # distinct sequences, as for a write
        gqa.attn_decode_append_meta(lib, [a, a], 4)
    assert e.value.name == "EINVAL"


def test_fp8_cache_description_and_pool_size():
    c = gqa.Cache(2, 128, 8, 2, 4, dtype="fp8", metadata_only=True)
    m = c.layout()
    assert m.dtype == gqa.DTYPE_FP8_E4M3
    assert not gqa.layout_compatible(m, gqa.Cache(2, 128, 8, 2, 4, dtype="bf16", metadata_only=True).layout())
    # Blocks of 16 one-byte rows of d_h codes, then one fp32 scale per row.
    assert gqa._lib.gqa_pool_bytes(ctypes.byref(c.desc)) == 8 * 2 * 2 * 16 * 128 + 8 * 2 * 2 * 16 * 4
    d96 = gqa.Cache(1, 96, 4, 1, 2, dtype="fp8", metadata_only=True)
    assert gqa._lib.gqa_pool_bytes(ctypes.byref(d96.desc)) == 4 * 2 * 16 * 128 + 4 * 2 * 16 * 4
    for kw in ({"head_dim": 100}, {"head_dim": 130}, {"rope": True}):
        args = dict(num_kv_heads=2, head_dim=128, num_pages=8, max_seqs=2, max_pages_per_seq=4, dtype="fp8",
                    metadata_only=True)
        args.update(kw)
        with pytest.raises(gqa.GqaError) as e:
            gqa.Cache(**args)
        assert e.value.name == "EINVAL", kw


def test_bounded_wait_selftest_arguments():
    c = gqa.Cache(2, 128, 8, 2, 4, dtype="bf16", metadata_only=True)
    with pytest.raises(gqa.GqaError) as e:
        c.selftest_bounded_wait(1000)
    assert e.value.name == "EINVAL"
    with pytest.raises(gqa.GqaError) as e:
        gqa._check(gqa._lib.gqa_selftest_bounded_wait(c.handle, 0, None))
    assert e.value.name == "ERANGE"
