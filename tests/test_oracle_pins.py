"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong scale, a wrong head map, a future key in the denominator, a transposed
operand) fails at least one of them.  None of them re-types the oracle's own
formula: they use printed values, closed forms, special cases and a second,
independently written form.
"""
import math

import numpy as np
import pytest

import oracle
import workloads


def _att(q, K, V, qpos):
    return oracle.attention(np.asarray(q, float), np.asarray(K, float), np.asarray(V, float),
                            np.asarray(qpos), nthreads=2)


# ---------------------------------------------------------------- worked example

def test_worked_example_second_position(golden):
    g = golden("worked_example_2d.txt")
    q = np.array([[g["q"]]])
    K = np.array([[g["k1"]], [g["k2"]]])
    V = np.array([[g["v1"]], [g["v2"]]])
    out = _att(q, K, V, [1])[0, 0]
    tol = 0.5 * 10 ** -int(g["decimals_out"])
    assert np.all(np.abs(out - np.array(g["out_pos2"])) <= tol), out
    # The weights: out = p1 v1 + p2 v2 with v1 = (10, 0), v2 = (0, 20).
    tol_p = 0.5 * 10 ** -int(g["decimals_p"])
    assert abs(out[0] / 10.0 - g["p1"]) <= tol_p
    assert abs(out[1] / 20.0 - g["p2"]) <= tol_p


def test_worked_example_first_position_excludes_future(golden):
    g = golden("worked_example_2d.txt")
    q = np.array([[g["q"]]])
    K = np.array([[g["k1"]], [g["k2"]]])
    V = np.array([[g["v1"]], [g["v2"]]])
    out = _att(q, K, V, [0])[0, 0]
    # Exactly v1: the second position must not enter the denominator either.
    assert np.array_equal(out, np.array(g["out_pos1"]))


def test_worked_example_scores_imply_weights(golden):
    # The page's printed scores (q.k/sqrt(2)) and weights agree with each other
    # through the two-element softmax (a logistic): an independent check that
    # the fixture was transcribed consistently.
    g = golden("worked_example_2d.txt")
    p1 = 1.0 / (1.0 + math.exp(g["score2"] - g["score1"]))
    assert abs(p1 - g["p1"]) <= 0.5e-6
    assert abs(g["score1"] - 1 / math.sqrt(2)) <= 0.5e-6


def test_workloads_worked_example_matches_fixture(golden):
    g = golden("worked_example_2d.txt")
    w = workloads.worked_example_2d()
    assert np.array_equal(w["k"][0, :, 0], np.array([g["k1"], g["k2"]], dtype=np.float32))
    assert np.array_equal(w["v"][0, :, 0], np.array([g["v1"], g["v2"]], dtype=np.float32))
    assert np.array_equal(w["q"][0, 1, 0], np.array(g["q"], dtype=np.float32))


# ---------------------------------------------------------------- closed forms

def test_scale_is_inverse_root_head_dim():
    # d = 4: q.k1 = 2 so the score is 2/sqrt(4) = 1; q.k2 = 0.  Two-key softmax
    # weight of key 1 is the logistic e/(e+1) = 0.7310585786300049.
    q = [[[2.0, 0, 0, 0]]]
    K = [[[1.0, 0, 0, 0]], [[0.0, 0, 0, 0]]]
    V = [[[1.0, 0, 0, 0]], [[0.0, 1, 0, 0]]]
    out = _att(q, K, V, [1])[0, 0]
    assert abs(out[0] - 0.7310585786300049) < 1e-15
    assert abs(out[1] - 0.2689414213699951) < 1e-15
    assert out[2] == 0 and out[3] == 0


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(1)
    q, K, V = rng.normal(size=(1, 3, 8)), rng.normal(size=(5, 1, 8)), rng.normal(size=(5, 1, 8))
    out = _att(q, K, V, [0])
    for h in range(3):
        assert np.array_equal(out[0, h], V[0, 0])


def test_zero_query_averages_visible_values():
    rng = np.random.default_rng(2)
    K, V = rng.normal(size=(9, 2, 6)), rng.normal(size=(9, 2, 6))
    q = np.zeros((3, 4, 6))
    pos = [0, 4, 8]
    out = _att(q, K, V, pos)
    for i, p in enumerate(pos):
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(out[i, h], V[: p + 1, g].mean(axis=0), rtol=0, atol=1e-14)


def test_identical_values_pass_through():
    rng = np.random.default_rng(3)
    c = rng.normal(size=5)
    K = rng.normal(size=(7, 1, 5))
    V = np.broadcast_to(c, (7, 1, 5)).copy()
    out = _att(rng.normal(size=(4, 2, 5)), K, V, [0, 2, 5, 6])
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-14)


def test_two_keys_logistic_large_scores_stable():
    # Scores around 700 would overflow exp() without the max subtraction; the
    # weights still follow the two-element closed form.
    d = 2
    q = [[[1.0, 0.0]]]
    K = [[[990.0, 0.0]], [[991.0, 0.0]]]
    V = [[[1.0, 0.0]], [[0.0, 1.0]]]
    out = _att(q, K, V, [1])[0, 0]
    s1, s2 = 990 / math.sqrt(d), 991 / math.sqrt(d)
    p1 = 1.0 / (1.0 + math.exp(s2 - s1))
    assert np.all(np.isfinite(out))
    assert abs(out[0] - p1) < 1e-14 and abs(out[1] - (1 - p1)) < 1e-14


def test_common_key_shift_leaves_output_unchanged():
    # Adding the same vector u to every key adds q.u/sqrt(d) to the whole row
    # of scores; softmax is invariant to that.
    rng = np.random.default_rng(4)
    q, K, V = rng.normal(size=(5, 4, 8)), rng.normal(size=(12, 2, 8)), rng.normal(size=(12, 2, 8))
    u = rng.normal(size=(1, 2, 8)) * 3
    pos = [3, 5, 7, 9, 11]
    np.testing.assert_allclose(_att(q, K + u, V, pos), _att(q, K, V, pos), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- GQA head map

@pytest.mark.parametrize("H_q,H_kv,expect", [
    (4, 2, [0, 0, 1, 1]),
    (6, 2, [0, 0, 0, 1, 1, 1]),
    (6, 3, [0, 0, 1, 1, 2, 2]),
    (3, 3, [0, 1, 2]),
    (4, 1, [0, 0, 0, 0]),
])
def test_query_heads_read_contiguous_kv_groups(H_q, H_kv, expect):
    # KV head g holds constant value rows equal to (g+1) * ones, so each query
    # head's output names the KV head it read.  Contiguous groups of H_q/H_kv
    # query heads share a KV head (the toy model's heads 0 and 1 both read KV
    # head 0; a kernel indexes the KV head rather than duplicating it).
    rng = np.random.default_rng(5)
    d, L = 4, 6
    V = np.stack([np.full((L, d), g + 1.0) for g in range(H_kv)], axis=1)
    out = _att(rng.normal(size=(2, H_q, d)), rng.normal(size=(L, H_kv, d)), V, [3, 5])
    got = [int(round(out[0, h, 0])) - 1 for h in range(H_q)]
    assert got == expect


def test_permuting_query_heads_within_a_group_permutes_outputs():
    rng = np.random.default_rng(6)
    q, K, V = rng.normal(size=(3, 8, 16)), rng.normal(size=(10, 2, 16)), rng.normal(size=(10, 2, 16))
    pos = [2, 6, 9]
    perm = [3, 1, 0, 2, 7, 5, 4, 6]           # stays inside the two groups of 4
    a = _att(q, K, V, pos)
    b = _att(q[:, perm], K, V, pos)
    assert np.array_equal(a[:, perm], b)


# ---------------------------------------------------------------- causality

def test_future_keys_do_not_change_a_row():
    rng = np.random.default_rng(7)
    q, K, V = rng.normal(size=(4, 2, 8)), rng.normal(size=(10, 1, 8)), rng.normal(size=(10, 1, 8))
    pos = [0, 3, 6, 9]
    a = _att(q, K, V, pos)
    K2, V2 = K.copy(), V.copy()
    K2[7:] = rng.normal(size=K2[7:].shape) * 100
    V2[7:] = np.nan                              # never read for rows at positions <= 6
    b = _att(q[:3], K2, V2, pos[:3])
    assert np.array_equal(a[:3], b)


def test_streaming_matches_dense_masked_form():
    rng = np.random.default_rng(8)
    for (n_q, H_q, H_kv, d, L) in [(1, 1, 1, 1, 1), (3, 2, 1, 4, 3), (6, 6, 2, 5, 9),
                                   (5, 8, 8, 3, 12), (4, 12, 3, 7, 20)]:
        q = rng.normal(size=(n_q, H_q, d))
        K, V = rng.normal(size=(L, H_kv, d)), rng.normal(size=(L, H_kv, d))
        pos = np.sort(rng.choice(L, size=n_q, replace=n_q > L))
        np.testing.assert_allclose(_att(q, K, V, pos), oracle.attention_dense(q, K, V, pos),
                                   rtol=0, atol=1e-13)


def test_brute_force_pure_python_tiny():
    # Plain nested loops over Python floats: math.exp of scores minus the row max.
    rng = np.random.default_rng(9)
    H_q, H_kv, d, L = 2, 1, 3, 5
    q, K, V = rng.normal(size=(L, H_q, d)), rng.normal(size=(L, H_kv, d)), rng.normal(size=(L, H_kv, d))
    out = _att(q, K, V, list(range(L)))
    for i in range(L):
        for h in range(H_q):
            sc = [sum(q[i, h, e] * K[j, 0, e] for e in range(d)) / math.sqrt(d) for j in range(i + 1)]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            ref = [sum(w[j] * V[j, 0, e] for j in range(i + 1)) / sum(w) for e in range(d)]
            np.testing.assert_allclose(out[i, h], ref, rtol=0, atol=1e-14)


def test_rejects_rows_without_visible_keys():
    with pytest.raises(ValueError):
        _att(np.zeros((1, 1, 2)), np.zeros((2, 1, 2)), np.zeros((2, 1, 2)), [2])
    with pytest.raises(ValueError):
        _att(np.zeros((1, 1, 2)), np.zeros((2, 1, 2)), np.zeros((2, 1, 2)), [-1])
    with pytest.raises(ValueError):   # H_kv must divide H_q
        _att(np.zeros((1, 3, 2)), np.zeros((2, 2, 2)), np.zeros((2, 2, 2)), [1])


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(10)
    q, K, V = rng.normal(size=(7, 4, 8)), rng.normal(size=(30, 2, 8)), rng.normal(size=(30, 2, 8))
    pos = np.arange(23, 30)
    a = oracle.attention(q, K, V, pos, nthreads=1)
    b = oracle.attention(q, K, V, pos, nthreads=5)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- cache drivers

def _model(dtype="f32", H_kv=1, d=4, pages=64):
    return oracle.CacheModel(pages, 8, 32, H_kv, d, dtype)


def test_decode_equals_last_row_of_full_recompute():
    # Cached decode must reproduce the last row of recomputing the whole
    # context: the toy decoder compares these after every step.
    w = workloads.tiny_fp32()
    cm = _model()
    s = cm.create()
    oracle.prefill(cm, [s], w["q"], w["k"], w["v"], w["valid_lengths"])
    allq, allk, allv = [w["q"][0]], [w["k"][0]], [w["v"][0]]
    for t in range(3):
        oracle.append(cm, [s], w["dec_k"][t], w["dec_v"][t])
        got = oracle.decode(cm, [s], w["dec_q"][t])[0]
        allq.append(w["dec_q"][t]); allk.append(w["dec_k"][t]); allv.append(w["dec_v"][t])
        Q = np.concatenate(allq).astype(float)
        Kf = np.concatenate(allk).astype(float)
        Vf = np.concatenate(allv).astype(float)
        L = Kf.shape[0]
        full = oracle.attention_dense(Q, Kf, Vf, np.arange(L))
        assert L == 5 + t
        np.testing.assert_allclose(got, full[-1], rtol=0, atol=1e-12)


def test_incremental_prefill_equals_one_shot_prefill():
    rng = np.random.default_rng(11)
    n1, n2, H_q, H_kv, d = 5, 7, 4, 2, 6
    q, k, v = rng.normal(size=(1, n1 + n2, H_q, d)), rng.normal(size=(1, n1 + n2, H_kv, d)), rng.normal(size=(1, n1 + n2, H_kv, d))
    q, k, v = (x.astype(np.float32) for x in (q, k, v))
    a = _model(H_kv=H_kv, d=d)
    s = a.create()
    one = oracle.prefill(a, [s], q, k, v, [n1 + n2])[0]
    b = _model(H_kv=H_kv, d=d)
    t = b.create()
    first = oracle.prefill(b, [t], q[:, :n1], k[:, :n1], v[:, :n1], [n1])[0]
    second = oracle.prefill(b, [t], q[:, n1:], k[:, n1:], v[:, n1:], [n2])[0]
    np.testing.assert_allclose(np.concatenate([first, second]), one, rtol=0, atol=1e-13)
    assert np.array_equal(a.raw_kv(s)[0], b.raw_kv(t)[0])


def test_padding_rows_never_matter():
    rng = np.random.default_rng(12)
    B, n, H_q, H_kv, d = 2, 9, 4, 2, 5
    q = rng.normal(size=(B, n, H_q, d)).astype(np.float32)
    k = rng.normal(size=(B, n, H_kv, d)).astype(np.float32)
    v = rng.normal(size=(B, n, H_kv, d)).astype(np.float32)
    nb = [4, 9]
    a = _model(H_kv=H_kv, d=d)
    sa = [a.create(), a.create()]
    ref = oracle.prefill(a, sa, q, k, v, nb)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[0, 4:], k2[0, 4:], v2[0, 4:] = np.nan, np.inf, np.nan
    b = _model(H_kv=H_kv, d=d)
    sb = [b.create(), b.create()]
    got = oracle.prefill(b, sb, q2, k2, v2, nb)
    assert np.array_equal(ref, got)
    assert np.all(got[0, 4:] == 0)
    assert a.length(sa[0]) == 4 and a.length(sa[1]) == 9


def test_edit_at_m_keeps_rows_before_m():
    # Changing the rows at positions >= m leaves every output row < m and the
    # cached K/V < m untouched (prefix stable, suffix invalid).
    rng = np.random.default_rng(13)
    n, m, H_q, H_kv, d = 24, 10, 4, 2, 6
    q = rng.normal(size=(1, n, H_q, d)).astype(np.float32)
    k = rng.normal(size=(1, n, H_kv, d)).astype(np.float32)
    v = rng.normal(size=(1, n, H_kv, d)).astype(np.float32)
    a = _model(H_kv=H_kv, d=d)
    s = a.create()
    ref = oracle.prefill(a, [s], q, k, v, [n])[0]
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for x in (q2, k2, v2):
        x[0, m:] = rng.normal(size=x[0, m:].shape)
    b = _model(H_kv=H_kv, d=d)
    t = b.create()
    got = oracle.prefill(b, [t], q2, k2, v2, [n])[0]
    assert np.array_equal(ref[:m], got[:m])
    assert not np.allclose(ref[m:], got[m:])
    # Truncate at m and re-prefill the suffix: identical to the full re-run.
    a.truncate(s, m)
    re = oracle.prefill(a, [s], q2[:, m:], k2[:, m:], v2[:, m:], [n - m])[0]
    np.testing.assert_allclose(re, got[m:], rtol=0, atol=1e-13)
    assert np.array_equal(a.raw_kv(s)[0], b.raw_kv(t)[0])


def test_bf16_inputs_are_read_exactly():
    x = np.array([1.0, -2.5, 3.140625, 1e-3], dtype=np.float32)
    bits = workloads.bf16_bits(x)
    back = oracle.to_f64(bits, "bf16")
    assert back[0] == 1.0 and back[1] == -2.5 and back[2] == 3.140625
    assert abs(back[3] - 1e-3) < 1e-3 * 2 ** -8


# ---------------------------------------------------------------- rotary positions
# The pages describe RoPE only in words ([P3], prefix caching): a rotation of
# Q/K fixed by the position ID, whose inner products depend only on the
# position difference; position 0 and equal positions leave inner products
# unchanged.  The pins check those properties, the pairing and direction
# read through a second form (complex multiplication), and the
# stored-key rounding rule against exact arithmetic.

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((4, 3, 16))
    assert np.array_equal(oracle.rope(x, np.zeros(4), 10000.0), x)


def test_rope_matches_complex_rotation_of_half_split_pairs():
    rng = np.random.default_rng(2)
    d, base = 12, 500.0
    x = rng.standard_normal((5, 2, d))
    pos = rng.integers(0, 4000, size=5)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    w = np.exp(1j * pos[:, None, None] * base ** (-np.arange(0, d, 2) / d))
    want = z * w
    got = oracle.rope(x, pos, base)
    assert np.allclose(got[..., : d // 2], want.real, rtol=0, atol=1e-12)
    assert np.allclose(got[..., d // 2:], want.imag, rtol=0, atol=1e-12)


def test_rope_pairs_dimension_k_with_k_plus_half():
    e0 = np.zeros((1, 1, 8))
    e0[..., 0] = 1.0
    r = oracle.rope(e0, [3], 10000.0)[0, 0]
    nz = set(np.flatnonzero(np.abs(r) > 1e-15))
    assert nz == {0, 4}
    assert math.isclose(r[0], math.cos(3.0), abs_tol=1e-15)      # theta_0 = 1
    assert math.isclose(r[4], math.sin(3.0), abs_tol=1e-15)


def test_rope_preserves_norms_and_composes():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 2, 32))
    a, b = rng.integers(0, 3000, 6), rng.integers(0, 3000, 6)
    r = oracle.rope(x, a, 10000.0)
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14, atol=0)
    assert np.allclose(oracle.rope(r, b, 10000.0), oracle.rope(x, a + b, 10000.0), rtol=0, atol=1e-10)


def test_rope_inner_products_depend_on_position_difference_only():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    base = 10000.0
    ref = float(np.sum(oracle.rope(q, [700], base) * oracle.rope(k, [650], base)))
    for shift in (1, 37, 1000, 5000):
        val = float(np.sum(oracle.rope(q, [700 + shift], base) * oracle.rope(k, [650 + shift], base)))
        assert abs(val - ref) <= 1e-10 * (1 + abs(ref))
    same = float(np.sum(oracle.rope(q, [123], base) * oracle.rope(k, [123], base)))
    assert abs(same - float(np.sum(q * k))) <= 1e-12


def test_rope_attention_is_invariant_to_a_common_position_shift():
    rng = np.random.default_rng(5)
    n, H_q, H_kv, d = 9, 4, 2, 16
    q = workloads.normal_bf16(rng, (1, n, H_q, d))
    k = workloads.normal_bf16(rng, (1, n, H_kv, d))
    v = workloads.normal_bf16(rng, (1, n, H_kv, d))
    # The same rows placed at positions 0.. and at 48..: the causal mask is
    # by relative index, the rotation by absolute position.
    K, V = oracle.to_f64(k[0], "bf16"), oracle.to_f64(v[0], "bf16")
    Q = oracle.to_f64(q[0], "bf16")
    res = []
    for p0 in (0, 48):
        pos = p0 + np.arange(n)
        res.append(_att(oracle.rope(Q, pos, 10000.0), oracle.rope(K, pos, 10000.0), V, np.arange(n)))
    assert np.allclose(res[0], res[1], rtol=0, atol=1e-12)


def test_rope_prefill_equals_rotated_definition_and_decode_last_row():
    rng = np.random.default_rng(6)
    n, H_q, H_kv, d, base = 7, 4, 2, 8, 10000.0
    q = workloads.normal_bf16(rng, (1, n, H_q, d))
    k = workloads.normal_bf16(rng, (1, n, H_kv, d))
    v = workloads.normal_bf16(rng, (1, n, H_kv, d))
    cm = oracle.CacheModel(4, 2, 4, H_kv, d, "bf16")
    s = cm.create()
    out = oracle.prefill(cm, [s], q, k, v, [n], nthreads=2, rope_base=base)
    Q, K, V = (oracle.to_f64(a[0], "bf16") for a in (q, k, v))
    pos = np.arange(n)
    want = oracle.attention_dense(oracle.rope(Q, pos, base), oracle.rope(K, pos, base), V, pos)
    assert np.allclose(out[0], want, rtol=0, atol=1e-12)
    # decode of the last token after appending it equals the last prefill row
    cm2 = oracle.CacheModel(4, 2, 4, H_kv, d, "bf16")
    s2 = cm2.create()
    oracle.prefill(cm2, [s2], q[:, : n - 1], k[:, : n - 1], v[:, : n - 1], [n - 1], nthreads=2, rope_base=base)
    oracle.append(cm2, [s2], k[:, n - 1], v[:, n - 1])
    dec = oracle.decode(cm2, [s2], q[:, n - 1], nthreads=2, rope_base=base)
    assert np.allclose(dec[0], out[0, n - 1], rtol=0, atol=1e-12)


def test_rope_stored_keys_round_to_within_one_bf16_step():
    rng = np.random.default_rng(7)
    k = workloads.normal_bf16(rng, (64, 2, 128))
    pos = rng.integers(0, 8192, 64)
    stored = oracle.rope_stored_bf16(k, pos, 10000.0)
    exact = oracle.rope(oracle.to_f64(k, "bf16"), pos, 10000.0)
    got = oracle.to_f64(stored, "bf16")
    # one bf16 step at |x| is 2^(floor(log2|x|) - 7); fp32 intermediate
    # rounding adds far less than that.
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(got - exact) <= step * 1.0001)
    # at position 0 the stored bytes are the input bytes
    assert np.array_equal(oracle.rope_stored_bf16(k, np.zeros(64), 10000.0), k)


# ---------------------------------------------------------------- pre-position keys
# [P1] 2.5: the cache records whether its keys were taken before or after the
# position transform.  A pre-position cache keeps each key as given and the
# reader rotates it by its position.  Pinned by: the stored bytes are the
# input bytes; in exact arithmetic the result is the post-position one; the
# stored keys read at a common offset give the same result (what a
# post-position cache cannot do: its keys carry their absolute positions,
# [P3] prefix caching); a pure-Python brute force on a tiny case.

def test_pre_position_cache_stores_the_input_bytes():
    rng = np.random.default_rng(21)
    k = workloads.normal_bf16(rng, (1, 37, 2, 8))
    v = workloads.normal_bf16(rng, (1, 37, 2, 8))
    q = workloads.normal_bf16(rng, (1, 37, 4, 8))
    cm = oracle.CacheModel(8, 1, 8, 2, 8, "bf16")
    s = cm.create()
    oracle.prefill(cm, [s], q, k, v, [37], nthreads=2, rope_base=10000.0)
    rk, rv = cm.raw_kv(s)
    assert np.array_equal(rk, k[0]) and np.array_equal(rv, v[0])
    # a post-position cache would hold other bytes for every position > 0
    post = oracle.rope_stored_bf16(k[0], np.arange(37), 10000.0)
    assert not np.array_equal(post[1:], k[0, 1:])


def test_pre_position_read_equals_post_position_definition():
    rng = np.random.default_rng(22)
    n, H_q, H_kv, d, base = 11, 6, 2, 16, 10000.0
    Q, K, V = rng.standard_normal((n, H_q, d)), rng.standard_normal((n, H_kv, d)), rng.standard_normal((n, H_kv, d))
    pos = np.arange(n)
    pre = oracle.attention_pre_position(Q, K, V, pos, base, nthreads=2)
    post = oracle.attention_dense(oracle.rope(Q, pos, base), oracle.rope(K, pos, base), V, pos)
    assert np.allclose(pre, post, rtol=0, atol=1e-12)
    # the window form too
    prew = oracle.attention_pre_position(Q, K, V, pos, base, window=3, nthreads=2)
    postw = oracle.attention_dense(oracle.rope(Q, pos, base), oracle.rope(K, pos, base), V, pos, window=3)
    assert np.allclose(prew, postw, rtol=0, atol=1e-12)


def test_pre_position_keys_read_at_an_offset_give_the_same_result():
    rng = np.random.default_rng(23)
    n, H_q, H_kv, d, base = 13, 4, 2, 32, 10000.0
    Q, K, V = rng.standard_normal((n, H_q, d)), rng.standard_normal((n, H_kv, d)), rng.standard_normal((n, H_kv, d))
    pos = np.arange(n)
    ref = oracle.attention_pre_position(Q, K, V, pos, base, nthreads=2)
    for off in (1, 100, 4096):
        got = oracle.attention_pre_position(Q, K, V, pos, base, offset=off, nthreads=2)
        assert np.allclose(got, ref, rtol=0, atol=1e-10)
    # post-position keys (rotated once at their original positions) read by
    # queries at an offset give a different result
    K_post = oracle.rope(K, pos, base)
    moved = _att(oracle.rope(Q, pos + 100, base), K_post, V, pos)
    assert np.abs(moved - ref).max() > 1e-3


def test_pre_position_read_brute_force_tiny():
    rng = np.random.default_rng(24)
    n, d, base = 4, 4, 10.0
    Q, K, V = rng.standard_normal((n, 1, d)), rng.standard_normal((n, 1, d)), rng.standard_normal((n, 1, d))
    got = oracle.attention_pre_position(Q, K, V, np.arange(n), base, nthreads=1)

    def rot(x, p):
        out = [0.0] * d
        for e in range(d // 2):
            a = p * base ** (-2.0 * e / d)
            out[e] = x[e] * math.cos(a) - x[e + d // 2] * math.sin(a)
            out[e + d // 2] = x[e] * math.sin(a) + x[e + d // 2] * math.cos(a)
        return out

    for i in range(n):
        qi = rot(list(Q[i, 0]), i)
        sc = [sum(a * b for a, b in zip(qi, rot(list(K[j, 0]), j))) / math.sqrt(d) for j in range(i + 1)]
        m = max(sc)
        w = [math.exp(x - m) for x in sc]
        o = [sum(w[j] * V[j, 0, e] for j in range(i + 1)) / sum(w) for e in range(d)]
        assert np.allclose(got[i, 0], o, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- sliding window
# [P3] sliding window: position t reads the most recent W positions, the
# current one included; K/V outside the window is never read again, so a
# ring cache holds O(W) of it.

def test_window_at_least_the_length_changes_nothing():
    rng = np.random.default_rng(11)
    q, K, V = rng.standard_normal((6, 2, 4)), rng.standard_normal((9, 1, 4)), rng.standard_normal((9, 1, 4))
    pos = np.array([0, 2, 4, 6, 7, 8])
    assert np.array_equal(oracle.attention(q, K, V, pos, 2, window=9), oracle.attention(q, K, V, pos, 2))
    assert np.array_equal(oracle.attention(q, K, V, pos, 2, window=1000), oracle.attention(q, K, V, pos, 2))


def test_window_of_one_returns_the_own_value():
    rng = np.random.default_rng(12)
    q, K, V = rng.standard_normal((4, 2, 4)), rng.standard_normal((7, 1, 4)), rng.standard_normal((7, 1, 4))
    pos = np.array([0, 3, 5, 6])
    out = oracle.attention(q, K, V, pos, 2, window=1)
    for i, p in enumerate(pos):
        assert np.allclose(out[i, :, :], V[p, 0][None, :], rtol=0, atol=1e-15)


def test_window_brute_force_pure_python():
    rng = np.random.default_rng(13)
    L, d, W = 7, 3, 3
    q, K, V = rng.standard_normal((L, 1, d)), rng.standard_normal((L, 1, d)), rng.standard_normal((L, 1, d))
    out = oracle.attention(q, K, V, np.arange(L), 1, window=W)
    for p in range(L):
        js = [j for j in range(L) if p - W < j <= p]
        sc = [sum(q[p, 0, e] * K[j, 0, e] for e in range(d)) / math.sqrt(d) for j in js]
        mx = max(sc)
        w = [math.exp(x - mx) for x in sc]
        z = sum(w)
        ref = [sum(w[a] * V[j, 0, e] for a, j in enumerate(js)) / z for e in range(d)]
        assert np.allclose(out[p, 0], ref, rtol=0, atol=1e-14)
    # the weight vector of a query whose window is full has W entries ([P3]: W = 4 -> length 4)
    assert len([j for j in range(L) if (L - 1) - W < j <= L - 1]) == W


def test_keys_outside_the_window_never_matter():
    rng = np.random.default_rng(14)
    L, W = 30, 8
    q, K, V = rng.standard_normal((L, 2, 8)), rng.standard_normal((L, 1, 8)), rng.standard_normal((L, 1, 8))
    base = oracle.attention(q, K, V, np.arange(L), 2, window=W)
    K2, V2 = K.copy(), V.copy()
    K2[:L - W] += 100.0
    V2[:L - W] -= 50.0
    moved = oracle.attention(q, K2, V2, np.arange(L), 2, window=W)
    assert np.array_equal(base[L - 1], moved[L - 1])      # the last row's window is L - W .. L - 1
    assert not np.array_equal(base[L - W - 1], moved[L - W - 1])


def test_windowed_cache_releases_pages_and_bounds_rewinds():
    cm = oracle.CacheModel(16, 2, 16, 1, 4, "f32", window=20)
    s = cm.create()
    rows = np.zeros((100, 1, 4), dtype=np.float32)
    cm.write([s], [rows], [rows])
    bt = cm.block_table(s)
    assert bt[:5] == [-1] * 5 and all(p >= 0 for p in bt[5:])   # positions 0..79 released (80 <= 100 - 20)
    assert cm.free_pages() == 16 - 2
    with pytest.raises(oracle.CacheError) as e:
        cm.truncate(s, 90)                                       # needs 70..89 but 0..79 are gone
    assert e.value.kind == "ERANGE"
    with pytest.raises(oracle.CacheError):
        cm.fork(s, 95)
    cm.truncate(s, 100)
    f = cm.fork(s, 100)
    assert cm.block_table(f) == bt
    cm.truncate(s, 0)
    assert cm.block_table(s) == []


def test_windowed_cache_holds_a_bounded_number_of_pages():
    W = 40
    cm = oracle.CacheModel(8, 1, 80, 1, 2, "f32", window=W)
    s = cm.create()
    one = np.zeros((1, 1, 2), dtype=np.float32)
    for _ in range(1000):
        cm.write([s], [one], [one])
        live = [p for p in cm.block_table(s) if p >= 0]
        assert len(live) <= -(-W // 16) + 1
    assert cm.length(s) == 1000


# --- quantised cache: FP8 E4M3 codes with a per-row fp32 scale -------------

def test_e4m3_decode_matches_torch_float8_for_every_code():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(mine)
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_known_codes_and_rounding():
    dec = oracle.e4m3_decode
    assert dec(0x7E) == 448.0 and dec(0xFE) == -448.0 and np.isnan(dec(0x7F))
    assert dec(0x38) == 1.0 and dec(0x08) == 2.0 ** -6 and dec(0x01) == 2.0 ** -9 and dec(0x00) == 0.0
    enc = lambda v: int(oracle.e4m3_encode(np.array([v]))[0])
    assert enc(1.0625) == 0x38            # halfway between 1 and 1.125: to the even mantissa (1)
    assert enc(1.1875) == 0x3A            # halfway between 1.125 and 1.25: to 1.25
    assert enc(1.5 * 2.0 ** -9) == 0x02   # subnormal tie: m = 1.5 -> 2
    assert enc(1000.0) == 0x7E and enc(-1000.0) == 0xFE and enc(460.0) == 0x7E
    finite = [c for c in range(256) if not np.isnan(dec(c))]
    assert all(enc(dec(c)) == c for c in finite)                    # every code round-trips
    # Brute force: the code is the nearest representable value (ties even).
    rng = np.random.default_rng(5)
    x = rng.standard_normal(4000) * np.exp2(rng.integers(-12, 9, 4000))
    x = x[np.abs(x) < 448]
    vals = np.array([dec(c) for c in finite])
    got = oracle.e4m3_decode(oracle.e4m3_encode(x))
    best = np.min(np.abs(vals[None, :] - x[:, None]), axis=1)
    assert np.all(np.abs(got - x) <= best + 1e-300)


def test_quantized_rows_scale_error_and_zero_rows():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((50, 4, 128)) * np.exp2(rng.integers(-6, 6, (50, 4, 1)))).astype(np.float32)
    x[3, 1] = 0.0
    codes, s = oracle.quantize_e4m3_rows(x)
    amax = np.max(np.abs(x), axis=-1)
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    assert s[3, 1] == 0 and not codes[3, 1].any()
    # The largest element of each non-zero row is coded as +-448.
    arg = np.argmax(np.abs(x), axis=-1)
    top = np.take_along_axis(codes, arg[..., None], axis=-1)[..., 0]
    nz = amax > 0
    assert np.all((top[nz] & 0x7F) == 0x7E)
    deq = oracle.dequantize_e4m3_rows(oracle.pack_e4m3_rows(codes, s)).astype(np.float64)
    # Round to nearest: half a unit in the last place (3 mantissa bits) for
    # normals, half the subnormal step (s * 2^-10) below 2^-6 * s.
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s[..., None] * 2.0 ** -10) * (1 + 1e-6) + 1e-30
    assert np.all(err <= bound)


def test_quantized_cache_model_serves_the_dequantized_rows():
    rng = np.random.default_rng(7)
    m = oracle.CacheModel(8, 1, 8, 2, 16, "fp8")
    s = m.create()
    k = workloads.normal_bf16(rng, (20, 2, 16))
    v = workloads.normal_bf16(rng, (20, 2, 16))
    m.write([s], [k], [v])
    K, V = m.kv(s)
    kc, ks = oracle.quantize_e4m3_rows(oracle.to_f64(k, "bf16").astype(np.float32))
    want = (oracle.e4m3_decode(kc).astype(np.float32) * ks[..., None]).astype(np.float64)
    assert np.array_equal(K, want)
    assert m.raw_kv(s)[0].shape == (20, 2, 20)
    m.truncate(s, 9)
    assert np.array_equal(m.kv(s)[0], want[:9])
    q = workloads.normal_bf16(rng, (1, 4, 16))
    got = oracle.decode(m, [s], q)
    ref = oracle.attention_dense(oracle.to_f64(q, "bf16"), m.kv(s)[0], m.kv(s)[1], [8])
    assert np.allclose(got, ref, atol=1e-12)
