"""Online softmax under large and growing scores.

"第二章 Prefill：整层状态演化与 KV 建立", section 2.3: the row softmax takes the
largest finite score m and exp(s - m); a tiled kernel meets the keys tile by
tile and must rescale what it has accumulated whenever a later tile raises
the maximum ("KV Cache 与 Prefill/Decode 推理路径", online softmax).  The
tensor-core kernel rescales O only when the running maximum grows by more
than 2^8 (in units of 2^x), and split decode merges ranges whose maxima
differ by far more than that.  N(0,1) inputs never get there, so these
cases scale q up and give later key tiles larger keys: the maximum grows by
far more than 2^8 from tile to tile (checked here from the oracle's scores),
in prefill, in split tensor-core decode and in the CUDA-core decode.  A
last case makes the maximum fall instead (early keys large), so the stale
maximum stays the reference across many tiles.
"""
import numpy as np
import pytest

import oracle
import workloads
from _helpers import assert_cache_matches, assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu

DT = "bf16"
LOG2E = 1.4426950408889634


def _scaled(rng, shape, scale):
    return workloads.bf16_bits(rng.standard_normal(size=shape, dtype=np.float32) * np.asarray(scale, np.float32))


def _key_scale(L, step, growing):
    """Per-position key scale: 1 + step * tile index (growing) or its mirror."""
    t = np.arange(L) // 128
    s = 1.0 + step * (t if growing else t.max() - t)
    return s.astype(np.float32)[:, None, None]


def _growth_log2(q_bits, K, qpos, H_kv, d):
    """Over the rows and heads given: the largest growth of a row's running
    maximum (log2 units) from one 128-key tile to the next, and the smallest
    total growth from the first tile's maximum to the row's maximum."""
    q = oracle.to_f64(q_bits, DT)
    H_q = q.shape[1]
    step, total = 0.0, np.inf
    for i, p in enumerate(qpos):
        for h in range(H_q):
            g = (h * H_kv) // H_q
            s = K[: p + 1, g, :] @ q[i, h] / np.sqrt(d) * LOG2E
            run = s[:128].max()
            first = run
            for j0 in range(128, p + 1, 128):
                tmax = s[j0:j0 + 128].max()
                step = max(step, tmax - run)
                run = max(run, tmax)
            total = min(total, run - first)
    return step, total


@pytest.mark.parametrize("growing", [True, False])
def test_prefill_with_growing_or_falling_maximum(growing):
    H_q, H_kv, d, n = 8, 2, 128, 900
    rng = np.random.default_rng(800 + growing)
    q = _scaled(rng, (1, n, H_q, d), 6.0)
    k = _scaled(rng, (1, n, H_kv, d), _key_scale(n, 0.75, growing)[None])
    v = workloads.normal_bf16(rng, (1, n, H_kv, d))
    K = oracle.to_f64(k[0], DT)
    if growing:
        rows = [300, 640, 899]
        step, _ = _growth_log2(q[0, rows], K, rows, H_kv, d)
        assert step > 12, "the case must drive the rescale path (growth > 8 from one tile to the next)"
    c = gqa.Cache(H_kv, d, 64, 1, 64, dtype=DT)
    s = c.seq_create()
    out = host_f64(gqa.attn_prefill(c, [s], dev(q, DT), dev(k, DT), dev(v, DT), [n]), DT)
    m = oracle.CacheModel(64, 1, 64, H_kv, d, DT)
    ms = m.create()
    ref = oracle.prefill(m, [ms], q, k, v, [n])
    assert_close(out, ref, DT, "prefill, %s maximum" % ("growing" if growing else "falling"))
    assert_cache_matches(c, m, [(s, ms)])
    assert c.check() == 0


@pytest.mark.parametrize("kernel", ["tensor_core", "cuda_core"])
def test_split_decode_merges_ranges_with_far_apart_maxima(kernel):
    # One long sequence: the decode splits its keys into ranges whose maxima
    # grow by far more than 2^8 from range to range; the merge weighs them.
    H_q, H_kv, d = 16, 2, 128
    L = 6000
    rng = np.random.default_rng(810)
    k = _scaled(rng, (L, H_kv, d), _key_scale(L, 0.1, True))
    v = workloads.normal_bf16(rng, (L, H_kv, d))
    q = _scaled(rng, (1, H_q, d), 6.0)
    K = oracle.to_f64(k, DT)
    _, total = _growth_log2(q, K, [L - 1], H_kv, d)
    assert total > 40, "the ranges' maxima must be far apart"
    pages = workloads.pages_for(L) + 4
    c = gqa.Cache(H_kv, d, pages, 1, pages, dtype=DT)
    c.set_decode_kernel(kernel)
    s = c.seq_create()
    gqa.kv_append(c, [s], dev(k[None], DT), dev(v[None], DT))
    c.profile_read()
    got = host_f64(gqa.attn_decode(c, [s], dev(q, DT)), DT)
    launched = c.profile_read()
    assert launched["prefill_tc" if kernel == "tensor_core" else "decode_split"][0] == 1, launched
    m = oracle.CacheModel(pages, 1, pages, H_kv, d, DT)
    ms = m.create()
    m.write([ms], [k], [v])
    assert_close(got, oracle.decode(m, [ms], q), DT, "%s decode merge" % kernel)
    assert_cache_matches(c, m, [(s, ms)])
    assert c.check() == 0


def test_incremental_prefill_new_rows_raise_the_maximum():
    # A 2048-token prefix of small keys, then new rows whose keys are much
    # larger: for every new row the maximum jumps on the first new tile.
    H_q, H_kv, d = 12, 2, 128
    P, n = 2048, 264
    rng = np.random.default_rng(820)
    pk = _scaled(rng, (P, H_kv, d), 0.5)
    pv = workloads.normal_bf16(rng, (P, H_kv, d))
    q = _scaled(rng, (1, n, H_q, d), 6.0)
    k = _scaled(rng, (1, n, H_kv, d), 4.0)
    v = workloads.normal_bf16(rng, (1, n, H_kv, d))
    pages = workloads.pages_for(P + n) + 4
    c = gqa.Cache(H_kv, d, pages, 1, pages, dtype=DT)
    s = c.seq_create()
    gqa.kv_append(c, [s], dev(pk[None], DT), dev(pv[None], DT))
    out = host_f64(gqa.attn_prefill(c, [s], dev(q, DT), dev(k, DT), dev(v, DT), [n]), DT)
    m = oracle.CacheModel(pages, 1, pages, H_kv, d, DT)
    ms = m.create()
    m.write([ms], [pk], [pv])
    ref = oracle.prefill(m, [ms], q, k, v, [n])
    assert_close(out, ref, DT, "incremental prefill, raised maximum")
    assert_cache_matches(c, m, [(s, ms)])
    assert c.check() == 0
