"""Failure detection on the GPU without a fault: the bounded wait every
pipeline wait uses gives up on a barrier phase that nothing completes,
records GQA_DEVERR_TIMEOUT in the cache's error word, and the context stays
usable for the next calls."""
import time

import numpy as np
import pytest

import oracle
import workloads
from _helpers import assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_a_timeout_and_the_context_stays_usable():
    c = gqa.Cache(2, 128, 16, 2, 8, dtype="bf16")
    m = oracle.CacheModel(16, 2, 8, 2, 128, "bf16")
    assert c.check() == 0
    t0 = time.perf_counter()
    c.selftest_bounded_wait(50_000_000)                # 50 ms
    flags = c.check()
    waited = time.perf_counter() - t0
    assert flags & gqa.DEVERR_TIMEOUT, flags
    assert 0.04 < waited < 5.0, waited
    assert c.check() == 0                              # reading the word clears it
    rng = np.random.default_rng(160)
    s, sm = c.seq_create(), m.create()
    q = workloads.normal_bf16(rng, (1, 50, 8, 128))
    k = workloads.normal_bf16(rng, (1, 50, 2, 128))
    v = workloads.normal_bf16(rng, (1, 50, 2, 128))
    out = host_f64(gqa.attn_prefill(c, [s], dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), [50]), "bf16")
    assert_close(out, oracle.prefill(m, [sm], q, k, v, [50]), "bf16", "prefill after a timeout")
    assert c.check() == 0
