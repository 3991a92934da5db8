"""GPU parity of the two decode kernels against the fp64 oracle: the
tensor-core kernel (the prefill kernel at one query row per sequence, key
tiles split across SMs and merged in the kernel) and the split-K CUDA-core
kernel.  Both within the bf16 tolerance; attn_decode_static gives the same
bits as attn_decode on either kernel."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _helpers import assert_close, dev, host_f64

gqa = pytest.importorskip("causal_gqa_attention_02_gb300")

pytestmark = pytest.mark.gpu


def _filled(rng, H_q, H_kv, lengths, window=0, rope=False):
    B, d = len(lengths), 128
    per_seq = workloads.pages_for(max(lengths)) + 1
    pages = sum(workloads.pages_for(L) for L in lengths) + 4
    c = gqa.Cache(H_kv, d, pages, B, per_seq, dtype="bf16", window=window, rope=rope)
    m = oracle.CacheModel(pages, B, per_seq, H_kv, d, "bf16", window=window)
    ids = [c.seq_create() for _ in range(B)]
    mids = [m.create() for _ in range(B)]
    for b, L in enumerate(lengths):
        k = workloads.normal_bf16(rng, (1, L, H_kv, d))
        v = workloads.normal_bf16(rng, (1, L, H_kv, d))
        gqa.kv_append(c, [ids[b]], dev(k, "bf16"), dev(v, "bf16"))
        oracle.append(m, [mids[b]], k, v)
    return c, m, ids, mids


CASES = [
    (48, 8, [8300]),                      # one long sequence: split into many key ranges
    (32, 8, [1, 17, 129, 2000, 5003]),    # ragged, from one token up
    (128, 8, [700, 3000]),                # g = 16 (tensor-core kernel only)
    (8, 8, [4097, 33]),                   # g = 1
]


@pytest.mark.parametrize("H_q,H_kv,lengths", CASES)
@pytest.mark.parametrize("kernel", ["tensor_core", "cuda_core"])
def test_decode_kernel_matches_oracle(kernel, H_q, H_kv, lengths):
    if kernel == "cuda_core" and H_q // H_kv > 8:
        pytest.skip("the split-K CUDA-core kernel serves H_q/H_kv <= 8")
    rng = np.random.default_rng(80 + H_q + len(lengths))
    c, m, ids, mids = _filled(rng, H_q, H_kv, lengths)
    c.set_decode_kernel(kernel)
    q = workloads.normal_bf16(rng, (len(lengths), H_q, 128))
    c.profile_read()
    o = gqa.attn_decode(c, ids, dev(q, "bf16"))
    launched = c.profile_read()
    assert launched["prefill_tc" if kernel == "tensor_core" else "decode_split"][0] == 1, launched
    assert_close(host_f64(o, "bf16"), oracle.decode(m, mids, q), "bf16", "%s decode" % kernel)
    s = gqa.attn_decode_static(c, ids, dev(q, "bf16"))
    assert torch.equal(o.view(torch.int16), s.view(torch.int16))
    assert c.check() == 0


@pytest.mark.parametrize("window,rope", [(500, False), (0, True), (300, True)])
def test_tensor_core_decode_with_window_and_rope(window, rope):
    rng = np.random.default_rng(90 + window)
    H_q, H_kv, lengths = 32, 8, [6000, 250, 1800]
    c, m, ids, mids = _filled(rng, H_q, H_kv, lengths, window=window, rope=rope)
    c.set_decode_kernel("tensor_core")
    q = workloads.normal_bf16(rng, (3, H_q, 128))
    o = host_f64(gqa.attn_decode(c, ids, dev(q, "bf16")), "bf16")
    assert_close(o, oracle.decode(m, mids, q, rope_base=10000.0 if rope else None), "bf16", "tc decode")
    assert c.check() == 0


def test_tensor_core_decode_repeated_sequences_and_steps():
    # Repeated ids in one batch (a read) and several steps: the merge
    # counters return to zero after every launch.
    rng = np.random.default_rng(95)
    H_q, H_kv = 32, 8
    c, m, ids, mids = _filled(rng, H_q, H_kv, [3000, 900])
    c.set_decode_kernel("tensor_core")
    for t in range(4):
        kt = workloads.normal_bf16(rng, (2, H_kv, 128))
        vt = workloads.normal_bf16(rng, (2, H_kv, 128))
        gqa.kv_append(c, ids, dev(kt, "bf16"), dev(vt, "bf16"))
        oracle.append(m, mids, kt, vt)
        q = workloads.normal_bf16(rng, (3, H_q, 128))
        o = host_f64(gqa.attn_decode(c, [ids[0], ids[1], ids[0]], dev(q, "bf16")), "bf16")
        ref = oracle.decode(m, [mids[0], mids[1], mids[0]], q)
        assert_close(o, ref, "bf16", "step %d" % t)
    assert c.check() == 0


@pytest.mark.parametrize("kernel", ["tensor_core", "cuda_core"])
def test_decode_over_caller_block_tables(kernel):
    # The caller's tables address the cache's pages directly: the cache's own
    # rows give the same bits as attn_decode, and rows that reuse a
    # sequence's first pages with a shorter length decode that prefix.
    rng = np.random.default_rng(170)
    H_q, H_kv, lengths = 32, 8, [3000, 129, 1700]
    c, m, ids, mids = _filled(rng, H_q, H_kv, lengths)
    c.set_decode_kernel(kernel)
    stride = c.max_pages_per_seq
    rows = []
    for s in ids:
        t = c.block_table(s)
        rows.append(t + [-1] * (stride - len(t)))
    q = workloads.normal_bf16(rng, (3, H_q, 128))
    own = gqa.attn_decode(c, ids, dev(q, "bf16"))
    tab = torch.tensor(rows, dtype=torch.int32, device="cuda")
    ext = gqa.attn_decode_tables(c, tab, lengths, dev(q, "bf16"))
    assert torch.equal(own.view(torch.int16), ext.view(torch.int16))
    # Prefixes of sequence 0 at lengths 1000 and 17, and sequence 2 reversed in the batch.
    tab2 = torch.tensor([rows[0], rows[0], rows[2]], dtype=torch.int32, device="cuda")
    q2 = workloads.normal_bf16(rng, (3, H_q, 128))
    o2 = host_f64(gqa.attn_decode_tables(c, tab2, [1000, 17, 1700], dev(q2, "bf16")), "bf16")
    K0, V0 = m.kv(mids[0])
    K2, V2 = m.kv(mids[2])
    ref = np.stack([oracle.attention(oracle.to_f64(q2[0][None], "bf16"), K0[:1000], V0[:1000], [999])[0],
                    oracle.attention(oracle.to_f64(q2[1][None], "bf16"), K0[:17], V0[:17], [16])[0],
                    oracle.attention(oracle.to_f64(q2[2][None], "bf16"), K2, V2, [1699])[0]])
    assert_close(o2, ref, "bf16", "caller tables")
    assert c.check() == 0
    with pytest.raises(gqa.GqaError) as e:
        gqa.attn_decode_tables(c, tab2, [1000, 0, 1700], dev(q2, "bf16"))
    assert e.value.name == "EMASK"
    with pytest.raises(gqa.GqaError) as e:
        gqa.attn_decode_tables(c, tab2, [1000, stride * 16 + 1, 1700], dev(q2, "bf16"))
    assert e.value.name == "ERANGE"
