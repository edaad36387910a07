"""Grouped query heads (GQA / MQA): CUDA path (C ABI) vs the fp64 oracle.

k, v (and dk, dv) have Hkv heads for Hq query heads; query head h attends
with key/value head h // (Hq/Hkv).  Tolerances as for the plain forward and
backward: |O - O_ref| <= 2e-2, |LSE - LSE_ref| <= 5e-3, gradients
<= 5e-2 * max |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import to64

pytestmark = pytest.mark.gpu


def _make(B, Hq, Hkv, N, d, dtype, seed):
    w = wl.Workload("g", "bwd", B, Hq, N, d, dtype, True, seed=seed)
    inp = wl.make_inputs(w)
    G = Hq // Hkv
    # the key/value heads: one head of each group of the seeded inputs
    k = inp["k"][:, ::G].contiguous()
    v = inp["v"][:, ::G].contiguous()
    return w, inp["q"], k, v, inp["do"]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64), ("bf16", 96)])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 2, 300), (2, 4, 1, 257), (1, 8, 2, 513)])
def test_gqa_forward_small(attn_lib, causal, dtype, d, B, Hq, Hkv, N):
    w, q, k, v, _ = _make(B, Hq, Hkv, N, d, dtype, seed=N + Hkv)
    o, lse = attn_lib.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
    assert attn_lib.poll_status() == (0, 0)
    O_ref, L_ref = oracle.attention_gqa(to64(q), to64(k), to64(v), causal, w.scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= 2e-2
    assert np.max(np.abs(to64(lse) - L_ref)) <= 5e-3


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64), ("bf16", 96)])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 2, 300), (2, 4, 1, 257), (1, 6, 3, 640)])
def test_gqa_backward_small(attn_lib, causal, dtype, d, B, Hq, Hkv, N):
    w, q, k, v, do = _make(B, Hq, Hkv, N, d, dtype, seed=7 * N + Hkv + d)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = attn_lib.fwd(qc, kc, vc, causal=causal, scale=w.scale)
    dq, dk, dv = attn_lib.bwd(qc, kc, vc, o, doc, lse, causal=causal, scale=w.scale)
    assert attn_lib.poll_status() == (0, 0)
    assert dk.shape == k.shape and dv.shape == v.shape
    refs = oracle.attention_backward_gqa(to64(q), to64(k), to64(v), to64(do), causal, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        err = np.max(np.abs(to64(g) - r)) / np.max(np.abs(r))
        assert err <= 5e-2, (name, err)


def test_gqa_full_size_sampled_heads(attn_lib):
    """[1,16,4096,128] bf16 causal with 4 key/value heads: forward on sampled
    rows of four query heads (the first and the last included), backward of
    the first key/value group (its 4 query heads) against the oracle."""
    w, q, k, v, do = _make(1, 16, 4, 4096, 128, "bf16", seed=99)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = attn_lib.fwd(qc, kc, vc, causal=True)
    dq, dk, dv = attn_lib.bwd(qc, kc, vc, o, doc, lse, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    rows = np.arange(0, w.N, 157)
    for h in (0, 6, 9, 15):
        g = oracle.kv_head_of(h, 16, 4)
        O_ref, L_ref = oracle.attention_rows(to64(q[0, h]), to64(k[0, g]), to64(v[0, g]), rows,
                                             True, w.scale)
        assert np.max(np.abs(to64(o[0, h])[rows] - O_ref)) <= 2e-2
        assert np.max(np.abs(to64(lse[0, h])[rows] - L_ref)) <= 5e-3
    refs = oracle.attention_backward_gqa(to64(q[:, :4]), to64(k[:, :1]), to64(v[:, :1]),
                                         to64(do[:, :4]), True, w.scale)
    for g, r in zip((dq[:, :4], dk[:, :1], dv[:, :1]), refs):
        assert np.max(np.abs(to64(g) - r)) / np.max(np.abs(r)) <= 5e-2


def test_gqa_rejects_non_dividing_heads(attn_lib):
    q = torch.zeros((1, 6, 128, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 4, 128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        attn_lib.fwd(q, k, k)
