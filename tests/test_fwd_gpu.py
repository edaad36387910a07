"""Forward parity: CUDA path (through the C ABI) vs the fp64 oracle.

Tolerances (stated for fp16/bf16 outputs): max |O - O_ref| <= 2e-2 and
max |LSE - LSE_ref| <= 5e-3, with the oracle fed the same 16-bit inputs
upcast to fp64.  Small shapes are compared element by element in full; the
full-size workloads are compared on seeded samples of heads and rows, which
the oracle computes one row at a time.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import sample_heads, sample_rows, to64

pytestmark = pytest.mark.gpu
O_TOL, LSE_TOL = 2e-2, 5e-3


def _run(attn, inp, w):
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device=dev)
    attn.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
    st, detail = attn.poll_status()
    assert st == 0, f"device status {st} detail 0x{detail:x}"
    return o, lse


def _full_compare(attn, w):
    inp = wl.make_inputs(w)
    o, lse = _run(attn, inp, w)
    O_ref, L_ref = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), w.causal,
                                    w.scale)
    O, L = to64(o), to64(lse)
    assert np.isfinite(O).all() and np.isfinite(L).all()
    eo, el = np.max(np.abs(O - O_ref)), np.max(np.abs(L - L_ref))
    assert eo <= O_TOL and el <= LSE_TOL, (w, eo, el)
    return eo, el


def test_tiny_fp16_causal_workload(attn_lib):
    _full_compare(attn_lib, wl.TINY_FWD_FP16)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 17), (2, 1, 128), (1, 3, 129), (2, 2, 255),
                                   (1, 2, 256), (1, 1, 300), (1, 2, 513), (2, 1, 1000)])
def test_small_shapes_full(attn_lib, dtype, d, causal, B, H, N):
    w = wl.Workload("t", "fwd", B, H, N, d, dtype, causal, seed=N + d)
    _full_compare(attn_lib, w)


@pytest.mark.parametrize("logit_gain", [4.0, 0.01])
@pytest.mark.parametrize("causal", [False, True])
def test_large_and_small_logits(attn_lib, logit_gain, causal):
    # Q and K multiplied by `logit_gain` (V unchanged, so the absolute O
    # tolerance keeps its meaning): large logits exercise the running-max
    # rescale path, tiny logits the near-uniform softmax.
    w = wl.Workload("t", "fwd", 1, 2, 700, 128, "bf16", causal, seed=5)
    inp = wl.make_inputs(w)
    for n in ("q", "k"):
        inp[n] = (inp[n].float() * logit_gain).to(torch.bfloat16)
    o, lse = _run(attn_lib, inp, w)
    O_ref, L_ref = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), w.causal,
                                    w.scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= O_TOL
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_TOL


def _sampled_compare(attn, w, n_heads=4, n_rows=48):
    inp = wl.make_inputs(w)
    o, lse = _run(attn, inp, w)
    O, L = o.cpu(), lse.cpu()
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
    worst_o = worst_l = 0.0
    for (b, h) in sample_heads(w.B, w.H, n_heads, seed=w.N):
        rows = sample_rows(w.N, n_rows, seed=b * 131 + h)
        Or, Lr = oracle.attention_rows(to64(inp["q"][b, h]), to64(inp["k"][b, h]),
                                       to64(inp["v"][b, h]), rows, w.causal, w.scale)
        worst_o = max(worst_o, float(np.max(np.abs(to64(O[b, h])[rows] - Or))))
        worst_l = max(worst_l, float(np.max(np.abs(to64(L[b, h])[rows] - Lr))))
    assert worst_o <= O_TOL and worst_l <= LSE_TOL, (w.name, worst_o, worst_l)


@pytest.mark.parametrize("causal", [True, False])
def test_fp16_d64_workload(attn_lib, causal):
    _sampled_compare(attn_lib, wl.FWD_FP16_D64.with_(causal=causal))


@pytest.mark.parametrize("causal", [True, False])
def test_bf16_d128_workload(attn_lib, causal):
    _sampled_compare(attn_lib, wl.FWD_BF16_D128.with_(causal=causal))


@pytest.mark.parametrize("causal", [True, False])
def test_d64_sweep(attn_lib, causal):
    for w in wl.sweep_d64(causal):
        _sampled_compare(attn_lib, w, n_heads=4, n_rows=16)


@pytest.mark.parametrize("causal", [True, False])
def test_d128_sweep(attn_lib, causal):
    for w in wl.sweep_d128(causal):
        _sampled_compare(attn_lib, w, n_heads=4, n_rows=16)


def test_q_zero_causal_prefix_mean_at_full_size(attn_lib):
    """Property that holds at any size: with Q = 0 the causal output row i
    is the mean of V[0..i] and LSE_i = log(i+1)."""
    w = wl.FWD_BF16_D128.with_(B=1, H=2)
    inp = wl.make_inputs(w)
    inp["q"] = torch.zeros_like(inp["q"])
    o, lse = _run(attn_lib, inp, w)
    v = to64(inp["v"][0, 1])
    prefix = np.cumsum(v, axis=0) / np.arange(1, w.N + 1)[:, None]
    np.testing.assert_allclose(to64(o[0, 1].cpu()), prefix, atol=O_TOL, rtol=0)
    np.testing.assert_allclose(to64(lse[0, 1].cpu()), np.log(np.arange(1, w.N + 1)),
                               atol=LSE_TOL, rtol=0)
    np.testing.assert_allclose(to64(o[0, 0, 0].cpu()), to64(inp["v"][0, 0, 0]), atol=1e-2)


def test_deterministic_and_status_clean(attn_lib):
    w = wl.Workload("t", "fwd", 2, 3, 777, 128, "bf16", True, seed=9)
    inp = wl.make_inputs(w)
    o1, l1 = _run(attn_lib, inp, w)
    o2, l2 = _run(attn_lib, inp, w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_invalid_arguments_rejected_before_launch(attn_lib):
    import ctypes
    L = attn_lib.lib()
    q = torch.zeros((1, 1, 64, 64), dtype=torch.float16, device="cuda")
    lse = torch.zeros((1, 1, 64), dtype=torch.float32, device="cuda")
    p, pl = ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(lse.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.attn_fwd(p, p, p, p, pl, 1, 1, 64, 80, 0, 0.1, 0, s) == 2      # d unsupported
    assert L.attn_fwd(p, p, p, p, pl, 1, 1, 0, 64, 0, 0.1, 0, s) == 1       # N = 0
    assert L.attn_fwd(None, p, p, p, pl, 1, 1, 64, 64, 0, 0.1, 0, s) == 1   # null
    mis = ctypes.c_void_p(q.data_ptr() + 2)
    assert L.attn_fwd(mis, p, p, p, pl, 1, 1, 64, 64, 0, 0.1, 0, s) == 1    # misaligned
    assert L.attn_fwd(p, p, p, p, pl, 1, 1, 64, 64, 2, 0.1, 0, s) == 1      # causal flag
    assert L.attn_fwd(p, p, p, p, pl, 1, 1, 64, 64, 0, -1.0, 0, s) == 1     # scale <= 0
    assert L.attn_fwd(p, p, p, p, pl, 1, 1, 64, 64, 0, 0.1, 7, s) == 1      # dtype
    assert attn_lib.poll_status()[0] == 0
