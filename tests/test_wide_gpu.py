"""Wide head dims d in {192, 256}: CUDA path (through the C ABI) vs the fp64
oracle, forward and backward.

Every formula is the one of the narrower head dims (scale = 1/sqrt(d)); only
the kernels differ (one query tile per forward work unit; 64-row sub-tiles
in the backward).  Tolerances as for the other head dims: |O - O_ref| <=
2e-2, |LSE - LSE_ref| <= 5e-3, gradients <= 5e-2 * max |ref|.  Small shapes
(ragged tails, several tiles, causal and not, both 16-bit types, grouped
query heads) are compared element by element in full; a longer sequence on
sampled rows of four heads, the oracle computing them one row at a time.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import sample_heads, sample_rows, to64

pytestmark = pytest.mark.gpu
O_TOL, LSE_TOL = 2e-2, 5e-3
WIDE = [192, 256]


def _fwd(attn, q, k, v, causal, scale, B, H, N):
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    attn.fwd(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
    st, detail = attn.poll_status()
    assert st == 0, f"device status {st} detail 0x{detail:x}"
    return o, lse


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 17), (2, 1, 128), (1, 3, 129),
                                   (2, 2, 255), (1, 2, 300), (1, 2, 513), (2, 1, 1000)])
def test_wide_forward_small_full(attn_lib, d, dtype, causal, B, H, N):
    w = wl.Workload("wide", "fwd", B, H, N, d, dtype, causal, seed=N + d)
    inp = wl.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = _fwd(attn_lib, q, k, v, causal, w.scale, B, H, N)
    O_ref, L_ref = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), causal,
                                    w.scale)
    O, L = to64(o), to64(lse)
    assert np.isfinite(O).all() and np.isfinite(L).all()
    assert np.max(np.abs(O - O_ref)) <= O_TOL
    assert np.max(np.abs(L - L_ref)) <= LSE_TOL


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("logit_gain", [4.0, 0.01])
def test_wide_forward_large_and_small_logits(attn_lib, d, logit_gain):
    """Large logits raise the running max often (the O rescale, which here
    waits for the previous P V), tiny logits give a near-uniform softmax."""
    w = wl.Workload("wide", "fwd", 1, 2, 700, d, "bf16", True, seed=5 + d)
    inp = wl.make_inputs(w)
    for n in ("q", "k"):
        inp[n] = (inp[n].float() * logit_gain).to(torch.bfloat16)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = _fwd(attn_lib, q, k, v, True, w.scale, 1, 2, 700)
    O_ref, L_ref = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), True,
                                    w.scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= O_TOL
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_TOL


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 2, 300), (2, 4, 1, 257)])
def test_wide_forward_grouped_heads(attn_lib, d, causal, B, Hq, Hkv, N):
    w = wl.Workload("wideg", "fwd", B, Hq, N, d, "bf16", causal, seed=N + Hkv + d)
    inp = wl.make_inputs(w)
    G = Hq // Hkv
    q = inp["q"]
    k, v = (inp[n][:, ::G].contiguous() for n in ("k", "v"))
    o, lse = _fwd(attn_lib, q.cuda(), k.cuda(), v.cuda(), causal, w.scale, B, Hq, N)
    O_ref, L_ref = oracle.attention_gqa(to64(q), to64(k), to64(v), causal, w.scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= O_TOL
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_TOL


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("causal", [True, False])
def test_wide_forward_long_sampled(attn_lib, d, causal):
    """[2, 8, 4096, d] bf16 on sampled rows of four heads (first and last
    included): many units per SM, so the persistent schedule, the ring wrap
    and the buffer parities all cycle."""
    w = wl.Workload("widel", "fwd", 2, 8, 4096, d, "bf16", causal, seed=d)
    inp = wl.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = _fwd(attn_lib, q, k, v, causal, w.scale, w.B, w.H, w.N)
    O, L = o.cpu(), lse.cpu()
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
    for (b, h) in sample_heads(w.B, w.H, 4, seed=d):
        rows = sample_rows(w.N, 32, seed=b * 17 + h)
        Or, Lr = oracle.attention_rows(to64(inp["q"][b, h]), to64(inp["k"][b, h]),
                                       to64(inp["v"][b, h]), rows, causal, w.scale)
        assert np.max(np.abs(to64(O[b, h])[rows] - Or)) <= O_TOL
        assert np.max(np.abs(to64(L[b, h])[rows] - Lr)) <= LSE_TOL


def test_wide_forward_deterministic(attn_lib):
    w = wl.Workload("wided", "fwd", 1, 3, 777, 256, "bf16", True, seed=9)
    inp = wl.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = _fwd(attn_lib, q, k, v, True, w.scale, 1, 3, 777)
    o2, l2 = _fwd(attn_lib, q, k, v, True, w.scale, 1, 3, 777)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_wide_modes_not_built_are_rejected(attn_lib):
    """The key split, the key cache and packed variable-length batches are
    built for d <= 128 only, except on the decoding kernel's shapes (at most
    128 query rows per key/value head): at d = 256 with 200 rows per head
    they return ATTN_ERR_UNSUPPORTED before any launch."""
    L = attn_lib.lib()
    x = torch.zeros((1, 1, 256, 256), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, 1, 1, 256), dtype=torch.float32, device="cuda")
    p, pl = ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(lse.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.attn_fwd_split(p, p, p, p, pl, 2, 1, 1, 200, 256, 1, 0.1, 1, s) == 2
    assert L.attn_fwd_kv(p, p, p, p, pl, 1, 1, 1, 1, 200, 256, 256, 1, 0.1, 1, s) == 2
    assert L.attn_fwd(p, p, p, p, pl, 1, 1, 64, 320, 1, 0.1, 1, s) == 2  # d = 320
    assert attn_lib.poll_status()[0] == 0


# ------------------------------------------------------------------ backward ---

BWD_TOL = 5e-2  # max |g - g_ref| <= 5e-2 * max |g_ref| for g in dQ, dK, dV


def _bwd_check(attn, inp, w, refs=None, k=None, v=None):
    q, do = inp["q"].cuda(), inp["do"].cuda()
    k = (inp["k"] if k is None else k).cuda()
    v = (inp["v"] if v is None else v).cuda()
    o, lse = attn.fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    attn.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv)
    st, detail = attn.poll_status()
    assert st == 0, f"device status {st} detail 0x{detail:x}"
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        g = to64(g)
        assert np.isfinite(g).all(), name
        ref_max = np.max(np.abs(r))
        if ref_max == 0.0:  # N = 1: the softmax of one key has zero Jacobian
            assert np.max(np.abs(g)) <= 1e-3, name
            continue
        err = np.max(np.abs(g - r)) / ref_max
        assert err <= BWD_TOL, (w.name, name, err)
    return dq, dk, dv


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 17), (1, 1, 64), (2, 1, 129),
                                   (1, 2, 300), (1, 1, 513), (2, 2, 1000)])
def test_wide_backward_small_full(attn_lib, d, dtype, causal, B, H, N):
    w = wl.Workload("wideb", "bwd", B, H, N, d, dtype, causal, seed=7 + N + d)
    inp = wl.make_inputs(w)
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), causal,
                                     w.scale)
    _bwd_check(attn_lib, inp, w, refs)


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 2, 300), (2, 4, 1, 257)])
def test_wide_backward_grouped_heads(attn_lib, d, causal, B, Hq, Hkv, N):
    """dK, dV of a shared key/value head sum over its query heads."""
    w = wl.Workload("widebg", "bwd", B, Hq, N, d, "bf16", causal, seed=3 * N + Hkv + d)
    inp = wl.make_inputs(w)
    G = Hq // Hkv
    k, v = (inp[n][:, ::G].contiguous() for n in ("k", "v"))
    refs = oracle.attention_backward_gqa(to64(inp["q"]), to64(k), to64(v), to64(inp["do"]),
                                         causal, w.scale)
    _bwd_check(attn_lib, inp, w, refs, k=k, v=v)


@pytest.mark.parametrize("d", WIDE)
@pytest.mark.parametrize("causal", [True, False])
def test_wide_backward_long_sampled(attn_lib, d, causal):
    """[1, 4, 4096, d] bf16: the first and the last head whole against the
    oracle; the other two on sampled dQ rows (the oracle computes each row's
    dQ on its own) and the dK / dV sum identities (every row of dS sums to
    zero, every row of P to one)."""
    w = wl.Workload("widebl", "bwd", 1, 4, 4096, d, "bf16", causal, seed=d + 1)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = attn_lib.fwd(q, k, v, causal=causal, scale=w.scale)
    dq, dk, dv = attn_lib.bwd(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    assert attn_lib.poll_status() == (0, 0)
    full = [(0, 0), (0, 3)]
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), causal,
                                     w.scale, heads=full)
    for g, r in zip((dq, dk, dv), refs):
        g64 = to64(g)
        for (b, h) in full:
            assert np.max(np.abs(g64[b, h] - r[b, h])) <= BWD_TOL * np.max(np.abs(r[b, h]))
    for h in (1, 2):
        qh, kh, vh, doh = (to64(inp[n][0, h]) for n in ("q", "k", "v", "do"))
        rows = sample_rows(w.N, 32, seed=h)
        dq_ref = oracle.attention_backward_dq_rows(qh, kh, vh, doh, rows, causal, w.scale)
        assert np.max(np.abs(to64(dq[0, h])[rows] - dq_ref)) <= BWD_TOL * np.max(np.abs(dq_ref))
        dkh, dvh = to64(dk[0, h]), to64(dv[0, h])
        assert np.all(np.abs(dkh.sum(axis=0)) <= 1e-2 * np.abs(dkh).sum(axis=0))
        assert np.all(np.abs(dvh.sum(axis=0) - doh.sum(axis=0)) <= 1e-2 * np.abs(dvh).sum(axis=0))


def test_wide_backward_deterministic(attn_lib):
    """One CTA owns each output tile (and column half), accumulating in a
    fixed order: two runs give the same bits."""
    w = wl.Workload("widebd", "bwd", 2, 2, 700, 256, "bf16", True, seed=21)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    g1 = attn_lib.bwd(q, k, v, o, do, lse, causal=True)
    g2 = attn_lib.bwd(q, k, v, o, do, lse, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
