"""Backward parity: CUDA path (through the C ABI) vs the fp64 oracle.

O and LSE come from the library's own forward pass on the same inputs (as in
the bf16 backward workload).  Tolerance, per gradient g in {dQ, dK, dV}:
max |g - g_ref| <= 5e-2 * max |g_ref|.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import sample_heads, sample_rows, to64

pytestmark = pytest.mark.gpu
REL_TOL = 5e-2


def _gpu_grads(attn, inp, w):
    dev = torch.device("cuda")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    attn.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv)
    st, detail = attn.poll_status()
    assert st == 0, f"device status {st} detail 0x{detail:x}"
    return dq, dk, dv


def _check(w, grads, refs, heads=None):
    for name, g, r in zip(("dQ", "dK", "dV"), grads, refs):
        g = to64(g)
        assert np.isfinite(g).all(), name
        if heads is not None:
            g = np.stack([g[b, h] for b, h in heads])
            r = np.stack([r[b, h] for b, h in heads])
        ref_max = np.max(np.abs(r))
        if ref_max == 0.0:
            # The gradient is exactly zero in exact arithmetic (e.g. N = 1:
            # the softmax over a single key has zero Jacobian); a relative
            # error is undefined, so bound the rounding noise absolutely.
            assert np.max(np.abs(g)) <= 1e-3, (w.name, name)
            continue
        err = np.max(np.abs(g - r)) / ref_max
        assert err <= REL_TOL, (w.name, name, err)


@pytest.mark.parametrize("d", [128, 64, 96])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 17), (1, 1, 128), (2, 1, 129),
                                   (1, 2, 300), (1, 1, 513), (2, 2, 1000)])
def test_small_shapes_full(attn_lib, dtype, causal, B, H, N, d):
    w = wl.Workload(f"bwd_{B}x{H}x{N}", "bwd", B, H, N, d, dtype, causal, seed=7 + N + d)
    inp = wl.make_inputs(w)
    grads = _gpu_grads(attn_lib, inp, w)
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), causal,
                                     w.scale)
    _check(w, grads, refs)


def _check_sampled_head(inp, grads, b, h, causal, scale, seed, n_rows=48):
    """One head of a workload too large for the full oracle: dQ on seeded
    sampled rows (the oracle computes each row's dQ on its own), and dK, dV
    through identities that hold at any size (every row of dS sums to zero,
    so the sum of dK over the keys vanishes; every row of P sums to one, so
    the sum of dV over the keys equals the sum of dO over the queries)."""
    N = inp["q"].shape[2]
    qh, kh, vh, doh = (to64(inp[n][b, h]) for n in ("q", "k", "v", "do"))
    rows = sample_rows(N, n_rows, seed=seed)
    dq_ref = oracle.attention_backward_dq_rows(qh, kh, vh, doh, rows, causal, scale)
    dq = to64(grads[0][b, h])
    assert np.max(np.abs(dq[rows] - dq_ref)) <= REL_TOL * np.max(np.abs(dq_ref)), (b, h)
    dkh, dvh = to64(grads[1][b, h]), to64(grads[2][b, h])
    assert np.all(np.abs(dkh.sum(axis=0)) <= 1e-2 * np.abs(dkh).sum(axis=0)), (b, h)
    assert np.all(np.abs(dvh.sum(axis=0) - doh.sum(axis=0)) <= 1e-2 * np.abs(dvh).sum(axis=0))


def test_bf16_backward_workload(attn_lib):
    """[2,16,8192,128] bf16 causal on four seeded heads including the first
    and the last: the oracle recomputes those two heads whole; the other two
    are checked on sampled dQ rows and the dK / dV sum identities."""
    w = wl.BWD_BF16_D128
    inp = wl.make_inputs(w)
    grads = _gpu_grads(attn_lib, inp, w)
    heads = sample_heads(w.B, w.H, 4, seed=4)
    full = [(0, 0), (w.B - 1, w.H - 1)]
    assert len(heads) == 4 and all(hd in heads for hd in full)
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), True,
                                     w.scale, heads=full)
    _check(w, grads, refs, full)
    for (b, h) in heads:
        if (b, h) not in full:
            _check_sampled_head(inp, grads, b, h, True, w.scale, seed=b * 131 + h)


def test_noncausal_medium(attn_lib):
    w = wl.Workload("bwd_nc", "bwd", 1, 4, 2048, 128, "bf16", False, seed=3)
    inp = wl.make_inputs(w)
    grads = _gpu_grads(attn_lib, inp, w)
    heads = sample_heads(1, 4, 4, seed=1)
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), False,
                                     w.scale, heads=heads)
    _check(w, grads, refs, heads)


def test_q_zero_closed_forms(attn_lib):
    """Q = 0, causal: dK = 0 exactly and dV_j = sum_{i>=j} dO_i / (i+1)."""
    w = wl.Workload("bwd_q0", "bwd", 1, 2, 1500, 128, "bf16", True, seed=11)
    inp = wl.make_inputs(w)
    inp["q"] = torch.zeros_like(inp["q"])
    dq, dk, dv = _gpu_grads(attn_lib, inp, w)
    assert torch.count_nonzero(dk) == 0
    do = to64(inp["do"][0, 1])
    want = np.cumsum((do / np.arange(1, w.N + 1)[:, None])[::-1], axis=0)[::-1]
    err = np.max(np.abs(to64(dv[0, 1]) - want)) / np.max(np.abs(want))
    assert err <= REL_TOL


def test_bwd_argument_errors(attn_lib):
    L = attn_lib.lib()
    x = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 64), dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p, pl, pw = (ctypes.c_void_p(t.data_ptr()) for t in (x, lse, ws))
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    need = attn_lib.bwd_workspace_bytes(1, 1, 64, 128)
    args = lambda d, wsz: (p, p, p, p, p, pl, p, p, p, pw, wsz, 1, 1, 64, d, 1, 0.1, 1, s)  # noqa
    assert L.attn_bwd(*args(80, need)) == 2            # d = 80 unsupported
    assert L.attn_bwd(*args(128, need - 1)) == 1       # workspace too small
    assert L.attn_bwd(*args(128, need)) == 0
    assert attn_lib.poll_status()[0] == 0


@pytest.mark.parametrize("causal", [True, False])
def test_backward_is_deterministic(attn_lib, causal):
    """dK, dV (per key tile) and dQ (per query tile) are each accumulated by
    one CTA in a fixed order, with no atomics: two runs give the same bits."""
    w = wl.Workload("det", "bwd", 2, 4, 2000, 128, "bf16", causal, seed=21)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = attn_lib.fwd(q, k, v, causal=causal)
    g1 = attn_lib.bwd(q, k, v, o, do, lse, causal=causal)
    g2 = attn_lib.bwd(q, k, v, o, do, lse, causal=causal)
    assert attn_lib.poll_status() == (0, 0)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d", [128, 256])
def test_workspace_contents_do_not_matter(attn_lib, d):
    """The kernels take their units from counters in the workspace, which the
    D pass zeroes first: a workspace full of 0xFF bytes gives the same bits as
    a zeroed one."""
    w = wl.Workload("ws", "bwd", 1, 4, 1100, d, "bf16", True, seed=31)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    nbytes = attn_lib.bwd_workspace_bytes(1, 4, 1100, d)
    ws0 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ws1 = torch.full((nbytes,), 255, dtype=torch.uint8, device="cuda")
    g0 = attn_lib.bwd(q, k, v, o, do, lse, causal=True, workspace=ws0)
    g1 = attn_lib.bwd(q, k, v, o, do, lse, causal=True, workspace=ws1)
    assert attn_lib.poll_status() == (0, 0)
    for a, b in zip(g0, g1):
        assert torch.isfinite(a).all()
        assert torch.equal(a, b)


def test_two_streams_with_their_own_workspaces(attn_lib):
    """Two backward calls in flight at once on two streams, each with its own
    workspace (and so its own work counters), match a call run alone."""
    w = wl.Workload("streams", "bwd", 2, 4, 2048, 128, "bf16", True, seed=33)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    ref = attn_lib.bwd(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for s in streams:
        with torch.cuda.stream(s):
            outs.append(attn_lib.bwd(q, k, v, o, do, lse, causal=True))
    torch.cuda.synchronize()
    assert attn_lib.poll_status() == (0, 0)
    for g in outs:
        for a, b in zip(g, ref):
            assert torch.equal(a, b)
