"""attn_bwd_noalloc: the backward pass for callers that cannot allocate.

Callers such as plugins whose host framework owns every device allocation,
or serving loops that may not call cudaMalloc on the request path, use this
entry point instead of attn_bwd: it keeps its scratch in a fixed device array
inside the library, so the call allocates nothing.  It runs the same
deterministic kernels as attn_bwd (only the address of the delta vector
differs), so this file requires its dQ, dK, dV to be bitwise equal to
attn_bwd's, through the C ABI, on two calls in a row for each of five
different problems (a stale or misplaced scratch would change the bits),
checks the first problem against the fp64 oracle at the backward tolerance
(5e-2 * max |reference|), and checks that oversized problems are rejected.
It is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from helpers import to64

pytestmark = pytest.mark.gpu
REL_TOL = 5e-2
MAX_ROWS = 4194304  # B * H * N limit of the fixed scratch array


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _noalloc_fn(attn):
    L = attn.lib()
    fn = L.attn_bwd_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp]
    fn.restype = i
    return fn


def _call(fn, q, k, v, o, do, lse, dq, dk, dv, w, stream):
    return fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
              _ptr(dv), w.B, w.H, w.N, w.d, int(w.causal), float(w.scale),
              1 if w.dtype == "bf16" else 0, stream)  # ATTN_BF16 / ATTN_F16


def test_noalloc_backward_matches_attn_bwd_twice(attn_lib):
    import oracle
    fn = _noalloc_fn(attn_lib)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # five different problems through the shared scratch array, each twice
    for n, w in enumerate((wl.Workload("na1", "bwd", 1, 4, 1000, 128, "bf16", True, seed=31),
                           wl.Workload("na2", "bwd", 2, 3, 4096, 128, "bf16", False, seed=32),
                           wl.Workload("na3", "bwd", 1, 2, 700, 64, "fp16", True, seed=33),
                           wl.Workload("na4", "bwd", 2, 1, 390, 96, "bf16", True, seed=34),
                           wl.Workload("na5", "bwd", 1, 2, 333, 256, "bf16", True, seed=35))):
        inp = wl.make_inputs(w)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = attn_lib.fwd(q, k, v, causal=w.causal, scale=w.scale)
        ref = attn_lib.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
        for call in range(2):
            got = [torch.full_like(q, float("nan")) for _ in range(3)]
            assert _call(fn, q, k, v, o, do, lse, *got, w, stream) == 0
            st, detail = attn_lib.poll_status()
            assert st == 0, hex(detail)
            for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
                if not torch.equal(g, r):
                    gd, rd = to64(g), to64(r)
                    raise AssertionError(
                        f"{w.name} call {call}: {name} differs from attn_bwd, max |diff| "
                        f"{np.nanmax(np.abs(gd - rd)):.3e} (max |ref| {np.max(np.abs(rd)):.3e})")
        if n == 0:
            refs = oracle.attention_backward(*(to64(inp[x]) for x in ("q", "k", "v", "do")),
                                             w.causal, w.scale)
            for g, r in zip(got, refs):
                assert np.max(np.abs(to64(g) - r)) <= REL_TOL * np.max(np.abs(r))


def test_noalloc_and_bwd_on_two_devices_in_turn(attn_lib):
    """The shared-memory opt-in of the kernels and the scratch array's
    address are per device: calls alternating between two GPUs in one
    process must each run on their own device with the same results as on
    the first.  Skipped on machines with a single GPU."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    fn = _noalloc_fn(attn_lib)
    w = wl.Workload("na2dev", "bwd", 1, 2, 700, 128, "bf16", True, seed=41)
    inp = wl.make_inputs(w)
    results = []
    for dev in (0, 1, 0, 1):
        with torch.cuda.device(dev):
            q, k, v, do = (inp[n].to(f"cuda:{dev}") for n in ("q", "k", "v", "do"))
            o, lse = attn_lib.fwd(q, k, v, causal=True, scale=w.scale)
            ref = attn_lib.bwd(q, k, v, o, do, lse, causal=True, scale=w.scale)
            got = [torch.empty_like(q) for _ in range(3)]
            stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
            assert _call(fn, q, k, v, o, do, lse, *got, w, stream) == 0
            assert attn_lib.poll_status()[0] == 0
            for g, r in zip(got, ref):
                assert torch.equal(g, r)
            results.append([t.cpu() for t in got])
    for a, b in zip(results[0], results[1]):
        assert torch.equal(a, b)


def test_noalloc_rejects_oversized_problems(attn_lib):
    fn = _noalloc_fn(attn_lib)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    x = torch.zeros((1, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 16), dtype=torch.float32, device="cuda")
    big = wl.Workload("big", "bwd", 1, 1, MAX_ROWS + 1, 128, "bf16", True)
    assert _call(fn, x, x, x, x, x, lse, x, x, x, big, stream) == 1  # ATTN_ERR_INVALID_ARG
    d80 = wl.Workload("d80", "bwd", 1, 1, 16, 80, "bf16", True)
    assert _call(fn, x, x, x, x, x, lse, x, x, x, d80, stream) == 2  # ATTN_ERR_UNSUPPORTED
    assert attn_lib.poll_status()[0] == 0
