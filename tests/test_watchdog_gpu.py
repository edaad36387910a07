"""Failure path on the GPU without a fault: a bounded pipeline wait that runs
out of time must record ATTN_ERR_TIMEOUT in the status word and let the
kernel exit normally, leaving the context usable."""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives(attn_lib):
    st, detail = attn_lib.selftest_wait_timeout(20000)
    assert st == 4, (st, hex(detail))        # ATTN_ERR_TIMEOUT
    assert (detail & 0xFF) == 4 and ((detail >> 8) & 0xFF) == 99
    assert attn_lib.poll_status() == (0, 0)  # polled once, then cleared
    # the context still works: a normal launch afterwards succeeds
    w = wl.Workload("t", "fwd", 1, 1, 256, 64, "fp16", True)
    inp = wl.make_inputs(w)
    o, lse = attn_lib.fwd(*(inp[n].cuda() for n in ("q", "k", "v")), causal=True)
    torch.cuda.synchronize()
    assert attn_lib.poll_status()[0] == 0
    assert torch.isfinite(o.float()).all()


def _expect_timeout(attn, launch, attempts=3):
    """Run `launch` with a 1 us pipeline-wait limit until a launch reports
    ATTN_ERR_TIMEOUT (status 4, timeout code in the low byte of the detail
    word).  Every attempt must end cleanly (0) or with that status, and at
    least one must time out: the wind-down path must have run."""
    seen = []
    attn.set_wait_limit_us(1)
    try:
        for _ in range(attempts):
            launch()
            st, detail = attn.poll_status()
            assert st in (0, 4), (st, hex(detail))
            seen.append((st, detail))
            if st == 4:
                assert (detail & 0xFF) == 4, hex(detail)
                break
    finally:
        attn.set_wait_limit_us(0)  # back to the default limit
    assert any(st == 4 for st, _ in seen), seen


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64)])
def test_forward_winds_down_when_waits_run_out(attn_lib, dtype, d):
    """With a 1 us wait limit, pipeline waits inside the forward kernel run out
    during an ordinary launch.  Every role must then walk the rest of its
    schedule without waiting (the issuer's named barriers still pair up), the
    kernel must end with ATTN_ERR_TIMEOUT in the status word, and the next
    launch at the normal limit must be correct."""
    import numpy as np
    import oracle
    from helpers import to64
    w = wl.Workload("t", "fwd", 2, 4, 2048, d, dtype, True, seed=d)
    inp = wl.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    attn_lib.poll_status()
    _expect_timeout(attn_lib, lambda: attn_lib.fwd(q, k, v, causal=True))
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    rows = np.arange(0, w.N, 97)
    O_ref, L_ref = oracle.attention_rows(to64(inp["q"][1, 2]), to64(inp["k"][1, 2]),
                                         to64(inp["v"][1, 2]), rows, True, w.scale)
    assert np.max(np.abs(to64(o[1, 2])[rows] - O_ref)) <= 2e-2
    assert np.max(np.abs(to64(lse[1, 2])[rows] - L_ref)) <= 5e-3


@pytest.mark.parametrize("d", [128, 64])
def test_backward_winds_down_when_waits_run_out(attn_lib, d):
    """The same for the backward main kernels: with a 1 us wait limit their
    roles walk their schedules to the end without waiting, the launch reports
    ATTN_ERR_TIMEOUT, and a following backward at the normal limit matches
    the oracle (d = 64 runs the dK/dV kernel with two S^T buffers)."""
    import numpy as np
    import oracle
    from helpers import to64
    # at d = 64 the small case's waits are all shorter than the limit; a
    # larger one gives every CTA several units, so some producer waits
    H, N = (2, 1024) if d == 128 else (8, 4096)
    w = wl.Workload("t", "bwd", 1, H, N, d, "bf16", True, seed=11)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    _expect_timeout(attn_lib, lambda: attn_lib.bwd(q, k, v, o, do, lse, causal=True))
    dq, dk, dv = attn_lib.bwd(q, k, v, o, do, lse, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    heads = [(0, 0), (0, H - 1)]
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), True,
                                     w.scale, heads=heads)
    for g, r in zip((dq, dk, dv), refs):
        g = np.stack([to64(g)[b, h] for b, h in heads])
        r = np.stack([r[b, h] for b, h in heads])
        assert np.max(np.abs(g - r)) <= 5e-2 * np.max(np.abs(r))


@pytest.mark.parametrize("d", [192, 256])
def test_wide_kernels_wind_down_when_waits_run_out(attn_lib, d):
    """The same for the wide head dims' forward and backward kernels (one
    query tile per forward unit; the 64-row backward rings), on enough work
    units that every CTA runs more than one (a producer then waits a whole
    unit for its next one, which outlasts any 1 us limit): a launch whose
    waits run out reports ATTN_ERR_TIMEOUT and the next launches at the
    normal limit match the oracle (two whole heads)."""
    import numpy as np
    import oracle
    from helpers import to64
    w = wl.Workload("tw", "bwd", 1, 8, 4096, d, "bf16", True, seed=d + 3)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    attn_lib.poll_status()
    _expect_timeout(attn_lib, lambda: attn_lib.fwd(q, k, v, causal=True))
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    _expect_timeout(attn_lib, lambda: attn_lib.bwd(q, k, v, o, do, lse, causal=True))
    dq, dk, dv = attn_lib.bwd(q, k, v, o, do, lse, causal=True)
    assert attn_lib.poll_status() == (0, 0)
    heads = [(0, 0), (0, 7)]
    refs = oracle.attention_backward(*(to64(inp[n]) for n in ("q", "k", "v", "do")), True,
                                     w.scale, heads=heads)
    for (b, h) in heads:
        O_ref, L_ref = oracle.attention_rows(to64(inp["q"][b, h]), to64(inp["k"][b, h]),
                                             to64(inp["v"][b, h]), np.arange(w.N), True,
                                             w.scale)
        assert np.max(np.abs(to64(o[b, h]) - O_ref)) <= 2e-2
        assert np.max(np.abs(to64(lse[b, h]) - L_ref)) <= 5e-3
        for g, r in zip((dq, dk, dv), refs):
            assert np.max(np.abs(to64(g[b, h]) - r[b, h])) <= 5e-2 * np.max(np.abs(r[b, h]))


def test_decoding_kernel_winds_down_when_waits_run_out(attn_lib):
    """The same for the decoding kernel (each warp streams its key/value
    blocks through a ring of its own): one query per head, 16 sequences x 16
    heads against an 8192-row cache in 4 splits, 1024 CTAs whose first copies
    queue behind each other's for longer than 1 us.  A launch whose waits run
    out reports ATTN_ERR_TIMEOUT; the next launch at the normal limit matches
    the oracle on the first and the last head."""
    import numpy as np
    import oracle
    from helpers import to64
    w = wl.DECODE_BF16_D128
    inp = wl.make_decode_inputs(w, kv_heads=w.H)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    attn_lib.poll_status()
    _expect_timeout(attn_lib, lambda: attn_lib.fwd_kv(q, k, v, 4, causal=w.causal, scale=w.scale))
    Op, Lp = attn_lib.fwd_kv(q, k, v, 4, causal=w.causal, scale=w.scale)
    assert attn_lib.poll_status() == (0, 0)
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        O_ref, L_ref = oracle.attention_kv(*(to64(inp[n][b:b + 1, h:h + 1]) for n in ("q", "k", "v")),
                                           w.causal, w.scale, 4)
        assert np.max(np.abs(to64(Op[:, b, h]) - O_ref[:, 0, 0])) <= 2e-2
        assert np.max(np.abs(to64(Lp[:, b, h]) - L_ref[:, 0, 0])) <= 5e-3
