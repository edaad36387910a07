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
