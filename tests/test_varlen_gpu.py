"""Variable-length batches: CUDA path (C ABI) vs the fp64 oracle.

Sequences of their own lengths are packed back to back ([H, total, d]);
sequence b owns rows cu_seqlens[b]..cu_seqlens[b+1] and attends only to
itself, causal counted from its first row.  Tolerances as for the plain
forward and backward: |O - O_ref| <= 2e-2, |LSE - LSE_ref| <= 5e-3, gradients
<= 5e-2 * max |ref| (per tensor).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import to64

pytestmark = pytest.mark.gpu

# ragged lengths around the 128-row tile, an empty sequence, one longer than
# four tiles
MIX = [1, 127, 128, 129, 0, 300, 513, 64]


def _run_fwd(attn, inp, max_seqlen, causal, scale):
    q, k, v, cu = (inp[n].cuda() for n in ("q", "k", "v", "cu_seqlens"))
    o, lse = attn.fwd_varlen(q, k, v, cu, max_seqlen, causal=causal, scale=scale)
    assert attn.poll_status() == (0, 0)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64), ("bf16", 96)])
@pytest.mark.parametrize("lengths,Hq,Hkv", [(MIX, 4, 2), (MIX, 2, 2), ([700], 2, 1),
                                            ([256, 256, 256], 3, 3)])
def test_varlen_forward(attn_lib, causal, dtype, d, lengths, Hq, Hkv):
    inp = wl.make_varlen_inputs(lengths, Hq, Hkv, d, dtype, seed=len(lengths) + d,
                                with_do=False)
    scale = d ** -0.5
    o, lse = _run_fwd(attn_lib, inp, max(lengths), causal, scale)
    O_ref, L_ref = oracle.attention_varlen(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]),
                                           inp["cu_seqlens"].numpy(), causal, scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= 2e-2
    assert np.max(np.abs(to64(lse) - L_ref)) <= 5e-3


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64), ("bf16", 96)])
@pytest.mark.parametrize("lengths,Hq,Hkv", [(MIX, 4, 2), ([129, 0, 384, 1], 2, 2)])
def test_varlen_backward(attn_lib, causal, dtype, d, lengths, Hq, Hkv):
    inp = wl.make_varlen_inputs(lengths, Hq, Hkv, d, dtype, seed=3 * len(lengths) + Hkv + d)
    scale = d ** -0.5
    q, k, v, do, cu = (inp[n].cuda() for n in ("q", "k", "v", "do", "cu_seqlens"))
    o, lse = attn_lib.fwd_varlen(q, k, v, cu, max(lengths), causal=causal, scale=scale)
    dq, dk, dv = attn_lib.bwd_varlen(q, k, v, o, do, lse, cu, max(lengths), causal=causal,
                                     scale=scale)
    assert attn_lib.poll_status() == (0, 0)
    refs = oracle.attention_backward_varlen(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]),
                                            to64(inp["do"]), inp["cu_seqlens"].numpy(), causal,
                                            scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        err = np.max(np.abs(to64(g) - r)) / np.max(np.abs(r))
        assert err <= 5e-2, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_the_dense_path_bitwise(attn_lib, causal):
    """B sequences of one length N packed into [H, B*N, d] give exactly the
    dense [B, H, N, d] results: every tile does the same arithmetic, rows of a
    neighbouring sequence are masked where the dense path reads zero fill."""
    B, H, N, d = 3, 4, 300, 128
    w = wl.Workload("vd", "bwd", B, H, N, d, "bf16", causal, seed=41)
    inp = wl.make_inputs(w)
    dense = {n: inp[n].cuda() for n in ("q", "k", "v", "do")}
    packed = {n: t.permute(1, 0, 2, 3).reshape(H, B * N, d).contiguous()
              for n, t in dense.items()}
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device="cuda")
    o, lse = attn_lib.fwd(dense["q"], dense["k"], dense["v"], causal=causal)
    dq, dk, dv = attn_lib.bwd(dense["q"], dense["k"], dense["v"], o, dense["do"], lse,
                              causal=causal)
    ov, lsev = attn_lib.fwd_varlen(packed["q"], packed["k"], packed["v"], cu, N, causal=causal)
    dqv, dkv, dvv = attn_lib.bwd_varlen(packed["q"], packed["k"], packed["v"], ov, packed["do"],
                                        lsev, cu, N, causal=causal)
    assert attn_lib.poll_status() == (0, 0)

    def pack(t):
        return t.permute(1, 0, 2, 3).reshape(H, B * N, d)

    assert torch.equal(ov, pack(o))
    assert torch.equal(lsev, lse.permute(1, 0, 2).reshape(H, B * N))
    for a, b in ((dqv, dq), (dkv, dk), (dvv, dv)):
        assert torch.equal(a, pack(b))


def test_larger_max_seqlen_changes_nothing(attn_lib):
    inp = wl.make_varlen_inputs(MIX, 2, 1, 128, "bf16", seed=5, with_do=False)
    T = int(sum(MIX))
    o1, l1 = _run_fwd(attn_lib, inp, max(MIX), True, 0.1)
    o2, l2 = _run_fwd(attn_lib, inp, T, True, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("cu", [[0, 200, 100, 300], [0, 100, 250], [5, 100, 300],
                                [0, 290, 300]])
def test_bad_offsets_are_reported(attn_lib, cu):
    """Offsets that are not a partition of [0, total) into runs of at most
    max_seqlen rows: the device check records ATTN_ERR_INVALID_ARG (the kernels
    clamp every sequence into the tensors, so nothing is accessed outside)."""
    T, H, d = 300, 2, 128
    q = torch.randn((H, T, d), device="cuda").to(torch.bfloat16)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    attn_lib.poll_status()
    attn_lib.fwd_varlen(q, q, q, cu_t, 256, causal=True)
    st, detail = attn_lib.poll_status()
    assert st == 1 and (detail & 0xFF) == 1 and ((detail >> 8) & 0xFF) == 60, (st, hex(detail))
    # the context is still usable
    inp = wl.make_varlen_inputs([100, 200], H, H, d, "bf16", seed=1, with_do=False)
    _run_fwd(attn_lib, inp, 200, True, d ** -0.5)


def test_varlen_measured_mix_sampled(attn_lib):
    """The measured batch (16 heads, d = 128, bf16, causal, 16384 tokens in the
    seeded length mix): forward on sampled rows of every sequence for two
    heads, backward of the shortest sequence for one head."""
    lengths = wl.varlen_lengths()
    H = wl.VARLEN_HEADS
    inp = wl.make_varlen_inputs(lengths, H, H, wl.VARLEN_D, "bf16", seed=0)
    scale = wl.VARLEN_D ** -0.5
    q, k, v, do, cu = (inp[n].cuda() for n in ("q", "k", "v", "do", "cu_seqlens"))
    o, lse = attn_lib.fwd_varlen(q, k, v, cu, max(lengths), causal=True)
    dq, dk, dv = attn_lib.bwd_varlen(q, k, v, o, do, lse, cu, max(lengths), causal=True)
    assert attn_lib.poll_status() == (0, 0)
    ranges = oracle.sequence_ranges(inp["cu_seqlens"].numpy())
    for h in (0, 11):
        for lo, hi in ranges:
            rows = np.unique(np.r_[np.arange(0, hi - lo, 97), hi - lo - 1])
            O_ref, L_ref = oracle.attention_rows(to64(inp["q"][h, lo:hi]),
                                                 to64(inp["k"][h, lo:hi]),
                                                 to64(inp["v"][h, lo:hi]), rows, True, scale)
            assert np.max(np.abs(to64(o[h, lo:hi])[rows] - O_ref)) <= 2e-2
            assert np.max(np.abs(to64(lse[h, lo:hi])[rows] - L_ref)) <= 5e-3
    b = int(np.argmin(lengths))
    lo, hi = ranges[b]
    h = 5
    sl = slice(lo, hi)
    refs = oracle.attention_backward_head(to64(inp["q"][h, sl]), to64(inp["k"][h, sl]),
                                          to64(inp["v"][h, sl]), to64(inp["do"][h, sl]), True,
                                          scale)[:3]
    for g, r in zip((dq[h, sl], dk[h, sl], dv[h, sl]), refs):
        assert np.max(np.abs(to64(g) - r)) / np.max(np.abs(r)) <= 5e-2
