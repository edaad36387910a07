"""Split over the keys + merge: CUDA path (through the C ABI) vs the oracle.

attn_fwd_split's partial results are compared with the oracle's partial
attention over the same key ranges (split s = key blocks [s nb / S,
(s+1) nb / S)); attn_merge with the oracle's merge; and the merge of the
split equals full attention (the oracle's pinned identity), checked against
the oracle and against attn_fwd.  Tolerances as for the forward pass:
|O - O_ref| <= 2e-2, |LSE - LSE_ref| <= 5e-3; rows that see no key of a split
must have LSE = -inf and O = 0 exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import to64

pytestmark = pytest.mark.gpu
O_TOL, LSE_TOL = 2e-2, 5e-3


def _inputs(w):
    inp = wl.make_inputs(w)
    return [inp[n].cuda() for n in ("q", "k", "v")], inp


def _check_partials(Op, Lp, O_ref, L_ref):
    Op, Lp = to64(Op), to64(Lp)
    empty = ~np.isfinite(L_ref)
    assert np.array_equal(empty, Lp == -np.inf), "rows without keys must have LSE = -inf"
    assert not Op[empty].any(), "rows without keys must have O = 0"
    full = ~empty
    assert np.isfinite(Op).all()
    assert np.max(np.abs(Op[full] - O_ref[full]), initial=0.0) <= O_TOL
    assert np.max(np.abs(Lp[full] - L_ref[full]), initial=0.0) <= LSE_TOL


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,n_split", [(1, 2, 300, 2), (2, 1, 513, 3), (1, 1, 1000, 8),
                                           (1, 2, 256, 5), (1, 1, 129, 1)])
def test_split_partials_and_merge_small(attn_lib, dtype, d, causal, B, H, N, n_split):
    w = wl.Workload("t", "fwd", B, H, N, d, dtype, causal, seed=N + n_split)
    (q, k, v), inp = _inputs(w)
    Op, Lp = attn_lib.fwd_split(q, k, v, n_split, causal=causal, scale=w.scale)
    assert attn_lib.poll_status() == (0, 0)
    q64, k64, v64 = (to64(inp[n]) for n in ("q", "k", "v"))
    O_ref_p, L_ref_p = oracle.attention_split(q64, k64, v64, causal, w.scale, n_split)
    _check_partials(Op, Lp, O_ref_p, L_ref_p)
    # merge of the device partials vs the oracle's full attention
    O, L = attn_lib.merge(Op, Lp)
    O_ref, L_ref = oracle.attention(q64, k64, v64, causal, w.scale)
    assert np.max(np.abs(to64(O) - O_ref)) <= O_TOL
    assert np.max(np.abs(to64(L) - L_ref)) <= LSE_TOL


@pytest.mark.parametrize("d", [64, 96, 128, 192, 256])
def test_merge_kernel_vs_oracle_merge(attn_lib, d):
    """The merge alone on synthetic partials: random O_s, LSE_s of spread
    magnitudes, some -inf (a split without keys) and one all -inf row."""
    g = torch.Generator().manual_seed(d)
    S, B, H, N = 5, 2, 3, 77
    Op = torch.randn((S, B, H, N, d), generator=g).to(torch.bfloat16)
    Lp = (torch.randn((S, B, H, N), generator=g) * 20.0).to(torch.float32)
    drop = torch.rand((S, B, H, N), generator=g) < 0.3
    Lp[drop] = float("-inf")
    Lp[:, 1, 2, 5] = float("-inf")
    O, L = attn_lib.merge(Op.cuda(), Lp.cuda())
    assert attn_lib.poll_status() == (0, 0)
    O_ref, L_ref = oracle.merge_partials(to64(Op), to64(Lp))
    assert np.max(np.abs(to64(O) - O_ref)) <= O_TOL
    fin = np.isfinite(L_ref)
    assert np.array_equal(fin, np.isfinite(to64(L)))
    assert np.max(np.abs(to64(L)[fin] - L_ref[fin])) <= 1e-4
    assert not to64(O)[~fin].any()


@pytest.mark.parametrize("d", [64, 128])
def test_merge_of_the_most_splits(attn_lib, d):
    """256 partials (the most attn_merge takes; its reads go four splits at a
    time) with most splits empty for some rows and rows of every kind of
    spread, against the oracle's merge."""
    g = torch.Generator().manual_seed(256 + d)
    S, B, H, N = 256, 1, 2, 45
    Op = torch.randn((S, B, H, N, d), generator=g).to(torch.bfloat16)
    Lp = (torch.randn((S, B, H, N), generator=g) * 8.0).to(torch.float32)
    Lp[torch.rand((S, B, H, N), generator=g) < 0.7] = float("-inf")
    Lp[:, 0, 1, 3] = float("-inf")      # a row without keys
    Lp[:, 0, 0, 7] = float("-inf")
    Lp[200, 0, 0, 7] = 3.0              # a row with one split only, late in the order
    O, L = attn_lib.merge(Op.cuda(), Lp.cuda())
    assert attn_lib.poll_status() == (0, 0)
    O_ref, L_ref = oracle.merge_partials(to64(Op), to64(Lp))
    assert np.max(np.abs(to64(O) - O_ref)) <= O_TOL
    fin = np.isfinite(L_ref)
    assert np.array_equal(fin, np.isfinite(to64(L)))
    assert np.max(np.abs(to64(L)[fin] - L_ref[fin])) <= 1e-4
    assert not to64(O)[~fin].any()


def test_split_one_equals_fwd(attn_lib):
    w = wl.Workload("t", "fwd", 1, 2, 700, 128, "bf16", True, seed=3)
    (q, k, v), _ = _inputs(w)
    o, lse = attn_lib.fwd(q, k, v, causal=True)
    Op, Lp = attn_lib.fwd_split(q, k, v, 1, causal=True)
    assert torch.equal(Op[0], o) and torch.equal(Lp[0], lse)


@pytest.mark.parametrize("causal", [True, False])
def test_split_workload_full_size(attn_lib, causal):
    """[2,16,8192,128] bf16 with 4 splits: the merge equals attn_fwd's O and
    LSE everywhere (a property at any size), and sampled rows of the merged
    result and of each partial match the oracle."""
    w = wl.FWD_BF16_D128.with_(causal=causal)
    (q, k, v), inp = _inputs(w)
    o, lse = attn_lib.fwd(q, k, v, causal=causal)
    Op, Lp = attn_lib.fwd_split(q, k, v, 4, causal=causal)
    O, L = attn_lib.merge(Op, Lp)
    assert attn_lib.poll_status() == (0, 0)
    assert (O.float() - o.float()).abs().max().item() <= O_TOL
    assert (L - lse).abs().max().item() <= LSE_TOL
    rows = np.arange(0, w.N, 331)
    for b, h in ((0, 0), (1, 15)):
        q64, k64, v64 = (to64(inp[n][b, h]) for n in ("q", "k", "v"))
        O_ref, L_ref = oracle.attention_rows(q64, k64, v64, rows, causal, w.scale)
        assert np.max(np.abs(to64(O[b, h])[rows] - O_ref)) <= O_TOL
        assert np.max(np.abs(to64(L[b, h])[rows] - L_ref)) <= LSE_TOL
        for s, (lo, hi) in enumerate(oracle.split_key_ranges(w.N, 4)):
            Os, Ls = oracle.attention_partial_head(q64[rows], k64, v64, False, w.scale, lo, hi) \
                if not causal else _partial_rows(q64, k64, v64, rows, w.scale, lo, hi)
            got_O, got_L = to64(Op[s, b, h])[rows], to64(Lp[s, b, h])[rows]
            fin = np.isfinite(Ls)
            assert np.array_equal(fin, np.isfinite(got_L))
            assert np.max(np.abs(got_O[fin] - Os[fin]), initial=0.0) <= O_TOL
            assert np.max(np.abs(got_L[fin] - Ls[fin]), initial=0.0) <= LSE_TOL


def _partial_rows(q, k, v, rows, scale, lo, hi):
    """Causal partial attention of selected rows over keys [lo, hi)."""
    O = np.zeros((len(rows), v.shape[1]))
    L = np.full(len(rows), -np.inf)
    for n, i in enumerate(rows):
        top = min(hi, i + 1)
        if top <= lo:
            continue
        s = scale * (k[lo:top] @ q[i])
        m = s.max()
        e = np.exp(s - m)
        L[n] = m + np.log(e.sum())
        O[n] = (e / e.sum()) @ v[lo:top]
    return O, L


def test_split_rejects_bad_arguments(attn_lib):
    x = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16, device="cuda")
    for n_split in (0, 257):
        with pytest.raises(attn_lib.AttnError):
            attn_lib.fwd_split(x, x, x, n_split)
    assert attn_lib.poll_status() == (0, 0)
