"""Seeded random combinations of the features, CUDA path vs the fp64 oracle.

The other parity tests vary one feature at a time; here every case draws a
head dim (64, 96, 128), a dtype, the masking, a grouped-query layout and
ragged sizes together, and runs one of three paths:
  dense  : forward and backward, [B, Hq, N, d] with Hkv key/value heads;
  varlen : forward and backward of a packed batch of random lengths
           (empty sequences allowed), grouped heads;
  split  : forward over n_split key ranges (partials against the oracle's
           partials) and the merge of the device partials against the
           oracle's full attention.
A second set of cases draws decoding shapes (at most 16 query rows per
key/value head, every head dim including 192 and 256, a ragged cache, 1-12
key splits) for the key-cache forward and the merge; at d = 192 and 256 a
third of them take 17-128 rows (groups of 16 rows on the decoding kernel).
Tolerances as everywhere: |O - O_ref| <= 2e-2, |LSE - LSE_ref| <= 5e-3,
gradients <= 5e-2 * max |ref| per tensor (an all-zero reference, e.g. N = 1,
bounds |g| <= 1e-3).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from helpers import to64

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, REL_TOL = 2e-2, 5e-3, 5e-2
CASES = 30


def _draw(seed):
    rng = np.random.default_rng(7000 + seed)
    c = {"mode": ("dense", "varlen", "split")[seed % 3],
         "d": int(rng.choice([64, 96, 128])),
         "dtype": str(rng.choice(["fp16", "bf16"])),
         "causal": bool(rng.integers(2)),
         "Hkv": int(rng.integers(1, 3)),
         "G": int(rng.integers(1, 4)),
         "B": int(rng.integers(1, 3)),
         "N": int(rng.integers(1, 700)),
         "n_split": int(rng.integers(1, 7)),
         "seed": seed}
    n_seq = int(rng.integers(1, 6))
    # about one sequence in five empty
    lengths = [0 if rng.random() < 0.2 else int(rng.integers(1, 420)) for _ in range(n_seq)]
    if sum(lengths) == 0:
        lengths[0] = 1
    c["lengths"] = lengths
    return c


def _check_grads(grads, refs, case):
    for name, g, r in zip(("dQ", "dK", "dV"), grads, refs):
        g = to64(g)
        assert np.isfinite(g).all(), (case, name)
        ref_max = np.max(np.abs(r))
        if ref_max == 0.0:
            assert np.max(np.abs(g)) <= 1e-3, (case, name)
            continue
        err = np.max(np.abs(g - r)) / ref_max
        assert err <= REL_TOL, (case, name, err)


def _dense(attn, c):
    Hq = c["Hkv"] * c["G"]
    w = wl.Workload("fuzz", "bwd", c["B"], Hq, c["N"], c["d"], c["dtype"], c["causal"],
                    seed=c["seed"])
    inp = wl.make_inputs(w)
    # key/value heads: the first head of each group of the seeded inputs
    q, do = inp["q"], inp["do"]
    k, v = inp["k"][:, ::c["G"]].contiguous(), inp["v"][:, ::c["G"]].contiguous()
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = attn.fwd(qc, kc, vc, causal=w.causal, scale=w.scale)
    grads = attn.bwd(qc, kc, vc, o, doc, lse, causal=w.causal, scale=w.scale)
    assert attn.poll_status() == (0, 0), c
    O_ref, L_ref = oracle.attention_gqa(to64(q), to64(k), to64(v), w.causal, w.scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= O_TOL, c
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_TOL, c
    refs = oracle.attention_backward_gqa(to64(q), to64(k), to64(v), to64(do), w.causal,
                                         w.scale)
    _check_grads(grads, refs, c)


def _varlen(attn, c):
    Hq, d = c["Hkv"] * c["G"], c["d"]
    inp = wl.make_varlen_inputs(c["lengths"], Hq, c["Hkv"], d, c["dtype"], seed=c["seed"])
    scale = d ** -0.5
    q, k, v, do, cu = (inp[n].cuda() for n in ("q", "k", "v", "do", "cu_seqlens"))
    mx = max(c["lengths"])
    o, lse = attn.fwd_varlen(q, k, v, cu, mx, causal=c["causal"], scale=scale)
    grads = attn.bwd_varlen(q, k, v, o, do, lse, cu, mx, causal=c["causal"], scale=scale)
    assert attn.poll_status() == (0, 0), c
    args = (to64(inp["q"]), to64(inp["k"]), to64(inp["v"]))
    O_ref, L_ref = oracle.attention_varlen(*args, inp["cu_seqlens"].numpy(), c["causal"], scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= O_TOL, c
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_TOL, c
    refs = oracle.attention_backward_varlen(*args, to64(inp["do"]), inp["cu_seqlens"].numpy(),
                                            c["causal"], scale)
    _check_grads(grads, refs, c)


def _split(attn, c):
    w = wl.Workload("fuzz", "fwd", c["B"], c["Hkv"], c["N"], c["d"], c["dtype"], c["causal"],
                    seed=c["seed"])
    inp = wl.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    Op, Lp = attn.fwd_split(q, k, v, c["n_split"], causal=w.causal, scale=w.scale)
    O, L = attn.merge(Op, Lp)
    assert attn.poll_status() == (0, 0), c
    q64, k64, v64 = (to64(inp[n]) for n in ("q", "k", "v"))
    O_ref_p, L_ref_p = oracle.attention_split(q64, k64, v64, w.causal, w.scale, c["n_split"])
    Lp64 = to64(Lp)
    # a split a row sees no key of: LSE = -inf and O = 0 on both sides
    assert np.array_equal(np.isneginf(Lp64), np.isneginf(L_ref_p)), c
    seen = ~np.isneginf(L_ref_p)
    assert np.max(np.abs(Lp64[seen] - L_ref_p[seen]), initial=0.0) <= LSE_TOL, c
    assert np.max(np.abs(to64(Op) - O_ref_p)) <= O_TOL, c
    O_ref, L_ref = oracle.attention(q64, k64, v64, w.causal, w.scale)
    assert np.max(np.abs(to64(O) - O_ref)) <= O_TOL, c
    assert np.max(np.abs(to64(L) - L_ref)) <= LSE_TOL, c


@pytest.mark.parametrize("seed", range(CASES))
def test_random_feature_combination(attn_lib, seed):
    c = _draw(seed)
    {"dense": _dense, "varlen": _varlen, "split": _split}[c["mode"]](attn_lib, c)


DECODE_CASES = 36


def _draw_decode(seed):
    rng = np.random.default_rng(9000 + seed)
    G = int(rng.integers(1, 9))
    Nq = int(rng.integers(1, 16 // G + 1))  # G * Nq <= 16 rows per key/value head
    d = int(rng.choice([64, 96, 128, 192, 256]))
    if d > 128 and seed % 3 == 0:
        Nq = int(rng.integers(16 // G + 1, 128 // G + 1))  # 17-128 rows
    return {"d": d,
            "dtype": str(rng.choice(["fp16", "bf16"])),
            "causal": bool(rng.integers(2)),
            "B": int(rng.integers(1, 3)),
            "Hkv": int(rng.integers(1, 3)),
            "G": G, "Nq": Nq,
            "Nk": int(rng.integers(Nq, 3000)),
            "n_split": int(rng.integers(1, 13)),
            "seed": seed}


@pytest.mark.parametrize("seed", range(DECODE_CASES))
def test_random_decoding_case(attn_lib, seed):
    c = _draw_decode(seed)
    Hq = c["Hkv"] * c["G"]
    w = wl.Workload("fuzzdec", "fwd", c["B"], Hq, c["Nk"], c["d"], c["dtype"], c["causal"],
                    seed=c["seed"])
    inp = wl.make_inputs(w)
    # the queries are the last Nq positions; key/value heads the first head of each group
    q = inp["q"][:, :, c["Nk"] - c["Nq"]:].contiguous()
    k, v = inp["k"][:, ::c["G"]].contiguous(), inp["v"][:, ::c["G"]].contiguous()
    Op, Lp = attn_lib.fwd_kv(q.cuda(), k.cuda(), v.cuda(), c["n_split"], causal=w.causal,
                             scale=w.scale)
    O, L = attn_lib.merge(Op, Lp)
    assert attn_lib.poll_status() == (0, 0), c
    q64, k64, v64 = to64(q), to64(k), to64(v)
    O_ref_p, L_ref_p = oracle.attention_kv(q64, k64, v64, w.causal, w.scale, c["n_split"])
    Lp64 = to64(Lp)
    assert np.array_equal(np.isneginf(Lp64), np.isneginf(L_ref_p)), c
    seen = ~np.isneginf(L_ref_p)
    assert np.max(np.abs(Lp64[seen] - L_ref_p[seen]), initial=0.0) <= LSE_TOL, c
    assert np.max(np.abs(to64(Op) - O_ref_p)) <= O_TOL, c
    O_ref, L_ref = oracle.attention_kv(q64, k64, v64, w.causal, w.scale, 1)
    assert np.max(np.abs(to64(O) - O_ref[0])) <= O_TOL, c
    assert np.max(np.abs(to64(L) - L_ref[0])) <= LSE_TOL, c
