"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: scalar brute force
written with ``math`` loops, closed forms, invariants of softmax attention,
finite differences, library special cases (torch SDPA / autograd in fp64),
and a brute-force search over all 256 E4M3 codes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _rand(*shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- forward ---

def _brute_force_head(q, k, v, causal, scale):
    """Scalar loops with math.exp/math.log, no numpy linear algebra."""
    N, d = len(q), len(q[0])
    O, L = [], []
    for i in range(N):
        js = [j for j in range(len(k)) if (not causal or j <= i)]
        s = [scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in js]
        z = sum(math.exp(x) for x in s)
        L.append(math.log(z))
        O.append([sum(math.exp(s[a]) / z * v[j][c] for a, j in enumerate(js))
                  for c in range(len(v[0]))])
    return np.array(O), np.array(L)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (5, 3), (9, 4), (13, 8)])
def test_forward_matches_scalar_brute_force(causal, N, d):
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    scale = 0.37
    O, L, _ = oracle.attention_head(q, k, v, causal, scale)
    Ob, Lb = _brute_force_head(q.tolist(), k.tolist(), v.tolist(), causal, scale)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


def test_forward_closed_form_two_keys():
    # N=2, d=1, scale=1: S = [[1*1, 1*0], [2*1, 2*0]] = [[1,0],[2,0]].
    q = np.array([[1.0], [2.0]])
    k = np.array([[1.0], [0.0]])
    v = np.array([[1.0], [3.0]])
    O, L, _ = oracle.attention_head(q, k, v, False, 1.0)
    e, e2 = math.e, math.e ** 2
    assert abs(O[0, 0] - (e * 1 + 1 * 3) / (e + 1)) < 1e-14
    assert abs(O[1, 0] - (e2 * 1 + 1 * 3) / (e2 + 1)) < 1e-14
    assert abs(L[0] - math.log(e + 1)) < 1e-14
    assert abs(L[1] - math.log(e2 + 1)) < 1e-14
    Oc, Lc, _ = oracle.attention_head(q, k, v, True, 1.0)
    assert abs(Oc[0, 0] - 1.0) < 1e-15 and abs(Lc[0] - 1.0) < 1e-15  # only key 0
    assert abs(Oc[1, 0] - O[1, 0]) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    S = _rand(40, 40) * 5
    P, _ = oracle.masked_softmax(S, oracle.allowed_mask(40, 40, causal))
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(P[np.triu_indices(40, 1)] == 0.0)


def test_q_zero_causal_is_prefix_mean():
    N, d = 37, 6
    v = _rand(N, d)
    O, L, _ = oracle.attention_head(np.zeros((N, d)), _rand(N, d), v, True, 0.5)
    for i in range(N):
        np.testing.assert_allclose(O[i], v[:i + 1].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(L[i] - math.log(i + 1)) < 1e-13


def test_q_zero_noncausal_is_mean():
    N, d = 29, 5
    v = _rand(N, d)
    O, L, _ = oracle.attention_head(np.zeros((N, d)), _rand(N, d), v, False, 0.5)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=0), O.shape), atol=1e-13)
    np.testing.assert_allclose(L, math.log(N), atol=1e-13)


def test_causal_row0_is_v0():
    q, k, v = _rand(20, 7), _rand(20, 7), _rand(20, 7)
    O, L, _ = oracle.attention_head(q, k, v, True, 1 / math.sqrt(7))
    np.testing.assert_allclose(O[0], v[0], rtol=0, atol=1e-15)
    assert abs(L[0] - q[0] @ k[0] / math.sqrt(7)) < 1e-13


def test_row_shift_invariance():
    S = _rand(16, 16)
    allowed = oracle.allowed_mask(16, 16, True)
    P, L = oracle.masked_softmax(S, allowed)
    c = _rand(16)[:, None] * 10
    P2, L2 = oracle.masked_softmax(S + c, allowed)
    np.testing.assert_allclose(P2, P, atol=1e-13)
    np.testing.assert_allclose(L2, L + c[:, 0], atol=1e-12)


def test_batch_head_permutation_equivariance():
    q, k, v = _rand(2, 3, 11, 4), _rand(2, 3, 11, 4), _rand(2, 3, 11, 4)
    O, L = oracle.attention(q, k, v, True, 0.5)
    pb, ph = [1, 0], [2, 0, 1]
    Op, Lp = oracle.attention(q[pb][:, ph], k[pb][:, ph], v[pb][:, ph], True, 0.5)
    np.testing.assert_array_equal(Op, O[pb][:, ph])
    np.testing.assert_array_equal(Lp, L[pb][:, ph])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 7, 64, 128])
def test_online_softmax_recurrence_equals_definition(causal, block):
    N, d = 150, 16
    q, k, v = _rand(N, d) * 2, _rand(N, d) * 2, _rand(N, d)
    O, L, _ = oracle.attention_head(q, k, v, causal, 0.25)
    O2, L2 = oracle.online_softmax_attention_head(q, k, v, causal, 0.25, block)
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_torch_sdpa_fp64(causal):
    q, k, v = _rand(2, 2, 33, 8), _rand(2, 2, 33, 8), _rand(2, 2, 33, 8)
    O, _ = oracle.attention(q, k, v, causal, 0.3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        is_causal=causal, scale=0.3).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_rows_matches_full(causal):
    q, k, v = _rand(50, 8), _rand(50, 8), _rand(50, 8)
    O, L, _ = oracle.attention_head(q, k, v, causal, 0.4)
    rows = [0, 1, 17, 49]
    Or, Lr = oracle.attention_rows(q, k, v, rows, causal, 0.4)
    np.testing.assert_allclose(Or, O[rows], atol=1e-13)
    np.testing.assert_allclose(Lr, L[rows], atol=1e-13)


# --------------------------------------------------------------- backward ---

def _loss(q, k, v, do, causal, scale):
    O, _, _ = oracle.attention_head(q, k, v, causal, scale)
    return float(np.sum(O * do))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(4, 3), (9, 8), (16, 5)])
def test_backward_finite_differences(causal, N, d):
    q, k, v, do = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    scale = 1 / math.sqrt(d)
    dQ, dK, dV, _ = oracle.attention_backward_head(q, k, v, do, causal, scale)
    h = 1e-6
    for name, X, G in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args = {"q": q, "k": k, "v": v}
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args[name] = Xp
            lp = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            args[name] = Xm
            lm = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - G)) / max(1e-30, np.max(np.abs(G)))
        assert err < 1e-6, (name, err)


def test_backward_q_zero_closed_forms():
    N, d = 12, 4
    k, v, do = _rand(N, d), _rand(N, d), _rand(N, d)
    dQ, dK, dV, _ = oracle.attention_backward_head(np.zeros((N, d)), k, v, do, True, 0.5)
    assert np.all(dK == 0.0)
    for j in range(N):
        want = sum(do[i] / (i + 1) for i in range(j, N))
        np.testing.assert_allclose(dV[j], want, atol=1e-13)


def test_backward_ds_rows_sum_to_zero():
    N, d = 30, 8
    _, _, _, dS = oracle.attention_backward_head(_rand(N, d), _rand(N, d), _rand(N, d),
                                                 _rand(N, d), True, 0.35)
    np.testing.assert_allclose(dS.sum(axis=1), 0.0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_fp64(causal):
    q, k, v, do = _rand(1, 2, 21, 8), _rand(1, 2, 21, 8), _rand(1, 2, 21, 8), _rand(1, 2, 21, 8)
    dQ, dK, dV = oracle.attention_backward(q, k, v, do, causal, 0.3)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.3)
    out.backward(torch.from_numpy(do))
    for mine, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=0, atol=1e-12)


# -------------------------------------------------------------------- FP8 ---

def _all_codes():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    return vals


def test_e4m3_decode_known_points():
    d = oracle.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3F, 0x7E, 0xFE, 0x80, 0xB8],
                                    np.uint8))
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.875, 448.0, -448.0, -0.0, -1.0]
    np.testing.assert_array_equal(d, want)
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    finite = _all_codes()[np.isfinite(_all_codes())]
    assert finite.max() == oracle.E4M3_MAX


def test_e4m3_encode_is_nearest_ties_to_even():
    vals = _all_codes()
    codes = np.arange(256)
    ok = np.isfinite(vals)
    vals, codes = vals[ok], codes[ok]
    x = np.concatenate([
        rng.standard_normal(4000) * 30, rng.standard_normal(2000) * 0.01,
        (vals[:, None] + vals[None, :]).ravel()[::37] / 2,       # exact midpoints
        np.array([500.0, -1000.0, 448.0, 0.0, 2.0 ** -10, 3 * 2.0 ** -10])]).astype(np.float32)
    enc = oracle.e4m3_encode(x)
    for xi, ci in zip(x.astype(np.float64), enc):
        xc = min(max(xi, -448.0), 448.0)
        dist = np.abs(vals - xc)
        best = np.flatnonzero(dist == dist.min())
        cand = codes[best]
        if len(cand) > 1:  # a tie: the even mantissa wins (zero: either sign)
            even = [c for c in cand if (c & 1) == 0]
            assert ci in even, (xi, ci, cand)
        else:
            assert ci == cand[0] or (vals[best[0]] == 0 and oracle.e4m3_decode(ci) == 0), (xi, ci)


def test_quantize_scales_and_error_bound():
    x = np.asarray(make_inputs(Workload("t", "fwd_fp8", 1, 2, 200, 32, "bf16", True,
                                        outliers=True))["q"].to(torch.float64))
    out = oracle.quantize_blocks(x, 64)
    x32 = out["x32"]
    for b in range(1):
        for h in range(2):
            for i in range(4):
                blk = x32[b, h, i * 64:(i + 1) * 64]
                s = np.float32(np.abs(blk).max()) / np.float32(448)
                assert out["scales"][b, h, i].view(np.uint32) == np.float32(s).view(np.uint32)
    deq = oracle.dequantize_blocks(out["codes"], out["scales"], 64)
    s_full = np.repeat(out["scales"].astype(np.float64), 64, axis=2)[:, :, :200, None]
    r = np.abs(x32 / s_full)
    bound = np.where(r >= 2.0 ** -6, s_full * r * 2.0 ** -4, s_full * 2.0 ** -10)
    assert np.all(np.abs(deq - x32) <= bound * (1 + 1e-6))
    # the largest element of every block is coded as +-448
    assert np.all(np.abs(oracle.e4m3_decode(out["codes"])).reshape(1, 2, -1).max(axis=2) == 448)


def test_quantize_all_zero_block_has_unit_scale():
    out = oracle.quantize_blocks(np.zeros((1, 1, 70, 16)), 64)
    assert np.all(out["scales"] == 1.0) and np.all(out["codes"] == 0)


def test_hadamard_orthogonality_and_invariance():
    for d in (1, 2, 8, 64, 128):
        Hd = oracle.hadamard_matrix(d)
        np.testing.assert_array_equal(Hd @ Hd.T, d * np.eye(d))
    signs = np.where(rng.random(16) < 0.5, -1, 1)
    R = oracle.rotation_matrix(signs)
    np.testing.assert_allclose(R @ R.T, np.eye(16), atol=1e-15)
    q, k, v = _rand(40, 16), _rand(40, 16), _rand(40, 16)
    O, L, _ = oracle.attention_head(q, k, v, True, 0.25)
    O2, L2, _ = oracle.attention_head(q @ R, k @ R, v, True, 0.25)
    np.testing.assert_allclose(O2, O, atol=1e-12)
    np.testing.assert_allclose(L2, L, atol=1e-12)


def test_hadamard_smears_outlier():
    # [FA3-8.3] 5.2: a single spike is spread evenly over all coordinates.
    x = np.zeros(128)
    x[5] = 20.0
    y = x @ oracle.rotation_matrix(np.ones(128))
    np.testing.assert_allclose(np.abs(y), 20 / math.sqrt(128), atol=1e-12)


def test_fp8_block_and_rotation_beat_per_tensor_on_outliers():
    """Directional pin of the [FA3-8.3] section-5 accuracy claim (2.6x there):
    per-block scales + Hadamard give lower O error than one per-tensor scale
    on inputs with 0.1% x20 outliers.  Emulated in fp64 on dequantized inputs.
    """
    w = Workload("t", "fwd_fp8", 1, 2, 512, 128, "bf16", True, outliers=True, hadamard=True)
    inp = make_inputs(w)
    q, k, v = (np.asarray(inp[n].to(torch.float64)) for n in ("q", "k", "v"))
    signs = inp["signs"].numpy()
    O_ref, _ = oracle.attention(q, k, v, True, w.scale)

    def per_tensor(x):
        out = oracle.quantize_blocks(x.reshape(1, 1, -1, x.shape[-1]), x.size // x.shape[-1])
        return oracle.dequantize_blocks(out["codes"], out["scales"], x.size // x.shape[-1]
                                        ).reshape(x.shape)

    def per_block(x, s=None):
        out = oracle.quantize_blocks(x, 64, s)
        return oracle.dequantize_blocks(out["codes"], out["scales"], 64)

    O_t, _ = oracle.attention(per_tensor(q), per_tensor(k), per_tensor(v), True, w.scale)
    O_b, _ = oracle.attention(per_block(q, signs), per_block(k, signs), per_block(v), True,
                              w.scale)
    e_t, e_b = oracle.rmse(O_t, O_ref), oracle.rmse(O_b, O_ref)
    assert e_b < e_t, (e_b, e_t)


# ------------------------------------------------------------ golden data ---

def test_golden_exp_vs_matmul_ratio():
    """[FA3-8.3] section 4: at head dim 128 the two matmuls need 512x the
    FLOPs of the exponentials.  Our FLOP count (4*N^2*d per head forward,
    one exp per score) must reproduce that ratio."""
    g = json.load(open(os.path.join(GOLDEN, "fa3_sec4_exp_ratio.json")))
    w = Workload("t", "fwd", 1, 1, 1024, g["head_dim"], "bf16", False)
    assert w.fwd_flops() / (w.N * w.N) == g["matmul_flops_per_exp"]
    assert abs(g["fp16_tensor_tflops"] / g["mufu_tflops"] - g["speed_ratio_approx"]) < 3


def test_golden_fa3_table_decoding():
    """[FA3-8.3] section 6.3 table (cell separators lost in extraction): the
    decoded columns must reproduce the printed speed-up column."""
    g = json.load(open(os.path.join(GOLDEN, "fa3_sec6_3_table.json")))
    for row in g["rows"]:
        raw = row["raw"]
        assert raw.startswith(row["seqlen"])
        assert raw == f'{row["seqlen"]}{row["fa2"]}{row["fa3"]}{row["speedup"]:.2f}x'
        assert abs(row["fa3"] / row["fa2"] - row["speedup"]) < 0.006


def test_fp8_recipe_error_floor():
    """The prescribed FP8 recipe (per-64-row E4M3 scales, Hadamard on Q and K)
    evaluated in fp64 on the dequantized inputs, with no kernel involved:
    on N(0,1) inputs its RMSE(O) is far below 3e-2; with 0.1% of entries x20
    it is already above 3e-2.  This is why the FP8 outlier workload is held to
    the quantization-aware oracle (see tests/test_fp8_gpu.py)."""
    res = {}
    for outl in (False, True):
        w = Workload("t", "fwd_fp8", 1, 1, 1024, 128, "bf16", True, outliers=outl,
                     hadamard=True, seed=3)
        inp = make_inputs(w)
        q, k, v = (np.asarray(inp[n].to(torch.float64)) for n in ("q", "k", "v"))
        s = inp["signs"].numpy()
        dq = lambda x, sg=None: oracle.dequantize_blocks(  # noqa: E731
            *[oracle.quantize_blocks(x, 64, sg)[y] for y in ("codes", "scales")], 64)
        O_ref, _ = oracle.attention(q, k, v, True, w.scale)
        O_q, _ = oracle.attention(dq(q, s), dq(k, s), dq(v), True, w.scale)
        res[outl] = oracle.rmse(O_q, O_ref)
    assert res[False] < 0.01 and res[True] > 0.03, res


# ---------------------------------------------------------------------------
# Split over the keys + merge (the single-GPU form of ring attention's
# exchange, [FA3-8.3] section 7.3; decoding split, [FA2-review] "Discussion
# Points").  Pins: the merge of partial results over a partition of the keys
# is, by the softmax definition, exactly the attention over all keys.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,block,n_split", [(300, 32, 2), (300, 32, 5), (257, 64, 3),
                                              (96, 32, 7), (128, 128, 1), (40, 16, 40)])
def test_split_then_merge_is_full_attention(causal, N, block, n_split):
    rng = np.random.default_rng(N + n_split)
    q, k, v = (rng.standard_normal((1, 2, N, 16)) for _ in range(3))
    Op, Lp = oracle.attention_split(q, k, v, causal, 0.3, n_split, block=block)
    O, L = oracle.merge_partials(Op, Lp)
    Or, Lr = oracle.attention(q, k, v, causal, 0.3)
    assert np.max(np.abs(O - Or)) < 1e-12 and np.max(np.abs(L - Lr)) < 1e-12


def test_split_merge_large_logits_stays_finite():
    # logits of order 1e3: a merge that exponentiates LSE_s without the
    # running maximum would overflow
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 1, 200, 8)) for _ in range(3))
    Op, Lp = oracle.attention_split(q, k, v, True, 400.0, 4, block=32)
    O, L = oracle.merge_partials(Op, Lp)
    Or, Lr = oracle.attention(q, k, v, True, 400.0)
    assert np.isfinite(O).all() and np.max(np.abs(O - Or)) < 1e-9
    assert np.max(np.abs(L - Lr) / np.abs(Lr)) < 1e-12


def test_partial_lse_brute_force():
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((9, 3)) for _ in range(3))
    O, L = oracle.attention_partial_head(q, k, v, True, 0.7, 3, 7)
    for i in range(9):
        keys = [j for j in range(3, 7) if j <= i]
        if not keys:
            assert L[i] == -np.inf and not O[i].any()
            continue
        e = [math.exp(0.7 * sum(q[i, c] * k[j, c] for c in range(3))) for j in keys]
        assert abs(L[i] - math.log(sum(e))) < 1e-13
        want = [sum(e[t] * v[j, c] for t, j in enumerate(keys)) / sum(e) for c in range(3)]
        assert np.max(np.abs(O[i] - want)) < 1e-13


def test_merge_order_free_and_associative():
    rng = np.random.default_rng(11)
    Op = rng.standard_normal((3, 5, 4))
    Lp = rng.standard_normal((3, 5)) * 3
    O, L = oracle.merge_partials(Op, Lp)
    Or, Lr = oracle.merge_partials(Op[::-1], Lp[::-1])
    O01, L01 = oracle.merge_partials(Op[:2], Lp[:2])
    Oa, La = oracle.merge_partials(np.stack([O01, Op[2]]), np.stack([L01, Lp[2]]))
    for a, b in ((O, Or), (L, Lr), (O, Oa), (L, La)):
        assert np.max(np.abs(a - b)) < 1e-13


def test_empty_split_is_neutral_and_all_empty_rows():
    rng = np.random.default_rng(13)
    Op = rng.standard_normal((2, 3, 4))
    Lp = rng.standard_normal((2, 3))
    O, L = oracle.merge_partials(Op, Lp)
    Oe, Le = oracle.merge_partials(np.concatenate([Op, np.full((1, 3, 4), 7.0)]),
                                   np.concatenate([Lp, np.full((1, 3), -np.inf)]))
    assert np.max(np.abs(O - Oe)) < 1e-15 and np.max(np.abs(L - Le)) < 1e-15
    Oz, Lz = oracle.merge_partials(np.ones((2, 3, 4)), np.full((2, 3), -np.inf))
    assert not Oz.any() and (Lz == -np.inf).all()


@pytest.mark.parametrize("n,ns", [(8192, 4), (300, 5), (100, 3), (129, 2)])
def test_split_key_ranges_tile_the_keys(n, ns):
    r = oracle.split_key_ranges(n, ns)
    assert r[0][0] == 0 and r[-1][1] == n and len(r) == ns
    for (a, b), (c, _) in zip(r, r[1:]):
        assert b == c and a <= b
    for a, _ in r:
        assert a % 128 == 0 or a == n


# ---------------------------------------------------------------------------
# Grouped query heads (GQA / MQA; linked from the "Insights" of [FA2-review]).
# Pins: identity with plain attention on K/V repeated over each group, the
# sum-over-group rule for dK/dV by finite differences, Hkv = Hq.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1), (8, 4), (3, 3)])
def test_gqa_equals_attention_on_repeated_kv(causal, Hq, Hkv):
    rng = np.random.default_rng(Hq * 10 + Hkv)
    q = rng.standard_normal((2, Hq, 33, 8))
    k, v = (rng.standard_normal((2, Hkv, 33, 8)) for _ in range(2))
    do = rng.standard_normal(q.shape)
    G = Hq // Hkv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    O, L = oracle.attention_gqa(q, k, v, causal, 0.4)
    Or, Lr = oracle.attention(q, kr, vr, causal, 0.4)
    assert np.max(np.abs(O - Or)) == 0.0 and np.max(np.abs(L - Lr)) == 0.0
    dQ, dK, dV = oracle.attention_backward_gqa(q, k, v, do, causal, 0.4)
    dQr, dKr, dVr = oracle.attention_backward(q, kr, vr, do, causal, 0.4)
    assert np.max(np.abs(dQ - dQr)) < 1e-14
    assert np.max(np.abs(dK - dKr.reshape(2, Hkv, G, 33, 8).sum(axis=2))) < 1e-13
    assert np.max(np.abs(dV - dVr.reshape(2, Hkv, G, 33, 8).sum(axis=2))) < 1e-13


def test_gqa_shared_kv_gradient_by_finite_differences():
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 4, 7, 3))
    k, v = (rng.standard_normal((1, 2, 7, 3)) for _ in range(2))
    do = rng.standard_normal(q.shape)
    _, dK, dV = oracle.attention_backward_gqa(q, k, v, do, True, 0.6)

    def loss(kk, vv):
        O, _ = oracle.attention_gqa(q, kk, vv, True, 0.6)
        return float(np.sum(O * do))

    eps = 1e-6
    for (g, i, c) in [(0, 3, 1), (1, 6, 2), (1, 0, 0)]:
        kp, km = k.copy(), k.copy()
        kp[0, g, i, c] += eps
        km[0, g, i, c] -= eps
        assert abs((loss(kp, v) - loss(km, v)) / (2 * eps) - dK[0, g, i, c]) < 1e-7
        vp, vm = v.copy(), v.copy()
        vp[0, g, i, c] += eps
        vm[0, g, i, c] -= eps
        assert abs((loss(k, vp) - loss(k, vm)) / (2 * eps) - dV[0, g, i, c]) < 1e-7


def test_kv_head_mapping_is_contiguous_groups():
    assert [oracle.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(h, 4, 1) for h in range(4)] == [0, 0, 0, 0]
    assert [oracle.kv_head_of(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]


# ---------------------------------------------------------------------------
# Variable-length batches (sequences packed back to back; "Discussion Points"
# of [FA2-review]).  Pins: attention over all packed rows with a
# block-diagonal (and, causal, per-sequence lower-triangular) mask built
# directly from the offsets; sequences do not see one another; the gradient
# by finite differences, an empty sequence included.
# ---------------------------------------------------------------------------

def _block_diagonal_mask(cu, causal):
    T = int(cu[-1])
    seq = np.full(T, -1)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    pos = np.arange(T) - np.asarray(cu)[np.maximum(seq, 0)]
    allowed = seq[:, None] == seq[None, :]
    if causal:
        allowed &= pos[None, :] <= pos[:, None]
    return allowed


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (3, 1)])
def test_varlen_equals_block_diagonal_masked_attention(causal, Hq, Hkv):
    rng = np.random.default_rng(7 * Hq + Hkv + causal)
    cu = np.array([0, 5, 5, 12, 13, 21])  # lengths 5, 0, 7, 1, 8
    T, d = int(cu[-1]), 6
    q = rng.standard_normal((Hq, T, d))
    k, v = (rng.standard_normal((Hkv, T, d)) for _ in range(2))
    O, L = oracle.attention_varlen(q, k, v, cu, causal, 0.5)
    allowed = _block_diagonal_mask(cu, causal)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        S = 0.5 * q[h] @ k[g].T
        S = np.where(allowed, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m)
        assert np.allclose(O[h], (e / e.sum(axis=1, keepdims=True)) @ v[g], rtol=0, atol=1e-13)
        assert np.allclose(L[h], np.log(e.sum(axis=1)) + m[:, 0], rtol=0, atol=1e-13)


def test_varlen_sequences_are_isolated():
    rng = np.random.default_rng(3)
    cu = np.array([0, 9, 20, 26])
    q, k, v = (rng.standard_normal((2, 26, 4)) for _ in range(3))
    O, L = oracle.attention_varlen(q, k, v, cu, True, 0.7)
    k2, v2 = k.copy(), v.copy()
    k2[:, 9:20] = rng.standard_normal((2, 11, 4))
    v2[:, 9:20] = rng.standard_normal((2, 11, 4))
    O2, L2 = oracle.attention_varlen(q, k2, v2, cu, True, 0.7)
    for lo, hi in [(0, 9), (20, 26)]:
        assert np.array_equal(O[:, lo:hi], O2[:, lo:hi]) and np.array_equal(L[:, lo:hi],
                                                                            L2[:, lo:hi])
    assert not np.allclose(O[:, 9:20], O2[:, 9:20])
    # the first row of every sequence sees only its own key under the causal mask
    for lo in (0, 9, 20):
        assert np.allclose(O[:, lo], v[:, lo], atol=1e-15)


def test_varlen_gradient_by_finite_differences():
    rng = np.random.default_rng(29)
    cu = np.array([0, 3, 3, 7])  # lengths 3, 0, 4
    q = rng.standard_normal((4, 7, 3))
    k, v = (rng.standard_normal((2, 7, 3)) for _ in range(2))
    do = rng.standard_normal(q.shape)
    dQ, dK, dV = oracle.attention_backward_varlen(q, k, v, do, cu, True, 0.6)

    def loss(qq, kk, vv):
        O, _ = oracle.attention_varlen(qq, kk, vv, cu, True, 0.6)
        return float(np.sum(O * do))

    eps = 1e-6
    for (h, i, c) in [(0, 0, 1), (3, 6, 2), (2, 4, 0), (1, 2, 2)]:
        qp, qm = q.copy(), q.copy()
        qp[h, i, c] += eps
        qm[h, i, c] -= eps
        assert abs((loss(qp, k, v) - loss(qm, k, v)) / (2 * eps) - dQ[h, i, c]) < 1e-7
    for (g, i, c) in [(0, 3, 1), (1, 6, 2), (1, 0, 0), (0, 2, 2)]:
        kp, km = k.copy(), k.copy()
        kp[g, i, c] += eps
        km[g, i, c] -= eps
        assert abs((loss(q, kp, v) - loss(q, km, v)) / (2 * eps) - dK[g, i, c]) < 1e-7
        vp, vm = v.copy(), v.copy()
        vp[g, i, c] += eps
        vm[g, i, c] -= eps
        assert abs((loss(q, k, vp) - loss(q, k, vm)) / (2 * eps) - dV[g, i, c]) < 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_dq_rows_equal_the_full_backward(causal):
    """The row-restricted dQ (for sampled rows of long sequences) equals the
    full-matrix backward, itself pinned by finite differences."""
    rng = np.random.default_rng(12 + causal)
    q, k, v, do = (rng.standard_normal((37, 5)) for _ in range(4))
    dQ, _, _, _ = oracle.attention_backward_head(q, k, v, do, causal, 0.45)
    rows = [0, 1, 17, 36]
    assert np.allclose(oracle.attention_backward_dq_rows(q, k, v, do, rows, causal, 0.45),
                       dQ[rows], rtol=0, atol=1e-13)


# ------------------------------------------------- queries against a cache ---

@pytest.mark.parametrize("nq,nk", [(1, 9), (3, 9), (5, 5), (4, 130)])
def test_kv_queries_are_the_suffix_of_full_causal_attention(nq, nk):
    """The Nq queries are the last Nq positions: their rows of the full
    causal attention over all Nk positions (top-left, pinned above) are the
    key-cache attention with the bottom-right offset."""
    d, scale = 6, 0.37
    q_full, k, v = _rand(nk, d), _rand(nk, d), _rand(nk, d)
    O_full, L_full, _ = oracle.attention_head(q_full, k, v, True, scale)
    O, L = oracle.attention_kv_head(q_full[nk - nq:], k, v, True, scale)
    assert np.allclose(O, O_full[nk - nq:], atol=1e-12, rtol=0)
    assert np.allclose(L, L_full[nk - nq:], atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_kv_head_brute_force(causal):
    nq, nk, d, scale = 3, 7, 4, 0.5
    q, k, v = _rand(nq, d), _rand(nk, d), _rand(nk, d)
    O, L = oracle.attention_kv_head(q, k, v, causal, scale)
    for i in range(nq):
        keys = [j for j in range(nk) if not causal or j <= nk - nq + i]
        s = [scale * sum(q[i, c] * k[j, c] for c in range(d)) for j in keys]
        m = max(s)
        tot = sum(math.exp(x - m) for x in s)
        assert abs(L[i] - (m + math.log(tot))) < 1e-12
        for c in range(d):
            o = sum(math.exp(x - m) / tot * v[j, c] for x, j in zip(s, keys))
            assert abs(O[i, c] - o) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_kv_split_merges_to_the_whole_and_matches_split_at_equal_lengths(causal):
    B, Hq, Hkv, nq, nk, d, scale = 1, 4, 2, 3, 300, 5, 0.3
    q, k, v = _rand(B, Hq, nq, d), _rand(B, Hkv, nk, d), _rand(B, Hkv, nk, d)
    Op, Lp = oracle.attention_kv(q, k, v, causal, scale, n_split=4)
    O1, L1 = oracle.attention_kv(q, k, v, causal, scale, n_split=1)
    O, L = oracle.merge_partials(Op, Lp)
    assert np.allclose(O, O1[0], atol=1e-12) and np.allclose(L, L1[0], atol=1e-12)
    # grouped heads = attention with each key/value head repeated per group
    rep = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
    O2, L2 = oracle.attention_kv(q, *rep, causal, scale, n_split=4)
    assert np.allclose(O2, Op, atol=1e-12) and np.array_equal(np.isneginf(L2), np.isneginf(Lp))
    # Nq = Nk: the key-cache attention is attention_split
    qn = _rand(B, Hkv, nk, d)
    Os, Ls = oracle.attention_split(qn, k, v, causal, scale, 3)
    Ok, Lk = oracle.attention_kv(qn, k, v, causal, scale, n_split=3)
    assert np.allclose(Os, Ok, atol=1e-12)
    assert np.array_equal(np.isneginf(Ls), np.isneginf(Lk))
    fin = ~np.isneginf(Ls)
    assert np.allclose(Ls[fin], Lk[fin], atol=1e-12)
