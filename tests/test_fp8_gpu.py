"""FP8 path: E4M3 block quantization (bit-exact against the oracle's
emulation) and the FP8 forward pass.

RMSE(O) <= 3e-2 is checked against the exact fp64 oracle on N(0,1) inputs.
On inputs with 0.1% x20 outliers the prescribed quantization by itself
(evaluated in fp64 by the oracle, no kernel involved) already exceeds that
bound, so there the kernel's own error is measured against the
quantization-aware oracle (fp64 attention on the oracle's dequantized,
rotated inputs) with the same 3e-2 bound, and its total error against the
exact oracle may exceed the recipe's own floor (the fp64 emulation of the
quantization, no kernel involved) by at most 25 % on the small cases and
10 % on the full-size workload (measured on a GB300: at most 1.17x and 1.03x)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import record, sample_heads, sample_rows, to64

pytestmark = pytest.mark.gpu
RMSE_TOL = 3e-2
FLOOR_RATIO_SMALL, FLOOR_RATIO_WORKLOAD = 1.25, 1.10


def _quant(attn, x, signs=None, transposed=False):
    codes, scales = attn.quantize_fp8(x.cuda(), None if signs is None else signs.cuda(),
                                      transposed=transposed)
    st, detail = attn.poll_status()
    assert st == 0, hex(detail)
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 64, 200, 1040])
def test_quantize_bit_exact_without_rotation(attn_lib, d, N):
    w = wl.Workload("q", "fwd_fp8", 2, 3, N, d, "bf16", False, outliers=True, seed=N)
    x = wl.make_inputs(w)["q"]
    ref = oracle.quantize_blocks(to64(x), 64)
    codes, scales = _quant(attn_lib, x)
    assert np.array_equal(scales.view(np.uint32), ref["scales"].view(np.uint32))
    assert np.array_equal(codes, ref["codes"])
    if N % 16 == 0:
        codes_t, scales_t = _quant(attn_lib, x, transposed=True)
        assert np.array_equal(scales_t, scales)
        assert np.array_equal(codes_t, np.swapaxes(ref["codes"], 2, 3))


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_many_blocks(attn_lib, d):
    """2048 blocks of 64 rows, more than the GPU holds at once, with a ragged
    32-row block ending every head: codes and scales bit-exact in both
    layouts."""
    w = wl.Workload("qm", "fwd_fp8", 2, 16, 4064, d, "bf16", False, outliers=True, seed=7 + d)
    x = wl.make_inputs(w)["q"]
    ref = oracle.quantize_blocks(to64(x), 64)
    codes, scales = _quant(attn_lib, x)
    assert np.array_equal(scales.view(np.uint32), ref["scales"].view(np.uint32))
    assert np.array_equal(codes, ref["codes"])
    codes_t, scales_t = _quant(attn_lib, x, transposed=True)
    assert np.array_equal(scales_t, scales)
    assert np.array_equal(codes_t, np.swapaxes(ref["codes"], 2, 3))


def test_quantize_all_zero_block(attn_lib):
    x = torch.zeros((1, 1, 130, 128), dtype=torch.bfloat16)
    x[0, 0, 128:] = 1.0
    codes, scales = _quant(attn_lib, x)
    assert scales[0, 0, 0] == 1.0 and scales[0, 0, 1] == 1.0 and not codes[0, 0, :64].any()
    assert scales[0, 0, 2] == np.float32(1.0) / np.float32(448.0)


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_with_hadamard_rotation(attn_lib, d):
    """The kernel rotates in fp32 (fast Walsh-Hadamard), the oracle in fp64, so
    values near an E4M3 rounding boundary may land one code apart; everything
    else must match, and the dequantized values stay within the E4M3 bound."""
    w = wl.Workload("qh", "fwd_fp8", 1, 4, 512, d, "bf16", False, outliers=True, hadamard=True,
                    seed=d)
    inp = wl.make_inputs(w)
    ref = oracle.quantize_blocks(to64(inp["q"]), 64, signs=inp["signs"].numpy())
    codes, scales = _quant(attn_lib, inp["q"], inp["signs"])
    np.testing.assert_allclose(scales, ref["scales"], rtol=4e-6, atol=0)
    mismatch = np.mean(codes != ref["codes"])
    assert mismatch < 2e-3, mismatch
    exact = to64(inp["q"]) @ oracle.rotation_matrix(inp["signs"].numpy())
    deq = oracle.dequantize_blocks(codes, scales, 64)
    s_full = np.repeat(scales.astype(np.float64), 64, axis=2)[:, :, :w.N, None]
    bound = np.maximum(np.abs(exact) * 2.0 ** -4, s_full * 2.0 ** -9) * 1.01 + 1e-6
    assert np.all(np.abs(deq - exact) <= bound)


def _fp8_forward(attn, inp, w, per_tensor=False):
    """Quantize (per 64-row block + optional Hadamard, or one scale per tensor
    prepared by the oracle's emulation) and run the FP8 forward kernel."""
    dev = torch.device("cuda")
    if per_tensor:
        ups = []
        for n in ("q", "k", "v"):
            x = to64(inp[n])
            out = oracle.quantize_blocks(x.reshape(1, 1, -1, w.d), x.size // w.d)
            nb = (w.N + 63) // 64
            codes = out["codes"].reshape(x.shape)
            sc = np.full((w.B, w.H, nb), out["scales"].ravel()[0], np.float32)
            if n == "v":
                codes = np.ascontiguousarray(np.swapaxes(codes, 2, 3))
            ups.append((torch.from_numpy(codes).to(dev), torch.from_numpy(sc).to(dev)))
        (q8, sq), (k8, sk), (v8t, sv) = ups
    else:
        signs = inp["signs"].to(dev) if "signs" in inp else None
        q8, sq = attn.quantize_fp8(inp["q"].to(dev), signs)
        k8, sk = attn.quantize_fp8(inp["k"].to(dev), signs)
        v8t, sv = attn.quantize_fp8(inp["v"].to(dev), None, transposed=True)
    o, lse = attn.fwd_fp8(q8, k8, v8t, sq, sk, sv, causal=w.causal, scale=w.scale)
    st, detail = attn.poll_status()
    assert st == 0, hex(detail)
    return o, lse


def _quant_aware_inputs(inp, hadamard):
    """fp64 values the prescribed recipe leaves of q, k, v: the oracle's own
    per-64-row E4M3 quantization (after the rotation for q and k)."""
    signs = inp["signs"].numpy() if hadamard else None
    out = []
    for n, sg in (("q", signs), ("k", signs), ("v", None)):
        qb = oracle.quantize_blocks(to64(inp[n]), 64, sg)
        out.append(oracle.dequantize_blocks(qb["codes"], qb["scales"], 64))
    return out


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [16, 128, 400, 1024])
def test_fp8_forward_normal_inputs(attn_lib, hadamard, causal, N):
    """N(0,1) q, k, v: RMSE(O) <= 3e-2 against the exact oracle."""
    w = wl.Workload("f8", "fwd_fp8", 1, 3, N, 128, "bf16", causal, hadamard=hadamard,
                    seed=N + 1)
    inp = wl.make_inputs(w)
    o, lse = _fp8_forward(attn_lib, inp, w)
    O_ref, L_ref = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), causal,
                                    w.scale)
    O = to64(o)
    assert np.isfinite(O).all() and np.isfinite(to64(lse)).all()
    e = oracle.rmse(O, O_ref)
    assert e <= RMSE_TOL, e
    assert np.max(np.abs(to64(lse) - L_ref)) < 0.1


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 400, 1024])
def test_fp8_forward_outlier_inputs(attn_lib, hadamard, causal, N):
    """0.1% x20 outliers.  The prescribed quantization alone (fp64 emulation,
    no kernel involved) already costs about 0.04 RMSE here, so the kernel is
    held to (a) RMSE <= 3e-2 against the quantization-aware fp64 oracle (its
    own error) and (b) RMSE against the exact oracle at most 1.25x that
    emulated floor."""
    w = wl.Workload("f8o", "fwd_fp8", 1, 3, N, 128, "bf16", causal, outliers=True,
                    hadamard=hadamard, seed=N + 1)
    inp = wl.make_inputs(w)
    o, lse = _fp8_forward(attn_lib, inp, w)
    O = to64(o)
    assert np.isfinite(O).all() and np.isfinite(to64(lse)).all()
    O_ref, _ = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), causal, w.scale)
    O_qa, L_qa = oracle.attention(*_quant_aware_inputs(inp, hadamard), causal, w.scale)
    floor = oracle.rmse(O_qa, O_ref)
    record(f"fp8_outliers_n{N}_c{int(causal)}_h{int(hadamard)}",
           {"e_exact": oracle.rmse(O, O_ref), "e_floor": floor, "e_kern": oracle.rmse(O, O_qa)})
    assert oracle.rmse(O, O_qa) <= RMSE_TOL
    assert oracle.rmse(O, O_ref) <= FLOOR_RATIO_SMALL * floor, (oracle.rmse(O, O_ref), floor)
    assert np.max(np.abs(to64(lse) - L_qa)) < 0.05


def test_fp8_forward_workload(attn_lib):
    """[2,16,8192,128] causal, 0.1% x20 outliers, Hadamard on Q and K: on
    seeded sampled rows of four heads, RMSE against the quantization-aware
    oracle <= 3e-2 and against the exact oracle at most 1.1x the floor."""
    w = wl.FWD_FP8_D128
    inp = wl.make_inputs(w)
    o, _ = _fp8_forward(attn_lib, inp, w)
    O = o.cpu()
    assert torch.isfinite(O.float()).all()
    signs = inp["signs"].numpy()
    d_kern, d_exact, d_floor = [], [], []
    for (b, h) in sample_heads(w.B, w.H, 4, seed=5):
        rows = sample_rows(w.N, 64, seed=b * 7 + h)
        head = {n: inp[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
        head["signs"] = inp["signs"]
        qa, ka, va = _quant_aware_inputs(head, True)
        Or, _ = oracle.attention_rows(to64(inp["q"][b, h]), to64(inp["k"][b, h]),
                                      to64(inp["v"][b, h]), rows, True, w.scale)
        Oq, _ = oracle.attention_rows(qa[0, 0], ka[0, 0], va[0, 0], rows, True, w.scale)
        Og = to64(O[b, h])[rows]
        d_kern.append((Og - Oq) ** 2)
        d_exact.append((Og - Or) ** 2)
        d_floor.append((Oq - Or) ** 2)
    rm = lambda xs: float(np.sqrt(np.mean(np.concatenate(xs))))  # noqa: E731
    e_kern, e_exact, e_floor = rm(d_kern), rm(d_exact), rm(d_floor)
    print(f"FP8 workload RMSE: vs exact {e_exact:.4f}, recipe floor {e_floor:.4f}, "
          f"kernel own {e_kern:.4f}")
    record("fp8_workload_rmse", {"e_exact": e_exact, "e_floor": e_floor, "e_kern": e_kern,
                                 "ratio_exact_to_floor": e_exact / e_floor,
                                 "rows": "64 seeded rows of 4 heads, (0,0) and (1,15) included"})
    assert e_kern <= RMSE_TOL
    assert e_exact <= FLOOR_RATIO_WORKLOAD * e_floor, (e_exact, e_floor)
    _ = signs


def test_fp8_block_scaling_and_rotation_reduce_error(attn_lib):
    """Direction of the accuracy claim of "8.3 FlashAttention-3" section 5
    (2.6x there): per-block scales + Hadamard beat one per-tensor scale on
    inputs with outliers, measured through the FP8 kernel.  The ratio is
    printed, not graded."""
    w = wl.Workload("f8cmp", "fwd_fp8", 1, 4, 2048, 128, "bf16", True, outliers=True,
                    hadamard=True, seed=21)
    inp = wl.make_inputs(w)
    O_ref, _ = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), True, w.scale)
    o_blk, _ = _fp8_forward(attn_lib, inp, w)
    o_pt, _ = _fp8_forward(attn_lib, inp, w, per_tensor=True)
    e_blk, e_pt = oracle.rmse(to64(o_blk), O_ref), oracle.rmse(to64(o_pt), O_ref)
    print(f"FP8 RMSE per-tensor {e_pt:.3e}  per-block+Hadamard {e_blk:.3e}  "
          f"ratio {e_pt / e_blk:.2f}")
    record("fp8_scaling_ratio", {"rmse_per_tensor": e_pt, "rmse_per_block_hadamard": e_blk,
                                 "ratio": e_pt / e_blk, "shape": [1, 4, 2048, 128]})
    assert e_blk < e_pt
