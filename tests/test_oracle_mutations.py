"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake of the kind a careful reader could still make
(a dropped term, a wrong sign, an off-by-one index, a transposed operand, a
wrong constant) in a copy of the oracle's source, loads the copy, and runs
checks written independently of it: scalar brute-force loops with math.exp,
central finite differences, the suffix identity of queries against a key
cache, a brute-force nearest-code search for E4M3, the Hadamard identity.
The unmodified oracle must pass every check and each planted mistake must
fail at least one.  Mistakes are planted only in this test's private copy.
"""
import math
import os

import numpy as np
import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "attention.py")

MUTATIONS = {
    "dropped scale": ("return scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)",
                      "return (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)"),
    "causal mask drops the diagonal": (
        "return np.arange(nk)[None, :] <= np.arange(nq)[:, None]",
        "return np.arange(nk)[None, :] < np.arange(nq)[:, None]"),
    "LSE without the row max": ("lse = (mx + np.log(rowsum))[:, 0]",
                                "lse = np.log(rowsum)[:, 0]"),
    "P V with P transposed": ("O = P @ np.asarray(v, np.float64)",
                              "O = P.T @ np.asarray(v, np.float64)"),
    "dS sign": ("    dS = P * (dP - D)\n    dQ = scale * (dS @ k)",
                "    dS = P * (dP + D)\n    dQ = scale * (dS @ k)"),
    "dK without the transpose": ("dK = scale * (dS.T @ q)", "dK = scale * (dS @ q)"),
    "dV without the transpose": ("dV = P.T @ do", "dV = P @ do"),
    "online softmax without the rescale of l": ("l = alpha * l + Pt.sum(axis=1)",
                                                "l = l + Pt.sum(axis=1)"),
    "key-cache offset off by one": ("position = nk - nq + np.arange(nq)",
                                    "position = nk - nq - 1 + np.arange(nq)"),
    "merge weight sign": ("w = np.where(np.isfinite(L), np.exp(L - safe[None]), 0.0)",
                          "w = np.where(np.isfinite(L), np.exp(safe[None] - L), 0.0)"),
    "split ranges overlap": ("lo, hi = (s * nb) // n_split, ((s + 1) * nb) // n_split",
                             "lo, hi = (s * nb) // n_split, ((s + 1) * nb) // n_split + 1"),
    "grouped heads interleaved": ("return h // (Hq // Hkv)", "return h % Hkv"),
    "E4M3 scale constant": (
        "s = np.float32(amax) / np.float32(E4M3_MAX) if amax > 0 else np.float32(1.0)",
        "s = np.float32(amax) / np.float32(240.0) if amax > 0 else np.float32(1.0)"),
    "Hadamard sign": ("H = np.block([[H, H], [H, -H]])", "H = np.block([[H, H], [-H, H]])"),
    "sequences end one row early": ("return list(zip(cu[:-1], cu[1:]))",
                                    "return list(zip(cu[:-1], [c - 1 for c in cu[1:]]))"),
    "sequence keys from the query head": (
        "attention_head(q[h, lo:hi], k[g, lo:hi], v[g, lo:hi],",
        "attention_head(q[h, lo:hi], k[h % np.shape(k)[0], lo:hi], v[g, lo:hi],"),
    "rotation signs on the wrong side": ("return hadamard_matrix(d) * s[None, :] / math.sqrt(d)",
                                         "return hadamard_matrix(d) * s[:, None] / math.sqrt(d)"),
    "rotation transposed": ("x = x @ rotation_matrix(signs)", "x = x @ rotation_matrix(signs).T"),
}


def _load(mutation=None):
    src = open(SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    ns = {"__name__": "oracle_copy"}
    exec(compile(src, "oracle_copy", "exec"), ns)
    return ns


# ------------------------------------------------------------- brute force ---

def _brute_rows(q, k, v, scale, visible):
    """O, LSE by scalar loops; visible(i, j) says whether key j is allowed."""
    nq, d = q.shape
    O = np.zeros((nq, v.shape[1]))
    L = np.zeros(nq)
    for i in range(nq):
        keys = [j for j in range(k.shape[0]) if visible(i, j)]
        s = [scale * sum(q[i, c] * k[j, c] for c in range(d)) for j in keys]
        m = max(s)
        tot = sum(math.exp(x - m) for x in s)
        L[i] = m + math.log(tot)
        for c in range(v.shape[1]):
            O[i, c] = sum(math.exp(x - m) / tot * v[j, c] for x, j in zip(s, keys))
    return O, L


def _rng():
    return np.random.default_rng(20)


def check_forward(m):
    r = _rng()
    q, k, v = r.standard_normal((6, 3)), r.standard_normal((6, 3)), r.standard_normal((6, 2))
    for causal in (False, True):
        O, L, _ = m["attention_head"](q, k, v, causal, 0.7)
        Ob, Lb = _brute_rows(q, k, v, 0.7, lambda i, j: not causal or j <= i)
        assert np.allclose(O, Ob, atol=1e-12) and np.allclose(L, Lb, atol=1e-12)
        for block in (1, 4):
            Oo, Lo = m["online_softmax_attention_head"](q, k, v, causal, 0.7, block)
            assert np.allclose(Oo, Ob, atol=1e-12) and np.allclose(Lo, Lb, atol=1e-12)


def check_backward(m):
    r = _rng()
    n, d, scale = 5, 3, 0.6
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, _ = m["attention_backward_head"](q, k, v, do, causal, scale)

        def loss(q_, k_, v_):
            O, _ = _brute_rows(q_, k_, v_, scale, lambda i, j: not causal or j <= i)
            return float(np.sum(O * do))
        h = 1e-6
        for g, idx in ((dq, 0), (dk, 1), (dv, 2)):
            for a in range(n):
                for c in range(d):
                    args_p = [q.copy(), k.copy(), v.copy()]
                    args_m = [q.copy(), k.copy(), v.copy()]
                    args_p[idx][a, c] += h
                    args_m[idx][a, c] -= h
                    fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
                    assert abs(fd - g[a, c]) < 1e-6 * max(1.0, abs(fd)), (idx, a, c)


def check_key_cache(m):
    r = _rng()
    nq, nk, d = 3, 8, 4
    q, k, v = r.standard_normal((nq, d)), r.standard_normal((nk, d)), r.standard_normal((nk, d))
    O, L = m["attention_kv_head"](q, k, v, True, 0.5)
    Ob, Lb = _brute_rows(q, k, v, 0.5, lambda i, j: j <= nk - nq + i)
    assert np.allclose(O, Ob, atol=1e-12) and np.allclose(L, Lb, atol=1e-12)


def check_split_and_merge(m):
    r = _rng()
    n, d = 300, 3
    q, k, v = (r.standard_normal((1, 1, n, d)) for _ in range(3))
    ranges = m["split_key_ranges"](n, 3, 128)
    # the ranges partition [0, n) in whole 128-key blocks
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    Op, Lp = m["attention_split"](q, k, v, False, 0.4, 3)
    O, L = m["merge_partials"](Op, Lp)
    rows = [0, 7, 299]
    Ob, Lb = _brute_rows(q[0, 0][rows], k[0, 0], v[0, 0], 0.4, lambda i, j: True)
    assert np.allclose(O[0, 0][rows], Ob, atol=1e-10)
    assert np.allclose(L[0, 0][rows], Lb, atol=1e-10)


def check_grouped_heads(m):
    r = _rng()
    Hq, Hkv, n, d = 4, 2, 4, 3
    q = r.standard_normal((1, Hq, n, d))
    k, v = r.standard_normal((1, Hkv, n, d)), r.standard_normal((1, Hkv, n, d))
    O, _ = m["attention_gqa"](q, k, v, False, 0.5)
    for h in range(Hq):
        g = h // (Hq // Hkv)  # contiguous groups
        Ob, _ = _brute_rows(q[0, h], k[0, g], v[0, g], 0.5, lambda i, j: True)
        assert np.allclose(O[0, h], Ob, atol=1e-12), h


def _e4m3_value(code):
    sign = -1.0 if code & 0x80 else 1.0
    e, f = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and f == 0x7:
        return math.nan
    if e == 0:
        return sign * f / 8.0 * 2.0 ** -6
    return sign * (1 + f / 8.0) * 2.0 ** (e - 7)


def check_quantize(m):
    r = _rng()
    x = (r.standard_normal((1, 1, 64, 4)) * 3).astype(np.float32)
    out = m["quantize_blocks"](x, 64)
    amax = np.float32(np.max(np.abs(x)))
    s = np.float32(amax / np.float32(448.0))
    assert out["scales"][0, 0, 0] == s
    finite = [c for c in range(256) if not math.isnan(_e4m3_value(c))]
    for val, code in zip((x[0, 0] / s).ravel(), out["codes"][0, 0].ravel()):
        best = min(abs(_e4m3_value(c) - float(val)) for c in finite)
        assert abs(_e4m3_value(int(code)) - float(val)) == best


def check_hadamard(m):
    for d in (2, 8):
        H = m["hadamard_matrix"](d)
        assert np.array_equal(H @ H.T, d * np.eye(d))
        assert np.all(H[0] == 1) and np.all(H[:, 0] == 1)  # Sylvester order


def check_varlen(m):
    r = _rng()
    lens = [3, 0, 5, 2]
    cu = np.cumsum([0] + lens)
    T, d, Hq, Hkv = int(cu[-1]), 3, 4, 2
    q = r.standard_normal((Hq, T, d))
    k, v = r.standard_normal((Hkv, T, d)), r.standard_normal((Hkv, T, d))
    O, L = m["attention_varlen"](q, k, v, cu, True, 0.5)
    for lo, hi in zip(cu[:-1], cu[1:]):
        if hi == lo:
            continue
        for h in range(Hq):
            g = h // (Hq // Hkv)
            Ob, Lb = _brute_rows(q[h, lo:hi], k[g, lo:hi], v[g, lo:hi], 0.5, lambda i, j: j <= i)
            assert np.allclose(O[h, lo:hi], Ob, atol=1e-12)
            assert np.allclose(L[h, lo:hi], Lb, atol=1e-12)


def check_rotation(m):
    """R = H_d diag(signs) / sqrt(d) built here from scalar loops; the
    quantizer rotates rows as x R."""
    d = 8
    signs = np.array([1, -1, -1, 1, 1, 1, -1, 1], np.float64)

    def h(i, j):  # Sylvester entry: (-1)^popcount(i & j)
        return -1.0 if bin(i & j).count("1") % 2 else 1.0
    R = np.array([[h(i, j) * signs[j] / math.sqrt(d) for j in range(d)] for i in range(d)])
    assert np.allclose(m["rotation_matrix"](signs), R, atol=1e-15)
    x = _rng().standard_normal((1, 1, 4, d))
    out = m["quantize_blocks"](x, 64, signs)
    assert np.array_equal(out["x32"], (x @ R).astype(np.float32))


CHECKS = [check_forward, check_backward, check_key_cache, check_split_and_merge,
          check_grouped_heads, check_varlen, check_quantize, check_hadamard, check_rotation]


def _failures(m):
    failed = []
    for c in CHECKS:
        try:
            c(m)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError):
            failed.append(c.__name__)
    return failed


def test_unmodified_oracle_passes_every_check():
    assert _failures(_load()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    failed = _failures(_load(MUTATIONS[name]))
    assert failed, f"no check caught: {name}"
