"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything under ``oracle/``.  The CUDA library never calls it and shares no code
with it.

Sources (the three web pages this implementation follows):

* [FA2-review]  "FlashAttention-2: Faster Attention with Better Parallelism and
  Work Partitioning" (paper review page): the flowchart under "프레임워크 개요"
  (Q,K,V in HBM -> tiles -> QK^T + online softmax statistics -> P V ->
  one final rescale -> O and log-sum-exp), the "Methods" section (defer the
  1/rowsum scaling to the end, keep only the log-sum-exp for the backward
  pass), "핵심 구성요소" (skip blocks entirely above the causal diagonal; the
  backward pass recomputes with the stored log-sum-exp), the glossary
  ("Online softmax", "Log-sum-exp (LSE)"), and the table "기존 접근법의 한계"
  naming standard (PyTorch) attention, which materialises the N x N matrix.
* [FA3-8.3]  "8.3 FlashAttention-3": section 5.1 (block quantization, one
  scale factor per block), section 5.2 (incoherent processing: multiply Q and
  K by a random orthogonal matrix built from a Hadamard transform with +-1
  entries).
* [Triton07]  "Triton 07: Flash Attention v3": section "Method" (un-scaled
  accumulation, exp2), the FP8 block-scaling + Hadamard item under the
  "Hopper" future-work list.

What this file computes, and how each function is pinned to something other
than itself, is listed per function.  All floating point is fp64 unless a
function is explicitly about the fp32/E4M3 encodings.

Readings where the pages are silent:

* LSE is the natural log of the sum of exp of the *scaled* scores.
* Causal masking is top-left aligned: key j is visible to query i iff j <= i.
* The softmax scale is the caller's (1/sqrt(d) in every workload).
* The backward pass is for the loss L = sum(O * dO), i.e. dO is the incoming
  gradient of O.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "scores", "allowed_mask", "masked_softmax", "attention_head", "attention",
    "attention_rows", "online_softmax_attention_head", "attention_backward_head",
    "attention_backward_dq_rows",
    "attention_backward", "E4M3_MAX", "e4m3_decode", "e4m3_encode", "hadamard_matrix",
    "rotation_matrix", "quantize_blocks", "dequantize_blocks", "rmse",
    "split_key_ranges", "attention_partial_head", "attention_split", "merge_partials",
    "kv_head_of", "attention_gqa", "attention_backward_gqa", "sequence_ranges",
    "attention_varlen", "attention_backward_varlen", "attention_kv_head", "attention_kv",
]


# ---------------------------------------------------------------------------
# Forward: the plain definition ("standard attention" in [FA2-review])
# ---------------------------------------------------------------------------

def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T for one head.  q: [Nq, d], k: [Nk, d] -> [Nq, Nk]."""
    return scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)


def allowed_mask(nq: int, nk: int, causal: bool) -> np.ndarray:
    """Boolean [nq, nk]; causal keeps key j for query i iff j <= i (top-left)."""
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    return np.arange(nk)[None, :] <= np.arange(nq)[:, None]


def masked_softmax(S: np.ndarray, allowed: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Row softmax over the allowed entries.

    Returns (P, LSE) with LSE_i = log(sum_{j allowed} exp(S_ij)) (natural log,
    glossary entry "Log-sum-exp" of [FA2-review]) and P_ij = exp(S_ij - LSE_i)
    on allowed entries, 0 elsewhere.  The row maximum is subtracted before
    exponentiating only to keep exp() in range; it cancels exactly.
    """
    Sm = np.where(allowed, S, -np.inf)
    mx = np.max(Sm, axis=1, keepdims=True)
    e = np.where(allowed, np.exp(Sm - mx), 0.0)
    rowsum = e.sum(axis=1, keepdims=True)
    lse = (mx + np.log(rowsum))[:, 0]
    P = e / rowsum
    return P, lse


def attention_head(q, k, v, causal: bool, scale: float):
    """O = softmax(scale Q K^T, masked) V for one head; returns (O, LSE, P)."""
    S = scores(q, k, scale)
    P, lse = masked_softmax(S, allowed_mask(S.shape[0], S.shape[1], causal))
    O = P @ np.asarray(v, np.float64)
    return O, lse, P


def attention(q, k, v, causal: bool, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Batched plain attention.  q,k,v: [B,H,N,d] -> O [B,H,N,d], LSE [B,H,N]."""
    q = np.asarray(q, np.float64)
    B, H, N, d = q.shape
    O = np.empty((B, H, N, v.shape[-1]), np.float64)
    L = np.empty((B, H, N), np.float64)
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h], _ = attention_head(q[b, h], k[b, h], v[b, h], causal, scale)
    return O, L


def attention_rows(q, k, v, rows: Sequence[int], causal: bool, scale: float):
    """Plain attention for selected query rows of one head (q,k,v: [N,d]).

    Row i needs only q_i and all of K, V, so large workloads can be checked on
    sampled rows.  Returns (O_rows [len(rows), d], LSE_rows [len(rows)]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    S = scale * (q[rows] @ k.T)
    allowed = np.ones_like(S, dtype=bool)
    if causal:
        allowed = np.arange(k.shape[0])[None, :] <= rows[:, None]
    P, lse = masked_softmax(S, allowed)
    return P @ v, lse


# ---------------------------------------------------------------------------
# Split over the keys, and the merge of the partial results
# ---------------------------------------------------------------------------
#
# [FA3-8.3] section 7.3 (ring attention) and the "Discussion Points" of
# [FA2-review] (a separate kernel that splits the keys for decoding) need
# attention over a subset of the keys and a way to combine such partial
# results; the "Insights" of [FA2-review] note that the log-sum-exp is all
# that has to be kept besides O.  The pages give no formula; the one below is
# the plain consequence of the softmax definition (a reading): over
# disjoint key sets K_s with partial results
# O_s = sum_{j in K_s} exp(S_ij - LSE_s) v_j and LSE_s = log sum_{j in K_s}
# exp(S_ij), the result over their union is
#   LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.

def split_key_ranges(n_keys: int, n_split: int, block: int = 128):
    """Key ranges [lo, hi) of the splits the library uses: the ceil(n/block)
    key blocks are cut into n_split contiguous runs, split s getting blocks
    floor(s nb / n_split) .. floor((s+1) nb / n_split) (a run may be empty)."""
    nb = -(-n_keys // block)
    out = []
    for s in range(n_split):
        lo, hi = (s * nb) // n_split, ((s + 1) * nb) // n_split
        out.append((min(lo * block, n_keys), min(hi * block, n_keys)))
    return out


def attention_partial_head(q, k, v, causal: bool, scale: float, key_lo: int, key_hi: int):
    """Attention of one head over the keys [key_lo, key_hi) only: the plain
    definition with every other key masked out (causal: key j visible to
    query i iff j <= i, with absolute positions).  A row that sees no key of
    the range gets LSE = -inf and O = 0.  Returns (O [N,d], LSE [N])."""
    q = np.asarray(q, np.float64)
    v = np.asarray(v, np.float64)
    n = q.shape[0]
    O = np.zeros((n, v.shape[1]), np.float64)
    lse = np.full(n, -np.inf)
    if key_hi <= key_lo:
        return O, lse
    S = scores(q, k[key_lo:key_hi], scale)
    allowed = np.ones(S.shape, dtype=bool)
    if causal:
        allowed = (key_lo + np.arange(key_hi - key_lo))[None, :] <= np.arange(n)[:, None]
    has = allowed.any(axis=1)
    if has.any():
        P, l = masked_softmax(S[has], allowed[has])
        O[has] = P @ v[key_lo:key_hi]
        lse[has] = l
    return O, lse


def attention_split(q, k, v, causal: bool, scale: float, n_split: int, block: int = 128):
    """Partial results of every split, batched.  q,k,v: [B,H,N,d] ->
    O_parts [n_split,B,H,N,d], LSE_parts [n_split,B,H,N]."""
    q = np.asarray(q, np.float64)
    B, H, N, d = q.shape
    ranges = split_key_ranges(N, n_split, block)
    O = np.zeros((n_split, B, H, N, np.shape(v)[-1]), np.float64)
    L = np.full((n_split, B, H, N), -np.inf)
    for s, (lo, hi) in enumerate(ranges):
        for b in range(B):
            for h in range(H):
                O[s, b, h], L[s, b, h] = attention_partial_head(q[b, h], k[b, h], v[b, h],
                                                                causal, scale, lo, hi)
    return O, L


def merge_partials(O_parts, LSE_parts):
    """Combine partial results over disjoint key sets (axis 0 = split):
    LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.  Rows where
    every LSE_s is -inf get LSE = -inf and O = 0."""
    O_parts = np.asarray(O_parts, np.float64)
    L = np.asarray(LSE_parts, np.float64)
    mx = np.max(L, axis=0)
    finite = np.isfinite(mx)
    safe = np.where(finite, mx, 0.0)
    w = np.where(np.isfinite(L), np.exp(L - safe[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    scale = np.where(finite, 1.0 / np.where(finite, tot, 1.0), 0.0)
    O = np.einsum("s...,s...d->...d", w * scale[None], O_parts)
    return O, lse


# ---------------------------------------------------------------------------
# Grouped query heads (GQA / MQA)
# ---------------------------------------------------------------------------
#
# The "Insights" of [FA2-review] link GQA ("Training Generalized Multi-Query
# Transformer Models") without spelling it out.  Reading: with Hq query
# heads and Hkv key/value heads, Hkv dividing Hq and
# G = Hq / Hkv, query head h attends with key/value head h // G (contiguous
# groups; Hkv = 1 is multi-query attention).  Each query head's attention is
# the plain definition; the gradient of a shared key/value head is the sum of
# the gradients it receives from the query heads of its group.

def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """Key/value head used by query head h."""
    return h // (Hq // Hkv)


def attention_gqa(q, k, v, causal: bool, scale: float):
    """q: [B,Hq,N,d], k, v: [B,Hkv,N,d] -> O [B,Hq,N,d], LSE [B,Hq,N]."""
    q = np.asarray(q, np.float64)
    B, Hq, N, d = q.shape
    Hkv = np.shape(k)[1]
    assert Hq % Hkv == 0
    O = np.empty((B, Hq, N, np.shape(v)[-1]), np.float64)
    L = np.empty((B, Hq, N), np.float64)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            O[b, h], L[b, h], _ = attention_head(q[b, h], k[b, g], v[b, g], causal, scale)
    return O, L


def attention_backward_gqa(q, k, v, do, causal: bool, scale: float):
    """dQ [B,Hq,N,d], dK / dV [B,Hkv,N,d]: per query head the plain backward,
    dK and dV summed over the query heads of each group."""
    q = np.asarray(q, np.float64)
    B, Hq, N, d = q.shape
    Hkv = np.shape(k)[1]
    dQ = np.empty(q.shape, np.float64)
    dK = np.zeros((B, Hkv) + np.shape(k)[2:], np.float64)
    dV = np.zeros((B, Hkv) + np.shape(v)[2:], np.float64)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            dq, dk, dv, _ = attention_backward_head(q[b, h], k[b, g], v[b, g], do[b, h], causal,
                                                    scale)
            dQ[b, h] = dq
            dK[b, g] += dk
            dV[b, g] += dv
    return dQ, dK, dV


# ---------------------------------------------------------------------------
# A block of queries against a longer key/value cache (decoding)
# ---------------------------------------------------------------------------
# [FA2-review] "Discussion Points" raises decoding with a KV cache, served by
# a kernel that splits the keys and combines the parts.  Reading: the Nq
# queries are the last Nq positions of a sequence whose Nk >= Nq keys and
# values are all cached, so with causal masking query i (position
# Nk - Nq + i) sees keys j <= Nk - Nq + i; without it, all Nk keys.  The
# split over the keys is the one of attention_split, over ceil(Nk/128) blocks.

def attention_kv_head(q, k, v, causal: bool, scale: float, key_lo: int = 0,
                      key_hi: Optional[int] = None):
    """One head: q [Nq,d], k, v [Nk,d], keys restricted to [key_lo, key_hi).
    Returns (O [Nq,d], LSE [Nq]); a row that sees no key of the range gets
    LSE = -inf and O = 0."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    nq, nk = q.shape[0], k.shape[0]
    key_hi = nk if key_hi is None else key_hi
    O = np.zeros((nq, v.shape[1]), np.float64)
    lse = np.full(nq, -np.inf)
    if key_hi <= key_lo:
        return O, lse
    S = scores(q, k[key_lo:key_hi], scale)
    allowed = np.ones(S.shape, dtype=bool)
    if causal:
        position = nk - nq + np.arange(nq)  # key position of each query
        allowed = (key_lo + np.arange(key_hi - key_lo))[None, :] <= position[:, None]
    has = allowed.any(axis=1)
    if has.any():
        P, l = masked_softmax(S[has], allowed[has])
        O[has] = P @ v[key_lo:key_hi]
        lse[has] = l
    return O, lse


def attention_kv(q, k, v, causal: bool, scale: float, n_split: int = 1, block: int = 128):
    """q [B,Hq,Nq,d], k, v [B,Hkv,Nk,d] (grouped heads as attention_gqa) ->
    O_parts [n_split,B,Hq,Nq,d], LSE_parts [n_split,B,Hq,Nq], split s over
    the keys of split_key_ranges(Nk, n_split, block)."""
    q = np.asarray(q, np.float64)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = np.shape(k)[1], np.shape(k)[2]
    O = np.zeros((n_split, B, Hq, Nq, np.shape(v)[-1]), np.float64)
    L = np.full((n_split, B, Hq, Nq), -np.inf)
    for s, (lo, hi) in enumerate(split_key_ranges(Nk, n_split, block)):
        for b in range(B):
            for h in range(Hq):
                g = kv_head_of(h, Hq, Hkv)
                O[s, b, h], L[s, b, h] = attention_kv_head(q[b, h], k[b, g], v[b, g], causal,
                                                           scale, lo, hi)
    return O, L


# ---------------------------------------------------------------------------
# Variable-length batches: independent sequences packed back to back
# ---------------------------------------------------------------------------
# [FA2-review] "Discussion Points" asks about many sequences, each with its
# own length (the decoding / KV-cache access pattern).  Plainest reading: each
# sequence is its own attention problem, the plain definition over its rows,
# with the causal diagonal counted from the sequence's first row.  Rows
# [cu[b], cu[b+1]) of every head belong to sequence b.

def sequence_ranges(cu_seqlens):
    """[(lo, hi)] row ranges of the sequences of a packed batch."""
    cu = [int(c) for c in np.asarray(cu_seqlens).ravel()]
    assert cu[0] == 0 and all(b >= a for a, b in zip(cu, cu[1:]))
    return list(zip(cu[:-1], cu[1:]))


def attention_varlen(q, k, v, cu_seqlens, causal: bool, scale: float):
    """q: [Hq,T,d], k, v: [Hkv,T,d] -> O [Hq,T,d], LSE [Hq,T] (rows outside
    every sequence stay NaN)."""
    q = np.asarray(q, np.float64)
    Hq, T, d = q.shape
    Hkv = np.shape(k)[0]
    O = np.full((Hq, T, np.shape(v)[-1]), np.nan)
    L = np.full((Hq, T), np.nan)
    for lo, hi in sequence_ranges(cu_seqlens):
        if hi == lo:
            continue
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            O[h, lo:hi], L[h, lo:hi], _ = attention_head(q[h, lo:hi], k[g, lo:hi], v[g, lo:hi],
                                                         causal, scale)
    return O, L


def attention_backward_varlen(q, k, v, do, cu_seqlens, causal: bool, scale: float):
    """dQ [Hq,T,d], dK / dV [Hkv,T,d] of attention_varlen: per sequence and
    query head the plain backward; dK, dV summed over each group."""
    q = np.asarray(q, np.float64)
    Hq, T, d = q.shape
    Hkv = np.shape(k)[0]
    dQ = np.full(q.shape, np.nan)
    dK = np.full((Hkv,) + np.shape(k)[1:], np.nan)
    dV = np.full((Hkv,) + np.shape(v)[1:], np.nan)
    for lo, hi in sequence_ranges(cu_seqlens):
        if hi == lo:
            continue
        dK[:, lo:hi] = 0.0
        dV[:, lo:hi] = 0.0
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            dq, dk, dv, _ = attention_backward_head(q[h, lo:hi], k[g, lo:hi], v[g, lo:hi],
                                                    do[h, lo:hi], causal, scale)
            dQ[h, lo:hi] = dq
            dK[g, lo:hi] += dk
            dV[g, lo:hi] += dv
    return dQ, dK, dV


# ---------------------------------------------------------------------------
# Forward: the tiled online-softmax recurrence, in the pages' order
# ---------------------------------------------------------------------------

def online_softmax_attention_head(q, k, v, causal: bool, scale: float, block: int):
    """Tiled attention with online softmax, fp64, following [FA2-review].

    Steps, for each block of ``block`` query rows (flowchart "프레임워크
    개요" and section "Methods"):
      1. load the Q tile;
      2. for each K/V tile (tiles entirely above the causal diagonal are
         skipped, "핵심 구성요소" causal-masking item):
           S = scale Q_tile K_tile^T, masked;
           m_new = max(m, rowmax(S));
           P~ = exp(S - m_new);
           l = exp(m - m_new) l + rowsum(P~);
           O~ = exp(m - m_new) O~ + P~ V_tile     (unnormalised);
           m = m_new;
      3. rescale once at the end: O = O~ / l;
      4. write O and LSE = m + log(l).
    Pinned by equality with ``attention_head`` (the plain definition) to
    1e-12 for several block sizes, in tests/test_oracle.py.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, dv = q.shape[0], v.shape[1]
    Nk = k.shape[0]
    O = np.zeros((N, dv))
    LSE = np.zeros(N)
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        qt = q[r0:r1]
        m = np.full(r1 - r0, -np.inf)
        l = np.zeros(r1 - r0)
        acc = np.zeros((r1 - r0, dv))
        for c0 in range(0, Nk, block):
            c1 = min(Nk, c0 + block)
            if causal and c0 > r1 - 1:
                break  # this and every later K/V tile lies above the diagonal
            S = scale * (qt @ k[c0:c1].T)
            if causal:
                ok = np.arange(c0, c1)[None, :] <= np.arange(r0, r1)[:, None]
                S = np.where(ok, S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))
            alpha = np.exp(m - m_new)           # exp(-inf) = 0 on the first tile
            Pt = np.exp(S - m_new[:, None])
            l = alpha * l + Pt.sum(axis=1)
            acc = alpha[:, None] * acc + Pt @ v[c0:c1]
            m = m_new
        O[r0:r1] = acc / l[:, None]
        LSE[r0:r1] = m + np.log(l)
    return O, LSE


# ---------------------------------------------------------------------------
# Backward: closed-form gradients of L = sum(O * dO)
# ---------------------------------------------------------------------------

def attention_backward_head(q, k, v, do, causal: bool, scale: float):
    """dQ, dK, dV for one head, recomputing P from the definition.

    [FA2-review] "핵심 구성요소" (backward item) recomputes P from the stored
    log-sum-exp; mathematically P is the same softmax as in the forward pass,
    so the oracle rebuilds it from the definition:
      dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij;
      dS = P o (dP - D);  dQ = scale dS K;  dK = scale dS^T Q.
    Pinned by central finite differences of L and by closed forms for Q = 0
    in tests/test_oracle.py.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    _, _, P = attention_head(q, k, v, causal, scale)
    dV = P.T @ do
    dP = do @ v.T
    D = np.sum(P * dP, axis=1, keepdims=True)
    dS = P * (dP - D)
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV, dS


def attention_backward_dq_rows(q, k, v, do, rows: Sequence[int], causal: bool, scale: float):
    """dQ of selected query rows of one head (q, k, v, do: [N, d]).

    Row i of dQ needs only row i of P: P_i = softmax(scale q_i K^T, masked),
    O_i = P_i V, D_i = dO_i . O_i, dP_i = dO_i V^T, dS_i = P_i o (dP_i - D_i),
    dQ_i = scale dS_i K (the formulas of attention_backward_head restricted
    to one row), so long sequences can be checked on sampled rows.
    Pinned against attention_backward_head in tests/test_oracle.py.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    S = scale * (q[rows] @ k.T)
    allowed = np.ones_like(S, dtype=bool)
    if causal:
        allowed = np.arange(k.shape[0])[None, :] <= rows[:, None]
    P, _ = masked_softmax(S, allowed)
    O = P @ v
    D = np.sum(do[rows] * O, axis=1, keepdims=True)
    dP = do[rows] @ v.T
    dS = P * (dP - D)
    return scale * (dS @ k)


def attention_backward(q, k, v, do, causal: bool, scale: float, heads=None):
    """Batched backward.  Returns dQ, dK, dV as [B,H,N,d] fp64.

    ``heads`` (optional iterable of (b, h)) restricts the work to those heads;
    the other entries are left as NaN.
    """
    q = np.asarray(q, np.float64)
    B, H, N, d = q.shape
    dQ = np.full(q.shape, np.nan)
    dK = np.full(q.shape, np.nan)
    dV = np.full(q.shape, np.nan)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        dQ[b, h], dK[b, h], dV[b, h], _ = attention_backward_head(
            q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
    return dQ, dK, dV


# ---------------------------------------------------------------------------
# FP8 E4M3 block quantization and the randomized Hadamard rotation
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0  # largest finite E4M3 value: 1.75 * 2^8


def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3 ("fn" variant: no infinities, 0x7F/0xFF are NaN) to fp64.

    Bit layout: sign (1) | exponent (4, bias 7) | mantissa (3).  Exponent 0
    is subnormal: value = m/8 * 2^-6.  Written from the format definition.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e4m3_encode(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to E4M3 (nearest, ties to even), saturating at +-448.

    Uses torch's float8_e4m3fn cast as the library rounding routine after a
    clamp to +-448 (the "satfinite" reading).  Pinned against a brute-force
    nearest-code search over all 256 codes in tests/test_oracle.py.
    """
    import torch
    x = np.clip(np.asarray(x32, np.float32), -E4M3_MAX, E4M3_MAX)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_d (d a power of two), entries +-1."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def rotation_matrix(signs) -> np.ndarray:
    """R = H_d diag(signs) / sqrt(d): orthogonal, so (Q R)(K R)^T = Q K^T.

    [FA3-8.3] section 5.2 multiplies Q and K by a random orthogonal matrix made
    from a Hadamard transform; the random part is the +-1 sign vector, drawn
    by the workload generator and passed in.
    """
    s = np.asarray(signs, np.float64)
    d = s.shape[0]
    return hadamard_matrix(d) * s[None, :] / math.sqrt(d)


def quantize_blocks(x, block_rows: int = 64, signs=None) -> Dict[str, np.ndarray]:
    """Per-block E4M3 quantization of one tensor [B,H,N,d] ([FA3-8.3] 5.1).

    For each (b, h) and each block of ``block_rows`` consecutive rows (the last
    block may be shorter):
      * optional rotation x <- x R (``signs`` given), computed in fp64 and
        rounded to fp32;
      * amax = max |x| over the block (fp32);
      * s = amax / 448 as one IEEE fp32 division (s = 1 when amax = 0);
      * code = E4M3(x / s), the division again in IEEE fp32.
    Returns dict(codes uint8 [B,H,N,d], scales fp32 [B,H,ceil(N/block_rows)],
    x32 = the fp32 values that were quantized).
    """
    x = np.asarray(x, np.float64)
    B, H, N, d = x.shape
    if signs is not None:
        x = x @ rotation_matrix(signs)
    x32 = x.astype(np.float32)
    nb = (N + block_rows - 1) // block_rows
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty((B, H, nb), np.float32)
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                blk = x32[b, h, i * block_rows:(i + 1) * block_rows]
                amax = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
                s = np.float32(amax) / np.float32(E4M3_MAX) if amax > 0 else np.float32(1.0)
                scales[b, h, i] = s
                codes[b, h, i * block_rows:(i + 1) * block_rows] = e4m3_encode(
                    (blk / np.float32(s)).astype(np.float32))
    return {"codes": codes, "scales": scales, "x32": x32}


def dequantize_blocks(codes, scales, block_rows: int = 64) -> np.ndarray:
    """Inverse of ``quantize_blocks`` up to rounding: code value * block scale."""
    vals = e4m3_decode(codes)
    s = np.repeat(np.asarray(scales, np.float64), block_rows, axis=2)[:, :, :vals.shape[2]]
    return vals * s[..., None]


def rmse(a, b) -> float:
    """Root-mean-square of (a - b) over all elements (absolute)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.sqrt(np.mean((a - b) ** 2)))
