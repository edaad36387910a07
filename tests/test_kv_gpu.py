"""A block of Nq queries against an Nk-row key/value cache (decoding), split
over the keys, through the C ABI (attn_fwd_kv) and the merge, against the
fp64 oracle (attention_kv).

Partials: |O_s - O_s,ref| <= 2e-2, |LSE_s - LSE_s,ref| <= 5e-3 where the
split sees a key, LSE_s = -inf exactly where it sees none; merged result
against the oracle's whole-cache attention at the same tolerances.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import to64

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL = 2e-2, 5e-3


def _check(attn, q, k, v, causal, n_split, scale):
    Op, Lp = attn.fwd_kv(q.cuda(), k.cuda(), v.cuda(), n_split, causal=causal, scale=scale)
    O, L = attn.merge(Op, Lp)
    assert attn.poll_status() == (0, 0)
    q64, k64, v64 = to64(q), to64(k), to64(v)
    O_ref_p, L_ref_p = oracle.attention_kv(q64, k64, v64, causal, scale, n_split)
    Lp64 = to64(Lp)
    assert np.array_equal(np.isneginf(Lp64), np.isneginf(L_ref_p))
    seen = ~np.isneginf(L_ref_p)
    assert np.max(np.abs(Lp64[seen] - L_ref_p[seen]), initial=0.0) <= LSE_TOL
    assert np.max(np.abs(to64(Op) - O_ref_p)) <= O_TOL
    O_ref, L_ref = oracle.attention_kv(q64, k64, v64, causal, scale, 1)
    assert np.max(np.abs(to64(O) - O_ref[0])) <= O_TOL
    assert np.max(np.abs(to64(L) - L_ref[0])) <= LSE_TOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dtype,n_split", [
    (1, 4, 2, 1, 1000, 128, "bf16", 1),
    (1, 4, 2, 1, 1000, 128, "bf16", 4),
    (2, 2, 2, 7, 300, 64, "fp16", 2),
    (1, 6, 3, 128, 513, 96, "bf16", 3),
    (1, 2, 1, 129, 129, 128, "bf16", 1),
    (1, 2, 2, 200, 777, 128, "fp16", 5),
    (1, 1, 1, 1, 1, 64, "bf16", 1),
    (1, 2, 1, 3, 257, 96, "fp16", 8),
    (2, 8, 2, 5, 300, 128, "bf16", 3),     # 4 heads x 5 queries share a tile
    (1, 16, 1, 8, 1000, 64, "fp16", 2),    # 16 x 8 = 128 rows: a full shared tile
    (1, 9, 3, 40, 700, 96, "bf16", 1),     # 3 x 40 = 120 rows
    (1, 8, 2, 20, 20, 128, "bf16", 1),     # Nq = Nk, shared tile, causal top-left
    # at most 16 rows per key/value head: the warp-level decoding kernel
    (2, 16, 1, 1, 1000, 128, "bf16", 3),   # 16 heads x 1 query = 16 rows
    (1, 8, 1, 2, 130, 64, "fp16", 2),      # 8 x 2 = 16 rows, the last key seen by one
    (1, 6, 2, 4, 333, 96, "fp16", 1),      # 3 x 4 = 12 rows: both halves of the M = 16
    (1, 5, 1, 3, 77, 128, "bf16", 7),      # 15 rows; 7 splits of one block, 6 empty
    (1, 2, 2, 5, 5, 64, "bf16", 1),        # Nk = Nq = 5, under one 16-key block
    (3, 4, 4, 1, 4099, 128, "fp16", 256),  # 33 blocks over 256 splits, most empty
    (1, 17, 1, 1, 300, 128, "bf16", 2),    # 17 rows: the tiled forward again
    # the wide head dims: only the decoding kernel's shapes
    (2, 8, 1, 1, 1000, 256, "bf16", 3),    # 8 rows, Q fragments from shared memory
    (1, 4, 2, 6, 555, 256, "fp16", 2),     # 12 rows, both halves of M
    (1, 16, 2, 2, 700, 192, "bf16", 5),    # 16 rows
    (2, 3, 3, 1, 130, 192, "fp16", 1),     # one row per key/value head
    # wide head dims, 17-128 rows: groups of 16 rows on the decoding kernel
    (1, 8, 1, 5, 900, 256, "bf16", 3),     # 40 rows: three groups, the last of 8
    (1, 2, 1, 64, 300, 192, "fp16", 2),    # 128 rows: eight groups
    (2, 4, 2, 9, 513, 256, "fp16", 1),     # 18 rows against a longer cache
    (1, 1, 1, 100, 100, 192, "bf16", 3),   # Nq = Nk: the key split of attn_fwd_split
])
def test_queries_against_a_cache(attn_lib, causal, B, Hq, Hkv, Nq, Nk, d, dtype, n_split):
    w = wl.Workload("kv", "fwd", B, Hq, Nk, d, dtype, causal, seed=Nq + Nk + d)
    inp = wl.make_inputs(w)
    # the queries are the cache's last Nq positions of the seeded q; the
    # key/value heads the first head of each group
    G = Hq // Hkv
    q = inp["q"][:, :, Nk - Nq:].contiguous()
    k, v = inp["k"][:, ::G].contiguous(), inp["v"][:, ::G].contiguous()
    _check(attn_lib, q, k, v, causal, n_split, w.scale)


def test_equal_lengths_match_the_split_forward_bitwise(attn_lib):
    w = wl.Workload("kv", "fwd", 1, 2, 700, 128, "bf16", True, seed=5)
    inp = wl.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    a = attn_lib.fwd_kv(q, k, v, 3, causal=True)
    b = attn_lib.fwd_split(q, k, v, 3, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("kv_heads", [16, wl.DECODE_GQA_KV_HEADS])
def test_decode_workload_sampled_heads(attn_lib, kv_heads):
    """The measured decode batches (one query per sequence against an
    8192-row cache, 16 sequences x 16 query heads with 16 or 2 key/value
    heads, d = 128, bf16, 4 splits + merge; with 2 the 8 query heads of a
    group share one query tile) in the launch configuration the bench times;
    eight (sequence, head) pairs, the first and the last among them, against
    the oracle."""
    w = wl.DECODE_BF16_D128
    inp = wl.make_decode_inputs(w, kv_heads=kv_heads)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    Op, Lp = attn_lib.fwd_kv(q, k, v, wl.DECODE_SPLITS, causal=w.causal, scale=w.scale)
    O, L = attn_lib.merge(Op, Lp)
    assert attn_lib.poll_status() == (0, 0)
    G = w.H // kv_heads
    for b, h in [(0, 0), (0, 15), (3, 7), (7, 1), (9, 12), (12, 4), (15, 8), (15, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        q64 = to64(inp["q"][sl])
        k64, v64 = (to64(inp[n][b:b + 1, h // G:h // G + 1]) for n in ("k", "v"))
        O_ref_p, L_ref_p = oracle.attention_kv(q64, k64, v64, w.causal, w.scale,
                                               wl.DECODE_SPLITS)
        assert np.max(np.abs(to64(Op[:, b, h]) - O_ref_p[:, 0, 0])) <= O_TOL
        assert np.max(np.abs(to64(Lp[:, b, h]) - L_ref_p[:, 0, 0])) <= LSE_TOL
        O_ref, L_ref = oracle.attention_kv(q64, k64, v64, w.causal, w.scale, 1)
        assert np.max(np.abs(to64(O[b, h]) - O_ref[0, 0, 0])) <= O_TOL
        assert np.max(np.abs(to64(L[b, h]) - L_ref[0, 0, 0])) <= LSE_TOL


@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (96, "fp16"), (128, "bf16"), (192, "fp16"),
                                     (256, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,N", [(3, 2), (1, 9), (2, 16)])
def test_short_sequences_through_the_plain_forward(attn_lib, d, dtype, causal, H, N):
    """attn_fwd on sequences of at most 16 rows (the decoding kernel: Nk =
    N, causal top-left), element by element against the oracle."""
    w = wl.Workload("short", "fwd", 2, H, N, d, dtype, causal, seed=N + d)
    inp = wl.make_inputs(w)
    o, lse = attn_lib.fwd(*(inp[n].cuda() for n in ("q", "k", "v")), causal=causal,
                          scale=w.scale)
    assert attn_lib.poll_status() == (0, 0)
    O_ref, L_ref = oracle.attention(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), causal,
                                    w.scale)
    assert np.max(np.abs(to64(o) - O_ref)) <= O_TOL
    assert np.max(np.abs(to64(lse) - L_ref)) <= LSE_TOL


@pytest.mark.parametrize("gain", [4.0, 0.01])
def test_decoding_with_large_and_small_logits(attn_lib, gain):
    """Queries scaled by `gain` (8 grouped heads, 2 queries each, against
    3000 keys in 2 splits): large logits make the running maximum rise block
    after block (the rescale of O in every warp), tiny ones give a nearly
    uniform softmax; results bitwise the same from run to run."""
    w = wl.Workload("kv", "fwd", 2, 16, 3000, 128, "bf16", True, seed=21)
    inp = wl.make_inputs(w)
    q = (inp["q"][:, :, -2:].float() * gain).to(torch.bfloat16).contiguous()
    k, v = inp["k"][:, ::8].contiguous(), inp["v"][:, ::8].contiguous()
    _check(attn_lib, q, k, v, True, 2, w.scale)
    a = attn_lib.fwd_kv(q.cuda(), k.cuda(), v.cuda(), 2, causal=True, scale=w.scale)
    b = attn_lib.fwd_kv(q.cuda(), k.cuda(), v.cuda(), 2, causal=True, scale=w.scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("d", [192, 256])
def test_decode_at_the_wide_head_dims(attn_lib, d):
    """One query per sequence, 8 sequences x 16 query heads on 2 key/value
    heads against a 4096-row bf16 cache at d = 192 / 256, 8 splits + merge
    (the decode batch's shape at the wide head dims): four (sequence, head)
    pairs, the first and the last among them, against the oracle."""
    w = wl.Workload("kvw", "fwd", 8, 16, 4096, d, "bf16", True, seed=d)
    inp = wl.make_decode_inputs(w, kv_heads=2)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    Op, Lp = attn_lib.fwd_kv(q, k, v, 8, causal=True, scale=w.scale)
    O, L = attn_lib.merge(Op, Lp)
    assert attn_lib.poll_status() == (0, 0)
    for b, h in [(0, 0), (2, 9), (5, 6), (7, 15)]:
        q64 = to64(inp["q"][b:b + 1, h:h + 1])
        k64, v64 = (to64(inp[n][b:b + 1, h // 8:h // 8 + 1]) for n in ("k", "v"))
        O_ref_p, L_ref_p = oracle.attention_kv(q64, k64, v64, True, w.scale, 8)
        assert np.max(np.abs(to64(Op[:, b, h]) - O_ref_p[:, 0, 0])) <= O_TOL
        assert np.max(np.abs(to64(Lp[:, b, h]) - L_ref_p[:, 0, 0])) <= LSE_TOL
        O_ref, L_ref = oracle.attention_kv(q64, k64, v64, True, w.scale, 1)
        assert np.max(np.abs(to64(O[b, h]) - O_ref[0, 0, 0])) <= O_TOL
        assert np.max(np.abs(to64(L[b, h]) - L_ref[0, 0, 0])) <= LSE_TOL


@pytest.mark.parametrize("kv_heads", [16, 2])
def test_merge_right_after_the_decoding_kernel(attn_lib, kv_heads):
    """The merge is launched as a programmatic dependent of the decoding
    kernel (its launch overlaps the decoding kernel's tail): back to back on
    the stream it gives the same bits as after a full synchronize."""
    w = wl.DECODE_BF16_D128
    inp = wl.make_decode_inputs(w, kv_heads=kv_heads)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    Op, Lp = attn_lib.fwd_kv(q, k, v, wl.DECODE_SPLITS, causal=True, scale=w.scale)
    O, L = attn_lib.merge(Op, Lp)
    for _ in range(3):
        O.zero_()
        Op.zero_()
        attn_lib.fwd_kv(q, k, v, wl.DECODE_SPLITS, causal=True, scale=w.scale, out=Op, lse=Lp)
        attn_lib.merge(Op, Lp, out=O, lse=L)
    torch.cuda.synchronize()
    O1, L1 = O.clone(), L.clone()
    O.zero_()
    attn_lib.fwd_kv(q, k, v, wl.DECODE_SPLITS, causal=True, scale=w.scale, out=Op, lse=Lp)
    torch.cuda.synchronize()
    attn_lib.merge(Op, Lp, out=O, lse=L)
    torch.cuda.synchronize()
    assert attn_lib.poll_status() == (0, 0)
    assert torch.equal(O1, O) and torch.equal(L1, L)


def test_more_queries_than_keys_is_rejected(attn_lib):
    L = attn_lib.lib()
    x = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 256), dtype=torch.float32, device="cuda")
    p, pl = ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(lse.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # Nq = 200 > Nk = 100: ATTN_ERR_INVALID_ARG before any launch
    assert L.attn_fwd_kv(p, p, p, p, pl, 1, 1, 1, 1, 200, 100, 64, 1, 0.125, 1, s) == 1
    assert attn_lib.poll_status() == (0, 0)
