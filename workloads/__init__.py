"""Seeded synthetic workloads for exact attention.

This module only draws numbers: shapes, seeds, distributions and the order of
the draws.  It holds none of the attention arithmetic, so both the fp64 oracle
(``oracle/``) and the CUDA path (``exact_attention_75_gb300``) can take their
inputs from here without sharing any code of the method itself.

Recipe (the same on every machine, because all draws come from a CPU
``torch.Generator``):

* ``torch.Generator().manual_seed(seed)``; fp32 standard normals drawn in the
  order q, k, v, then dO (backward workloads only), each with shape [B,H,N,d].
* optional multiplication of q, k, v by ``input_scale`` in fp32 (0.5 for the
  d=128 bf16 forward workload);
* optional outliers: after the normals, one uniform draw per element of q, k
  and v (in that order); entries whose draw is < ``outlier_prob`` (0.001) are
  multiplied by ``outlier_mult`` (20);
* optional Hadamard sign vector: after everything else, ``d`` draws of
  {0, 1} mapped to {+1, -1}; these are the random signs of the randomized
  Hadamard rotation, passed to both sides as an input;
* finally a cast to the workload dtype (fp16 / bf16) with round-to-nearest.

The workloads themselves are the five shapes the attention kernels are
measured on (fp16 and bf16 forward at d=64 and d=128, the bf16 backward, the
FP8 forward with outliers), plus the sequence-length sweeps that keep B*N at
16384 tokens.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

TOKENS_PER_SWEEP = 16384


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "fwd", "bwd" or "fwd_fp8"
    B: int
    H: int
    N: int
    d: int
    dtype: str           # "fp16" or "bf16" (dtype of q, k, v, o, do)
    causal: bool
    input_scale: float = 1.0
    outliers: bool = False
    hadamard: bool = False
    seed: int = 0

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d) used by every workload."""
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"fp16": torch.float16, "bf16": torch.bfloat16}[self.dtype]

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def fwd_flops(self) -> float:
        """4*B*H*N^2*d, halved for causal attention."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """2.5x the forward count."""
        return 2.5 * self.fwd_flops()


# The five measured workloads.
TINY_FWD_FP16 = Workload("fwd_fp16_causal_b1h2n256d64", "fwd", 1, 2, 256, 64, "fp16", True)
FWD_FP16_D64 = Workload("fwd_fp16_b4h16n4096d64", "fwd", 4, 16, 4096, 64, "fp16", True)
FWD_BF16_D128 = Workload("fwd_bf16_b2h16n8192d128", "fwd", 2, 16, 8192, 128, "bf16", True,
                         input_scale=0.5)
BWD_BF16_D128 = Workload("bwd_bf16_causal_b2h16n8192d128", "bwd", 2, 16, 8192, 128, "bf16", True)
FWD_FP8_D128 = Workload("fwd_fp8_causal_b2h16n8192d128", "fwd_fp8", 2, 16, 8192, 128, "bf16",
                        True, outliers=True, hadamard=True)

WORKLOADS = [TINY_FWD_FP16, FWD_FP16_D64, FWD_BF16_D128, BWD_BF16_D128, FWD_FP8_D128]

# Decoding against a key/value cache (split over the keys, then merged): one
# new query per sequence, 16 sequences x 16 heads, an 8192-row cache of the
# bf16 d=128 workload's head size.  N is the cache length.
DECODE_BF16_D128 = Workload("decode_bf16_b16h16nk8192d128", "fwd_kv", 16, 16, 8192, 128, "bf16",
                            True)
DECODE_NQ = 1
# Key splits of the decode batches: 8 (256 CTAs with grouped heads, 2048 for
# the multi-head batch) timed fastest of 1 ... 32 for both.
DECODE_SPLITS = 8
# The same batch with grouped heads: 16 query heads sharing 2 key/value heads
# (a group's 8 queries share one query tile).
DECODE_GQA_KV_HEADS = 2


def sweep_d64(causal: bool) -> List[Workload]:
    """fp16 d=64 forward at N in {512..8192}, B = 16384 / N, H = 16."""
    return [FWD_FP16_D64.with_(name=f"fwd_fp16_d64_n{n}", B=TOKENS_PER_SWEEP // n, N=n,
                               causal=causal)
            for n in (512, 1024, 2048, 4096, 8192)]


def sweep_d128(causal: bool) -> List[Workload]:
    """bf16 d=128 forward at N in {1024..16384} (powers of two), B = 16384 / N."""
    return [FWD_BF16_D128.with_(name=f"fwd_bf16_d128_n{n}", B=TOKENS_PER_SWEEP // n, N=n,
                                causal=causal)
            for n in (1024, 2048, 4096, 8192, 16384)]


def make_inputs(w: Workload, with_do: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Draw the seeded inputs of workload ``w`` on the CPU.

    Returns a dict with ``q``, ``k``, ``v`` (and ``do`` for backward workloads)
    as CPU tensors of the workload dtype, and ``signs`` (int8, length d, values
    +-1) when the workload uses the randomized Hadamard rotation.
    """
    if with_do is None:
        with_do = w.kind == "bwd"
    g = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    names = ["q", "k", "v"] + (["do"] if with_do else [])
    raw = {n: torch.randn(shape, generator=g, dtype=torch.float32) for n in names}
    if w.input_scale != 1.0:
        for n in ("q", "k", "v"):
            raw[n] = raw[n] * w.input_scale
    if w.outliers:
        for n in ("q", "k", "v"):
            u = torch.rand(shape, generator=g, dtype=torch.float32)
            raw[n] = torch.where(u < 0.001, raw[n] * 20.0, raw[n])
    out = {n: t.to(w.torch_dtype) for n, t in raw.items()}
    if w.hadamard:
        bits = torch.randint(0, 2, (w.d,), generator=g)
        out["signs"] = (1 - 2 * bits).to(torch.int8)
    return out


# Variable-length batch measured beside the dense step: 16 heads, d = 128,
# bf16, causal, the same 16384 tokens per head as the dense [2,16,8192,128]
# workload, cut into sequences whose lengths are drawn uniformly from
# [VARLEN_MIN, VARLEN_MAX] (seed 0; the last one is cut to fill the total).
VARLEN_TOTAL, VARLEN_MIN, VARLEN_MAX, VARLEN_HEADS, VARLEN_D = 16384, 256, 4096, 16, 128


def varlen_lengths(total: int = VARLEN_TOTAL, lo: int = VARLEN_MIN, hi: int = VARLEN_MAX,
                   seed: int = 0) -> List[int]:
    """Sequence lengths drawn uniformly from [lo, hi] until they sum to total."""
    g = torch.Generator().manual_seed(seed)
    out: List[int] = []
    while sum(out) < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(min(n, total - sum(out)))
    return out


def make_varlen_inputs(lengths: List[int], Hq: int, Hkv: int, d: int, dtype: str,
                       seed: int = 0, with_do: bool = True) -> Dict[str, torch.Tensor]:
    """Packed inputs of a variable-length batch on the CPU: q (and do)
    [Hq, T, d], k, v [Hkv, T, d] fp32 standard normals drawn in the order q,
    k, v, do and cast to ``dtype``; ``cu_seqlens`` int32 [n+1] (row offsets)."""
    g = torch.Generator().manual_seed(seed)
    T = int(sum(lengths))
    tdt = {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype]
    shapes = {"q": (Hq, T, d), "k": (Hkv, T, d), "v": (Hkv, T, d)}
    if with_do:
        shapes["do"] = (Hq, T, d)
    out = {n: torch.randn(sh, generator=g, dtype=torch.float32).to(tdt)
           for n, sh in shapes.items()}
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    return out


def make_decode_inputs(w: Workload, nq: int = DECODE_NQ,
                       kv_heads: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Inputs of a decode step on the CPU: q [B,H,nq,d], k, v [B,Hkv,N,d] (N the
    cache length, Hkv = kv_heads or H), fp32 standard normals drawn in the
    order q, k, v and cast to the workload's dtype."""
    hkv = w.H if kv_heads is None else kv_heads
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.H, nq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, hkv, w.N, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, hkv, w.N, w.d), generator=g, dtype=torch.float32)
    return {n: t.to(w.torch_dtype) for n, t in (("q", q), ("k", k), ("v", v))}


def head_range(rank: int, world: int, BH: int) -> range:
    """Contiguous share of the B*H independent heads given to ``rank``."""
    per = (BH + world - 1) // world
    lo = min(BH, rank * per)
    return range(lo, min(BH, lo + per))
