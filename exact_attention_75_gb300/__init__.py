"""GB300-native exact attention (sm_103a): Python binding of ``libattn``.

Every function here only marshals arguments: it checks tensors, takes their
device pointers and the current CUDA stream, and calls the C ABI declared in
``include/attn.h``.  All computation runs in the library's CUDA kernels.  If
the library has not been built, or no sm_103a GPU is present, calls raise —
there is no fallback path.

Build the library first::

    python -m exact_attention_75_gb300.build
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

__all__ = ["AttnError", "lib", "lib_path", "fwd", "fwd_split", "fwd_kv", "merge", "bwd", "fwd_varlen",
           "bwd_varlen", "bwd_workspace_bytes", "quantize_fp8", "fwd_fp8", "poll_status", "set_wait_limit_us",
           "selftest_wait_timeout", "num_sms", "STATUS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_CUDA", 4: "ATTN_ERR_TIMEOUT"}
_F16, _BF16 = 0, 1
_lib = None


class AttnError(RuntimeError):
    def __init__(self, what: str, status: int, detail: int = 0):
        super().__init__(f"{what} failed: {STATUS.get(status, status)} (detail 0x{detail:x})")
        self.status = status
        self.detail = detail


def lib_path() -> str:
    return os.path.join(_HERE, "_build", "libattn.so")


def lib() -> ctypes.CDLL:
    """Load libattn.so (built in-tree) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m exact_attention_75_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    u32p = ctypes.POINTER(ctypes.c_uint32)
    sigs = {
        "attn_fwd": ([vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp], i),
        "attn_fwd_split": ([vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp], i),
        "attn_fwd_gqa": ([vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp], i),
        "attn_fwd_kv": ([vp] * 5 + [i] * 8 + [f, i, vp], i),
        "attn_bwd_gqa": ([vp] * 10 + [sz, i, i, i, i, i, i, f, i, vp], i),
        "attn_merge": ([vp, vp, i, vp, vp, i, i, i, i, i, vp], i),
        "attn_fwd_varlen": ([vp] * 6 + [i, i, i, i, i, i, i, f, i, vp], i),
        "attn_bwd_varlen": ([vp] * 10 + [sz, vp, i, i, i, i, i, i, i, f, i, vp], i),
        "attn_bwd_workspace_bytes": ([i, i, i, i], sz),
        "attn_bwd": ([vp] * 10 + [sz, i, i, i, i, i, f, i, vp], i),
        "attn_quantize_fp8": ([vp, vp, vp, i, i, i, i, i, vp, i, vp], i),
        "attn_fwd_fp8": ([vp] * 8 + [i, i, i, i, i, f, vp], i),
        "attn_poll_device_status": ([vp, u32p], i),
        "attn_set_wait_limit_us": ([ctypes.c_uint64], i),
        "attn_selftest_wait_timeout": ([ctypes.c_uint64, vp, u32p], i),
        "attn_status_string": ([i], ctypes.c_char_p),
        "attn_num_sms": ([], i),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(status: int, what: str) -> None:
    if status != 0:
        raise AttnError(what, status)


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return _F16
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"q/k/v must be float16 or bfloat16, got {t.dtype}")


def _check_qkv(*ts: torch.Tensor) -> Tuple[int, int, int, int]:
    q = ts[0]
    if q.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    for t in ts:
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("q, k, v (and o, dO) must share shape and dtype")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")
    B, H, N, d = q.shape
    return B, H, N, d


def _check_kv_heads(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> int:
    """Key/value heads of k, v for query tensor q (GQA when fewer than q's)."""
    if k.dim() != 4 or k.shape != v.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must share shape and q's dtype")
    if k.shape[0] != q.shape[0] or k.shape[2:] != q.shape[2:]:
        raise ValueError("k, v must be [B, Hkv, N, d] with q's B, N, d")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("the number of key/value heads must divide the query heads")
    for t in (k, v):
        if not t.is_cuda or t.device != q.device or not t.is_contiguous():
            raise ValueError("k, v must be contiguous tensors on q's device")
    return int(k.shape[1])


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE = attention(q, k, v).  q: [B,H,N,d], k, v: [B,Hkv,N,d] (Hkv
    divides H; fewer heads = grouped query heads) fp16/bf16, d in {64,96,128,192,256}."""
    if k.dim() == 4 and q.dim() == 4 and k.shape[1] != q.shape[1]:
        return _fwd_gqa(q, k, v, causal, scale, out, lse)
    B, H, N, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv(q, out)
    with torch.cuda.device(q.device):
        st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                            int(bool(causal)), float(scale), _dtype_code(q), _stream(q))
    _check(st, "attn_fwd")
    return out, lse


def fwd_split(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_split: int,
              causal: bool = False, scale: Optional[float] = None,
              out: Optional[torch.Tensor] = None,
              lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Partial results of attention over n_split runs of whole 128-key blocks:
    O_parts [n_split,B,H,N,d] (q's dtype), LSE_parts [n_split,B,H,N] fp32
    (-inf where a row sees no key of the split)."""
    B, H, N, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((n_split, B, H, N, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((n_split, B, H, N), dtype=torch.float32, device=q.device)
    if tuple(out.shape) != (n_split, B, H, N, d) or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [n_split, B, H, N, d] tensor of q's dtype")
    if tuple(lse.shape) != (n_split, B, H, N) or lse.dtype != torch.float32:
        raise ValueError("lse must be a float32 [n_split, B, H, N] tensor")
    with torch.cuda.device(q.device):
        st = lib().attn_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(n_split),
                                  B, H, N, d, int(bool(causal)), float(scale), _dtype_code(q),
                                  _stream(q))
    _check(st, "attn_fwd_split")
    return out, lse


def fwd_kv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_split: int = 1,
           causal: bool = False, scale: Optional[float] = None,
           out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Nq queries (the last Nq positions) against an Nk-row key/value cache,
    split over the keys: q [B,Hq,Nq,d], k, v [B,Hkv,Nk,d] (Hkv divides Hq,
    Nq <= Nk).  Returns O_parts [n_split,B,Hq,Nq,d], LSE_parts
    [n_split,B,Hq,Nq] (combine with merge; n_split = 1 holds the result).
    causal: query i sees keys j <= i + Nk - Nq."""
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, Hq, Nq, d] and k, v [B, Hkv, Nk, d]")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = int(k.shape[1]), int(k.shape[2])
    if k.shape[0] != B or k.shape[3] != d or Hq % Hkv != 0 or Nq > Nk:
        raise ValueError("k, v must be [B, Hkv, Nk, d] with Hkv dividing Hq and Nk >= Nq")
    for t in (q, k, v):
        if not t.is_cuda or t.device != q.device or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous tensors of one dtype on one device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((n_split, B, Hq, Nq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((n_split, B, Hq, Nq), dtype=torch.float32, device=q.device)
    if tuple(out.shape) != (n_split, B, Hq, Nq, d) or out.dtype != q.dtype \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous [n_split, B, Hq, Nq, d] tensor of q's dtype")
    if tuple(lse.shape) != (n_split, B, Hq, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be a float32 [n_split, B, Hq, Nq] tensor")
    with torch.cuda.device(q.device):
        st = lib().attn_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(n_split),
                               B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
                               _dtype_code(q), _stream(q))
    _check(st, "attn_fwd_kv")
    return out, lse


def merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: Optional[torch.Tensor] = None,
          lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Combine partial results over disjoint key sets: LSE = log sum exp(LSE_s),
    O = sum_s exp(LSE_s - LSE) O_s.  o_parts [S,B,H,N,d], lse_parts [S,B,H,N]."""
    if o_parts.dim() != 5 or not o_parts.is_cuda or not o_parts.is_contiguous():
        raise ValueError("o_parts must be a contiguous CUDA [n_split, B, H, N, d] tensor")
    S, B, H, N, d = o_parts.shape
    if tuple(lse_parts.shape) != (S, B, H, N) or lse_parts.dtype != torch.float32 \
            or not lse_parts.is_contiguous():
        raise ValueError("lse_parts must be a contiguous float32 [n_split, B, H, N] tensor")
    if out is None:
        out = torch.empty((B, H, N, d), dtype=o_parts.dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):
        st = lib().attn_merge(_ptr(o_parts), _ptr(lse_parts), int(S), _ptr(out), _ptr(lse),
                              B, H, N, d, _dtype_code(o_parts), _stream(o_parts))
    _check(st, "attn_merge")
    return out, lse


def _fwd_gqa(q, k, v, causal, scale, out, lse):
    B, H, N, d = _check_qkv(q)
    Hkv = _check_kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv(q, out)
    with torch.cuda.device(q.device):
        st = lib().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                                int(bool(causal)), float(scale), _dtype_code(q), _stream(q))
    _check(st, "attn_fwd_gqa")
    return out, lse


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, H, N, d))


def bwd(q, k, v, o, do, lse, causal: bool = False, scale: Optional[float] = None,
        workspace: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None):
    """dQ, dK, dV of the loss with gradient ``do`` w.r.t. O (d in {64, 96, 128, 192, 256}).  k, v
    (and dk, dv) may have fewer heads than q (grouped query heads)."""
    B, H, N, d = _check_qkv(q, o, do)
    Hkv = _check_kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws = bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be contiguous fp32 [B, H, N]")
    if dk.shape != k.shape or dv.shape != v.shape:
        raise ValueError("dk, dv must have the shape of k, v")
    with torch.cuda.device(q.device):
        if Hkv == H:
            st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, H, N,
                                d, int(bool(causal)), float(scale), _dtype_code(q), _stream(q))
        else:
            st = lib().attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                    workspace.numel(), B, H, Hkv, N, d, int(bool(causal)),
                                    float(scale), _dtype_code(q), _stream(q))
    _check(st, "attn_bwd" if Hkv == H else "attn_bwd_gqa")
    return dq, dk, dv


def quantize_fp8(x: torch.Tensor, signs: Optional[torch.Tensor] = None,
                 transposed: bool = False, block_rows: int = 64):
    """E4M3 codes (uint8) and per-64-row fp32 scales of a bf16 [B,H,N,d] tensor.

    ``signs``: optional int8 CUDA tensor of d values +-1 (randomized Hadamard).
    ``transposed``: write the codes as [B,H,d,N] (the layout attn_fwd_fp8 wants
    for V).
    """
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.dim() != 4:
        raise ValueError("x must be a contiguous bf16 CUDA tensor [B,H,N,d]")
    B, H, N, d = x.shape
    codes = torch.empty((B, H, d, N) if transposed else (B, H, N, d), dtype=torch.uint8,
                        device=x.device)
    scales = torch.empty((B, H, (N + block_rows - 1) // block_rows), dtype=torch.float32,
                         device=x.device)
    if signs is not None:
        if signs.dtype != torch.int8 or not signs.is_cuda or signs.numel() != d:
            raise ValueError("signs must be an int8 CUDA tensor of d values")
    with torch.cuda.device(x.device):
        st = lib().attn_quantize_fp8(_ptr(x), _ptr(codes), _ptr(scales), B, H, N, d, block_rows,
                                     _ptr(signs), int(bool(transposed)), _stream(x))
    _check(st, "attn_quantize_fp8")
    return codes, scales


def fwd_fp8(q8, k8, v8t, q_scale, k_scale, v_scale, causal: bool = False,
            scale: Optional[float] = None, out=None, lse=None):
    """FP8 forward: E4M3 q8, k8 [B,H,N,d], v8t [B,H,d,N] + block scales -> bf16 O, fp32 LSE."""
    B, H, N, d = q8.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (q8, k8, v8t, q_scale, k_scale, v_scale):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    with torch.cuda.device(q8.device):
        st = lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(q_scale), _ptr(k_scale),
                                _ptr(v_scale), _ptr(out), _ptr(lse), B, H, N, d,
                                int(bool(causal)), float(scale), _stream(q8))
    _check(st, "attn_fwd_fp8")
    return out, lse


def poll_status(device=None) -> Tuple[int, int]:
    """Synchronise the current stream and read/clear the device status word."""
    detail = ctypes.c_uint32(0)
    s = torch.cuda.current_stream(device)
    st = lib().attn_poll_device_status(ctypes.c_void_p(s.cuda_stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def set_wait_limit_us(us: int) -> None:
    _check(lib().attn_set_wait_limit_us(int(us)), "attn_set_wait_limit_us")


def selftest_wait_timeout(limit_us: int = 20000, device=None) -> Tuple[int, int]:
    detail = ctypes.c_uint32(0)
    s = torch.cuda.current_stream(device)
    st = lib().attn_selftest_wait_timeout(int(limit_us), ctypes.c_void_p(s.cuda_stream),
                                          ctypes.byref(detail))
    return int(st), int(detail.value)


def _check_varlen(q, k, v, cu_seqlens, max_seqlen, *more) -> Tuple[int, int, int, int, int]:
    """Shapes of a packed variable-length batch: q (and more) [H, total, d],
    k, v [Hkv, total, d], cu_seqlens int32 [n_seq + 1] on q's device."""
    if q.dim() != 3:
        raise ValueError("packed tensors must be [H, total, d]")
    H, T, d = q.shape
    if k.dim() != 3 or k.shape != v.shape or k.shape[1:] != q.shape[1:]:
        raise ValueError("k, v must be [Hkv, total, d] with q's total and d")
    if H % k.shape[0] != 0:
        raise ValueError("the number of key/value heads must divide the query heads")
    for t in (q, k, v) + more:
        if not t.is_cuda or t.device != q.device or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q, k, v, o, dO must be contiguous CUDA tensors of one dtype")
    for t in more:
        if t.shape != q.shape:
            raise ValueError("o and dO must have q's shape")
    if (cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2
            or cu_seqlens.device != q.device or not cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 [n_seq + 1] tensor on q's device")
    if not 1 <= int(max_seqlen) <= T:
        raise ValueError("max_seqlen must lie in [1, total]")
    return H, int(k.shape[0]), T, d, cu_seqlens.numel() - 1


def fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
               max_seqlen: int, causal: bool = False, scale: Optional[float] = None,
               out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention over a packed batch of sequences of their own lengths.
    q [H, total, d], k, v [Hkv, total, d]; sequence b is rows
    cu_seqlens[b]..cu_seqlens[b+1] and attends only to itself.  Returns
    O [H, total, d] and LSE [H, total] fp32.  max_seqlen >= every length."""
    H, Hkv, T, d, n_seq = _check_varlen(q, k, v, cu_seqlens, max_seqlen)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    _check_varlen(q, k, v, cu_seqlens, max_seqlen, out)
    if tuple(lse.shape) != (H, T) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, total] tensor")
    with torch.cuda.device(q.device):
        st = lib().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                   _ptr(cu_seqlens), n_seq, int(max_seqlen), T, H, Hkv, d,
                                   int(bool(causal)), float(scale), _dtype_code(q), _stream(q))
    _check(st, "attn_fwd_varlen")
    return out, lse


def bwd_varlen(q, k, v, o, do, lse, cu_seqlens: torch.Tensor, max_seqlen: int,
               causal: bool = False, scale: Optional[float] = None,
               workspace: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None):
    """dQ, dK, dV of fwd_varlen (d in {64, 96, 128}); layouts as fwd_varlen."""
    H, Hkv, T, d, n_seq = _check_varlen(q, k, v, cu_seqlens, max_seqlen, o, do)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if tuple(lse.shape) != (H, T) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, total] tensor")
    ws = bwd_workspace_bytes(1, H, T, d)
    if workspace is None:
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape:
        raise ValueError("dq, dk, dv must have the shapes of q, k, v")
    with torch.cuda.device(q.device):
        st = lib().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                   workspace.numel(), _ptr(cu_seqlens), n_seq, int(max_seqlen),
                                   T, H, Hkv, d, int(bool(causal)), float(scale),
                                   _dtype_code(q), _stream(q))
    _check(st, "attn_bwd_varlen")
    return dq, dk, dv


def num_sms() -> int:
    return int(lib().attn_num_sms())
