"""The C-ABI library builds here (nvcc cross-compiles sm_103a without a GPU),
loads, and exports every entry point include/attn.h declares.  No compute
call is made, so this runs on CPU-only machines."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_75_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path():
    names = _declared()
    for need in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_quantize_fp8",
                 "attn_fwd_fp8", "attn_poll_device_status", "attn_status_string"):
        assert need in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_workspace_size_without_gpu(lib):
    lib.attn_status_string.restype = ctypes.c_char_p
    assert lib.attn_status_string(0) == b"ATTN_OK"
    assert lib.attn_status_string(4) == b"ATTN_ERR_TIMEOUT"
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    B, H, N, d = 2, 16, 8192, 128
    want = B * H * N * 4 + 256  # the fp32 delta vector D (a 256-byte multiple here), counters
    assert lib.attn_bwd_workspace_bytes(B, H, N, d) == want
    assert lib.attn_bwd_workspace_bytes(0, 1, 1, 128) == 0
    assert lib.attn_bwd_workspace_bytes(1, 1, 1, 80) == 0
    assert lib.attn_bwd_workspace_bytes(1, 1, 3, 128) == 512  # D rounded up, counters


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import exact_attention_75_gb300 as attn
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        attn.lib()


def test_argument_checks_return_before_any_launch(lib):
    """Shapes the library does not take are refused on the host, before the
    device is touched, so these calls run on a machine without a GPU (the
    pointers are never dereferenced).  Status 1 = ATTN_ERR_INVALID_ARG,
    2 = ATTN_ERR_UNSUPPORTED."""
    p = ctypes.c_void_p(0x10000)       # 16-byte aligned, never read
    bad = ctypes.c_void_p(0x10008)     # not 16-byte aligned
    s = ctypes.c_void_p(0)
    f = lib.attn_fwd_kv
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_void_p]
    #   q  k  v  o  lse n_split B Hq Hkv Nq  Nk   d  causal scale bf16 stream
    assert f(p, p, p, p, p, 1, 1, 1, 1, 200, 256, 256, 1, 0.1, 1, s) == 2  # 200 rows at d=256
    assert f(p, p, p, p, p, 1, 1, 8, 1, 17, 300, 192, 1, 0.1, 1, s) == 2   # 136 rows at d=192
    assert f(p, p, p, p, p, 1, 1, 1, 1, 4, 300, 80, 1, 0.1, 1, s) == 2     # d = 80
    assert f(p, p, p, p, p, 1, 1, 1, 1, 300, 200, 128, 1, 0.1, 1, s) == 1  # Nq > Nk
    assert f(p, p, p, p, p, 0, 1, 1, 1, 1, 200, 128, 1, 0.1, 1, s) == 1    # n_split = 0
    assert f(p, p, p, p, p, 257, 1, 1, 1, 1, 200, 128, 1, 0.1, 1, s) == 1  # n_split > 256
    assert f(p, p, p, p, p, 1, 1, 3, 2, 1, 200, 128, 1, 0.1, 1, s) == 1    # Hkv does not divide Hq
    assert f(p, bad, p, p, p, 1, 1, 1, 1, 1, 200, 128, 1, 0.1, 1, s) == 1  # misaligned k
    m = lib.attn_merge
    m.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int] * 5 + [ctypes.c_void_p]
    assert m(p, p, 4, p, p, 1, 1, 1, 80, 1, s) == 2    # d = 80
    assert m(p, p, 0, p, p, 1, 1, 1, 128, 1, s) == 1   # n_split = 0
    assert m(p, p, 4, p, p, 0, 1, 1, 128, 1, s) == 1   # B = 0
