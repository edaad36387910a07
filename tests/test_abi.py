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
