"""The boundary from plain C: include/attn.h compiles as strict C99 (CPU), and
a C program links against the built library and runs a small forward pass
through it (GPU; tests/c_abi/abi_example.c states what it checks)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_example.c")
CC = shutil.which("gcc") or shutil.which("cc")


@pytest.mark.skipif(CC is None, reason="no C compiler")
def test_header_and_example_compile_as_c99(tmp_path):
    r = subprocess.run([CC, "-std=c99", "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), SRC], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
@pytest.mark.skipif(CC is None, reason="no C compiler")
def test_c_program_runs_the_forward(attn_lib, tmp_path):
    libdir = os.path.dirname(attn_lib.lib_path())
    cuda_lib = "/usr/local/cuda/lib64"
    exe = str(tmp_path / "abi_example")
    r = subprocess.run([CC, "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
                        "-L", libdir, "-l:" + os.path.basename(attn_lib.lib_path()),
                        "-Wl,-rpath," + libdir, "-L", cuda_lib, "-Wl,-rpath," + cuda_lib,
                        "-lcudart", "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "OK", (run.stdout, run.stderr)
