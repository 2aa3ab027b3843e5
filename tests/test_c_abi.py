"""The C ABI from a plain C11 program (no Python, no torch in the caller)."""
import os
import shutil
import subprocess

import pytest

from moe_finalize_rmsnorm_gb300.build import LIB, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_closed_form.c")
CUDA = "/usr/local/cuda"


def _compile(out, syntax_only=False):
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", f"-I{ROOT}/include",
           f"-I{CUDA}/include", SRC]
    if syntax_only:
        cmd.append("-fsyntax-only")
    else:
        cmd += ["-o", out, f"-L{os.path.dirname(LIB)}", "-lmoe_finalize",
                f"-Wl,-rpath,{os.path.dirname(LIB)}", f"-L{CUDA}/lib64", "-lcudart",
                f"-Wl,-rpath,{CUDA}/lib64"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_header_is_plain_c11():
    _compile(None, syntax_only=True)


@pytest.mark.gpu
def test_c_program_closed_forms(tmp_path):
    build()
    exe = str(tmp_path / "abi_closed_form")
    _compile(exe)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "c abi: ok" in p.stdout
