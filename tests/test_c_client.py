"""The C ABI used from plain C: the header compiles as C99 and as C++, and
on a GPU a C program linked against libgemm07.so computes exact products."""
import os
import shutil
import subprocess

import pytest

from dense_gemm_07_gb300 import _abi, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CLIENT = os.path.join(ROOT, "tests", "c_client", "gemm_client.c")
INCLUDE = os.path.join(ROOT, "include")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("no CUDA headers")
    return cc


def test_header_compiles_as_c99_and_cxx(tmp_path):
    cc = _cc()
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", INCLUDE,
                    "-I", os.path.join(CUDA, "include"), CLIENT], check=True)
    cxx = shutil.which("g++")
    if cxx:
        src = tmp_path / "h.cpp"
        src.write_text('#include "gemm07.h"\nint main() { return gemm_abi_version() > 0 ? 0 : 1; }\n')
        subprocess.run([cxx, "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-I", INCLUDE,
                        str(src)], check=True)


@pytest.mark.gpu
def test_c_program_gets_exact_products(tmp_path):
    cc = _cc()
    _abi.lib()  # builds the library if needed
    libdir = os.path.dirname(_build.LIB_PATH)
    exe = tmp_path / "gemm_client"
    subprocess.run([cc, "-std=c99", "-O2", "-I", INCLUDE, "-I", os.path.join(CUDA, "include"),
                    CLIENT, "-L", libdir, "-lgemm07", "-L", os.path.join(CUDA, "lib64"),
                    "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}",
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gemm_f32: 78000 elements exact" in r.stdout
    assert "gemm_bf16_f32acc: 78000 elements exact" in r.stdout
