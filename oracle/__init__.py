"""The CPU oracle for dense GEMM (C = A*B), as a small ctypes wrapper.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library under ``dense_gemm_07_gb300/`` and imports nothing from
it; the two meet only in the seeded input generators, which hold none of the
GEMM arithmetic.

The arithmetic lives in ``gemm_oracle.c`` (plain C, FP64 accumulation, loop
order i, k, j); see that file's header for the definition it follows and the
passages it cites.  This wrapper only builds the shared library, checks array
shapes and dtypes, and passes pointers.

Parity of every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, exact rational arithmetic and the worked examples the
pages print; no function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into _build/liboracle.so (OpenMP if available).

    Flags: -O2 with FP contraction off and no fast-math, so every product and
    sum is a separate IEEE double operation as written.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler (gcc) found")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
            "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            for name in ("oracle_gemm_f32", "oracle_gemm_bf16"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [i64, i64, i64, vp, i64, vp, i64, dp, i64, dp]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_gemm_flops.restype = ctypes.c_double
            lib.oracle_gemm_flops.argtypes = [i64, i64, i64]
            lib.oracle_gemm_epilogue.restype = ctypes.c_int
            lib.oracle_gemm_epilogue.argtypes = [i64, i64, vp, i64, ctypes.c_double,
                                                 ctypes.c_double, vp, i64, vp,
                                                 ctypes.c_int, vp, i64]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


def _rows(a: np.ndarray, name: str):
    """(rows, cols, leading dimension in elements) of a 2-D row-major view."""
    if a.ndim != 2:
        raise ValueError(f"oracle: {name} must be 2-D")
    if a.size == 0:
        return a.shape[0], a.shape[1], max(a.shape[1], 1)
    if a.shape[1] > 1 and a.strides[1] != a.itemsize:
        raise ValueError(f"oracle: {name} must have unit stride along rows")
    ld = a.strides[0] // a.itemsize if a.shape[0] > 1 else max(a.shape[1], 1)
    if ld < a.shape[1]:
        raise ValueError(f"oracle: {name} rows overlap")
    return a.shape[0], a.shape[1], ld


def _gemm(fn_name, A, B, want_s):
    lib = _load()
    M, K, lda = _rows(A, "A")
    K2, N, ldb = _rows(B, "B")
    if K2 != K:
        raise ValueError(f"oracle: inner sizes differ ({K} vs {K2})")
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64) if want_s else None
    rc = getattr(lib, fn_name)(M, N, K, _ptr(A), lda, _ptr(B), ldb,
                               _ptr(C), max(N, 1), _ptr(S))
    if rc != 0:
        raise ValueError(f"oracle: {fn_name} rejected its arguments")
    return (C, S) if want_s else C


def gemm_f32(A: np.ndarray, B: np.ndarray, with_abs: bool = False):
    """C = A*B in FP64 from FP32 inputs; with_abs also returns S = sum|a*b|."""
    if A.dtype != np.float32 or B.dtype != np.float32:
        raise TypeError("oracle.gemm_f32 takes float32 arrays")
    return _gemm("oracle_gemm_f32", A, B, with_abs)


def gemm_bf16(A_bits: np.ndarray, B_bits: np.ndarray, with_abs: bool = False):
    """C = A*B in FP64 from BF16 inputs given as their uint16 bit patterns."""
    if A_bits.dtype != np.uint16 or B_bits.dtype != np.uint16:
        raise TypeError("oracle.gemm_bf16 takes uint16 (BF16 bit) arrays")
    return _gemm("oracle_gemm_bf16", A_bits, B_bits, with_abs)


def gemm_epilogue(AB: np.ndarray, alpha: float = 1.0, beta: float = 0.0,
                  C0: np.ndarray | None = None, bias: np.ndarray | None = None,
                  act: int = 0) -> np.ndarray:
    """act(alpha * AB + beta * C0 + bias) in double; AB from gemm_f32/gemm_bf16.

    C0 (FP32, M x N) None means C is not read; bias (FP32, N) None means no
    bias; act 0 = identity, 1 = ReLU, 2 = GELU (x * Phi(x), erf form).
    """
    lib = _load()
    AB = np.ascontiguousarray(AB, dtype=np.float64)
    M, N = AB.shape
    c0 = None if C0 is None else np.ascontiguousarray(C0, dtype=np.float32)
    bs = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if c0 is not None and c0.shape != (M, N):
        raise ValueError("oracle: C0 must be M x N")
    if bs is not None and bs.shape != (N,):
        raise ValueError("oracle: bias must have N elements")
    out = np.zeros((M, N), dtype=np.float64)
    rc = lib.oracle_gemm_epilogue(M, N, _ptr(AB), max(N, 1), float(alpha), float(beta),
                                  _ptr(c0), max(N, 1), _ptr(bs), int(act), _ptr(out),
                                  max(N, 1))
    if rc != 0:
        raise ValueError("oracle: gemm_epilogue rejected its arguments")
    return out


def bf16_to_double(bits: int) -> float:
    """Exact value of one BF16 bit pattern."""
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def gemm_flops(M: int, N: int, K: int) -> float:
    """2*M*N*K, the operation count of one GEMM."""
    return float(_load().oracle_gemm_flops(M, N, K))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))
