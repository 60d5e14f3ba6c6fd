"""ctypes declarations of libgemm07.so -- one Python name per C entry point.

Argument marshalling only: every function here forwards its integers and
addresses to the C symbol of the same name and returns its result.  The
library is loaded on first use; if it has not been built, or cannot be
loaded, the call raises (there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import threading

from . import _build

_lib = None
_lock = threading.Lock()

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_MISALIGNED = 2          # reserved, never returned
GEMM_ERR_UNSUPPORTED_DEVICE = 3
GEMM_ERR_LAUNCH = 4
GEMM_ERR_TIMEOUT = 5
GEMM_ERR_INTERNAL = 6
GEMM_ERR_NO_MEMORY = 7
GEMM_ERR_SCRATCH_TOO_SMALL = 8
NOALLOC_SCRATCH_BYTES = 64 << 20

PATHS = {0: "none", 1: "zero_fill", 2: "f32_simt", 3: "bf16_tma",
         4: "bf16_packed", 5: "bf16_skinny", 6: "bf16_gemv", 7: "bf16_small",
         8: "bf16_narrow"}


class GemmPlan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("pack_a", ctypes.c_int32), ("pack_b", ctypes.c_int32),
                ("dp_tiles", ctypes.c_int64), ("sk_tiles", ctypes.c_int64),
                ("sk_pairs", ctypes.c_int32), ("pairs", ctypes.c_int32)]


class GemmEpilogue(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("bias", ctypes.c_void_p), ("activation", ctypes.c_int32)]


ACT_NONE = 0
ACT_RELU = 1
ACT_GELU = 2


# (name, restype, argtypes)
_i64, _vp, _i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
_GEMM_ARGS = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
SIGNATURES = [
    ("gemm_f32", _i32, _GEMM_ARGS),
    ("gemm_bf16_f32acc", _i32, _GEMM_ARGS),
    ("gemm_bf16_f32acc_noalloc", _i32, _GEMM_ARGS),
    ("gemm_f32_ex", _i32, _GEMM_ARGS[:-1] + [ctypes.POINTER(GemmEpilogue), _vp]),
    ("gemm_bf16_f32acc_ex", _i32, _GEMM_ARGS[:-1] + [ctypes.POINTER(GemmEpilogue), _vp]),
    ("gemm_f32_host", _i32, _GEMM_ARGS),
    ("gemm_f32_ladder", _i32, [_i32] + _GEMM_ARGS),
    ("gemm_bf16_f32acc_host", _i32, _GEMM_ARGS),
    ("gemm_status_string", ctypes.c_char_p, [_i32]),
    ("gemm_get_device_status", _i32, [_vp]),
    ("gemm_shutdown", None, []),
    ("gemm_abi_version", _i32, []),
    ("gemm_launch_count", ctypes.c_uint64, []),
    ("gemm_debug_inject", _i32, [_i32, ctypes.c_uint64]),
    ("gemm_tile_order", _i32, [_i64, _i64, _i64, _i64,
                               ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    ("gemm_plan_bf16", _i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                              ctypes.POINTER(GemmPlan)]),
    ("gemm_plan_f32", _i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                             ctypes.POINTER(GemmPlan)]),
    ("gemm_pair_units", _i64, [_i64, _i64, _i64, _i32, _i32, _i32, _vp, _i64]),
    ("gemm_set_bf16_schedule", _i32, [_i32]),
    ("gemm_set_bf16_small_limit", _i64, [_i64]),
]


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded library (built first if needed and allowed)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                path = _build.build()
            else:
                path = _build.LIB_PATH
            try:
                handle = ctypes.CDLL(path)
            except OSError as exc:
                raise RuntimeError(f"libgemm07.so could not be loaded from "
                                   f"{path}: {exc}") from exc
            for name, res, args in SIGNATURES:
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def library_path() -> str:
    return _build.LIB_PATH


def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream):
    return lib().gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_bf16_f32acc(M, N, K, A, lda, B, ldb, C, ldc, stream):
    return lib().gemm_bf16_f32acc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def _epi(epilogue):
    return None if epilogue is None else ctypes.byref(epilogue)


def gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, epilogue, stream):
    """gemm_f32 with a fused epilogue (GemmEpilogue or None)."""
    return lib().gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, _epi(epilogue), stream)


def gemm_bf16_f32acc_ex(M, N, K, A, lda, B, ldb, C, ldc, epilogue, stream):
    """gemm_bf16_f32acc with a fused epilogue (GemmEpilogue or None)."""
    return lib().gemm_bf16_f32acc_ex(M, N, K, A, lda, B, ldb, C, ldc, _epi(epilogue),
                                     stream)


def gemm_bf16_f32acc_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream):
    """gemm_bf16_f32acc without any device allocation (fixed scratch)."""
    return lib().gemm_bf16_f32acc_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f32_ladder(rung, M, N, K, A, lda, B, ldb, C, ldc, stream):
    """Teaching rung 0 (naive), 1 (smem-tiled) or 2 (1-D register tiles)."""
    return lib().gemm_f32_ladder(rung, M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f32_host(M, N, K, A, lda, B, ldb, C, ldc, stream):
    return lib().gemm_f32_host(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_bf16_f32acc_host(M, N, K, A, lda, B, ldb, C, ldc, stream):
    return lib().gemm_bf16_f32acc_host(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_status_string(status: int) -> str:
    return lib().gemm_status_string(status).decode()


def gemm_get_device_status(stream) -> int:
    return lib().gemm_get_device_status(stream)


def gemm_shutdown() -> None:
    lib().gemm_shutdown()


def gemm_abi_version() -> int:
    return lib().gemm_abi_version()


def gemm_debug_inject(mode: int, wait_ns: int) -> int:
    """Test hook: bounded-wait limit and fault mode (see include/gemm07.h)."""
    return lib().gemm_debug_inject(mode, wait_ns)


def gemm_launch_count() -> int:
    return int(lib().gemm_launch_count())


def gemm_tile_order(tiles_m, tiles_n, group, linear):
    tm, tn = _i64(), _i64()
    s = lib().gemm_tile_order(tiles_m, tiles_n, group, linear,
                              ctypes.byref(tm), ctypes.byref(tn))
    return s, tm.value, tn.value


def _plan(fn, M, N, K, A, lda, B, ldb, C, ldc):
    p = GemmPlan()
    s = fn(M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(p))
    return s, p


def gemm_plan_bf16(M, N, K, A, lda, B, ldb, C, ldc):
    return _plan(lib().gemm_plan_bf16, M, N, K, A, lda, B, ldb, C, ldc)


def gemm_plan_f32(M, N, K, A, lda, B, ldb, C, ldc):
    return _plan(lib().gemm_plan_f32, M, N, K, A, lda, B, ldb, C, ldc)


SCHEDULE_AUTO = 0
SCHEDULE_STREAM_K = 1
SCHEDULE_COLUMN_SPLIT = 2


def gemm_set_bf16_schedule(schedule: int) -> int:
    return lib().gemm_set_bf16_schedule(schedule)


def gemm_set_bf16_small_limit(max_macs: int) -> int:
    """Largest M*N*K (M >= 2) sent to the CUDA-core small-problem path;
    0 sends every BF16 call to the tensor-core kernels.  Returns the
    previous limit."""
    return lib().gemm_set_bf16_small_limit(max_macs)


def gemm_pair_units(M, N, K, max_pairs, pair, schedule=SCHEDULE_AUTO):
    """The BF16 paired-SM kernel's work units for one pair, in order, as a
    list of (tile, k0, k1, slot, first_pair, segments, stream_k, n_off,
    width) tuples; raises on bad arguments."""
    n = lib().gemm_pair_units(M, N, K, max_pairs, schedule, pair, None, 0)
    if n < 0:
        raise ValueError("gemm_pair_units: argument out of range")
    buf = (ctypes.c_int64 * (9 * max(n, 1)))()
    n2 = lib().gemm_pair_units(M, N, K, max_pairs, schedule, pair, buf, n)
    assert n2 == n
    return [tuple(buf[9 * i:9 * i + 9]) for i in range(n)]
