"""The C-ABI library on the CPU: it builds, loads, exports every symbol the
header declares, and its host-only logic (tile order, path planning,
argument checks, status strings) behaves as documented.  No GPU work."""
import ctypes
import os
import re

import contextlib

import pytest

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import _abi, _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "gemm07.h")


@pytest.fixture(scope="module")
def lib():
    return _abi.lib()


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GEMM07_API\s+[\w\s\*]*?\b(gemm_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_symbols()
    for must in ["gemm_f32", "gemm_bf16_f32acc", "gemm_status_string",
                 "gemm_get_device_status", "gemm_f32_host", "gemm_bf16_f32acc_host"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
        assert name in {n for n, _, _ in _abi.SIGNATURES}, f"no binding for {name}"
        assert hasattr(_abi, name), f"no Python function named {name}"


def test_library_is_in_tree_and_for_sm103a():
    assert os.path.dirname(_build.LIB_PATH).startswith(os.path.dirname(g7.__file__))
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.NVCC_FLAGS)


def test_abi_version(lib):
    assert _abi.gemm_abi_version() == 5


def test_status_numbering_follows_the_boundary_table():
    # the codes of the boundary's definition, then this library's additions
    assert (_abi.GEMM_OK, _abi.GEMM_ERR_INVALID_ARG, _abi.GEMM_ERR_MISALIGNED,
            _abi.GEMM_ERR_UNSUPPORTED_DEVICE, _abi.GEMM_ERR_LAUNCH,
            _abi.GEMM_ERR_TIMEOUT, _abi.GEMM_ERR_INTERNAL) == (0, 1, 2, 3, 4, 5, 6)
    assert (_abi.GEMM_ERR_NO_MEMORY, _abi.GEMM_ERR_SCRATCH_TOO_SMALL) == (7, 8)


def test_status_strings(lib):
    seen = set()
    for code in range(9):
        s = _abi.gemm_status_string(code)
        assert s and s not in seen
        seen.add(s)
    assert _abi.gemm_status_string(99) == "unknown status"


@pytest.mark.parametrize("tm,tn,group", [(32, 16, 8), (7, 5, 3), (1, 9, 8),
                                         (24, 1, 8), (13, 17, 4), (32, 32, 1)])
def test_tile_order_is_a_bijection_in_bands(tm, tn, group):
    seen = set()
    for lin in range(tm * tn):
        s, m, n = _abi.gemm_tile_order(tm, tn, group, lin)
        assert s == 0 and 0 <= m < tm and 0 <= n < tn
        # index `lin` lies in band lin // (group*tn): rows [band*group, +group)
        band = lin // (group * tn)
        assert band * group <= m < min(tm, (band + 1) * group)
        seen.add((m, n))
    assert len(seen) == tm * tn


def test_tile_order_runs_down_columns_first():
    # inside a band, consecutive indices step down the rows of one column
    coords = [_abi.gemm_tile_order(32, 16, 8, i)[1:] for i in range(16)]
    assert coords[:8] == [(r, 0) for r in range(8)]
    assert coords[8:16] == [(r, 1) for r in range(8)]


def test_tile_order_rejects_bad_arguments():
    assert _abi.gemm_tile_order(0, 4, 2, 0)[0] == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_tile_order(4, 4, 0, 0)[0] == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_tile_order(4, 4, 2, 16)[0] == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_tile_order(4, 4, 2, -1)[0] == _abi.GEMM_ERR_INVALID_ARG


def _path(kind, *a, **k):
    s, p = g7.plan(kind, *a, **k)
    assert s == 0
    return _abi.PATHS[p.path], p


def test_plan_paths():
    assert _path("bf16", 0, 5, 5)[0] == "none"
    assert _path("bf16", 5, 0, 5)[0] == "none"
    assert _path("bf16", 5, 5, 0)[0] == "zero_fill"
    assert _path("f32", 5, 5, 0)[0] == "zero_fill"
    path, p = _path("bf16", 4096, 4096, 4096)
    # three whole waves on 76 pairs, then each of the last 28 tiles halved
    # along K over two pairs (scratch: partial-sum slots and flags, which
    # the halves need only when they cannot be added in C itself)
    assert path == "bf16_tma" and p.tiles == 16 * 16
    assert p.workspace_bytes == 56 * 4 * 128 * 1024 + (28 * 8 + 56 * 16) * 8
    assert (p.dp_tiles, p.sk_tiles, p.sk_pairs, p.pairs) == (228, 28, 56, 76)
    assert (p.tile_m, p.tile_n, p.tile_k, p.stages) == (256, 256, 64, 6)
    path, p = _path("bf16", 129, 4096, 1024)
    assert path == "bf16_tma" and (p.tile_m, p.tile_n, p.stages) == (256, 256, 6)
    # few 128 x 128 tiles (at most half the SMs) and K >= 1536: the narrow-N
    # kernel with 128 x 128 tiles, K split over clusters; not for a short K,
    # more tiles, or a schedule other than the automatic one
    path, p = _path("bf16", 129, 4096, 4096)
    assert path == "bf16_narrow" and (p.tile_m, p.tile_n, p.split_k) == (128, 128, 2)
    assert p.tiles == 64 * 2 and p.workspace_bytes == 0
    path, p = _path("bf16", 512, 1024, 8192)
    assert path == "bf16_narrow" and p.split_k == 4 and p.tiles == 32 * 4
    assert _path("bf16", 512, 512, 4096)[1].split_k == 8
    assert _path("bf16", 1024, 1024, 1528)[0] == "bf16_tma"
    # the limits exactly: 4 x 19 = 76 tiles, K 1536 / 1528
    assert _path("bf16", 512, 2432, 1536)[0] == "bf16_narrow"
    assert _path("bf16", 512, 2433, 1536)[0] == "bf16_packed"   # 4 x 20 tiles (B copied)
    assert _path("bf16", 512, 2432, 1528)[0] == "bf16_tma"
    assert _path("bf16", 1280, 1024, 4096)[0] == "bf16_tma"   # 80 tiles
    prev = _abi.gemm_set_bf16_schedule(_abi.SCHEDULE_STREAM_K)
    try:
        assert _path("bf16", 512, 1024, 8192)[0] == "bf16_tma"
    finally:
        _abi.gemm_set_bf16_schedule(prev)
    # M <= 128: small-M path, 128-column tiles, K split 4 ways over 32 tiles
    path, p = _path("bf16", 16, 4096, 4096)
    assert path == "bf16_skinny" and (p.tile_m, p.tile_n, p.split_k) == (16, 128, 4)
    assert p.tiles == 32 * 4
    # M = 1 takes the same small-M path (a 16-row MMA, rows 1..15 read as
    # zeros), with no scratch for aligned operands
    path, p = _path("bf16", 1, 4096, 4096)
    assert path == "bf16_skinny" and (p.tile_m, p.tile_n, p.split_k) == (16, 128, 4)
    assert p.tiles == 32 * 4 and p.workspace_bytes == 0
    path, p = _path("bf16", 1, 1000, 16)
    assert path == "bf16_skinny" and p.split_k == 1 and p.workspace_bytes == 0
    # N <= 128 < M: narrow-N path, 128-row tiles by all N columns (MMA N 64
    # or 128), K split 4 ways over 32 row tiles
    path, p = _path("bf16", 4096, 128, 4096)
    assert path == "bf16_narrow" and (p.tile_m, p.tile_n, p.split_k) == (128, 128, 4)
    assert p.tiles == 32 * 4 and p.workspace_bytes == 0
    assert _path("bf16", 4096, 64, 4096)[1].tile_n == 64
    assert _path("bf16", 4096, 65, 4096)[1].tile_n == 128
    assert _path("bf16", 20000, 100, 4096)[1].split_k == 1     # 157 tiles: no split
    assert _path("bf16", 4096, 136, 1024)[0] == "bf16_tma"     # wider, short K: SM pairs
    # sizes whose M * N * K overflows 64 bits are not mistaken for small
    # problems: their tile count is refused
    huge = 1 << 30
    assert _abi.gemm_plan_bf16(huge, huge, 4096, 16, 4096, 16, huge, 16, huge)[0] == \
        _abi.GEMM_ERR_INVALID_ARG
    # a matrix spanning more than 2^60 elements (rows x leading dimension)
    # is refused, whatever M, N and K are
    for fn in (_abi.gemm_plan_bf16, _abi.gemm_plan_f32):
        assert fn(1 << 20, 64, 64, 16, 1 << 41, 16, 64, 16, 64)[0] == _abi.GEMM_ERR_INVALID_ARG
        assert fn(64, 64, 1 << 20, 16, 1 << 20, 16, 1 << 41, 16, 64)[0] == \
            _abi.GEMM_ERR_INVALID_ARG
        assert fn(1 << 20, 64, 64, 16, 64, 16, 64, 16, 1 << 41)[0] == _abi.GEMM_ERR_INVALID_ARG
        assert fn(1 << 20, 64, 64, 16, 1 << 40, 16, 64, 16, 64)[0] == _abi.GEMM_OK
    assert _path("bf16", 4096, 136, 4096)[0] == "bf16_narrow"  # 64 tiles, long K
    assert _path("bf16", 8192, 136, 4096)[0] == "bf16_tma"     # 128 tiles: SM pairs
    assert _path("bf16", 128, 64, 4096)[0] == "bf16_skinny"    # M <= 128 first
    assert _path("bf16", 33, 4096, 4096)[1].tile_m == 64
    assert _path("bf16", 128, 4096, 4096)[1].tile_m == 128
    with _small_limit(0):                                   # tensor-core kernels only
        assert _path("bf16", 2, 4096, 4096)[1].tile_m == 16
        assert _path("bf16", 16, 100, 64)[1].split_k == 1  # one k slice only
    path, p = _path("f32", 4096, 4096, 4096)
    assert path == "f32_simt" and p.tiles == 32 * 32
    # small problems: 64 x 64 tiles (split along K on the device)
    path, p = _path("f32", 256, 256, 256)
    assert path == "f32_simt" and (p.tile_m, p.tile_n, p.tiles) == (64, 64, 16)
    assert _path("f32", 512, 512, 2048)[1].tile_m == 64     # 2^29 multiply-adds
    assert _path("f32", 512, 512, 4096)[1].tile_m == 128    # 2^30
    assert _path("f32", 2048, 300, 100)[1].tile_m == 128    # 48 tiles of 128 x 128
    # K = 3001: A rows are not a multiple of 16 bytes -> A is packed
    path, p = _path("bf16", 127, 1000, 3001)
    assert path == "bf16_skinny" and p.pack_a == 1 and p.pack_b == 0
    path, p = _path("bf16", 3001, 1000, 3001)
    assert path == "bf16_packed" and p.pack_a == 1 and p.pack_b == 0
    assert p.workspace_bytes >= 3001 * 3008 * 2
    # few tiles and a long K: the narrow-N kernel, A still copied first
    path, p = _path("bf16", 300, 1000, 3001)
    assert path == "bf16_narrow" and p.pack_a == 1 and p.pack_b == 0
    assert p.workspace_bytes >= 300 * 3008 * 2
    # misaligned base address -> packed
    path, p = _path("bf16", 3001, 1000, 3001, A=16 + 2)
    assert path == "bf16_packed" and p.pack_a == 1 and p.pack_b == 0
    with _small_limit(0):
        path, p = _path("bf16", 256, 256, 256, A=16 + 2)
        assert path == "bf16_packed" and p.pack_a == 1 and p.pack_b == 0


@contextlib.contextmanager
def _small_limit(v):
    prev = _abi.gemm_set_bf16_small_limit(v)
    try:
        yield
    finally:
        _abi.gemm_set_bf16_small_limit(prev)


def test_plan_small_bf16_path():
    # M >= 2, few multiply-adds: 64 x 64 tiles on the CUDA cores, operands
    # read in place (no copies even with rows of 127 elements or a base off
    # 16 bytes), K split so that the blocks cover about two per SM
    path, p = _path("bf16", 127, 127, 127)
    assert path == "bf16_small" and p.pack_a == 0 and p.pack_b == 0
    assert (p.tile_m, p.tile_n, p.tile_k) == (64, 64, 32)
    assert p.split_k == 4 and p.tiles == 4 * 4          # 4 slices of K, 4 tiles
    assert p.workspace_bytes == 4096 + 4 * 4 * 64 * 64 * 4   # fixed counter area first
    path, p = _path("bf16", 256, 256, 256, A=16 + 2)
    assert path == "bf16_small" and p.pack_a == 0
    path, p = _path("bf16", 3001, 127, 127)
    assert path == "bf16_small" and p.split_k == 3 and p.tiles == 47 * 2 * 3   # 304 // 94 = 3
    # an operand would be copied: up to 2^26 with K <= 512, else up to 2^24
    path, p = _path("bf16", 1000, 500, 127)             # 63.5 M, A would be copied
    assert path == "bf16_small" and p.pack_a == 0 and p.split_k == 2   # 304 // 128 tiles
    assert _path("bf16", 1000, 1000, 127)[0] == "bf16_packed"     # 127 M: tensor cores
    assert _path("bf16", 127, 127, 1000)[0] == "bf16_small"       # 16.1 M, long K
    assert _path("bf16", 127, 127, 3001)[0] == "bf16_skinny"      # 48 M, long K
    assert _path("bf16", 1000, 127, 1000)[0] == "bf16_narrow"     # 127 M
    # operands the tensor-core kernels read in place: only up to 2^24
    assert _path("bf16", 256, 256, 256)[0] == "bf16_small"        # 2^24
    assert _path("bf16", 256, 256, 264)[0] == "bf16_tma"
    assert _path("bf16", 127, 1000, 1000)[0] == "bf16_skinny"     # aligned rows, 1.3e8
    assert _path("bf16", 1000, 1000, 1000)[0] == "bf16_tma"       # 10^9: tensor cores
    # few rows and a larger B: the small-M tensor-core kernel streams B
    assert _path("bf16", 2, 1000, 1000)[0] == "bf16_skinny"
    assert _path("bf16", 8, 3001, 3001)[0] == "bf16_skinny"
    assert _path("bf16", 2, 8, 8)[0] == "bf16_small"
    assert _path("bf16", 1, 127, 127)[0] == "bf16_skinny"        # M = 1: tensor cores
    # the limit is process-wide and settable; negative values are refused
    with _small_limit(1000):
        assert _path("bf16", 10, 10, 10)[0] == "bf16_small"      # lda = 10: A would be copied
        assert _path("bf16", 10, 10, 11)[0] == "bf16_skinny"
    assert _abi.gemm_set_bf16_small_limit(-1) == -1
    assert _path("bf16", 127, 127, 127)[0] == "bf16_small"


def test_plan_and_calls_reject_bad_arguments(lib):
    bad = [(-1, 4, 4, 4, 4, 4), (4, 4, 8, 7, 4, 4), (4, 8, 4, 4, 7, 8),
           (4, 8, 4, 4, 8, 7), (1 << 31, 4, 4, 4, 4, 4)]
    for (M, N, K, lda, ldb, ldc) in bad:
        for kind in ("bf16", "f32"):
            s, _ = g7.plan(kind, M, N, K, lda=lda, ldb=ldb, ldc=ldc)
            assert s == _abi.GEMM_ERR_INVALID_ARG, (kind, M, N, K, lda, ldb, ldc)
        # the entry points check before touching any device
        for fn in (_abi.gemm_f32, _abi.gemm_bf16_f32acc):
            assert fn(M, N, K, 16, lda, 16, ldb, 16, ldc, None) == \
                _abi.GEMM_ERR_INVALID_ARG
    # null data pointer with a nonzero extent
    assert _abi.gemm_f32(4, 4, 4, None, 4, 16, 4, 16, 4, None) == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_bf16_f32acc(4, 4, 4, 16, 4, 16, 4, None, 4, None) == \
        _abi.GEMM_ERR_INVALID_ARG
    # empty problems are fine without a GPU: nothing is launched
    assert _abi.gemm_f32(0, 4, 4, None, 4, None, 4, None, 4, None) == _abi.GEMM_OK


def test_binding_row_strides():
    # the binding passes a tensor's row stride as the leading dimension: rows
    # must be contiguous and must not overlap (a broadcast row has stride 0)
    torch = pytest.importorskip("torch")
    assert g7._ld(torch.zeros(4, 3), "A") == 3
    assert g7._ld(torch.zeros(4, 8)[:, 2:5], "A") == 8     # a column slice
    assert g7._ld(torch.zeros(1, 5), "A") == 5
    assert g7._ld(torch.zeros(4, 1).t(), "A") == 4          # one row
    with pytest.raises(ValueError):
        g7._ld(torch.zeros(4, 3).t(), "A")                  # transposed
    with pytest.raises(ValueError):
        g7._ld(torch.zeros(1, 3).expand(4, 3), "A")         # broadcast rows
    with pytest.raises(ValueError):
        g7._ld(torch.zeros(12).as_strided((4, 6), (2, 1)), "A")  # overlapping rows


def test_epilogue_entry_points_validate_on_host(lib):
    epi = _abi.GemmEpilogue(1.0, 0.0, None, 9)
    assert _abi.gemm_bf16_f32acc_ex(4, 4, 4, 16, 4, 16, 4, 16, 4, epi, None) == \
        _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_f32_ex(-1, 4, 4, 16, 4, 16, 4, 16, 4, None, None) == \
        _abi.GEMM_ERR_INVALID_ARG


def test_ladder_rejects_bad_rungs(lib):
    assert _abi.gemm_f32_ladder(3, 4, 4, 4, 16, 4, 16, 4, 16, 4, None) == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_f32_ladder(-1, 4, 4, 4, 16, 4, 16, 4, 16, 4, None) == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_f32_ladder(0, 600000, 4, 4, 16, 4, 16, 4, 16, 4, None) == \
        _abi.GEMM_ERR_INVALID_ARG


def test_debug_hook_rejects_unknown_modes(lib):
    assert _abi.gemm_debug_inject(7, 0) == _abi.GEMM_ERR_INVALID_ARG
    assert _abi.gemm_debug_inject(-1, 0) == _abi.GEMM_ERR_INVALID_ARG


def test_no_gpu_means_a_loud_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    buf = (ctypes.c_float * 16)()
    addr = ctypes.addressof(buf)
    s = _abi.gemm_f32(2, 2, 2, addr, 2, addr, 2, addr, 2, None)
    assert s == _abi.GEMM_ERR_UNSUPPORTED_DEVICE
    with pytest.raises(Exception):
        g7.gemm_f32(torch.ones(2, 2), torch.ones(2, 2))
