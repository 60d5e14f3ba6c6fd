"""GPU parity: the CUDA path, called through the C ABI, against the oracle.

Every case uses the seeded generators of dense_gemm_07_gb300.inputs and the
bounds stated in tests/gemm_check.py.  Small and medium shapes are compared
element by element; the full 4096-class shapes (the ones the benchmark times)
are compared in full as well, element by element (the FP64 oracle takes a
few seconds per 4096^3 product on the host cores).
"""
import numpy as np
import pytest
import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import _abi
from dense_gemm_07_gb300 import inputs
from gemm_check import (ROUTES, assert_guards_intact, assert_within, guarded_output,
                        oracle_ref, route_limit)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _dtype(kind):
    return torch.float32 if kind == "f32" else torch.bfloat16


def _run(kind, a, b, out=None):
    a_d, b_d = a.to(DEV), b.to(DEV)
    fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
    c = fn(a_d, b_d, out=out)
    torch.cuda.synchronize()
    return c


def _check(kind, M, N, K, seed, dist, dist_b=None, exact=False, rows=None, route="default"):
    a, b = inputs.make_pair(M, N, K, seed, dist, dist_b, dtype=_dtype(kind))
    with route_limit(route):
        c = _run(kind, a, b).cpu().numpy()
    if rows is not None:
        c = c[rows]
    c_ref, s_ref = oracle_ref(kind, a, b, rows=rows, with_abs=not exact)
    assert_within(kind, c, c_ref, s_ref, exact=exact, what=f"{kind} {M}x{N}x{K}")
    assert g7.gemm_get_device_status() == 0


# ------------------------------------------------------------ FP32 (SIMT)

@pytest.mark.parametrize("shape,tile", [
    ((512, 512, 512), 64), ((513, 512, 512), 128), ((512, 512, 2049), 128),
    ((1, 4096, 4096), 128), ((4096, 1, 4096), 128), ((1, 1, 1), 64), ((2048, 2048, 1), 128)])
def test_f32_path_transitions_exact(shape, tile):
    # each side of the small-problem limit (16 tiles of 128 x 128 and 2^29
    # multiply-adds), a single row or column over a long K, and K = 1
    M, N, K = shape
    s, p = g7.plan("f32", M, N, K)
    assert s == 0 and p.tile_m == tile
    _check("f32", M, N, K, 24, inputs.INT3, exact=True)


def test_f32_256_uniform():
    _check("f32", 256, 256, 256, 0, inputs.UNIFORM)


def test_f32_256_integers_exact():
    _check("f32", 256, 256, 256, 0, inputs.INT4, exact=True)


@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (1000, 700, 1024),
                                   (1000, 700, 1000)])
def test_f32_ragged_lab_shapes(shape):
    M, N, K = shape
    _check("f32", M, N, K, 7, inputs.INT4, exact=True)


@pytest.mark.parametrize("K", [1, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127])
def test_f32_small_and_ragged_k(K):
    _check("f32", 130, 131, K, 11, inputs.UNIFORM)


@pytest.mark.parametrize("shape", [(2560, 2048, 136), (2432, 2055, 77),
                                   (4096, 1024, 40)])
def test_f32_full_and_split_waves_exact(shape):
    # more tiles than resident blocks: whole waves of 128 x 128 tiles plus a
    # last wave of half-width tiles, with ragged N and K in the second case
    M, N, K = shape
    _check("f32", M, N, K, 16, inputs.INT4, exact=True)


def test_f32_4096_every_element():
    M = N = K = 4096
    _check("f32", M, N, K, 1, inputs.UNIFORM)


@pytest.mark.parametrize("rung", [0, 1, 2])
@pytest.mark.parametrize("shape", [(256, 256, 256), (1000, 700, 1000), (65, 129, 33)])
def test_f32_ladder_rungs_exact(rung, shape):
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 20, inputs.INT4, dtype=torch.float32)
    c = g7.gemm_f32_ladder(rung, a.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    c_ref, _ = oracle_ref("f32", a, b, with_abs=False)
    assert_within("f32", c.cpu().numpy(), c_ref, None, exact=True, what=f"rung {rung}")


def test_f32_ladder_rung_uniform():
    a, b = inputs.make_pair(300, 200, 500, 21, inputs.UNIFORM, dtype=torch.float32)
    for rung in range(3):
        c = g7.gemm_f32_ladder(rung, a.to(DEV), b.to(DEV))
        torch.cuda.synchronize()
        c_ref, s_ref = oracle_ref("f32", a, b)
        assert_within("f32", c.cpu().numpy(), c_ref, s_ref, what=f"rung {rung}")


# --------------------------------------------------- BF16 (tensor cores)

@pytest.mark.parametrize("route", ROUTES)
def test_bf16_256_normal(route):
    _check("bf16", 256, 256, 256, 2, inputs.NORMAL, route=route)


@pytest.mark.parametrize("route", ROUTES)
def test_bf16_integers_exact_tiles(route):
    # several tiles, several k slices and ragged tails on either route
    _check("bf16", 300, 600, 200, 4, inputs.INT3, exact=True, route=route)


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("K", [1, 8, 16, 63, 64, 65, 200])
def test_bf16_small_and_ragged_k(K, route):
    _check("bf16", 130, 260, K, 5, inputs.INT3, exact=True, route=route)


def test_bf16_full_and_split_waves_exact():
    # 256 pair tiles: whole waves of 256 x 256 tiles, then the last wave as
    # 256 x 128 units (rows 3072..4095 hold some of them)
    M, N, K = 4096, 4096, 136
    _check("bf16", M, N, K, 17, inputs.INT3, exact=True)


def test_bf16_4096_every_element():
    M = N = K = 4096
    _check("bf16", M, N, K, 2, inputs.NORMAL)


@pytest.mark.parametrize("NK", [(4096, 4096), (11008, 4096), (4096, 11008)])
def test_bf16_linear_layer_shapes_every_element(NK):
    N, K = NK
    _check("bf16", 2048, N, K, 3, inputs.NORMAL, inputs.NORMAL_W)


# Stream-K: tiles split into runs of k-slices over several SM pairs, finished
# by adding the segments' partial sums.  Integer inputs make every order of
# summation exact, so the split must not change a single bit.
@pytest.fixture
def stream_k():
    prev = g7.abi.gemm_set_bf16_schedule(g7.abi.SCHEDULE_STREAM_K)
    yield
    g7.abi.gemm_set_bf16_schedule(prev)


@pytest.mark.parametrize("shape", [(512, 1024, 8192),    # 8 tiles halved over 16 pairs
                                   (512, 512, 8192),     # 4 tiles, long K
                                   (2560, 2304, 1024),   # 90 tiles: 1 wave + 14, all shared
                                   (2560, 2302, 640),    # N % 4: direct stores
                                   (3100, 3100, 700),    # 169 tiles, ragged edges
                                   (2900, 3300, 1000)])  # 156 tiles, ragged K
def test_bf16_stream_k_exact(stream_k, shape):
    M, N, K = shape
    s, p = g7.plan("bf16", M, N, K)
    assert p.sk_tiles > 0
    _check("bf16", M, N, K, 23, inputs.INT3, exact=True)


def test_bf16_stream_k_chosen_automatically_for_long_k():
    # 20 tiles of 256 x 256 (80 of 128 x 128, too many for the narrow-N
    # kernel) and a long K: the automatic schedule halves each tile along K
    M, N, K = 1280, 1024, 4096
    s, p = g7.plan("bf16", M, N, K)
    assert g7.abi.PATHS[p.path] == "bf16_tma" and (p.sk_tiles, p.sk_pairs) == (20, 40)
    _check("bf16", M, N, K, 27, inputs.NORMAL)


def test_bf16_stream_k_after_whole_waves_exact(stream_k):
    # 128 tiles: one whole wave and 52 more, shared as k-slice runs
    M, N, K = 4096, 2048, 1024
    _check("bf16", M, N, K, 24, inputs.INT3, exact=True)


@pytest.mark.parametrize("shape,dp,sk,skp", [
    ((2560, 2048, 6200), 0, 80, 76),     # one wave + 4 tiles: all 80 shared as k runs
    ((2530, 2040, 6150), 0, 80, 76),     # the same with ragged edges and K
    ((2530, 2030, 6150), 0, 80, 76),     # and N % 4 != 0: row stores, partial sums
    ((2600, 2100, 4100), 76, 23, 46),    # one wave, then 23 ragged tiles halved along K
    ((2560, 2560, 4096), 76, 24, 48),    # one wave, then 24 tiles halved along K
    ((4096, 4096, 4096), 228, 28, 56)])  # three waves, then 28 tiles halved along K
def test_bf16_auto_k_splits_after_whole_waves_exact(shape, dp, sk, skp):
    # automatic schedule after a whole wave: stream-K over every tile, or
    # the last wave's tiles halved along K; every element is compared
    M, N, K = shape
    s, plan = g7.plan("bf16", M, N, K)
    assert (plan.dp_tiles, plan.sk_tiles, plan.sk_pairs) == (dp, sk, skp)
    a, b = inputs.make_pair(M, N, K, 27, inputs.INT3, dtype=torch.bfloat16)
    c = g7.gemm_bf16_f32acc(a.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


def test_bf16_halved_tail_deterministic_bits():
    # 4096^3, automatic schedule: both halves of a split tile add into C
    # (cleared first) in whichever order they finish; the bits never change
    M = N = K = 4096
    s, plan = g7.plan("bf16", M, N, K)
    assert (plan.sk_tiles, plan.sk_pairs) == (28, 56)
    a, b = inputs.make_pair(M, N, K, 26, inputs.NORMAL, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    first = g7.gemm_bf16_f32acc(a_d, b_d).clone()
    for _ in range(5):
        again = g7.gemm_bf16_f32acc(a_d, b_d)
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    assert g7.gemm_get_device_status() == 0


@pytest.mark.parametrize("shape", [(2560, 2304, 1024), (4096, 4096, 1024)])
def test_bf16_stream_k_deterministic_bits(stream_k, shape):
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 25, inputs.NORMAL, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    first = g7.gemm_bf16_f32acc(a_d, b_d).clone()
    for _ in range(5):
        again = g7.gemm_bf16_f32acc(a_d, b_d)
        assert torch.equal(again.view(torch.int32), first.view(torch.int32))
    c_ref, s_ref = oracle_ref("bf16", a, b)
    assert_within("bf16", first.cpu().numpy(), c_ref, s_ref)


@pytest.mark.parametrize("shape", [(3100, 3100, 700), (2048, 4096, 1024), (700, 1300, 6200)])
def test_bf16_every_schedule_same_bits_on_integers(shape):
    # column split, stream-K and the automatic choice: exact sums everywhere
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 28, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    outs = []
    prev = g7.abi.gemm_set_bf16_schedule(g7.abi.SCHEDULE_AUTO)
    try:
        for sched in (g7.abi.SCHEDULE_AUTO, g7.abi.SCHEDULE_STREAM_K,
                      g7.abi.SCHEDULE_COLUMN_SPLIT):
            g7.abi.gemm_set_bf16_schedule(sched)
            outs.append(g7.gemm_bf16_f32acc(a_d, b_d).clone())
            assert g7.gemm_get_device_status() == 0
    finally:
        g7.abi.gemm_set_bf16_schedule(prev)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", outs[0].cpu().numpy(), c_ref, None, exact=True)


@pytest.mark.parametrize("M", [127, 1000, 3001])
@pytest.mark.parametrize("N", [127, 1000, 3001])
@pytest.mark.parametrize("K", [127, 1000, 3001])
def test_bf16_boundary_sweep_exact(M, N, K):
    _check("bf16", M, N, K, 4, inputs.INT3, exact=True)
    # shapes under the small-problem limit run on the CUDA cores by default:
    # check the tensor-core kernels on them as well
    s, plan = g7.plan("bf16", M, N, K)
    if _abi.PATHS[plan.path] == "bf16_small":
        _check("bf16", M, N, K, 4, inputs.INT3, exact=True, route="tensor_cores")


@pytest.mark.parametrize("M", [1, 16])
def test_bf16_skinny_exact(M):
    _check("bf16", M, 4096, 4096, 4, inputs.INT3, exact=True)


@pytest.mark.parametrize("shape", [(1, 4096, 4096), (1, 1000, 3001), (1, 3001, 1000),
                                   (1, 127, 127), (1, 11008, 4096), (1, 4096, 11008),
                                   (1, 4096, 1), (1, 4096, 16), (1, 4096, 17), (1, 1, 64),
                                   (1, 256, 65536), (1, 1100, 40), (1, 4096, 64),
                                   (1, 1000, 100), (1, 2048, 200), (1, 3000, 4096)])
def test_bf16_vector_times_matrix_exact(shape):
    # M = 1 on the small-M kernel (one row of A in a 16-row MMA, the other
    # rows zero-filled by the copy engine): ragged N (a partial or wholly
    # out-of-range column tile), ragged K, B copied first (N = 3001, 127),
    # K below one k-slice, long K (the K split over a cluster)
    M, N, K = shape
    s, plan = g7.plan("bf16", M, N, K)
    assert _abi.PATHS[plan.path] == "bf16_skinny"
    _check("bf16", M, N, K, 19, inputs.INT3, exact=True)


def test_bf16_vector_times_matrix_general_values_and_bits():
    # N(0,1) inputs within the BF16 bound; the range sums are added in a
    # fixed order, so repeated calls give the same bits
    a, b = inputs.make_pair(1, 4096, 11008, 20, inputs.NORMAL, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    first = g7.gemm_bf16_f32acc(a_d, b_d).clone()
    for _ in range(3):
        again = g7.gemm_bf16_f32acc(a_d, b_d)
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    c_ref, s_ref = oracle_ref("bf16", a, b)
    assert_within("bf16", first.cpu().numpy(), c_ref, s_ref)
    assert g7.gemm_get_device_status() == 0


@pytest.mark.parametrize("shape", [(2, 300, 1000), (17, 1000, 777), (33, 257, 4096),
                                   (64, 4096, 64), (65, 999, 130), (100, 128, 3001),
                                   (128, 2048, 2048), (5, 50, 1)])
@pytest.mark.parametrize("route", ROUTES)
def test_bf16_small_m_paths_exact(shape, route):
    # every MMA width (16/32/64/128), ragged N and K, K below the split
    # count; and the same shapes on the CUDA-core small-problem path
    M, N, K = shape
    _check("bf16", M, N, K, 18, inputs.INT3, exact=True, route=route)


@pytest.mark.parametrize("shape,path", [
    ((128, 4096, 512), "bf16_skinny"), ((129, 4096, 512), "bf16_tma"),
    ((4096, 128, 512), "bf16_narrow"), ((4096, 129, 512), "bf16_packed"),
    ((128, 128, 512), "bf16_skinny"), ((129, 128, 512), "bf16_narrow"),
    ((129, 129, 64), "bf16_packed"), ((1, 1, 1), "bf16_skinny"), ((129, 1, 1), "bf16_narrow"),
    ((128, 129, 65), "bf16_skinny"), ((129, 4096, 1), "bf16_packed"),
    ((4096, 129, 65), "bf16_packed")])
def test_bf16_path_transitions_exact(shape, path):
    # each side of the points where the plan changes kernel: M = 128 / 129
    # (small-M kernel / SM pairs), N = 128 / 129 (narrow-N kernel / SM
    # pairs), both together, and K of one element or just over one k-slice
    M, N, K = shape
    with route_limit("tensor_cores"):
        s, p = g7.plan("bf16", M, N, K)
        assert s == 0 and g7.abi.PATHS[p.path] == path
        _check("bf16", M, N, K, 23, inputs.INT3, exact=True, route="tensor_cores")


def test_bf16_small_m_normal_values():
    _check("bf16", 24, 3000, 4096, 19, inputs.NORMAL, inputs.NORMAL_W)


@pytest.mark.parametrize("shape", [(129, 1, 64), (300, 16, 1000), (1000, 64, 3001),
                                   (1000, 65, 777), (3001, 127, 3001), (3001, 127, 1000),
                                   (4096, 128, 4096), (2048, 96, 4096), (20000, 100, 200),
                                   (257, 128, 8192), (700, 33, 1)])
@pytest.mark.parametrize("route", ROUTES)
def test_bf16_narrow_n_paths_exact(shape, route):
    # N <= 128 < M on the narrow-N kernel: both MMA widths (64, 128), ragged
    # M (a partial 128-row tile), N and K, copied operands (127, 3001), a K
    # split of up to 8 per cluster, more tiles than SMs (no split), K below
    # one slice; and the same shapes on the CUDA-core path where they are
    # small
    M, N, K = shape
    with route_limit(route):
        s, plan = g7.plan("bf16", M, N, K)
    if route == "tensor_cores":
        assert _abi.PATHS[plan.path] == "bf16_narrow"
    _check("bf16", M, N, K, 21, inputs.INT3, exact=True, route=route)


@pytest.mark.parametrize("shape", [(512, 1024, 8192), (512, 512, 4096), (256, 1024, 4096),
                                   (1000, 1000, 3001), (129, 4096, 4096), (4096, 136, 4096),
                                   (300, 1000, 3001), (1023, 1025, 1536), (700, 1300, 6200)])
def test_bf16_few_tiles_long_k_exact(shape):
    # M, N > 128 with at most half as many 128 x 128 tiles as SMs and a long
    # K run on the narrow-N kernel as 128 x 128 tiles, K split over clusters
    # (ragged M, N and K, copied A, a last column tile of 8 columns)
    M, N, K = shape
    s, p = g7.plan("bf16", M, N, K)
    assert s == 0 and g7.abi.PATHS[p.path] == "bf16_narrow" and p.tile_n == 128
    _check("bf16", M, N, K, 34, inputs.INT3, exact=True)


def test_bf16_few_tiles_normal_values():
    _check("bf16", 700, 900, 4000, 35, inputs.NORMAL)


def test_bf16_narrow_n_normal_values_and_bits():
    # N(0,1) inputs within the BF16 bound; the split's partial sums are added
    # in rank order, so repeated calls give the same bits
    a, b = inputs.make_pair(3000, 96, 4096, 22, inputs.NORMAL, inputs.NORMAL_W,
                            dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    first = g7.gemm_bf16_f32acc(a_d, b_d).clone()
    for _ in range(3):
        again = g7.gemm_bf16_f32acc(a_d, b_d)
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    c_ref, s_ref = oracle_ref("bf16", a, b)
    assert_within("bf16", first.cpu().numpy(), c_ref, s_ref)
    assert g7.gemm_get_device_status() == 0


# ------------------------------------------------------------- edge cases

@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_zero_k_writes_zeros(kind):
    buf, c = guarded_output(37, 45, 50, DEV)
    a = torch.empty((37, 0), dtype=_dtype(kind), device=DEV)
    b = torch.empty((0, 45), dtype=_dtype(kind), device=DEV)
    (g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc)(a, b, out=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)
    assert_guards_intact(buf, 37, 45, 50)


@pytest.mark.parametrize("kind,M,N,K,route", [
    ("f32", 300, 260, 200, "default"), ("f32", 700, 900, 1000, "default"),
    ("bf16", 520, 600, 448, "tensor_cores"), ("bf16", 16, 1200, 448, "tensor_cores"),
    ("bf16", 1000, 100, 1200, "tensor_cores"), ("bf16", 200, 300, 150, "default")])
def test_non_finite_inputs_propagate(kind, M, N, K, route):
    # A NaN in A[i0, k0] and +Inf in B[k1, j1] (k1 != k0): row i0 of C is NaN
    # (NaN times anything), column j1 is not finite (+-Inf, or NaN where
    # A[i, k1] = 0), and every other element is finite and exact, as the
    # two entries do not enter it
    a, b = inputs.make_pair(M, N, K, 25, inputs.INT3, dtype=_dtype(kind))
    i0, k0, k1, j1 = M // 2, K // 3, (2 * K) // 3, N - 1
    a_bad, b_bad = a.clone(), b.clone()
    a_bad[i0, k0] = float("nan")
    b_bad[k1, j1] = float("inf")
    with route_limit(route):
        c = _run(kind, a_bad, b_bad).cpu().numpy()
    assert np.all(np.isnan(c[i0])), "row of the NaN"
    assert not np.any(np.isfinite(c[:, j1])), "column of the Inf"
    c_ref, _ = oracle_ref(kind, a, b, with_abs=False)
    keep = np.ones((M, N), dtype=bool)
    keep[i0] = False
    keep[:, j1] = False
    assert np.all(np.isfinite(c[keep]))
    assert np.array_equal(c[keep].astype(np.float64), c_ref[keep])
    assert g7.gemm_get_device_status() == 0


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_empty_m_or_n_is_noop(kind):
    buf, c = guarded_output(0, 5, 8, DEV)
    a = torch.ones((0, 3), dtype=_dtype(kind), device=DEV)
    b = torch.ones((3, 5), dtype=_dtype(kind), device=DEV)
    (g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc)(a, b, out=c)
    torch.cuda.synchronize()
    assert_guards_intact(buf, 0, 5, 8)


@pytest.mark.parametrize("kind,route", [("f32", "default"), ("bf16", "default"),
                                        ("bf16", "tensor_cores")])
@pytest.mark.parametrize("shape", [(129, 257, 70), (300, 600, 200)])
def test_guard_bands_untouched(kind, route, shape):
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 9, inputs.INT3, dtype=_dtype(kind))
    ldc = N + 7
    buf, c = guarded_output(M, N, ldc, DEV)
    with route_limit(route):
        (g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc)(a.to(DEV), b.to(DEV), out=c)
        torch.cuda.synchronize()
    assert_guards_intact(buf, M, N, ldc)
    c_ref, s_ref = oracle_ref(kind, a, b)
    assert_within(kind, c.cpu().numpy(), c_ref, s_ref, exact=True)


@pytest.mark.parametrize("shape,schedule,route", [
    ((2048, 2561, 320), g7.abi.SCHEDULE_AUTO, "default"),      # 88 tiles: half-width tail units
    ((2560, 2302, 640), g7.abi.SCHEDULE_STREAM_K, "default"),  # partial sums combined on the way out
    ((300, 258, 200), g7.abi.SCHEDULE_AUTO, "tensor_cores"),
    ((1000, 127, 127), g7.abi.SCHEDULE_AUTO, "tensor_cores"),
    ((300, 258, 200), g7.abi.SCHEDULE_AUTO, "default"),        # small-problem path
    ((1000, 127, 127), g7.abi.SCHEDULE_AUTO, "default")])
def test_bf16_row_store_epilogue_guarded(shape, schedule, route):
    # a row stride that is not a multiple of 16 bytes: C is written through
    # the staging boxes with ordinary row stores (no TMA store), and nothing
    # outside [0, M) x [0, N) may change
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 29, inputs.INT3, dtype=torch.bfloat16)
    ldc = N + 1 if (N + 1) % 4 else N + 2
    buf, c = guarded_output(M, N, ldc, DEV)
    prev = g7.abi.gemm_set_bf16_schedule(schedule)
    try:
        with route_limit(route):
            g7.gemm_bf16_f32acc(a.to(DEV), b.to(DEV), out=c)
            torch.cuda.synchronize()
    finally:
        g7.abi.gemm_set_bf16_schedule(prev)
    assert g7.gemm_get_device_status() == 0
    assert_guards_intact(buf, M, N, ldc)
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


@pytest.mark.parametrize("kind,route", [("f32", "default"), ("bf16", "default"),
                                        ("bf16", "tensor_cores")])
def test_leading_dims_and_misaligned_bases(kind, route):
    M, N, K = 150, 270, 90
    a, b = inputs.make_pair(M, N, K, 12, inputs.INT3, dtype=_dtype(kind))
    # operands placed at odd element offsets inside wider rows
    a_buf = torch.zeros((M, K + 11), dtype=a.dtype, device=DEV)
    b_buf = torch.zeros((K, N + 13), dtype=b.dtype, device=DEV)
    a_buf[:, 1:K + 1] = a.to(DEV)
    b_buf[:, 3:N + 3] = b.to(DEV)
    a_v, b_v = a_buf[:, 1:K + 1], b_buf[:, 3:N + 3]
    assert a_v.stride(0) == K + 11 and b_v.stride(0) == N + 13
    with route_limit(route):
        c = (g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc)(a_v, b_v)
        torch.cuda.synchronize()
        if kind == "bf16":
            # read in place by the small-problem kernel, copied first for
            # the tensor-core kernels
            s, p = g7.plan("bf16", M, N, K, a_v.data_ptr(), a_v.stride(0),
                           b_v.data_ptr(), b_v.stride(0), c.data_ptr(), N)
            if route == "default":
                assert g7.abi.PATHS[p.path] == "bf16_small" and not p.pack_a and not p.pack_b
            else:
                assert g7.abi.PATHS[p.path] == "bf16_packed" and p.pack_a and p.pack_b
    c_ref, s_ref = oracle_ref(kind, a, b)
    assert_within(kind, c.cpu().numpy(), c_ref, s_ref, exact=True)


@pytest.mark.parametrize("a_off,b_off", [(1, 0), (0, 3), (8, 8)])
def test_bf16_vector_times_matrix_misaligned_bases(a_off, b_off):
    # M = 1 with A and/or B at element offsets: a base off 16 bytes is
    # copied first; an aligned A with any stride is read in place
    M, N, K = 1, 2000, 1000
    a, b = inputs.make_pair(M, N, K, 14, inputs.INT3, dtype=torch.bfloat16)
    a_buf = torch.zeros((M, K + 16), dtype=a.dtype, device=DEV)
    b_buf = torch.zeros((K, N + 16), dtype=b.dtype, device=DEV)
    a_buf[:, a_off:K + a_off] = a.to(DEV)
    b_buf[:, b_off:N + b_off] = b.to(DEV)
    a_v, b_v = a_buf[:, a_off:K + a_off], b_buf[:, b_off:N + b_off]
    s, p = g7.plan("bf16", M, N, K, a_v.data_ptr(), a_v.stride(0),
                   b_v.data_ptr(), b_v.stride(0), 16, N)
    assert g7.abi.PATHS[p.path] == "bf16_skinny"
    assert (p.pack_a, p.pack_b) == (a_off % 8 != 0, b_off % 8 != 0)
    c = g7.gemm_bf16_f32acc(a_v, b_v)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_deterministic_bits(kind):
    a, b = inputs.make_pair(512, 768, 1000, 13, inputs.NORMAL, dtype=_dtype(kind))
    a_d, b_d = a.to(DEV), b.to(DEV)
    fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
    first = fn(a_d, b_d).clone()
    for _ in range(10):
        again = fn(a_d, b_d)
        assert torch.equal(again.view(torch.int32), first.view(torch.int32))


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_host_buffer_variant_matches_device(kind):
    a, b = inputs.make_pair(333, 444, 555, 14, inputs.NORMAL, dtype=_dtype(kind))
    dev_fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
    host_fn = g7.gemm_f32_host if kind == "f32" else g7.gemm_bf16_f32acc_host
    c_dev = dev_fn(a.to(DEV), b.to(DEV)).cpu()
    c_host = host_fn(a.pin_memory(), b.pin_memory())
    assert c_host.device.type == "cpu"
    assert torch.equal(c_host.view(torch.int32), c_dev.view(torch.int32))


@pytest.mark.parametrize("kind,shape", [("f32", (2048, 300, 700)), ("bf16", (2048, 520, 333)),
                                        ("bf16", (3000, 1000, 1000))])
def test_host_buffer_variant_in_row_blocks_exact(kind, shape):
    # large enough that the host variant overlaps copies with per-block GEMMs
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 22, inputs.INT3, dtype=_dtype(kind))
    host_fn = g7.gemm_f32_host if kind == "f32" else g7.gemm_bf16_f32acc_host
    c = host_fn(a.pin_memory(), b.pin_memory())
    c_ref, _ = oracle_ref(kind, a, b, with_abs=False)
    assert_within(kind, c.numpy(), c_ref, None, exact=True)
    # a strided host C: rows ldc apart, padding untouched
    ldc = N + 3
    buf = torch.full((M, ldc), -7.0).pin_memory()
    host_fn(a.pin_memory(), b.pin_memory(), out=buf[:, :N])
    assert torch.all(buf[:, N:] == -7.0)
    assert_within(kind, buf[:, :N].numpy(), c_ref, None, exact=True)


@pytest.mark.parametrize("kind,shape", [("f32", (2048, 300, 2100)), ("f32", (2100, 256, 4099)),
                                        ("bf16", (2048, 256, 4099))])
def test_host_buffer_variant_k_pieces(kind, shape):
    # several row blocks and a long K: B and the first block of A go up in
    # pieces along K and the first block accumulates piece by piece
    # (K = 4099: ragged last piece and odd row strides)
    M, N, K = shape
    host_fn = g7.gemm_f32_host if kind == "f32" else g7.gemm_bf16_f32acc_host
    a, b = inputs.make_pair(M, N, K, 29, inputs.INT3, dtype=_dtype(kind))
    c = host_fn(a.pin_memory(), b.pin_memory())
    c_ref, _ = oracle_ref(kind, a, b, with_abs=False)
    assert_within(kind, c.numpy(), c_ref, None, exact=True)
    # general values: the piecewise sums stay within the FP32 bound
    a, b = inputs.make_pair(M, N, K, 30, inputs.NORMAL if kind == "bf16" else inputs.UNIFORM,
                            dtype=_dtype(kind))
    c = host_fn(a.pin_memory(), b.pin_memory())
    c_ref, s_ref = oracle_ref(kind, a, b)
    assert_within(kind, c.numpy(), c_ref, s_ref)
    assert g7.gemm_get_device_status() == 0


@pytest.mark.parametrize("shape", [(4096, 2048, 2304), (4096, 2048, 640)])
def test_f32_host_whole_wave_head_block(shape):
    # FP32 host variant with a head block of whole waves: 2432 rows (19 tile
    # rows x 16 tile columns = two waves of 304 resident blocks), then the
    # other 1664 rows; with K = 2304 the head block goes up and accumulates
    # in four K pieces
    M, N, K = shape
    a, b = inputs.make_pair(M, N, K, 31, inputs.INT4, dtype=torch.float32)
    c = g7.gemm_f32_host(a.pin_memory(), b.pin_memory())
    c_ref, _ = oracle_ref("f32", a, b, with_abs=False)
    assert_within("f32", c.numpy(), c_ref, None, exact=True)
    assert g7.gemm_get_device_status() == 0


def test_streams_are_respected():
    a, b = inputs.make_pair(1024, 1024, 1024, 15, inputs.INT3, dtype=torch.bfloat16)
    s = torch.cuda.Stream()
    a_d, b_d = a.to(DEV), b.to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        c = g7.gemm_bf16_f32acc(a_d, b_d)
    s.synchronize()
    c_ref, s_ref = oracle_ref("bf16", a, b)
    assert_within("bf16", c.cpu().numpy(), c_ref, s_ref, exact=True)


@pytest.mark.parametrize("kind,M,N,K,route", [
    ("bf16", 4096, 1024, 4096, "default"),        # paired SMs, operands read in place
    ("bf16", 3001, 1000, 1001, "default"),        # operand copy kernel first
    ("bf16", 16, 4096, 4096, "default"),          # small M
    ("bf16", 4096, 100, 4096, "default"),         # narrow N
    ("bf16", 300, 258, 200, "default"),           # small problem, CUDA cores
    ("f32", 2048, 2048, 2048, "default"), ("f32", 256, 256, 256, "default")])
def test_reads_wait_for_the_previous_kernel(kind, M, N, K, route):
    # Every kernel is launched as a programmatic dependent of the one before
    # it and may start early: it must not read A or B before that kernel has
    # finished.  Here the kernels just before the GEMM overwrite A and B
    # (zeros before), queued behind a spin so the GEMM is launched while they
    # run; the result must be that of the new operands.
    dtype = _dtype(kind)
    a, b = inputs.make_pair(M, N, K, 26, inputs.INT3, dtype=dtype)
    a_new, b_new = a.to(DEV), b.to(DEV)
    a_d = torch.zeros_like(a_new)
    b_d = torch.zeros_like(b_new)
    torch.cuda.synchronize()
    with route_limit(route):
        torch.cuda._sleep(2_000_000)
        a_d.copy_(a_new)
        b_d.copy_(b_new)
        c = (g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc)(a_d, b_d)
        torch.cuda.synchronize()
    c_ref, _ = oracle_ref(kind, a, b, with_abs=False)
    assert_within(kind, c.cpu().numpy(), c_ref, None, exact=True)
    assert g7.gemm_get_device_status() == 0


def test_chained_gemms_read_the_previous_result():
    # Back-to-back launches of the library on one stream, each reading what
    # the one before wrote: FP32 C1 = A.B (128 x 128 blocks) feeds
    # C2 = C1.D (small-problem tiles); BF16 C = A1.B1 on SM pairs, then
    # C += A2.B2 (beta = 1) on SM pairs, then on the narrow-N kernel for its
    # first 100 columns.  Integer values keep every sum exact.
    a, b = inputs.make_pair(512, 520, 64, 27, inputs.INT3, dtype=torch.float32)
    d = torch.randint(-3, 4, (520, 256), generator=torch.Generator().manual_seed(28)).float()
    c1 = g7.gemm_f32(a.to(DEV), b.to(DEV))
    c2 = g7.gemm_f32(c1, d.to(DEV))
    torch.cuda.synchronize()
    ab, _ = oracle_ref("f32", a, b, with_abs=False)
    # C1's values are integers below 2^24: exact in FP32
    want, _ = oracle_ref("f32", torch.from_numpy(ab.astype(np.float32)), d, with_abs=False)
    assert np.array_equal(c2.cpu().numpy().astype(np.float64), want)

    M, N = 1000, 1000
    a1, b1 = inputs.make_pair(M, N, 512, 29, inputs.INT3, dtype=torch.bfloat16)
    a2, b2 = inputs.make_pair(M, N, 256, 30, inputs.INT3, dtype=torch.bfloat16)
    a3, b3 = inputs.make_pair(M, 100, 192, 32, inputs.INT3, dtype=torch.bfloat16)
    c = torch.empty((M, N), dtype=torch.float32, device=DEV)
    with route_limit("tensor_cores"):
        g7.gemm_bf16_f32acc(a1.to(DEV), b1.to(DEV), out=c)
        g7.gemm_bf16_f32acc_ex(a2.to(DEV), b2.to(DEV), out=c, beta=1.0)
        g7.gemm_bf16_f32acc_ex(a3.to(DEV), b3.to(DEV), out=c[:, :100], beta=1.0)
        torch.cuda.synchronize()
    want = oracle_ref("bf16", a1, b1, with_abs=False)[0] + \
        oracle_ref("bf16", a2, b2, with_abs=False)[0]
    want[:, :100] += oracle_ref("bf16", a3, b3, with_abs=False)[0]
    assert np.array_equal(c.cpu().numpy().astype(np.float64), want)
    assert g7.gemm_get_device_status() == 0


def test_invalid_arguments_rejected_before_launch():
    a = torch.ones((4, 8), dtype=torch.bfloat16, device=DEV)
    b = torch.ones((8, 4), dtype=torch.bfloat16, device=DEV)
    c = torch.zeros((4, 4), dtype=torch.float32, device=DEV)
    st = torch.cuda.current_stream().cuda_stream
    assert g7.abi.gemm_bf16_f32acc(4, 4, 8, a.data_ptr(), 7, b.data_ptr(), 4,
                                   c.data_ptr(), 4, st) == g7.abi.GEMM_ERR_INVALID_ARG
    assert g7.abi.gemm_f32(-1, 4, 8, a.data_ptr(), 8, b.data_ptr(), 4,
                           c.data_ptr(), 4, st) == g7.abi.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(c == 0)


def test_bf16_stream_k_in_cuda_graph_replays_exact(stream_k):
    # A captured stream-K launch replays with the same launch tag; the
    # finishing warps leave the synchronisation words clean, so every replay
    # is exact.
    M, N, K = 2560, 2304, 1024
    a, b = inputs.make_pair(M, N, K, 33, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    c = torch.empty((M, N), dtype=torch.float32, device=DEV)
    g7.gemm_bf16_f32acc(a_d, b_d, out=c)      # warm-up: scratch and tensor maps
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g7.gemm_bf16_f32acc(a_d, b_d, out=c)
    torch.cuda.current_stream().wait_stream(s)
    for r in range(3):
        # new operand values each replay: stale partial sums or tickets from
        # the previous replay would show
        a_r, _ = inputs.make_pair(M, N, K, 34 + r, inputs.INT3, dtype=torch.bfloat16)
        a_d.copy_(a_r.to(DEV))
        c.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g7.gemm_get_device_status() == 0
        c_ref, _ = oracle_ref("bf16", a_r, b, with_abs=False)
        assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


@pytest.mark.parametrize("case", ["f32_split_k", "bf16_stream_k", "bf16_packed",
                                  "bf16_m1_packed", "bf16_narrow", "bf16_small"])
def test_capture_on_fresh_stream_then_replay(case):
    # Captured on a stream the library has never seen: its scratch is then
    # allocated inside the graph (owned by it) rather than kept, and every
    # replay on new operand values is exact.
    kind = "f32" if case.startswith("f32") else "bf16"
    M, N, K = {"f32_split_k": (2560, 2048, 640), "bf16_stream_k": (2560, 2304, 1024),
               "bf16_packed": (1000, 600, 1333), "bf16_m1_packed": (1, 3001, 1000),
               "bf16_narrow": (3001, 100, 1000),
               "bf16_small": (300, 258, 200)}[case]
    dtype = _dtype(kind)
    fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
    a, b = inputs.make_pair(M, N, K, 35, inputs.INT3, dtype=dtype)
    a_d, b_d = a.to(DEV), b.to(DEV)
    c = torch.empty((M, N), dtype=torch.float32, device=DEV)
    prev = g7.abi.gemm_set_bf16_schedule(
        g7.abi.SCHEDULE_STREAM_K if case == "bf16_stream_k" else g7.abi.SCHEDULE_AUTO)
    want = {"bf16_packed": "bf16_packed", "bf16_m1_packed": "bf16_skinny",
            "bf16_narrow": "bf16_narrow", "bf16_small": "bf16_small",
            "bf16_stream_k": "bf16_tma", "f32_split_k": "f32_simt"}[case]
    assert g7.abi.PATHS[g7.plan(kind, M, N, K)[1].path] == want
    try:
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                fn(a_d, b_d, out=c)
        torch.cuda.current_stream().wait_stream(s)
        for r in range(2):
            a_r, _ = inputs.make_pair(M, N, K, 36 + r, inputs.INT3, dtype=dtype)
            a_d.copy_(a_r.to(DEV))
            c.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert g7.gemm_get_device_status() == 0
            c_ref, _ = oracle_ref(kind, a_r, b, with_abs=False)
            assert_within(kind, c.cpu().numpy(), c_ref, None, exact=True)
        del graph
    finally:
        g7.abi.gemm_set_bf16_schedule(prev)


# ------------------------------------------- BF16 small problems (CUDA cores)

@pytest.mark.parametrize("shape", [(127, 127, 127), (2, 8, 8), (3001, 127, 127),
                                   (127, 3001, 127), (1000, 500, 127), (64, 64, 4001),
                                   (65, 63, 33), (5, 50, 1), (256, 256, 256)])
def test_bf16_small_problem_path_normal_values(shape):
    # general values: every element within the BF16 bound, on the path that
    # reads operands in place and splits K over the SMs
    M, N, K = shape
    s, plan = g7.plan("bf16", M, N, K)
    assert _abi.PATHS[plan.path] == "bf16_small"
    _check("bf16", M, N, K, 41, inputs.NORMAL)


def test_bf16_small_problem_deterministic_bits():
    # the K ranges are added in a fixed order by whichever block finishes
    # last, so repeated calls give the same bits
    a, b = inputs.make_pair(200, 300, 500, 42, inputs.NORMAL, dtype=torch.bfloat16)
    s, plan = g7.plan("bf16", 200, 300, 500)
    assert _abi.PATHS[plan.path] == "bf16_small" and plan.split_k > 1
    a_d, b_d = a.to(DEV), b.to(DEV)
    first = g7.gemm_bf16_f32acc(a_d, b_d).clone()
    for _ in range(5):
        assert torch.equal(g7.gemm_bf16_f32acc(a_d, b_d).view(torch.int32),
                           first.view(torch.int32))
    c_ref, s_ref = oracle_ref("bf16", a, b)
    assert_within("bf16", first.cpu().numpy(), c_ref, s_ref)


def test_bf16_small_problem_odd_strides_and_offsets_read_in_place():
    # rows of odd length at odd element offsets in every operand, C at an
    # odd offset too: nothing is copied, nothing outside C changes
    M, N, K = 77, 91, 133
    a, b = inputs.make_pair(M, N, K, 43, inputs.INT3, dtype=torch.bfloat16)
    a_buf = torch.zeros((M, K + 5), dtype=a.dtype, device=DEV)
    b_buf = torch.zeros((K, N + 3), dtype=b.dtype, device=DEV)
    a_buf[:, 1:K + 1] = a.to(DEV)
    b_buf[:, 2:N + 2] = b.to(DEV)
    a_v, b_v = a_buf[:, 1:K + 1], b_buf[:, 2:N + 2]
    ldc = N + 3
    buf, c = guarded_output(M, N, ldc, DEV)
    s, p = g7.plan("bf16", M, N, K, a_v.data_ptr(), a_v.stride(0),
                   b_v.data_ptr(), b_v.stride(0), c.data_ptr(), ldc)
    assert _abi.PATHS[p.path] == "bf16_small" and not p.pack_a and not p.pack_b
    g7.gemm_bf16_f32acc(a_v, b_v, out=c)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    assert_guards_intact(buf, M, N, ldc)
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)
