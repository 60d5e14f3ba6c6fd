"""The fused epilogue C := act(alpha * A@B + beta * C + bias) on every path,
against the oracle's epilogue step applied to its exact product.

Bound: |C - C_ref| <= rtol * (|alpha| * S + |beta * C0| + |bias|) + atol, the
product's bound scaled by alpha plus one rounding of the added terms; with
integer-valued operands, alpha, beta and bias the result is exact."""
import numpy as np
import pytest
import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import _abi, inputs
import oracle
from gemm_check import ATOL, RTOL, oracle_ref, route_limit

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(kind, M, N, K, seed, alpha, beta, use_bias, act, exact, dist,
          schedule=None, route="default"):
    dtype = torch.float32 if kind == "f32" else torch.bfloat16
    a, b = inputs.make_pair(M, N, K, seed, dist, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 1000)
    c0 = torch.randint(-5, 6, (M, N), generator=g).float()
    bias = torch.randint(-4, 5, (N,), generator=g).float() if use_bias else None
    out = c0.to(DEV).clone()
    fn = g7.gemm_f32_ex if kind == "f32" else g7.gemm_bf16_f32acc_ex
    prev = _abi.gemm_set_bf16_schedule(schedule) if schedule is not None else None
    try:
        with route_limit(route):
            fn(a.to(DEV), b.to(DEV), out=out, alpha=alpha, beta=beta,
               bias=bias.to(DEV) if bias is not None else None, activation=act)
            torch.cuda.synchronize()
    finally:
        if prev is not None:
            _abi.gemm_set_bf16_schedule(prev)
    assert g7.gemm_get_device_status() == 0
    ab, s = oracle_ref(kind, a, b)
    want = oracle.gemm_epilogue(ab, alpha=alpha, beta=beta,
                                C0=c0.numpy() if beta != 0 else None,
                                bias=bias.numpy() if bias is not None else None,
                                act=1 if act == "relu" else 0)
    got = out.cpu().numpy().astype(np.float64)
    if exact:
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{len(bad)} mismatches, first {tuple(bad[0])}"
    else:
        scale = abs(alpha) * s + abs(beta) * np.abs(c0.numpy()) + \
            (np.abs(bias.numpy())[None, :] if bias is not None else 0)
        err = np.abs(got - want)
        lim = RTOL[kind] * scale + ATOL[kind]
        assert np.all(err <= lim), float(np.max(err - lim))


TC = "tensor_cores"
PATHS = [
    ("bf16", 512, 768, 320, None, TC),   # SM pairs, TMA-store epilogue
    ("bf16", 300, 258, 200, None, TC),   # SM pairs, N % 4 != 0: row stores
    ("bf16", 2048, 2561, 320, None, TC),  # half-width tail units, row stores
    ("bf16", 2560, 2304, 512, _abi.SCHEDULE_STREAM_K, TC),  # stream-K + TMA stores
    ("bf16", 2560, 2302, 512, _abi.SCHEDULE_STREAM_K, TC),  # stream-K + row stores
    ("bf16", 1280, 1024, 4096, None, TC),  # tiles halved along K; alpha-only: finished in C
    ("bf16", 512, 1024, 8192, None, TC),   # few tiles, long K: 128 x 128 tiles, K split
    ("bf16", 2560, 2048, 4096, _abi.SCHEDULE_STREAM_K, TC),  # stream-K over every tile
    ("bf16", 48, 1000, 777, None, TC),   # small M, cluster reduction
    ("bf16", 1, 4096, 4096, None, TC),   # M = 1 on the small-M kernel, K split
    ("bf16", 1, 1000, 40, None, TC),     # M = 1, one k-slice: no split
    ("bf16", 1000, 100, 777, None, TC),  # narrow N (MMA N = 128), cluster reduction
    ("bf16", 3001, 64, 2000, None, TC),  # narrow N (MMA N = 64), rows of A copied
    ("bf16", 300, 258, 200, None, "default"),   # small problem on the CUDA cores, split K
    ("bf16", 2000, 500, 60, None, "default"),   # small problem, no split: finished in place
    ("f32", 200, 190, 300, None, "default"),    # FP32 small problem: 64 x 64 tiles split along K
    ("f32", 640, 520, 2000, None, "default"),   # FP32, one partial wave split along K
    ("f32", 2560, 2048, 640, None, "default"),  # FP32, whole waves + split tail
]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: f"{p[0]}-{p[1]}x{p[2]}x{p[3]}-{p[5]}")
@pytest.mark.parametrize("epi", [(2.0, -1.0, True, "none"), (1.0, 0.0, True, "relu"),
                                 (-3.0, 2.0, False, "relu"), (0.5, 0.0, False, "none"),
                                 (0.0, 1.0, True, "none")],
                         ids=["ab+c+bias", "bias+relu", "beta_relu", "alpha_only",
                              "no_product"])
def test_epilogue_exact_integers(path, epi):
    kind, M, N, K, schedule, route = path
    alpha, beta, use_bias, act = epi
    _case(kind, M, N, K, 50, alpha, beta, use_bias, act, exact=True,
          dist=inputs.INT3, schedule=schedule, route=route)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_epilogue_general_values(kind):
    _case(kind, 700, 900, 1000, 51, 0.75, -1.25, True, "none", exact=False,
          dist=inputs.NORMAL if kind == "bf16" else inputs.UNIFORM)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_epilogue_with_zero_k(kind):
    _case(kind, 33, 45, 0, 52, 2.0, 3.0, True, "relu", exact=True, dist=inputs.INT3)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_identity_epilogue_equals_plain_entry_point_bitwise(kind):
    dtype = torch.float32 if kind == "f32" else torch.bfloat16
    a, b = inputs.make_pair(600, 500, 300, 53, inputs.NORMAL, dtype=dtype)
    a, b = a.to(DEV), b.to(DEV)
    plain = (g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc)(a, b)
    ex = (g7.gemm_f32_ex if kind == "f32" else g7.gemm_bf16_f32acc_ex)(a, b)
    assert torch.equal(plain.view(torch.int32), ex.view(torch.int32))


def test_beta_zero_does_not_read_c():
    a, b = inputs.make_pair(300, 260, 100, 54, inputs.INT3, dtype=torch.bfloat16)
    out = torch.full((300, 260), float("nan"), device=DEV)
    g7.gemm_bf16_f32acc_ex(a.to(DEV), b.to(DEV), out=out, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()


def test_unknown_activation_rejected():
    epi = _abi.GemmEpilogue(1.0, 0.0, None, 5)
    a = torch.ones((4, 4), device=DEV)
    c = torch.zeros((4, 4), device=DEV)
    st = torch.cuda.current_stream().cuda_stream
    assert _abi.gemm_f32_ex(4, 4, 4, a.data_ptr(), 4, a.data_ptr(), 4, c.data_ptr(), 4,
                            epi, st) == _abi.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("kind,M,N,K,schedule,route", [
    ("f32", 700, 900, 1000, None, "default"), ("f32", 200, 190, 300, None, "default"),
    ("bf16", 700, 900, 1000, None, "default"), ("bf16", 300, 258, 200, None, TC),
    ("bf16", 48, 1000, 777, None, TC), ("bf16", 1, 3000, 3001, None, "default"),
    ("bf16", 2560, 2304, 512, _abi.SCHEDULE_STREAM_K, "default"),
    ("bf16", 300, 258, 200, None, "default"), ("bf16", 48, 500, 777, None, "default"),
    ("bf16", 2000, 100, 1000, None, TC)])
def test_epilogue_gelu(kind, M, N, K, schedule, route):
    # GELU after alpha, beta and the bias on every path.  Bound: GELU's slope
    # is at most 1.13, so the pre-activation bound grows by that factor; the
    # FP32 erff and the final products add a few units in the last place of
    # |v|.
    dtype = torch.float32 if kind == "f32" else torch.bfloat16
    dist = inputs.NORMAL if kind == "bf16" else inputs.UNIFORM
    a, b = inputs.make_pair(M, N, K, 52, dist, dtype=dtype)
    g = torch.Generator().manual_seed(1052)
    c0 = torch.randn((M, N), generator=g).float()
    bias = torch.randn((N,), generator=g).float()
    out = c0.to(DEV).clone()
    fn = g7.gemm_f32_ex if kind == "f32" else g7.gemm_bf16_f32acc_ex
    prev = _abi.gemm_set_bf16_schedule(schedule) if schedule is not None else None
    try:
        with route_limit(route):
            fn(a.to(DEV), b.to(DEV), out=out, alpha=0.5, beta=0.75, bias=bias.to(DEV),
               activation="gelu")
            torch.cuda.synchronize()
    finally:
        if prev is not None:
            _abi.gemm_set_bf16_schedule(prev)
    assert g7.gemm_get_device_status() == 0
    ab, s = oracle_ref(kind, a, b)
    pre = oracle.gemm_epilogue(ab, alpha=0.5, beta=0.75, C0=c0.numpy(), bias=bias.numpy())
    want = oracle.gemm_epilogue(ab, alpha=0.5, beta=0.75, C0=c0.numpy(), bias=bias.numpy(),
                                act=2)
    got = out.cpu().numpy().astype(np.float64)
    scale = 0.5 * s + 0.75 * np.abs(c0.numpy()) + np.abs(bias.numpy())[None, :]
    lim = 1.13 * (RTOL[kind] * scale + ATOL[kind]) + 1e-6 * np.abs(pre) + 1e-6
    err = np.abs(got - want)
    assert np.all(err <= lim), float(np.max(err - lim))


@pytest.mark.parametrize("epi", [(2.0, -1.0, True, "relu"), (1.0, 0.0, False, "none")],
                         ids=["workspace", "in_c"])
def test_epilogue_halved_after_whole_waves_sampled(epi):
    # 2560 x 2560 x 8192: one whole wave of 76 tiles, then the last 24 halved
    # along K over 48 pairs.  With beta, a bias and ReLU the halves meet in
    # the partial-sum workspace; the plain product adds them in C itself.
    # Sampled rows cover the halved tiles (rows 1024..2559).
    M, N, K = 2560, 2560, 8192
    alpha, beta, use_bias, act = epi
    a, b = inputs.make_pair(M, N, K, 56, inputs.INT3, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(1056)
    c0 = torch.randint(-5, 6, (M, N), generator=g).float()
    bias = torch.randint(-4, 5, (N,), generator=g).float() if use_bias else None
    out = c0.to(DEV).clone()
    g7.gemm_bf16_f32acc_ex(a.to(DEV), b.to(DEV), out=out, alpha=alpha, beta=beta,
                           bias=bias.to(DEV) if bias is not None else None,
                           activation=act)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    rows = np.unique(np.concatenate([np.arange(0, M, 211), np.arange(1024, 2048, 97),
                                     np.arange(2048, M, 41), [M - 1]]))
    ab, _ = oracle_ref("bf16", a, b, rows=rows, with_abs=False)
    want = oracle.gemm_epilogue(ab, alpha=alpha, beta=beta,
                                C0=c0.numpy()[rows] if beta != 0 else None,
                                bias=bias.numpy() if bias is not None else None,
                                act=1 if act == "relu" else 0)
    got = out.cpu().numpy().astype(np.float64)[rows]
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {tuple(bad[0])}"
