"""Helpers shared by the GPU parity tests: run a GEMM through the C ABI on
seeded inputs and compare it with the oracle.

Acceptance (the stated bounds, elementwise, against the FP64 oracle run on
exactly the inputs the GPU saw):
  * FP32 path:            |C - C_ref| <= 1e-5 * S + 1e-7
  * BF16 -> FP32 path:    |C - C_ref| <= 4e-3 * S + 1e-6
  * integer-valued inputs: C == C_ref exactly (every partial sum is an
    integer below 2^24, so any summation order is exact in FP32)
where S[i][j] = sum_k |A[i][k] * B[k][j]| comes from the oracle as well.
"""
from __future__ import annotations

import contextlib

import numpy as np
import torch

import oracle
from dense_gemm_07_gb300 import inputs

RTOL = {"f32": 1e-5, "bf16": 4e-3}
ATOL = {"f32": 1e-7, "bf16": 1e-6}

SENTINEL_BITS = 0x7FC0DEAD  # a NaN payload no GEMM result can produce


def oracle_ref(kind, a_cpu, b_cpu, rows=None, with_abs=True):
    """Oracle result (C_ref, S) for all rows, or for the listed rows only;
    S is None when with_abs is False."""
    if rows is not None:
        a_cpu = a_cpu[rows]
    if kind == "f32":
        r = oracle.gemm_f32(a_cpu.contiguous().numpy(), b_cpu.contiguous().numpy(),
                            with_abs=with_abs)
    else:
        r = oracle.gemm_bf16(inputs.bf16_bits(a_cpu.contiguous()),
                             inputs.bf16_bits(b_cpu.contiguous()), with_abs=with_abs)
    return r if with_abs else (r, None)


def assert_within(kind, c_gpu, c_ref, s_ref, exact=False, what=""):
    c = np.asarray(c_gpu, dtype=np.float64)
    assert c.shape == c_ref.shape, (c.shape, c_ref.shape)
    assert np.all(np.isfinite(c)), f"{what}: non-finite output"
    if exact:
        bad = np.argwhere(c != c_ref)
        assert bad.size == 0, (f"{what}: {len(bad)} mismatches, first at "
                               f"{tuple(bad[0])}: {c[tuple(bad[0])]} vs {c_ref[tuple(bad[0])]}")
        return
    err = np.abs(c - c_ref)
    lim = RTOL[kind] * s_ref + ATOL[kind]
    bad = np.argwhere(err > lim)
    assert bad.size == 0, (f"{what}: {len(bad)} elements outside the bound, first at "
                           f"{tuple(bad[0])}: err {err[tuple(bad[0])]:.3e} > {lim[tuple(bad[0])]:.3e}")


def guarded_output(M, N, ldc, device):
    """C with one guard row above and below and ldc-N guard columns, all set
    to a sentinel NaN; returns (buffer, C view)."""
    buf = torch.empty((M + 2) * ldc, dtype=torch.int32, device=device)
    buf.fill_(SENTINEL_BITS - (1 << 32) if SENTINEL_BITS >= 1 << 31 else SENTINEL_BITS)
    full = buf.view(torch.float32).view(M + 2, ldc)
    return buf, full[1:M + 1, :N]


def assert_guards_intact(buf, M, N, ldc):
    bits = buf.view(M + 2, ldc).cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    assert np.all(bits[0] == SENTINEL_BITS), "row above C written"
    assert np.all(bits[M + 1] == SENTINEL_BITS), "row below C written"
    assert np.all(bits[1:M + 1, N:] == SENTINEL_BITS), "padding columns written"


@contextlib.contextmanager
def small_limit(max_macs):
    """BF16 calls inside the block take the CUDA-core small-problem path
    only up to max_macs multiply-adds (0: always the tensor-core kernels)."""
    from dense_gemm_07_gb300 import _abi
    prev = _abi.gemm_set_bf16_small_limit(max_macs)
    try:
        yield
    finally:
        _abi.gemm_set_bf16_small_limit(prev)


# Routes for BF16 shapes under the small-problem limit: the default (the
# CUDA-core small-problem kernel) and the tensor-core kernels.
ROUTES = ("default", "tensor_cores")


def route_limit(route):
    return small_limit(0) if route == "tensor_cores" else contextlib.nullcontext()
