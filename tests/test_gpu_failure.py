"""Failure detection on the GPU without a fault: every mbarrier wait in the
tensor-core kernels is bounded.  The test hook makes a kernel withhold the
copy of its first k-slice (paired-SM kernel, small-M cluster kernel) or
first stage (M = 1 kernel), so a wait for it runs out (after a 20 ms limit);
the kernel must unwind and return, the host must read GEMM_ERR_TIMEOUT from
the device status word, and the context must stay usable: the next GEMM is
exact against the oracle and the status is clean again."""
import numpy as np
import pytest
import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import _abi, inputs
from gemm_check import assert_within, oracle_ref

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_gpu_stays_usable():
    M, N, K = 512, 768, 640           # paired-SM path, several tiles per pair
    a, b = inputs.make_pair(M, N, K, 31, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.cuda(), b.cuda()
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    assert _abi.gemm_debug_inject(1, 20_000_000) == _abi.GEMM_OK
    try:
        g7.gemm_bf16_f32acc(a_d, b_d)
        assert g7.gemm_get_device_status() == _abi.GEMM_ERR_TIMEOUT
        # the status word is cleared by reading it
        assert g7.gemm_get_device_status() == _abi.GEMM_OK
    finally:
        assert _abi.gemm_debug_inject(0, 0) == _abi.GEMM_OK
    c = g7.gemm_bf16_f32acc(a_d, b_d)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


def test_stream_k_timeout_then_next_launch_exact():
    # Stream-K schedule: the timed-out launch leaves its tickets and flags
    # half-counted; the next launch carries a new tag, so they read as zero
    # and its fix-up is exact.
    M, N, K = 2560, 2304, 512        # 90 tiles shared as k-slice runs by 76 pairs
    a, b = inputs.make_pair(M, N, K, 32, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.cuda(), b.cuda()
    prev = _abi.gemm_set_bf16_schedule(_abi.SCHEDULE_STREAM_K)
    try:
        s, plan = g7.plan("bf16", M, N, K)
        assert plan.sk_tiles > 0
        assert g7.gemm_get_device_status() == _abi.GEMM_OK
        assert _abi.gemm_debug_inject(1, 20_000_000) == _abi.GEMM_OK
        try:
            g7.gemm_bf16_f32acc(a_d, b_d)
            assert g7.gemm_get_device_status() == _abi.GEMM_ERR_TIMEOUT
        finally:
            assert _abi.gemm_debug_inject(0, 0) == _abi.GEMM_OK
        c = g7.gemm_bf16_f32acc(a_d, b_d)
        torch.cuda.synchronize()
        assert g7.gemm_get_device_status() == _abi.GEMM_OK
    finally:
        _abi.gemm_set_bf16_schedule(prev)
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


def test_vector_times_matrix_timeout_then_next_launch_exact():
    # M = 1 (on the small-M kernel): its first stage is withheld, the MMA
    # issuers' bounded waits run out, every cluster unwinds; the next launch
    # is exact.
    M, N, K = 1, 4096, 4096
    a, b = inputs.make_pair(M, N, K, 33, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.cuda(), b.cuda()
    s, plan = g7.plan("bf16", M, N, K)
    assert _abi.PATHS[plan.path] == "bf16_skinny" and plan.split_k > 1
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    assert _abi.gemm_debug_inject(1, 20_000_000) == _abi.GEMM_OK
    try:
        g7.gemm_bf16_f32acc(a_d, b_d)
        assert g7.gemm_get_device_status() == _abi.GEMM_ERR_TIMEOUT
    finally:
        assert _abi.gemm_debug_inject(0, 0) == _abi.GEMM_OK
    c = g7.gemm_bf16_f32acc(a_d, b_d)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


def test_narrow_n_cluster_timeout_then_next_launch_exact():
    # Narrow-N kernel: every CTA withholds its first k-slice, the MMA
    # issuers' bounded waits run out, every cluster unwinds and meets at its
    # final barrier; the next launch is exact.
    M, N, K = 4096, 128, 4096
    a, b = inputs.make_pair(M, N, K, 36, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.cuda(), b.cuda()
    s, plan = g7.plan("bf16", M, N, K)
    assert _abi.PATHS[plan.path] == "bf16_narrow" and plan.split_k > 1
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    assert _abi.gemm_debug_inject(1, 20_000_000) == _abi.GEMM_OK
    try:
        g7.gemm_bf16_f32acc(a_d, b_d)
        assert g7.gemm_get_device_status() == _abi.GEMM_ERR_TIMEOUT
    finally:
        assert _abi.gemm_debug_inject(0, 0) == _abi.GEMM_OK
    c = g7.gemm_bf16_f32acc(a_d, b_d)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)


@pytest.mark.parametrize("M", [16, 100])
def test_small_m_cluster_timeout_then_next_launch_exact(M):
    # Small-M kernel (clusters of CTAs splitting K): every CTA withholds its
    # first k-slice, the MMA issuers' bounded waits run out, all roles
    # unwind and each cluster still meets at its final barrier (the launch
    # returns); the next launch on the same context is exact.
    N, K = 4096, 4096
    a, b = inputs.make_pair(M, N, K, 34, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.cuda(), b.cuda()
    s, plan = g7.plan("bf16", M, N, K)
    assert _abi.PATHS[plan.path] == "bf16_skinny" and plan.split_k > 1
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    assert _abi.gemm_debug_inject(1, 20_000_000) == _abi.GEMM_OK
    try:
        g7.gemm_bf16_f32acc(a_d, b_d)
        assert g7.gemm_get_device_status() == _abi.GEMM_ERR_TIMEOUT
        assert g7.gemm_get_device_status() == _abi.GEMM_OK
    finally:
        assert _abi.gemm_debug_inject(0, 0) == _abi.GEMM_OK
    c = g7.gemm_bf16_f32acc(a_d, b_d)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == _abi.GEMM_OK
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert_within("bf16", c.cpu().numpy(), c_ref, None, exact=True)
