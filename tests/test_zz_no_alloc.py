"""gemm_bf16_f32acc_noalloc: the BF16 GEMM for callers that may not allocate
device memory.

Some callers cannot call cudaMalloc: a plug-in running inside a host
application that owns all device memory through its own allocator and
forbids others from allocating, or a latency-critical loop in which an
allocation could synchronise the device.  For them the library offers one
entry point whose operand copies go into a fixed scratch array declared in
device memory instead of a memory pool.

These tests call it through the C ABI, twice in a row on each input (the
second call runs on scratch left over from the first), and check every
element of each output against the FP64 oracle -- exactly on integer inputs,
within the BF16 bound otherwise -- and against the ordinary (pool-using)
entry point, within the same bound (bit for bit where both run the same
schedule).  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import _abi, inputs
from gemm_check import assert_within, oracle_ref, small_limit

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _noalloc(a, b, out):
    """Call the no-allocation entry point on (possibly strided) CUDA tensors."""
    M, K = a.shape
    N = b.shape[1]
    st = torch.cuda.current_stream().cuda_stream
    return _abi.gemm_bf16_f32acc_noalloc(M, N, K, a.data_ptr(), a.stride(0),
                                         b.data_ptr(), b.stride(0),
                                         out.data_ptr(), out.stride(0), st)


def _misaligned(t, extra_cols, offset):
    """Copy of t placed `offset` elements into rows `extra_cols` wider."""
    rows, cols = t.shape
    buf = torch.zeros((rows, cols + extra_cols), dtype=t.dtype, device=DEV)
    buf[:, offset:offset + cols] = t.to(DEV)
    return buf[:, offset:offset + cols]


# (M, N, K, seed, distribution, exact): K = 333 makes A's rows a
# non-multiple of 16 bytes; the second case offsets both operands by odd
# element counts, so both copies land in the scratch array.
CASES = [(300, 520, 333, 21, inputs.INT3, True),
         (257, 300, 200, 22, inputs.NORMAL, False)]


def _against_oracle_and_pooled(a, b, a_d, b_d, exact, what):
    """Two no-allocation calls in a row, each compared in full with the
    oracle and with the pooled entry point."""
    M, K = a.shape
    N = b.shape[1]
    c_ref, s_ref = oracle_ref("bf16", a, b, with_abs=not exact)
    pooled = g7.gemm_bf16_f32acc(a_d, b_d).cpu().numpy()
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(a_d, b_d, out) == _abi.GEMM_OK
        torch.cuda.synchronize()
        assert g7.gemm_get_device_status() == 0
        got = out.cpu().numpy()
        assert_within("bf16", got, c_ref, s_ref, exact=exact,
                      what=f"{what}, call {call + 1} against the oracle")
        if exact:
            assert np.array_equal(got, pooled), f"{what}: differs from the pooled call"
        else:
            # the same bound, taken around the pooled entry point's output
            assert_within("bf16", got, pooled.astype(np.float64), s_ref,
                          what=f"{what}, call {call + 1} against the pooled call")


def test_noalloc_copied_operands_two_calls_in_a_row():
    for (M, N, K, seed, dist, exact) in CASES:
        a, b = inputs.make_pair(M, N, K, seed, dist, dtype=torch.bfloat16)
        if exact:
            a_d, b_d = a.to(DEV), b.to(DEV)
        else:
            a_d, b_d = _misaligned(a, 9, 3), _misaligned(b, 11, 1)
        # this entry point never takes the small-problem path: planned with
        # that path off, the call copies A (and B) into the fixed array
        with small_limit(0):
            s, plan = g7.plan("bf16", M, N, K, a_d.data_ptr(), a_d.stride(0),
                              b_d.data_ptr(), b_d.stride(0), 16, N)
        assert s == 0 and plan.pack_a == 1, "case must exercise the scratch copies"
        _against_oracle_and_pooled(a, b, a_d, b_d, exact, f"{M}x{N}x{K}")


@pytest.mark.parametrize("dist,exact", [(inputs.INT3, True), (inputs.NORMAL, False)])
def test_noalloc_stream_k_two_calls_in_a_row(dist, exact):
    # 90 tiles shared as k-slice runs by 76 SM pairs: the partial sums
    # and the synchronisation words live in the fixed scratch array too
    M, N, K = 2560, 2304, 1024
    a, b = inputs.make_pair(M, N, K, 26, dist, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    prev = _abi.gemm_set_bf16_schedule(_abi.SCHEDULE_STREAM_K)
    try:
        s, plan = g7.plan("bf16", M, N, K)
        assert s == 0 and plan.sk_tiles > 0
        _against_oracle_and_pooled(a, b, a_d, b_d, exact, "stream-K 2560x2304x1024")
    finally:
        _abi.gemm_set_bf16_schedule(prev)


def test_noalloc_default_schedule_4096_aligned_operands():
    # 4096^3 with aligned operands: no copies, but the default schedule halves
    # the last wave's 28 tiles along K and their cleared flags live in the
    # array
    M = N = K = 4096
    a, b = inputs.make_pair(M, N, K, 2, inputs.NORMAL, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    s, plan = g7.plan("bf16", M, N, K)
    assert s == 0 and plan.sk_tiles == 28 and plan.pack_a == 0 and plan.pack_b == 0
    _against_oracle_and_pooled(a, b, a_d, b_d, False, "4096^3 default schedule")


def test_noalloc_rejects_requests_beyond_its_scratch():
    # A needs a copy (lda odd); 4096 rows of 8200 BF16 exceed the 64 MiB scratch
    M, K, N = 4096, 8199, 64
    a = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((K, N), dtype=torch.bfloat16, device=DEV)
    c = torch.full((M, N), 7.0, dtype=torch.float32, device=DEV)
    s, plan = g7.plan("bf16", M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N)
    assert plan.workspace_bytes > _abi.NOALLOC_SCRATCH_BYTES
    assert _noalloc(a, b, c) == _abi.GEMM_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(c == 7.0)   # nothing was enqueued


def test_noalloc_single_row_exact():
    # M = 1 runs on the small-M kernel; A's single row of 3001 elements (not
    # a multiple of 16 bytes) is read in place, and so is B
    M, N, K = 1, 1000, 3001
    a, b = inputs.make_pair(M, N, K, 23, inputs.INT3, dtype=torch.bfloat16)
    a_d, b_d = a.to(DEV), b.to(DEV)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    assert _noalloc(a_d, b_d, out) == _abi.GEMM_OK
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), c_ref)


@pytest.mark.parametrize("M,N,K,packed", [(3001, 100, 1000, "b"), (300, 1000, 3001, "a")])
def test_noalloc_narrow_n_exact(M, N, K, packed):
    # N <= 128 < M runs on the narrow-N kernel (cluster reduction, nothing in
    # the array); B's rows of 100 elements are copied into it first.  So do
    # few 128 x 128 tiles with a long K, here with A's rows copied.
    a, b = inputs.make_pair(M, N, K, 24, inputs.INT3, dtype=torch.bfloat16)
    s, plan = g7.plan("bf16", M, N, K)
    assert _abi.PATHS[plan.path] == "bf16_narrow"
    assert (plan.pack_a, plan.pack_b) == ((1, 0) if packed == "a" else (0, 1))
    a_d, b_d = a.to(DEV), b.to(DEV)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    for _ in range(2):
        assert _noalloc(a_d, b_d, out) == _abi.GEMM_OK
        torch.cuda.synchronize()
        assert g7.gemm_get_device_status() == 0
        c_ref, _ = oracle_ref("bf16", a, b, with_abs=False)
        assert np.array_equal(out.cpu().numpy().astype(np.float64), c_ref)
