"""Large sizes: outputs with more than 2^31 elements (64-bit element
offsets in every store path) and very long K (k-slice indices and copy
coordinates far from zero), compared with the oracle on sampled rows plus
exact row and column sums over every element, or with an exact closed
form."""
import numpy as np
import pytest
import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import inputs
from gemm_check import assert_within, oracle_ref

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_output_beyond_2_31_elements(kind):
    # C is 70000 x 32000 = 2.24e9 elements (9 GB): rows from 67109 on start
    # past element 2^31.  Ragged tiles along M.
    M, N, K = 70000, 32000, 64
    dtype = torch.float32 if kind == "f32" else torch.bfloat16
    a, b = inputs.make_pair(M, N, K, 40, inputs.INT3, dtype=dtype)
    fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
    c = fn(a.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    rows = np.array([0, 1, 127, 128, 35000, 67107, 67108, 67109, 68000, 69887,
                     69888, 69999])
    got = c[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    # Every element, through two properties of the exact product that hold at
    # any size: its row sums equal A (B 1) and its column sums (1^T A) B.  The
    # inputs are small integers, so every sum below is exact in FP64.
    row_sums = c.sum(dim=1, dtype=torch.float64).cpu().numpy()
    col_sums = c.sum(dim=0, dtype=torch.float64).cpu().numpy()
    del c
    a64, b64 = a.to(torch.float64).numpy(), b.to(torch.float64).numpy()
    assert np.array_equal(row_sums, a64 @ b64.sum(axis=1)), "row sums of C differ"
    assert np.array_equal(col_sums, a64.sum(axis=0) @ b64), "column sums of C differ"
    c_ref, _ = oracle_ref(kind, a, b, rows=rows, with_abs=False)
    assert_within(kind, got, c_ref, None, exact=True, what=f"{kind} {M}x{N}x{K}")


def _closed_form(sign, N, K):
    # C[i][j] = sign[i] * sum_{k<K} (((k + j) mod 3) - 1): per residue class
    out = np.empty((len(sign), N), dtype=np.float64)
    for j in range(N):
        counts = [0, 0, 0]
        for r in range(3):
            # number of k in [0, K) with (k + j) % 3 == r
            first = (r - j) % 3
            counts[r] = 0 if first >= K else (K - 1 - first) // 3 + 1
        out[:, j] = sign * float(counts[2] - counts[0])
    return out


@pytest.mark.parametrize("kind,M,N,K", [("bf16", 16, 64, 1 << 25), ("bf16", 300, 64, 1 << 22),
                                        ("f32", 8, 8, 1 << 23)])
def test_very_long_k_exact(kind, M, N, K):
    # A[i][k] = +-1 by row, B[k][j] = ((k + j) mod 3) - 1: every partial sum
    # stays within [-2, 2] (2^25 = 33.5 M k-steps for the small-M path, split
    # over a cluster; 2^22 on the paired-SM path; 2^23 on the FP32 path), so
    # the sums are exact in FP32.
    dtype = torch.float32 if kind == "f32" else torch.bfloat16
    sign = np.where(np.arange(M) % 2 == 0, 1.0, -1.0)
    A = torch.from_numpy(sign).to(DEV, torch.float32)[:, None].expand(M, K).to(dtype).contiguous()
    kk = torch.arange(K, device=DEV, dtype=torch.int32)[:, None]
    jj = torch.arange(N, device=DEV, dtype=torch.int32)[None, :]
    B = ((kk + jj) % 3 - 1).to(dtype)
    del kk, jj
    fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
    c = fn(A, B)
    torch.cuda.synchronize()
    assert g7.gemm_get_device_status() == 0
    want = _closed_form(sign, N, K)
    got = c.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {tuple(bad[0])}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"
