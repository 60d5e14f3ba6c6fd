"""Calls from several host threads at once, each thread on a CUDA stream of
its own: every result exact against the oracle (integer inputs) and no
bounded wait runs out.  The host-buffer entry points, whose copies share two
helper streams per device, run among them.

The threads race on each kernel's first-call set-up (shared-memory
attributes and occupancy queries cached per device), and their calls run
side by side on the GPU, each with its stream's own scratch (operand copies,
stream-K partial sums and flags, FP32 split-K partial tiles and counters)."""
import random
import threading

import numpy as np
import pytest
import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import inputs
import oracle
from gemm_check import oracle_ref

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (kind, M, N, K, with a bias): one shape per path
CASES = [
    ("bf16", 3001, 1000, 1000, False),  # operands copied to aligned rows, paired kernel
    ("bf16", 1280, 1024, 4096, False),  # tiles halved along K, finished in C
    ("bf16", 1280, 1024, 4096, True),   # halved tiles meeting in the partial-sum workspace
    ("bf16", 512, 1024, 8192, False),   # few tiles, long K: 128 x 128 tiles, K split
    ("bf16", 1000, 3001, 777, False),   # row-store epilogue
    ("bf16", 16, 4096, 4096, False),    # small-M kernel, cluster reduction
    ("bf16", 1000, 100, 1200, False),   # narrow-N kernel
    ("bf16", 300, 258, 200, False),     # small problem on the CUDA cores
    ("f32", 640, 520, 2000, False),     # FP32, partial wave split along K
    ("f32", 256, 256, 256, False),      # FP32 small problem
    ("bf16_host", 1024, 1536, 2048, False),  # host buffers: copies on shared helper streams
    ("f32_host", 700, 900, 1000, False),
]
THREADS = 4
REPS = 3


def _case_inputs(i):
    kind, M, N, K, with_bias = CASES[i]
    kind = kind.replace("_host", "")
    dtype = torch.bfloat16 if kind == "bf16" else torch.float32
    a, b = inputs.make_pair(M, N, K, 70 + i, inputs.INT3, dtype=dtype)
    bias = (torch.randint(-4, 5, (N,), generator=torch.Generator().manual_seed(170 + i))
            .float() if with_bias else None)
    ab, _ = oracle_ref(kind, a, b, with_abs=False)
    want = oracle.gemm_epilogue(ab, bias=bias.numpy()) if with_bias else ab
    return a, b, bias, want


def test_concurrent_calls_from_host_threads_exact():
    data = [_case_inputs(i) for i in range(len(CASES))]
    dev_data = [(a.pin_memory(), b.pin_memory(), None) if CASES[i][0].endswith("_host")
                else (a.to(DEV), b.to(DEV), None if bias is None else bias.to(DEV))
                for i, (a, b, bias, _) in enumerate(data)]
    torch.cuda.synchronize()
    results = {}
    errors = []
    start = threading.Barrier(THREADS)

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            order = [i for _ in range(REPS) for i in range(len(CASES))]
            random.Random(t).shuffle(order)
            outs = []
            start.wait()
            with torch.cuda.stream(stream):
                for i in order:
                    kind, M, N, K, _ = CASES[i]
                    a, b, bias = dev_data[i]
                    if kind == "bf16_host":
                        c = g7.gemm_bf16_f32acc_host(a, b)
                    elif kind == "f32_host":
                        c = g7.gemm_f32_host(a, b)
                    elif bias is not None:
                        c = g7.gemm_bf16_f32acc_ex(a, b, bias=bias)
                    elif kind == "bf16":
                        c = g7.gemm_bf16_f32acc(a, b)
                    else:
                        c = g7.gemm_f32(a, b)
                    outs.append((i, c))
            stream.synchronize()
            results[t] = [(i, c.cpu().numpy()) for i, c in outs]
        except Exception as e:  # reported on the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a thread did not finish"
    assert not errors, errors
    assert g7.gemm_get_device_status() == 0
    assert sorted(results) == list(range(THREADS))
    for t in range(THREADS):
        assert len(results[t]) == REPS * len(CASES)
        for i, got in results[t]:
            want = data[i][3]
            bad = np.argwhere(got.astype(np.float64) != want)
            assert bad.size == 0, (t, CASES[i], len(bad), tuple(bad[0]))
