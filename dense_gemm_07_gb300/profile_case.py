"""Run one GEMM configuration a few times, for profiler captures.

    python -m dense_gemm_07_gb300.profile_case --kind bf16 --m 4096 --n 4096 --k 4096 --reps 3

Inputs are the seeded synthetic ones of the benchmark (BF16: N(0,1), seed 2;
FP32: U[-1,1), seed 1); an L2 flush (256 MiB write) precedes every call so a
captured launch reads its operands from HBM.
"""
from __future__ import annotations

import argparse

import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import inputs


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--kind", choices=["bf16", "f32"], default="bf16")
    p.add_argument("--m", type=int, default=4096)
    p.add_argument("--n", type=int, default=4096)
    p.add_argument("--k", type=int, default=4096)
    p.add_argument("--reps", type=int, default=3)
    a = p.parse_args()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if a.kind == "bf16":
        x, y = inputs.make_pair(a.m, a.n, a.k, 2, inputs.NORMAL, dtype=torch.bfloat16)
        fn = g7.gemm_bf16_f32acc
    else:
        x, y = inputs.make_pair(a.m, a.n, a.k, 1, inputs.UNIFORM, dtype=torch.float32)
        fn = g7.gemm_f32
    X, Y = x.to(dev), y.to(dev)
    C = torch.empty((a.m, a.n), dtype=torch.float32, device=dev)
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
    for i in range(a.reps):
        flush.fill_(float(i))
        fn(X, Y, out=C)
    torch.cuda.synchronize()
    status = g7.gemm_get_device_status()
    print(f"{a.kind} {a.m}x{a.n}x{a.k} x{a.reps}: status {status}")
    if status != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
