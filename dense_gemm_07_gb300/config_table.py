"""Time every workload configuration of the method on one GPU and print a
markdown table (CUDA events on the calling stream, 3 warm-up calls, a
256 MiB L2 flush before every call).  Two measures:
  * batched: events around `--reps` x (flush, call) minus events around
    `--reps` flushes alone, per call -- the kernels' own time, resolved below
    the ~2 us step of CUDA event timestamps on this GPU; the TFLOP/s, GB/s
    and roofline columns use it;
  * per call: events around each call, queued behind a short spin so that
    host call overhead is not timed; mean and best of `--reps` (includes
    the GPU's launch latency after the flush, and is quantised to ~2 us).

    python -m dense_gemm_07_gb300.config_table [--reps 40] [--peaks MEASURED_PEAKS.json]

Configurations (the workloads of "How a Matrix Multiply Runs on a GPU",
"The problem and the roofline", "A06 -- Tiled Matrix Multiply (GEMM)",
section 4, and the linear-layer and boundary shapes of "GEMM
Optimization"):
  C1   FP32 256^3 (U[-1,1) and integers in [-4, 4])
  C2   FP32 4096^3, U[-1,1)
  C3   BF16 4096^3, N(0, 1)
  C4   BF16 linear layers, M = 2048: (N, K) = (4096, 4096), (11008, 4096),
       (4096, 11008); A ~ N(0, 1), B ~ N(0, 0.02)
  C5a  BF16 {127, 1000, 3001}^3, integers in [-3, 3]
  C5b  BF16 M = 1, N = K = 4096 (bandwidth-bound: reported in GB/s)
  C5c  BF16 M = 16, N = K = 4096 (bandwidth-bound)
Roofline per configuration: min(peak compute, I * HBM bandwidth) with
I = 2MNK / (minimum bytes), every matrix crossing HBM once.  Peaks: the
measured ones when the file is given, else 80.5 TFLOP/s FP32 (152 SMs x
128 lanes x 2 x 2.07 GHz), 1900 TFLOP/s BF16 and 6800 GB/s.
"""
from __future__ import annotations

import argparse
import json
import os

import torch

import dense_gemm_07_gb300 as g7
from dense_gemm_07_gb300 import inputs, roofline


def configs():
    out = [("C1a", "f32", (256, 256, 256), inputs.UNIFORM, None, 0),
           ("C1b", "f32", (256, 256, 256), inputs.INT4, None, 0),
           ("C2", "f32", (4096, 4096, 4096), inputs.UNIFORM, None, 1),
           ("C3", "bf16", (4096, 4096, 4096), inputs.NORMAL, None, 2)]
    for (n, k) in ((4096, 4096), (11008, 4096), (4096, 11008)):
        out.append(("C4", "bf16", (2048, n, k), inputs.NORMAL, inputs.NORMAL_W, 3))
    for m in (127, 1000, 3001):
        for n in (127, 1000, 3001):
            for k in (127, 1000, 3001):
                out.append(("C5a", "bf16", (m, n, k), inputs.INT3, None, 4))
    out.append(("C5b", "bf16", (1, 4096, 4096), inputs.INT3, None, 4))
    out.append(("C5c", "bf16", (16, 4096, 4096), inputs.INT3, None, 4))
    return out


def time_batched(fn, reps, flush):
    """Per-call device time without the ~2 us granularity of CUDA event
    timestamps on this GPU: events around `reps` x (L2 flush, call) minus
    events around `reps` flushes alone, divided by reps.  The stream is held
    by a spin kernel until the host has queued the whole batch, so host
    call overhead never shows; a call's launch latency is hidden behind the
    flush before it, so this is close to the kernels' own duration."""
    for _ in range(3):
        fn()
    out = []
    for with_call in (True, False):
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000 * reps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            flush.fill_(1.0)
            if with_call:
                fn()
        e1.record()
        e1.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3)
    return (out[0] - out[1]) / reps


def time_call(fn, reps, flush):
    for _ in range(3):
        fn()
    ts = []
    for _ in range(reps):
        # a ~0.2 ms torch spin kernel holds the stream while the host queues
        # the flush and the call, so the host's call overhead stays outside
        # the events
        torch.cuda._sleep(400_000)
        flush.fill_(1.0)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return sum(ts) / len(ts), min(ts)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--reps", type=int, default=40)
    p.add_argument("--peaks", default=None)
    a = p.parse_args()
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    src = "fallback"
    if a.peaks and os.path.exists(a.peaks):
        with open(a.peaks) as f:
            peaks.update(json.load(f))
        src = "measured"
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak = roofline.fp32_simt_peak(sms, float(peaks.get("sm_max_mhz", 2070.0))) / 1e12
    bf16_peak = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
    print(f"peaks ({src}): FP32 {fp32_peak:.1f} TFLOP/s, BF16 {bf16_peak:.1f} TFLOP/s, "
          f"HBM {hbm:.0f} GB/s")
    print("| cfg | kind | M x N x K | us (batched) | mean us (per call) | best us | TFLOP/s "
          "| GB/s (min bytes) | roofline | % of roofline |")
    print("|---|---|---|---|---|---|---|---|---|---|")
    for name, kind, (M, N, K), dist, dist_b, seed in configs():
        dtype = torch.float32 if kind == "f32" else torch.bfloat16
        x, y = inputs.make_pair(M, N, K, seed, dist, dist_b, dtype=dtype)
        X, Y = x.to(dev), y.to(dev)
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
        fn = g7.gemm_f32 if kind == "f32" else g7.gemm_bf16_f32acc
        mean, best = time_call(lambda: fn(X, Y, out=C), a.reps, flush)
        batched = time_batched(lambda: fn(X, Y, out=C), a.reps, flush)
        eb = 4 if kind == "f32" else 2
        flops = roofline.gemm_flops(M, N, K)
        nbytes = roofline.min_bytes(M, N, K, eb, 4)
        tf = flops / (batched * 1e-6) / 1e12
        gbs = nbytes / (batched * 1e-6) / 1e9
        peak = fp32_peak if kind == "f32" else bf16_peak
        roof = min(peak, roofline.intensity(M, N, K, eb, 4) * hbm / 1e3)
        bound = "compute" if roof >= peak else "HBM"
        print(f"| {name} | {kind} | {M}x{N}x{K} | {batched:.1f} | {mean:.1f} | {best:.1f} | "
              f"{tf:.1f} | {gbs:.0f} | {roof:.0f} TF ({bound}) | {100 * tf / roof:.1f} |")
    if g7.gemm_get_device_status() != 0:
        raise SystemExit("device status error")


if __name__ == "__main__":
    main()
