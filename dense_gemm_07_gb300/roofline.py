"""Operation counts, traffic models and roofline arithmetic for dense GEMM.

Pure host arithmetic used by the benchmark to turn a measured time into
TFLOP/s and a fraction of the roofline.  Nothing here touches the GPU.

* FLOPs of one GEMM: 2*M*N*K, one multiply and one add per (i, j, k)
  ("A06 -- Tiled Matrix Multiply (GEMM)", section 6, Pitfall 4; "How a Matrix
  Multiply Runs on a GPU", "The problem and the roofline").  The direct
  kernel's 2MNK - MN count ("GEMM", inference-book, first cost section) is the
  same work without the first add; the 2MNK convention is used throughout.
* Algorithmic minimum traffic: every element of A, B and C crosses HBM once,
  e_in*(MK + KN) + e_out*MN bytes ("How a Matrix Multiply Runs on a GPU",
  "The problem and the roofline"; "GEMM Optimization", section 1).
* Roofline: attainable rate = min(peak, intensity * bandwidth); the ridge is
  peak / bandwidth ("A06", section 2, "Where the ridge point is").
* The per-k-tile traffic model of "GEMM, step by step" (section "Code"):
  a staged block moves e*(bm*bk + bk*bn) bytes from global memory per k-tile
  and reads that tile plus, for every thread, e*bk*(tm+tn) bytes back from
  shared memory; an unstaged kernel moves e*bm*bn*2*bk bytes from global
  memory.  C is written once per block (4 bytes per element).  The model's
  time is the largest of FLOPs/ALU peak, global bytes/HBM bandwidth and
  shared bytes/shared-memory bandwidth.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def min_bytes(M: int, N: int, K: int, e_in: int, e_out: int = 4) -> float:
    """Each of A (MxK), B (KxN) read once and C (MxN) written once."""
    return float(e_in * (M * K + K * N) + e_out * M * N)


def intensity(M: int, N: int, K: int, e_in: int, e_out: int = 4) -> float:
    b = min_bytes(M, N, K, e_in, e_out)
    return gemm_flops(M, N, K) / b if b else math.inf


def roof(peak_flops: float, bw_bytes: float, flop_per_byte: float) -> float:
    """min(peak, I * BW), in the units of peak_flops."""
    return min(peak_flops, flop_per_byte * bw_bytes)


def ridge(peak_flops: float, bw_bytes: float) -> float:
    return peak_flops / bw_bytes


def block_intensity(bm: int, bn: int, e: int) -> float:
    """Global intensity of one block's own loads: 2/(e(1/bn + 1/bm)).

    "GEMM, step by step", section "Maths": the slice depth bk cancels.
    """
    return 2.0 / (e * (1.0 / bn + 1.0 / bm))


def thread_smem_intensity(tm: int, tn: int) -> float:
    """2*tm*tn / (4*(tm+tn)) FLOP per shared byte (FP32 operands)."""
    return 2.0 * tm * tn / (4.0 * (tm + tn))


@dataclass(frozen=True)
class TileModel:
    """One kernel of the per-k-tile model (tm = tn = 0: no per-thread reads)."""

    staged: bool
    bm: int
    bn: int
    bk: int
    tm: int
    tn: int
    eb: int
    c_bytes: int = 4


def tile_model_bytes(m: TileModel, M: int, N: int, K: int):
    """(global bytes, shared bytes) of the whole GEMM under the page's model."""
    blocks = math.ceil(M / m.bm) * math.ceil(N / m.bn)
    ktiles = math.ceil(K / m.bk)
    if m.staged:
        tile = m.eb * (m.bm * m.bk + m.bk * m.bn)
        glob = tile
        smem = tile
        if m.tm and m.tn:
            threads = (m.bm * m.bn) // (m.tm * m.tn)
            smem += m.eb * m.bk * threads * (m.tm + m.tn)
    else:
        glob = m.eb * m.bm * m.bn * 2 * m.bk
        smem = 0
    c_store = m.c_bytes * m.bm * m.bn
    return (blocks * (ktiles * glob + c_store), blocks * ktiles * smem)


def tile_model_time(m: TileModel, M: int, N: int, K: int, peak_flops: float,
                    hbm_bw: float, smem_bw: float):
    """(seconds, which roof binds) under the page's max-of-roofs model."""
    glob, smem = tile_model_bytes(m, M, N, K)
    t = {"alu": gemm_flops(M, N, K) / peak_flops, "hbm": glob / hbm_bw}
    if smem:
        t["smem"] = smem / smem_bw
    bound = max(t, key=t.get)
    return t[bound], bound


def fp32_simt_peak(sms: int, mhz: float, lanes_per_sm: int = 128) -> float:
    """FP32 CUDA-core peak: SMs x FP32 lanes x 2 FLOP (one FMA) x clock."""
    return sms * lanes_per_sm * 2.0 * mhz * 1e6


def smem_bandwidth(sms: int, mhz: float, bytes_per_clk: int = 128) -> float:
    """Shared-memory bandwidth: SMs x 32 banks x 4 bytes x clock."""
    return sms * bytes_per_clk * mhz * 1e6
