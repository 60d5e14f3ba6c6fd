"""The benchmark's FLOP, byte and roofline arithmetic against the numbers the
pages print (fixtures under tests/golden/, each naming its page and section).

Device constants that the pages use but do not print are public datasheet
figures: A100 (108 SMs, 1410 MHz boost, 1.555 TB/s HBM2) and H100 SXM
(132 SMs, 1980 MHz boost); shared memory moves 32 banks x 4 bytes per clock
per SM on both.
"""
import json
import math
import os

import pytest

from dense_gemm_07_gb300 import roofline as rl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


A100 = dict(fp32=19.5e12, tensor=312e12, hbm=1.555e12,
            smem=rl.smem_bandwidth(108, 1410))
H100 = dict(fp32=67e12, tensor=989e12, hbm=3.35e12,
            smem=rl.smem_bandwidth(132, 1980))


def _close(x, printed):
    """Equal to the printed value at the precision it is printed with."""
    s = f"{printed}"
    digits = len(s.split(".")[1]) if "." in s else 0
    return round(x, digits) == printed or math.isclose(x, printed, rel_tol=6e-3)


def test_p1_model_table():
    g = _load("p1_model_table.json")
    p = g["problem"]
    M, N, K = p["M"], p["N"], p["K"]
    for r in g["rows"]:
        m = rl.TileModel(r["staged"], r["bm"], r["bn"], r["bk"], r["tm"],
                         r["tn"], r["eb"])
        glob, _ = rl.tile_model_bytes(m, M, N, K)
        assert _close(rl.gemm_flops(M, N, K) / glob, r["flop_per_byte"]), r
        for dev, key in ((A100, "ms_a100"), (H100, "ms_h100")):
            peak = dev["tensor"] if r["alu"] == "tensor" else dev["fp32"]
            smem_bw = dev["smem"] if r["alu"] != "tensor" else math.inf
            t, bound = rl.tile_model_time(m, M, N, K, peak, dev["hbm"], smem_bw)
            assert _close(t * 1e3, r[key]), (r["kernel"], key, t * 1e3)
            if dev is A100:
                assert bound == r["bound_a100"], (r["kernel"], bound)
    # the A100 tensor ridge: 312 TFLOP/s over 1.555 TB/s
    assert round(rl.ridge(A100["tensor"], A100["hbm"])) == \
        g["printed_rates"]["a100_tensor_ridge_flop_per_byte"]


def test_p1_block_and_thread_intensity():
    # b/e for square blocks: b/4 FP32, b/2 BF16; 1/4 -> 2 for an 8x8 patch
    assert rl.block_intensity(128, 128, 4) == 32
    assert rl.block_intensity(128, 128, 2) == 64
    assert rl.block_intensity(32, 32, 4) == 8
    assert rl.thread_smem_intensity(1, 1) == 0.25
    assert rl.thread_smem_intensity(8, 8) == 2.0


def test_p5_traffic_table():
    g = _load("p5_traffic_table.json")
    n = g["N"]
    naive = rl.TileModel(False, 1, 1, 1, 1, 1, 4, c_bytes=0)
    glob, _ = rl.tile_model_bytes(naive, n, n, n)
    assert round(glob / 1e9, 1) == g["naive"]["traffic_gb"]
    assert rl.gemm_flops(n, n, n) / glob == g["naive"]["flop_per_byte"]
    for row in g["tiled"]:
        T = row["T"]
        m = rl.TileModel(True, T, T, T, 0, 0, 4, c_bytes=0)
        glob, _ = rl.tile_model_bytes(m, n, n, n)
        assert round(glob / 1e9, 1) == row["traffic_gb"]
        assert rl.gemm_flops(n, n, n) / glob == row["flop_per_byte"]
        assert rl.block_intensity(T, T, 4) == row["flop_per_byte"]
    # A, B and C once each, FP32
    assert round(rl.min_bytes(n, n, n, 4, 4) / 1e6) == g["footprint_mb"]
    assert round(2 * n / 3) == g["times_moved"]
    for d in g["ridge"]:
        assert round(rl.ridge(d["fp32_tflops"], d["hbm_tbs"])) == d["ridge"]
    for d, row in zip(g["ridge_crossing_tile"], g["ridge"][::-1]):
        assert 4 * row["ridge"] == d["T"]


def test_p2_roofline_numbers():
    g = _load("p2_roofline.json")
    n = g["square_bf16"]["n"]
    assert rl.gemm_flops(n, n, n) == pytest.approx(g["square_bf16"]["flops"], rel=5e-3)
    b = rl.min_bytes(n, n, n, 2, 2)          # FP16/BF16 C as well
    assert b / 1e6 >= g["square_bf16"]["min_mb"]
    assert round(rl.gemm_flops(n, n, n) / b) == g["square_bf16"]["flop_per_byte"]
    h = g["h100_sxm"]
    assert round(rl.ridge(h["bf16_tflops"], h["hbm_tbs"])) == h["ridge_bf16"]
    assert round(rl.ridge(h["fp32_tflops"], h["hbm_tbs"])) == h["ridge_fp32"]
    assert rl.block_intensity(32, 32, 4) == g["level1_fp32_T32_flop_per_byte"]
    assert rl.block_intensity(128, 128, 2) == g["level2_bf16_128x128_flop_per_byte"]


def test_roof_and_min_bytes():
    assert rl.roof(100.0, 10.0, 5.0) == 50.0
    assert rl.roof(100.0, 10.0, 50.0) == 100.0
    # BF16 in, FP32 out, 4096^3: 2*2*4096^2 + 4*4096^2 bytes
    assert rl.min_bytes(4096, 4096, 4096, 2, 4) == 8 * 4096**2
    assert rl.intensity(4096, 4096, 4096, 2, 4) == 2 * 4096**3 / (8 * 4096**2)
    assert rl.fp32_simt_peak(152, 2070) == pytest.approx(80.55e12, rel=1e-3)
