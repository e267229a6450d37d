"""The roofline arithmetic of bench.py: the slower of bytes at the measured
HBM bandwidth and FLOPs at the dense FP4 peak decides the bound, and the
fraction is that time over the measured one.  Hand-computed cases."""
import sys
from pathlib import Path

import pytest

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6786.6, "bf16_tflops": 1917.4, "source": "measured"}


def test_fp4_peak_is_six_times_bf16():
    assert bench.fp4_peak_tflops(PEAKS) == pytest.approx(6 * 1917.4)


def test_bytes_bound_case():
    # 1 GB in 0.2 ms with 1 GFLOP: bytes take 1e9 / 6786.6e9 s = 0.14735 ms
    r = bench.roofline(1e9, 1e9, 0.2, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(5000.0)
    assert r["frac"] == pytest.approx(5000.0 / 6786.6)
    assert r["roofline_ms"] == pytest.approx(1e9 / 6786.6e9 * 1e3)


def test_flops_bound_case():
    # 12.99 TFLOP and 4.7 GB in 4.17 ms: FLOPs take 12.99e12 / 11504.4e12 s = 1.129 ms > 0.69 ms of bytes
    r = bench.roofline(4.7e9, 12.99e12, 4.17, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(12.99e12 / 4.17e-3 / 1e12)
    assert r["frac"] == pytest.approx((12.99e12 / 11504.4e12 * 1e3) / 4.17, rel=1e-4)
    assert r["frac"] == pytest.approx(r["roofline_ms"] / r["ms"])


def test_layer_work_counts():
    """Per route 2 * 3 * I * H FLOPs; gate/up two thirds of them; the layer's
    bytes add the router weights, x and the bf16 output to the GEMMs'."""
    H, I, E, T = 7168, 2048, 384, 8
    w = bench.layer_work(H, I, E, T, "mxfp4", "a4w4", touched=44, routes=64)
    assert w["gateup"][1] == 2.0 * 2 * I * H * 64 and w["down"][1] == 2.0 * H * I * 64
    assert w["layer"][1] == w["gateup"][1] + w["down"][1]
    gu, dn = bench.algorithmic_bytes(H, I, "mxfp4", "a4w4", 44, 64, T)
    assert w["layer"][0] == gu + dn + E * H * 2 + 2 * T * H * 2
