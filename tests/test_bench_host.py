"""Host logic of bench.py (no GPU): the roofline classification of each timed part and the
algorithmic byte counts it rests on."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0, "bf16_tflops_sustained": 1800.0, "source": "test"}


def test_roofline_classifies_by_intensity_against_the_ridge():
    ridge = 2000e12 / 8000e9  # 250 flop/B
    t = bench.roofline_of(flops=4.0e12, algo_bytes=4.0e12 / 500, ms=2.5, peaks=PEAKS)  # AI 500 > ridge
    assert t["bound"] == "tensor" and t["ridge_flop_per_byte"] == pytest.approx(ridge)
    assert t["attainable_tflops"] == pytest.approx(2000.0)
    assert t["tflops"] == pytest.approx(1600.0) and t["frac_of_attainable"] == pytest.approx(0.8)
    h = bench.roofline_of(flops=4.0e12, algo_bytes=4.0e12 / 125, ms=4.0, peaks=PEAKS)  # AI 125 < ridge
    assert h["bound"] == "hbm"
    assert h["attainable_tflops"] == pytest.approx(125 * 8000e9 / 1e12)  # 1000 TFLOP/s
    assert h["frac_of_attainable"] == pytest.approx(1000.0 / 1000.0)
    assert h["achieved_gbs"] == pytest.approx(4.0e12 / 125 / 4.0e-3 / 1e9)
    tiny = bench.roofline_of(flops=6.7e7, algo_bytes=2e6, ms=0.02, peaks=PEAKS)
    assert tiny["bound"] == "launch"


def test_algorithmic_bytes_of_the_deepseek_wgrad():
    from moe_grouped_gemm_persistent_gb300 import synth
    _, w = synth.workload_specs("deepseek")

    class P:
        dspec, wspec = None, w

    b = bench.Problem.algorithmic_bytes(P())
    want = 7168 * w.T * 2 + w.T * 2048 * 2 + 256 * 7168 * 2048 * 4  # A, B, FP32 outputs written once
    assert b["wgrad"] == want
