"""bench.py's roofline bookkeeping (no GPU): which roof bounds a launch, and the
achieved figure it divides by that roof."""

import pytest

import bench

PEAKS = {"hbm_gbs": 6785.5, "bf16_tflops": 1866.5, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}


def roof(kind, variant, M, N, K, seconds):
    return bench.roofline_for(kind, variant, M, N, K, seconds, PEAKS, "test", None, 152, "none")


def test_large_tensor_problem_is_tensor_bound():
    r = roof("umma", "bf16_rm", 8192, 8192, 8192, 1e-3)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(2 * 8192 ** 3 / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1866.5)


def test_skinny_tensor_problem_is_hbm_bound():
    """M = 32 does 64 FLOPs per weight byte pair, far below the ridge point
    (1866.5e12 / 6785.5e9 = 275 FLOP/byte): the HBM roof applies."""
    M, N, K, t = 32, 12288, 4096, 21.5e-6
    r = roof("umma", "bf16_rm", M, N, K, t)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    bytes_ = 2 * (M * K + K * N + M * N)
    assert r["achieved"] == pytest.approx(bytes_ / t / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6785.5)


def test_fp8_peak_is_twice_the_bf16_burst():
    r = roof("umma", "e4m3_rowscale", 8192, 8192, 8192, 1e-3)
    assert r["bound"] == "tensor" and r["peak"] == pytest.approx(2 * 1866.5)


def test_gemv_is_hbm_bound_and_simt_is_alu_bound():
    assert roof("gemv", "bf16_rm", 1, 12288, 4096, 19e-6)["bound"] == "hbm"
    r = roof("simt", "f32_rm", 4096, 4096, 4096, 2.2e-3)
    assert r["bound"] == "alu"
    assert r["peak"] == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
