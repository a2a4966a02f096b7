"""The bench's metric arithmetic against the worked numbers the pages print."""

import os

import pytest

from dense_matrix_multiply_gb300 import metrics

MIB = 1 << 20


def golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "gemm_model_numbers.txt")
    out = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            name, value, _cite = line.split()
            out[name] = float(value)
    return out


def test_flops_and_bytes_k1_walkthrough():
    g = golden()
    assert metrics.gemm_flops(4096, 4096, 4096) == g["flops_4096_cubed"]
    assert metrics.min_bytes(4096, 4096, 4096, 2) == g["min_bytes_fp16_4096_cubed"]
    assert metrics.tiled_bytes(4096, 4096, 4096, 2, 128, 128) == g["tiled_bytes_fp16_4096_cubed_128x128"]


def test_ffn_bytes_chapter5():
    g = golden()
    M, K, N = 1024, 4096, 12288
    assert metrics.min_bytes(M, N, K, 2) == g["v_once_mib_ffn"] * MIB
    for t in (32, 64, 128):
        assert metrics.tiled_bytes(M, N, K, 2, t, t) == g[f"tiled_mib_ffn_{t}x{t}"] * MIB
    assert metrics.tile_working_set(64, 64, 32) == g["smem_kib_ffn_64x64_k32"] * 1024
    assert metrics.tile_working_set(128, 128, 32) == g["smem_kib_ffn_128x128_k32"] * 1024


def test_fp32_peak_gflops_and_beat_sgemm_ledgers():
    g = golden()
    assert round(metrics.simt_fp32_peak(128, 2.52e9) / 1e9) == g["fp32_peak_gflops_4090_2.52GHz"]
    assert round(metrics.simt_fp32_peak(128, 2.64e9) / 1e9) == g["fp32_peak_gflops_4090_2.64GHz"]
    t = 22.225e-3
    assert round(metrics.flops_per_s(4096, 4096, 4096, t) / 1e9, 1) == g["gflops_4096_cubed_22.225ms"]
    assert round(metrics.beat(128, 2.52e9, t, 4096, 4096, 4096), 3) == g["beat_4096_cubed_22.225ms_128sm_2.52GHz"]


def test_wave_accounting():
    # 1024 tiles on 46 SMs at one CTA each: 23 waves, the last holding 12 tiles
    assert metrics.wave_count(1024, 46) == pytest.approx(22.26, abs=0.01)
    assert metrics.wave_efficiency(1024, 46) == pytest.approx(1024 / (23 * 46))
    assert metrics.wave_efficiency(0, 10) == 1.0


def test_fp8_quantisation_traffic_example_5_8():
    g = golden()
    t = metrics.fp8_rowscale_traffic(4096, 4096, 1536, 128)
    assert t["separate_input"] == g["fp8_separate_input_mib"] * MIB
    assert t["fused_input"] == g["fp8_fused_input_mib"] * MIB
    assert t["weights_output"] == g["fp8_weights_output_mib"] * MIB
    assert t["separate_total"] == g["fp8_separate_total_mib"] * MIB
    assert t["fused_total"] == g["fp8_fused_total_mib"] * MIB
