"""bench.py's JSON line (no GPU): the keys the benchmark contract asks for, and
whole-job figures over replicas, from a measurement shaped like the one the
GPU run produces."""

import json

import pytest

import bench
import synthetic

FLOPS = 2 * 4096 ** 3


def fake_measurement():
    return {
        "workload": "sgemm_f32_rm_4096", "variant": "f32_rm", "M": 4096, "N": 4096, "K": 4096,
        "kernel": "simt_f32_vec4", "flops_per_step": FLOPS, "ms_per_step": 2.12, "tflops": FLOPS / 2.12e-3 / 1e12,
        "steps": 10, "ms_total": 21.2,
        "roofline": {"bound": "alu", "achieved": 64.8, "peak": 80.55, "unit": "TFLOP/s", "frac": 64.8 / 80.55,
                     "traffic": 403020032},
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 12, "power_w_max": 900.0},
        "footprint_bytes": 3 * 4096 * 4096 * 4, "gpu_launches": 20, "l2": "no flush: 192 MiB of operands > 129 MB L2",
        "e2e": {"value": FLOPS / 2.17e-3 / 1e12, "unit": "TFLOP/s", "ms_per_step": 2.17, "steps": 10,
                "overlap": "pipelined", "h2d_bytes_per_step": 134217728, "d2h_bytes_per_step": 67108864},
        "e2e_serial": {"value": FLOPS / 3.12e-3 / 1e12, "unit": "TFLOP/s", "ms_per_step": 3.12, "steps": 10,
                       "h2d_bytes_per_step": 134217728, "d2h_bytes_per_step": 67108864},
        "cpu_baseline": {"value": 0.043, "unit": "TFLOP/s", "cores": 16, "kind": "oracle",
                         "sample": "64 of 4096 output rows"},
        "cublas": {"tflops": 66.8, "ms_per_step": 2.06, "mode": "FP32, CUBLAS_PEDANTIC_MATH"},
    }


def test_single_gpu_line_carries_every_contract_key():
    res = fake_measurement()
    line = bench.bench_line(res, "sgemm_f32_rm_4096", 10, 3, 1, 21.2, {}, [])
    json.dumps(line)  # serialisable
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks", "e2e",
                "cpu_baseline"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["warmup"] == 3
    assert line["value"] == pytest.approx(FLOPS * 10 / 21.2e-3 / 1e12)
    assert line["ms_per_step"] == pytest.approx(2.12)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["dtype"] == "f32" and line["data"] == "synthetic"
    assert line["config"]["workload"] == "sgemm_f32_rm_4096" and "l2" in line["config"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in line["roofline"]
    assert set(("sm_mhz", "sm_max_mhz", "reasons")) <= set(line["clocks"])
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in line["e2e"]
    assert line["e2e"]["value"] == pytest.approx(FLOPS / 2.17e-3 / 1e12)
    assert line["e2e"]["unit"] == line["unit"]
    assert line["gpu_launches"] == 20
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in line["cpu_baseline"]


def test_replicas_aggregate_over_ranks():
    """Two replicas: FLOPs of both ranks over the slowest rank's time, the same
    for the end-to-end figures; launches summed."""
    res = fake_measurement()
    line = bench.bench_line(res, "sgemm_f32_rm_4096", 10, 3, 2, 25.0, {"e2e": 2.5, "e2e_serial": 3.5}, [])
    assert line["n_gpus"] == 2 and line["config"]["parallelism"] == "replicas x2"
    assert line["value"] == pytest.approx(FLOPS * 10 * 2 / 25.0e-3 / 1e12)
    assert line["e2e"]["value"] == pytest.approx(FLOPS * 2 / 2.5e-3 / 1e12)
    assert line["e2e"]["ms_per_step"] == 2.5
    assert line["e2e_serial"]["value"] == pytest.approx(FLOPS * 2 / 3.5e-3 / 1e12)
    assert line["gpu_launches"] == 40
    # the measurement itself is left as it was
    assert res["e2e"]["ms_per_step"] == 2.17


def test_half_precision_workloads_name_their_dtype_and_layout():
    res = fake_measurement()
    res.update(variant="f16_cm", workload="hgemm_f16_cm_8192")
    for key in ("e2e", "e2e_serial", "cpu_baseline"):
        res.pop(key)
    path = {"workload": "x", "kernel": "umma_bf16", "ms_per_step": 0.5, "tflops": 100.0,
            "roofline": {"frac": 0.5, "bound": "tensor", "traffic": None, "algorithmic_bytes": 10}}
    line = bench.bench_line(res, "hgemm_f16_cm_8192", 10, 3, 1, 6.0, {}, [path])
    assert line["dtype"] == "f16" and line["config"]["layout"] == "column-major"
    assert "e2e" not in line and line["paths_detail"] == [path]
    assert line["paths"] == {"x": {"kernel": "umma_bf16", "us": 500.0, "tflops": 100.0, "frac": 0.5,
                                   "bound": "tensor"}}
    # the compact summary is the line's last key (the end of the output)
    assert list(line)[-1] == "paths"


def test_k4100_rows_carry_their_k4096_control():
    def rec(name, ms, tf):
        return {"workload": name, "kernel": "simt_f32_vec4", "ms_per_step": ms, "tflops": tf,
                "roofline": {"frac": 0.8, "bound": "alu", "traffic": 300, "algorithmic_bytes": 150},
                "cublas": {"tflops": 60.0}}
    paths = [rec("edge_f32_rm_8192x4096x4100", 4.4, 62.5), rec("edge_f32_rm_8192x4096x4096", 4.2, 65.0),
             rec("edge_bf16_rm_8192x4096x4100", 0.2, 1400.0)]
    bench.add_k4096_controls(paths)
    c = paths[0]["k4096_control"]
    assert c["workload"] == "edge_f32_rm_8192x4096x4096" and c["slowdown_vs_k4096"] == pytest.approx(65.0 / 62.5)
    assert "k4096_control" not in paths[1] and "k4096_control" not in paths[2]  # no bf16 control measured
    compact = bench.compact_paths(paths)
    assert compact["edge_f32_rm_8192x4096x4100"] == {
        "kernel": "simt_f32_vec4", "us": 4400.0, "tflops": 62.5, "frac": 0.8, "bound": "alu", "traffic_x": 2.0,
        "cublas_tflops": 60.0, "slowdown_vs_k4096": 1.04}


def test_default_paths_cover_every_configuration_shape():
    """Every workload of the five configurations is the headline or a path."""
    names = set(bench.DEFAULT_PATHS) | {bench.DEFAULT_WORKLOAD}
    for wl in synthetic.WORKLOADS:
        assert wl in names
    for (M, N, K) in synthetic.EDGE_SHAPES:
        for v in ("f32_rm", "bf16_rm"):
            if (M, N, K) == (32, 12288, 4096) and v == "f32_rm":
                continue  # M = 32 decode: a 16-bit addition of this library's sweep
            assert f"edge_{v}_{M}x{N}x{K}" in names


def test_per_call_spread_statistics():
    s = bench.spread_stats([1.0] * 9 + [1.1])
    assert s["calls"] == 10 and s["median_ms"] == 1.0 and s["p10_ms"] == 1.0
    assert s["p90_ms"] == pytest.approx(1.01)
    assert s["cv"] == pytest.approx(0.03 / 1.01)  # population std 0.03 over mean 1.01
    assert s["noisy"] is True
    assert bench.spread_stats([2.0, 2.0, 2.0])["noisy"] is False


def test_per_call_spread_reaches_the_line():
    res = fake_measurement()
    res["per_call"] = bench.spread_stats([2.1, 2.12, 2.11])
    line = bench.bench_line(res, "sgemm_f32_rm_4096", 10, 3, 1, 21.2, {}, [])
    assert line["per_call"]["calls"] == 3 and not line["per_call"]["noisy"]
