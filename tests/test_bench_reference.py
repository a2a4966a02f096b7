"""bench.py's reference arm on the host (no GPU): the CPU oracle timed on a
bounded sample of the workload, one JSON line with the contract's keys; ranks
other than 0 print nothing."""

import json

import bench


def test_reference_arm_prints_one_contract_line(capsys, monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    bench.main(["--impl", "reference", "--workload", "sgemm_f32_rm_256", "--steps", "2", "--warmup", "1",
                "--ref-seconds", "0.5"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == "sgemm_f32_rm_256"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_is_silent_on_other_ranks(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--workload", "sgemm_f32_rm_256", "--steps", "1", "--warmup", "0",
                "--ref-seconds", "0.1"])
    assert capsys.readouterr().out.strip() == ""
