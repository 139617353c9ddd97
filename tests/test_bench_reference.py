"""The benchmark's reference arm (the CPU oracle timed on a bounded sample) on the
host: the JSON line carries the keys of the benchmark contract, and a rank other
than 0 does no work and prints nothing."""
import json

import bench


def test_reference_arm_prints_one_complete_line(capsys, monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "sample" in cb
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert abs(d["ms_per_step"] - 1 / d["value"] * 1e3) < 1e-9 * d["ms_per_step"] + 1e-12


def test_reference_arm_on_another_rank_does_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out.strip() == ""
