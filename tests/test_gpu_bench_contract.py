"""bench.py's JSON line (our arm) on a reduced workload: one line, the keys the driver reads, and
their consistency (value = windows / time, e2e with its copy sizes, the roofline object, clocks,
the launch count, the read probe). The full default run takes minutes; this one, seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line():
    cmd = [sys.executable, "bench.py", "--tokens", "2048", "--steps", "5", "--warmup", "3", "--no-sweep", "--no-next",
           "--no-cpu-baseline", "--workload-calls", "20"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "e2e", "roofline", "clocks", "gpu_launches", "hbm_read_probe"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["unit"] == "windows/s" and d["scaling"] == "weak" and d["vs_baseline"] is None  # not the 16374 workload
    assert abs(d["value"] - 2048 / (d["ms_per_step"] * 1e-3)) <= 1e-6 * d["value"]
    assert d["config"]["token_num"] == 2048 and "workload" in d["config"]
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert abs(rf["frac_of_read_probe"] - rf["achieved"] / rf["read_probe_gbs"]) < 1e-9
    assert rf["algorithmic_bytes_per_launch"] == 2048 * (128 * 1024 * 4 + 64 + 256 + 584)
    assert d["gpu_launches"] == 2 * 5  # planning pass and compress kernel per step (2048 > 8 per SM)
    assert d["hbm_read_probe"]["gbs"] == rf["read_probe_gbs"] and d["hbm_read_probe"]["bytes"] > 0
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    # the five synthetic workloads: windows/s = active windows / µs per call, GB/s = bytes / µs per call
    w = d["workloads"]
    assert set(w) == {"tiny", "decode", "mixed", "varlen", "varlen16k"}
    assert [w[k]["windows"] for k in ("tiny", "decode")] == [4, 128]
    for name, row in w.items():
        assert row["windows"] > 0 and row["tokens"] >= row["windows"], name
        for col in ("cold", "l2_hot"):
            c = row[col]
            assert c["calls"] == 20 and c["us_min_chunk"] <= c["us_median_chunk"], (name, col)
            assert abs(c["windows_per_s"] - row["windows"] / (c["us_per_call"] * 1e-6)) <= 1e-3 * c["windows_per_s"]
            gbs = row["algorithmic_bytes_per_call"] / (c["us_per_call"] * 1e-6) / 1e9
            assert abs(c["algorithmic_gbs"] - gbs) <= 1e-3 * gbs + 0.1, (name, col)
