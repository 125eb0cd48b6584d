"""bench.py on a GPU prints one JSON line with every field of its contract."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_prints_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5",
                          "--warmup", "3", "--no-extras", "--no-cpu"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches", "ceilings"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # one or two launches per step (the long-context headline adds a summary pass)
    import selective_state_space_132_b300 as ssm
    c = d["config"]
    per_call = ssm.scan_launches_per_call(c["batch"], c["seqlen"], c["d_inner"], c["d_state"])
    assert d["gpu_launches"] == 5 * per_call
    # the scan is dispatch-bound: the ALU roofline, with the HBM one beside it
    r = d["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "state-updates/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert abs(r["achieved"] - d["value"]) <= 0.05 * d["value"]
    h = r["hbm"]
    assert h["bound"] == "hbm" and h["unit"] == "GB/s" and 0 < h["frac"] < 1.5
    assert abs(h["frac"] - h["achieved"] / h["peak"]) < 1e-9
    # ncu occupancy figures only for the sources they were captured on
    occ = r["profiled_occupancy"]
    import bench
    if r["source_hash"] in bench.PROFILED_OCCUPANCY:
        assert occ == bench.PROFILED_OCCUPANCY[r["source_hash"]].get(c["workload"])
    else:
        assert occ is None
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "workload" in d["config"] and "l2" in d["config"]
