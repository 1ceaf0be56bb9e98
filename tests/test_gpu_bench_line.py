"""bench.py's native JSON line on a GB300: one line, with every key the
benchmark contract asks for and the types it asks for (a short run of the
decode workload: 5 timed steps after 3 warm-up steps, one other workload's
clocked loop)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _number(v):
    return isinstance(v, (int, float)) and not isinstance(v, bool)


def test_native_line_keeps_the_contract():
    proc = subprocess.run([sys.executable, os.path.join(REPO, "bench.py"), "--workload", "decode", "--steps", "5",
                           "--warmup", "3", "--e2e-steps", "5", "--e2e-trials", "3", "--breakdown-steps", "5",
                           "--cpu-seconds", "1", "--cpu-max-passes", "1", "--per-config-only", "decode/non-expand",
                           "--per-config-steps", "20"],
                          cwd=REPO, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, proc.stdout
    d = json.loads(lines[0])
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert _number(d["value"]) and d["value"] > 0 and _number(d["ms_per_step"]) and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "bf16" and d["data"] == "synthetic" and d["config"]["workload"] == "decode"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert _number(rf["achieved"]) and _number(rf["peak"]) and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None or _number(rf["traffic"])
    e2e = d["e2e"]
    assert _number(e2e["value"]) and e2e["value"] > 0 and e2e["unit"] == "tokens/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert isinstance(d["gpu_launches"], int) and d["gpu_launches"] >= 5 * 3
    assert "clocks" in d
    assert e2e["link_ceiling_tokens_per_s"] > 0 and 0 < e2e["frac_of_link"]
    assert len(e2e["trials"]) == 3 and e2e["steps"] == 5
    assert sorted(t["tokens_per_s"] for t in e2e["trials"])[1] == pytest.approx(e2e["value"])
    for t in e2e["trials"]:
        assert t["steady_step_ms"] > 0 and t["link_steady_step_ms"] > 0
        assert isinstance(t["stalls_ms"], list) and isinstance(t["link_stalls_ms"], list)
    assert e2e["link"]["steps_both_directions"] == 5 and e2e["link"]["steady_step_ms_both_directions"] > 0
    assert _number(d["host_enqueue_us_per_step"]) and d["host_enqueue_us_per_step"] > 0
    gr = d["graph"]
    assert gr["steps"] == 5 and gr["ms_per_step"] > 0 and gr["host_us_per_replay"] > 0
    assert set(d["rooflines"]) == {"permute", "combine"}
    N = d["config"]["num_tokens"]
    assert d["combine_tokens_per_s"] == pytest.approx(N / (d["kernels_ms"]["combine"] / 1e3))
    assert d["dispatch_tokens_per_s"] == pytest.approx(N / ((d["kernels_ms"]["layout"] + d["kernels_ms"]["permute"]) / 1e3))
    for r in d["rooflines"].values():
        assert r["bound"] == "hbm" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    clk = d["clocks"]
    assert clk is not None and clk["samples"] >= 1 and _number(clk["sm_mhz"]) and isinstance(clk["reasons"], list)
    pc = d["per_config"]
    assert list(pc) == ["decode/non-expand"]
    ne = pc["decode/non-expand"]
    assert ne["steps"] == 20 and ne["config"]["layout_mode"] == "non-expand"
    assert "permute_ranks" in ne["kernels_ms"] and ne["clocks"] is not None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["unit"] == "tokens/s" and _number(cb["value"])
