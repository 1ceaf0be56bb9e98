"""bench.py host logic on the CPU: the oracle slice runner, the reference arm's
JSON line, and the max-over-ranks timing across two gloo ranks."""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, REPO)

import bench  # noqa: E402
import oracle  # noqa: E402
from counting_sort_bucketization_gb300 import workloads as wl  # noqa: E402


@pytest.mark.parametrize("S", [256, 64, 100])
def test_slices_of_a_pass_equal_the_pass(S):
    w = wl.WORKLOADS["tiny"]
    inp = wl.make(w)
    r = bench.OracleRunner(w, inp)
    r.recv[:] = 0xEE
    r.out[:] = 0xEEEE
    nslices = -(-w.num_tokens // S)
    done = sum(r.step(i, S) for i in range(nslices))
    assert done == w.num_tokens
    full = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment)
    rows = full["total_rows"]
    x = inp["x"].view(torch.uint8).numpy().reshape(w.num_tokens, -1)
    _, recv, _ = oracle.permute(x, full["dst_slot"], full["expert_offset"], full["expert_count"], rows)
    np.testing.assert_array_equal(r.recv[:rows], recv)
    eo = oracle.expert_scale(recv.view(np.uint16), full["expert_offset"], inp["expert_scale"].numpy())
    np.testing.assert_array_equal(r.out, oracle.combine(eo, full["dst_slot"], inp["weights"].numpy()))


def test_reference_arm_prints_one_line(capsys):
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "4", "--warmup", "1",
                "--ref-seconds", "2"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["steps"] == 4 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    got = bench.reduce_max(float(rank + 1) * 1.5, world, torch.device("cpu"))
    bench.barrier(world)
    results[rank] = got
    torch.distributed.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(results) == {0: 3.0, 1: 3.0}



def test_reference_arm_other_ranks_exit_without_work(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "0"])
    assert capsys.readouterr().out.strip() == ""


def test_clock_window_summarises_only_its_region_and_waits_for_a_short_one():
    """The clock record of a timed region: the samples taken inside it, their
    median, maximum and throttle reasons; a region shorter than the sampling
    period gets the first sample after its start, which the summary waits for."""
    import threading
    import time

    cs = bench.ClockSampler(0)
    cs.source, cs.period = "synthetic", 0.005
    t = time.perf_counter()
    cs.samples = [(t - 2.0, 1500.0, 2070.0, 0x0, 100.0),          # before: not counted
                  (t - 1.0, 2070.0, 2070.0, 0x4, 900.0),          # inside [t-1.5, t-0.5]
                  (t - 0.9, 2000.0, 2070.0, 0x8 | 0x20, 950.0)]   # inside, two slowdown reasons
    w = cs.window(t - 1.5, t - 0.5)
    assert w["samples"] == 2 and w["sm_mhz"] == 2035.0 and w["sm_max_mhz"] == 2070.0 and w["sm_mhz_min"] == 2000.0
    assert w["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"] and w["power_w_max"] == 950.0

    def late():
        time.sleep(0.01)
        cs.samples.append((time.perf_counter(), 2070.0, 2070.0, 0x0, 400.0))

    threading.Thread(target=late).start()
    t0 = time.perf_counter()
    w = cs.window(t0, t0 + 0.001)          # ends before any sample: waits for the next one
    assert w["samples"] == 1 and w["sm_mhz"] == 2070.0 and w["reasons"] == []


def test_step_gaps_steady_state_and_stalls():
    # completion times of a loop: 6.3 ms steps with one 34.1 ms stall; the
    # first step (ramp) is left out of the statistics
    g = bench.step_gaps([7.0, 13.3, 19.6, 25.9, 60.0, 66.3, 72.6])
    assert g["median_ms"] == pytest.approx(6.3)
    assert g["mean_ms"] == pytest.approx((72.6 - 7.0) / 6)
    assert g["stalls_ms"] == [34.1]
    assert bench.step_gaps([1.0, 2.0, 3.0])["stalls_ms"] == []
