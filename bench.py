"""Benchmark of the MoE dispatch layout hot path on GB300.

One step = one pass of the whole path over one batch of the workload:
count -> scan (offsets + slot maps) -> permute (expand-mode row scatter with
zero padding) -> combine (weighted top-k gather back to token order), each a
launch of this library through its C ABI.  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Multi-GPU (torchrun, one process per GPU): replicas.  Logical ranks are
partitions of one GPU's buffer, so there is no data-path collective; each
process runs its own batch (weak scaling) and timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

from counting_sort_bucketization_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE dispatch permute tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20          # > 2x the 129 MB L2

# DRAM traffic of the permute kernel from ncu captures (dram__bytes_read.sum +
# dram__bytes_write.sum) per launch, by workload and layout mode, tied to the
# kernel sources they were measured on.  bench reports null if they changed
# or the workload was not captured.
PERMUTE_TRAFFIC = {"sha256": "84d1af49c0472e56db817dec3fd9e137f27bff7bb16289179472e7b8226b4aae",
                   "bytes_per_launch": {"decode": 58_915_840 + 646_384_640,
                                        "decode/non-expand": 58_925_568 + 249_672_704,
                                        "skewed": 235_471_616 + 1_841_223_936,
                                        "prefill_fp8": 243_337_984 + 1_997_432_064}}
PERMUTE_SOURCES = ["counting_sort_bucketization_gb300/csrc/permute_kernel.cu",
                   "counting_sort_bucketization_gb300/csrc/ptx.cuh",
                   "counting_sort_bucketization_gb300/csrc/common.cuh"]


# ---------------------------------------------------------------- helpers
def host_info() -> dict:
    """The host the CPU baseline ran on: its CPU count and RAM (for the record; the
    baseline itself is single-threaded)."""
    info = {"host_cpus": os.cpu_count(), "host_arch": platform.machine()}
    try:
        pages, size = os.sysconf("SC_PHYS_PAGES"), os.sysconf("SC_PAGE_SIZE")
        info["host_ram_gb"] = round(pages * size / 1e9, 1)
    except (ValueError, OSError, AttributeError):
        info["host_ram_gb"] = None
    return info


def sources_sha256(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(REPO, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def reduce_max(v: float, world: int, device) -> float:
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def measured_peaks() -> dict:
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def config_of(w: wl.Workload) -> dict:
    return {"workload": w.name, "num_tokens": w.num_tokens, "topk": w.topk, "num_experts": w.num_experts,
            "num_ranks": w.num_ranks, "alignment": w.alignment, "hidden": w.hidden, "row_dtype": w.row_dtype,
            "routing": w.routing, "mask_prob": w.mask_prob,
            "l2": "flushed before every step, outside the step's events: 256 MiB written, then a second "
                  "256 MiB buffer read, so each step starts with a cold L2 holding no dirty lines"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict | None:
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags) if fl == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ CPU oracle
class OracleRunner:
    """The oracle (oracle/oracle.c as it stands, single-threaded) on a workload.

    A full pass = layout of all N tokens, permute of every row with zero
    padding, combine of every token.  ``step(i, S)`` runs slice i of S tokens
    of a pass: the first slice of each pass also does the layout and the
    gap-row zeroing, so ceil(N / S) consecutive steps are exactly one pass.
    """

    def __init__(self, w: wl.Workload, inp: dict):
        import oracle
        self.oracle = oracle
        self.w = w
        self.idx = inp["topk_idx"].numpy()
        self.x = inp["x"].contiguous().view(torch.uint8).numpy().reshape(w.num_tokens, -1)
        self.sf = inp["sf"].contiguous().view(torch.uint8).numpy().reshape(w.num_tokens, -1) \
            if inp["sf"] is not None else None
        self.weights = inp["weights"].numpy()
        self.cap = wl.worst_case_rows(w)
        self.lay = oracle.layout(self.idx, w.num_experts, w.num_ranks, w.alignment, capacity_rows=self.cap)
        rows = self.lay["total_rows"]
        self.recv = np.zeros((self.cap, self.x.shape[1]), np.uint8)
        self.recv_sf = np.zeros((self.cap, self.sf.shape[1]), np.uint8) if self.sf is not None else None
        oracle.permute(self.x, self.lay["dst_slot"], self.lay["expert_offset"], self.lay["expert_count"], rows,
                       sf_bytes=self.sf, out=self.recv, out_sf=self.recv_sf)
        self.combine = w.row_dtype == "bf16"
        if self.combine:   # the stand-in expert's output (harness, untimed)
            self.eo = oracle.expert_scale(self.recv[:rows].view(np.uint16), self.lay["expert_offset"],
                                          inp["expert_scale"].numpy())
            self.out = np.zeros((w.num_tokens, w.hidden), np.uint16)

    def step(self, i: int, S: int) -> int:
        o, w = self.oracle, self.w
        N = w.num_tokens
        nslices = -(-N // S)
        j = i % nslices
        t0, t1 = j * S, min(N, (j + 1) * S)
        if j == 0:
            self.lay = o.layout(self.idx, w.num_experts, w.num_ranks, w.alignment, capacity_rows=self.cap)
        lay = self.lay
        rows = lay["total_rows"]
        o.permute(self.x[t0:t1], lay["dst_slot"][t0:t1], lay["expert_offset"], lay["expert_count"], rows,
                  sf_bytes=None if self.sf is None else self.sf[t0:t1], zero_pad=(j == 0),
                  out=self.recv, out_sf=self.recv_sf)
        if self.combine:
            o.combine(self.eo, lay["dst_slot"][t0:t1], self.weights[t0:t1], out=self.out[t0:t1])
        return t1 - t0

    def time_passes(self, min_seconds: float, max_passes: int) -> tuple[float, int]:
        """Full passes until min_seconds elapsed (at least one); returns (tokens/s, passes)."""
        N = self.w.num_tokens
        passes, t_start = 0, time.perf_counter()
        while True:
            self.step(0, N)
            passes += 1
            el = time.perf_counter() - t_start
            if el >= min_seconds or passes >= max_passes:
                return passes * N / el, passes


# ------------------------------------------------------------ native run
def algorithmic_bytes(w: wl.Workload, lay, sf_col_major: bool = False) -> dict:
    """Bytes each kernel must move, from the layout of this batch.  With
    ``sf_col_major`` the permute moves the rows only and the scale factors
    go column-major in their own kernel (reads each routed token's scale
    row, writes every receive row's words, reads the inverse map)."""
    N, K, E = w.num_tokens, w.topk, w.num_experts
    dst = lay.dst_slot[: N * K].view(N, K)
    valid = dst >= 0
    P = int(valid.sum().item())
    n_tok = int(valid.any(dim=1).sum().item())
    rows = int(lay.total_rows.item())
    rb = w.row_bytes + (0 if sf_col_major else w.sf_row_bytes)
    permute = n_tok * rb + P * rb + (rows - P) * rb + N * K * 4 + 2 * (E + 1) * 4
    sf_cm = n_tok * w.sf_row_bytes + rows * w.sf_row_bytes + rows * 4 if sf_col_major else 0
    combine = P * w.hidden * 2 + N * K * 8 + N * w.hidden * 2 if w.row_dtype == "bf16" else 0
    count = N * K * 8
    scan = N * K * 8 + N * K * 4 + rows * 4
    return {"permute": permute, "combine": combine, "count": count, "scan": scan, "sf_col_major": sf_cm,
            "P": P, "rows": rows,
            "tokens_routed": n_tok}


def run_layout_only(args, local):
    """Time the layout step alone (ids in, maps out): small on the device at any
    workload size, so it is also the command to profile the layout kernels with."""
    from counting_sort_bucketization_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    if args.tokens is not None:
        w = w.replace(num_tokens=args.tokens)
    idx = wl.draw_topk_idx(w, wl.SEEDS[w.name]).to(dev)
    if args.ids_int32:
        idx = idx.to(torch.int32)
    lay = binding.Layout(w, wl.worst_case_rows(w), device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    times = {}
    # The two-call API (count, then scan) takes int64 ids only.
    for fused in ((True,) if args.ids_int32 else (True, False)):
        evs = []
        for i in range(args.warmup + args.steps):
            flush_w.zero_()
            flush_r.max()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            lay.build(idx, fused=fused)
            b.record()
            if i >= args.warmup:
                evs.append((a, b))
        torch.cuda.synchronize(dev)
        times["one_call" if fused else "two_calls"] = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    assert lay.error() == 0
    cfg = config_of(w)
    cfg["ids"] = "int32" if args.ids_int32 else "int64"
    print(json.dumps({"mode": "layout-only", "config": cfg, "steps": args.steps, "warmup": args.warmup,
                      "layout_ms": times, "tokens_per_s": {k: w.num_tokens / (v / 1e3) for k, v in times.items()}}),
          flush=True)


def run_native(args, rank, world, local):
    from counting_sort_bucketization_gb300 import binding

    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    seed = wl.SEEDS[w.name] + 1000 * rank
    inp = wl.make(w, seed)
    N, K, H = w.num_tokens, w.topk, w.hidden
    cap = wl.worst_case_rows(w)
    stream = torch.cuda.current_stream(dev)

    idx_d = inp["topk_idx"].to(dev)
    x_d = inp["x"].to(dev)
    sf_d = inp["sf"].to(dev) if inp["sf"] is not None else None
    wt_d = inp["weights"].to(dev)
    lay = binding.Layout(w, cap, device=dev)
    recv = torch.empty((cap, H), dtype=x_d.dtype, device=dev)
    recv_sf = torch.empty((cap, sf_d.shape[1]), dtype=sf_d.dtype, device=dev) if sf_d is not None else None
    sf_cm = args.sf_col_major and sf_d is not None
    # Column-major scale factors: the permute moves rows only, then its own kernel.
    recv_sf_cm = binding.new_sf_col_major(sf_d.shape[1], cap, device=dev) if sf_cm else None
    perm_sf, perm_recv_sf = (None, None) if sf_cm else (sf_d, recv_sf)
    do_combine = w.row_dtype == "bf16"
    out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    # The combine's input: the round-trip stand-in expert applied once to a
    # dispatched buffer (harness, untimed): rows of expert e scaled by 1 + e/384.
    lay.build(idx_d)
    lay.permute(x_d, recv, sf_d, recv_sf)
    rows = int(lay.total_rows.item())
    eo = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
    if do_combine:
        off = lay.expert_offset.to(torch.int64)
        row_e = torch.searchsorted(off[1:], torch.arange(rows, device=dev), right=True)
        eo[:rows] = (recv[:rows].float() * inp["expert_scale"].to(dev)[row_e][:, None]).to(torch.bfloat16)
    assert lay.error() == 0, "device error during set-up"
    # Non-expand mode: one row per (token, rank reached), rank-contiguous, no padding.
    ne = args.non_expand
    if ne:
        ne_cap = N * w.num_ranks
        lay.rank_rows(idx_d, capacity_rows=ne_cap)
        recv_ne = torch.empty((ne_cap, H), dtype=x_d.dtype, device=dev)
        recv_ne_sf = torch.empty((ne_cap, sf_d.shape[1]), dtype=sf_d.dtype, device=dev) if sf_d is not None else None
        lay.permute_ranks(x_d, recv_ne, sf_d, recv_ne_sf)
        assert lay.error() == 0, "device error during set-up"
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.max()

    # The step's kernels in order, one event after each (and one before the
    # first): every timed interval holds exactly one step of the path.
    stages = [("layout", lambda: lay.build(idx_d))]
    if ne:
        stages += [("rank_rows", lambda: lay.rank_rows(idx_d, capacity_rows=ne_cap)),
                   ("permute_ranks", lambda: lay.permute_ranks(x_d, recv_ne, sf_d, recv_ne_sf))]
    else:
        stages.append(("permute", lambda: lay.permute(x_d, recv, perm_sf, perm_recv_sf)))
        if sf_cm:
            stages.append(("sf_col_major", lambda: lay.permute_sf_col_major(sf_d, recv_sf_cm)))
        if do_combine:
            stages.append(("combine", lambda: lay.combine(eo, wt_d, out)))

    # The timed steps carry one event before and one after the whole step: an
    # event between two kernels would stand between them in the stream and
    # stop the next one from starting during the previous one's tail (the
    # programmatic dependent launch the kernels are built for).  Per-kernel
    # times come from a second loop with an event after every kernel.
    def step(ev):
        ev[0].record(stream)
        for _, run in stages:
            run()
        ev[1].record(stream)

    def step_per_kernel(ev):
        ev[0].record(stream)
        for i, (_, run) in enumerate(stages):
            run()
            ev[i + 1].record(stream)

    new_events = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for _ in range(args.warmup):
        flush_l2()
        step(new_events(2))
    torch.cuda.synchronize(dev)
    assert lay.error() == 0, "device error during warm-up"

    evs = [new_events(2) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = binding.kernel_launches()
    sampler = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.__enter__()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        step(evs[i])
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
    launches = binding.kernel_launches() - launches0
    err = lay.error()
    assert err == 0, f"device error {err} in the timed region"

    step_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])   # ms
    ms_per_step = reduce_max(float(step_ms.mean()), world, dev)
    # Per-kernel breakdown (untimed for the headline): the same steps with an event after each kernel.
    n_break = min(args.steps, args.breakdown_steps)
    kevs = [new_events(len(stages) + 1) for _ in range(n_break)]
    for i in range(n_break):
        flush_l2()
        step_per_kernel(kevs[i])
    torch.cuda.synchronize(dev)
    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(stages))] for e in kevs])   # ms
    kern_ms = dict(zip([name for name, _ in stages], per.mean(axis=0).tolist()))
    ab = algorithmic_bytes(w, lay, sf_cm)
    if ne:
        # each routed token's row read once, one row written per (token, rank reached), the slots read
        rows_ne = int(lay.rank_psum[-1].item())
        rb_all = w.row_bytes + w.sf_row_bytes
        ab["permute_ranks"] = ab["tokens_routed"] * rb_all + rows_ne * rb_all + N * w.topk * 4
        ab["rows_non_expand"] = rows_ne
    value = world * N / (ms_per_step / 1e3)
    dispatch_ms = sum(v for k, v in kern_ms.items() if k != "combine")

    # End to end through the public API with host buffers: pinned ids, rows
    # and weights in, the combined tokens back (dispatch-only workloads: the
    # receive rows back).  moe_dispatch_from_host and moe_combine_to_host
    # overlap the copies with the kernels in chunks, and HostPipeline keeps
    # `--e2e-lanes` batches in flight so one batch's copy back overlaps the
    # next one's copy in.  Every copy is inside the timed region; each
    # step's working set (rows, receive buffer) is larger than L2.
    idx_h = inp["topk_idx"].pin_memory()
    x_h = inp["x"].pin_memory()
    sf_h = inp["sf"].pin_memory() if inp["sf"] is not None else None
    wt_h = inp["weights"].pin_memory()
    out_shape, out_dtype = ((N, H), torch.bfloat16) if do_combine else ((cap, H), x_d.dtype)
    lanes = max(1, args.e2e_lanes)
    outs_h = [torch.empty(out_shape, dtype=out_dtype).pin_memory() for _ in range(lanes)]
    h2d = idx_h.numel() * 8 + x_h.numel() * x_h.element_size() + wt_h.numel() * 4 + \
        (sf_h.numel() * 4 if sf_h is not None else 0)
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    chunk_of = lambda n_chunks: -(-N // max(1, n_chunks))
    e2e_line = None
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    expert = (lambda lay_, recv_, recv_sf_: eo) if do_combine else None

    def e2e_ms_per_step(n_lanes, n_chunks):
        pipe = binding.HostPipeline(w, cap, H, x_dtype=x_d.dtype, sf_cols=sf_d.shape[1] if sf_d is not None else 0,
                                    lanes=n_lanes, chunk_tokens=chunk_of(n_chunks), device=dev)
        for i in range(2 * n_lanes):
            pipe.submit(idx_h, x_h, wt_h, outs_h[i % n_lanes], expert, sf_h)
        pipe.join(stream)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(e2e_steps):
            pipe.submit(idx_h, x_h, wt_h, outs_h[i % n_lanes], expert, sf_h)
        pipe.join(stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        assert pipe.errors() == [0] * n_lanes, "device error in the end-to-end steps"
        return a.elapsed_time(b) / e2e_steps

    if not ne:   # the end-to-end leg is the expand path's
        e2e_step_ms = reduce_max(e2e_ms_per_step(lanes, args.e2e_chunks), world, dev)
        # One batch in flight, its copies overlapped with the kernels in 4 chunks: the reference point.
        e2e_one_ms = reduce_max(e2e_ms_per_step(1, 4), world, dev)
        e2e_line = {"value": world * N / (e2e_step_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps, "chunks": args.e2e_chunks,
                    "batches_in_flight": lanes,
                    "value_one_batch_in_flight_4_chunks": world * N / (e2e_one_ms / 1e3),
                    "api": "HostPipeline: moe_dispatch_from_host + moe_combine_to_host" if do_combine
                    else "HostPipeline: moe_dispatch_from_host + receive rows copied back"}

    if rank != 0:
        return
    peaks = measured_peaks()
    dom = "permute_ranks" if ne else "permute"
    permute_s = kern_ms[dom] / 1e3
    achieved = ab[dom] / permute_s / 1e9
    traffic = None
    if PERMUTE_TRAFFIC.get("sha256") == sources_sha256(PERMUTE_SOURCES):
        traffic = PERMUTE_TRAFFIC["bytes_per_launch"].get(w.name + ("/non-expand" if ne else ""))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w),
        "roofline": {"kernel": "permute_dyn_kernel", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "peak_source": peaks["source"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic, "algorithmic_bytes_per_launch": ab[dom],
                     "note": "algorithmic bytes include the launch's last writes, still dirty in L2 when it "
                             "ends (written back during the next kernel): frac can read a little above 1 and "
                             "traffic below the algorithmic bytes"},
        "kernels_ms": dict(kern_ms) if ne else {
            "layout": kern_ms["layout"], "permute": kern_ms["permute"],
            "sf_col_major": kern_ms.get("sf_col_major"), "combine": kern_ms.get("combine")},
        "kernels_gbs": {"permute_ranks": achieved} if ne else {
            "permute": ab["permute"] / permute_s / 1e9,
            "sf_col_major": (ab["sf_col_major"] / (kern_ms["sf_col_major"] / 1e3) / 1e9) if sf_cm else None,
            "combine": (ab["combine"] / (kern_ms["combine"] / 1e3) / 1e9) if do_combine else None},
        "breakdown": {"steps": n_break, "sum_of_kernels_ms": float(sum(kern_ms.values())),
                      "note": "kernels_ms come from separate steps with an event after every kernel; those "
                              "events keep each kernel from starting during the previous one's tail, so their "
                              "sum exceeds ms_per_step, which is timed per whole step"},
        "dispatch_tokens_per_s": world * N / (dispatch_ms / 1e3),
        "layout": {"valid_pairs": ab["P"], "rows": ab["rows"], "tokens_routed": ab["tokens_routed"]},
        "e2e": e2e_line,
        "gpu_launches": launches,
        "wall_s_timed_region": t_wall,
        "clocks": sampler.summary() if sampler else None,
    }
    if ne:
        line["config"]["layout_mode"] = "non-expand: one row per (token, rank reached), rank-contiguous, no padding"
        line["layout"]["rows_non_expand"] = ab["rows_non_expand"]
    if sf_d is not None:
        line["config"]["sf_layout"] = ("column-major, ld = capacity rounded up to 4 words (e2e leg: row-major)"
                                       if sf_cm else "row-major, moved by the permute")
    if world == 1 and not args.no_cpu_baseline and not ne:
        runner = OracleRunner(w, inp)
        tps, passes = runner.time_passes(args.cpu_seconds, args.cpu_max_passes)
        line["cpu_baseline"] = {"value": tps, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{passes} full pass(es) of the {w.name} workload ({N} tokens): "
                                          f"layout, permute with zero padding, combine; single-threaded C",
                                **host_info()}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: rank 0 times it, other ranks exit."""
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    inp = wl.make(w, wl.SEEDS[w.name])
    runner = OracleRunner(w, inp)
    N = w.num_tokens
    # Size each step so that warm-up + timed steps take about args.ref_seconds.
    t0 = time.perf_counter()
    runner.step(0, N)
    t_full = time.perf_counter() - t0
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    S = N
    while S > 1 and t_full * S / N > budget:
        S //= 2
    for i in range(args.warmup):
        runner.step(i, S)
    nslices = -(-N // S)
    tokens = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        tokens += runner.step(i, S)   # step 0 is the first slice of a pass
    el = time.perf_counter() - t0
    value = tokens / el
    sample = (f"each step: {S} of the {N} tokens of the {w.name} workload through the oracle's permute and "
              f"combine; every {nslices} steps also the full layout and gap-row zeroing, so {nslices} steps "
              f"= one full pass; single-threaded C")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                         **host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(wl.WORKLOADS), default="decode")
    ap.add_argument("--e2e-steps", type=int, default=200,
                    help="timed end-to-end steps (enough that filling and draining the batches in flight is ~1 %%)")
    ap.add_argument("--e2e-chunks", type=int, default=1, help="token chunks the host copies are split into")
    ap.add_argument("--e2e-lanes", type=int, default=3, help="batches in flight in the end-to-end leg")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-max-passes", type=int, default=20)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--sf-col-major", action="store_true",
                    help="fp8 workloads: scale factors column-major (TMA-aligned) by their own kernel")
    ap.add_argument("--ids-int32", action="store_true", help="--layout-only: int32 routing ids")
    ap.add_argument("--tokens", type=int, default=None,
                    help="--layout-only: tokens per batch instead of the workload's (same routing recipe)")
    ap.add_argument("--breakdown-steps", type=int, default=300,
                    help="steps of the per-kernel breakdown loop (after the timed steps)")
    ap.add_argument("--non-expand", action="store_true",
                    help="time the non-expand layout instead: layout, rank rows, rank-contiguous permute")
    ap.add_argument("--layout-only", action="store_true",
                    help="time only the layout step (count, scan, maps) on the chosen workload")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    assert args.steps >= 1 and args.warmup >= 0
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.layout_only:
        if rank == 0:
            run_layout_only(args, local)
    else:
        run_native(args, rank, world, local)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
