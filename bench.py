"""Benchmark of the MoE dispatch layout hot path on GB300.

One step = one pass of the whole path over one batch of the workload:
layout (count -> aligned prefix sums -> slot maps) -> permute (expand-mode
row scatter with zero padding) -> combine (weighted top-k gather back to
token order), each a launch of this library through its C ABI.  Prints ONE
JSON line.  The default workload is the largest single-GPU one, round-trip
(131072 tokens, top-8 of 384 experts, hidden 4096 bf16); the line also
carries a clocked entry for every other large workload (``per_config``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload roundtrip]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm
    python bench.py --profile --workload roundtrip --tokens 16384 ...   # small footprint, for ncu

Multi-GPU (torchrun, one process per GPU): replicas.  Logical ranks are
partitions of one GPU's buffer, so there is no data-path collective; each
process runs its own batch (weak scaling) and timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import threading
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
DEFAULT_WORKLOAD = "roundtrip"      # the largest workload that fits one GPU

# DRAM traffic per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum,
# one metric pass) of each HBM-bound kernel, by workload, tied to the sources
# it was measured on: a kernel whose sources changed since reports null.  The
# captures ran `bench.py --profile` at full size, caches flushed before each
# captured kernel (ncu's default); each figure is the mean of two launches.
HOW = "ncu, one metric pass (dram__bytes_read.sum + dram__bytes_write.sum), full size, bench.py --profile, caches flushed before the kernel (ncu default); mean of two launches"
TRAFFIC = {
    "permute_dyn_kernel": {
        "sources": ["counting_sort_bucketization_gb300/csrc/permute_kernel.cu",
                    "counting_sort_bucketization_gb300/csrc/ptx.cuh",
                    "counting_sort_bucketization_gb300/csrc/common.cuh"],
        "sha256": "1fffee62edae026b5ca95720bf44f6a7005c57c475b74538e2986c35734c6757",
        "bytes_per_launch": {"roundtrip": {"bytes": 9273815552, "how": HOW}, "decode": {"bytes": 704104576, "how": HOW}, "skewed": {"bytes": 2075054464, "how": HOW}, "prefill_fp8": {"bytes": 2239759872, "how": HOW}, "prefill_fp8/sf-col-major": {"bytes": 2169645440, "how": HOW}, "decode/non-expand": {"bytes": 306171264, "how": HOW}},
    },
    "combine": {   # combine_bulk_kernel (round-trip, skewed) or combine_kernel (decode), by batch size
        "sources": ["counting_sort_bucketization_gb300/csrc/combine_kernel.cu",
                    "counting_sort_bucketization_gb300/csrc/ptx.cuh",
                    "counting_sort_bucketization_gb300/csrc/common.cuh"],
        "sha256": "088673f399f2a3677b81538aed54aeb2aa922f9fefa85e7585eeec034566d335",
        "bytes_per_launch": {"roundtrip": {"bytes": 9192338560, "how": HOW}, "skewed": {"bytes": 1876517888, "how": HOW}, "decode": {"bytes": 477036800, "how": HOW}},
    },
    "sf_col_major_kernel": {
        "sources": ["counting_sort_bucketization_gb300/csrc/sf_layout_kernel.cu",
                    "counting_sort_bucketization_gb300/csrc/ptx.cuh",
                    "counting_sort_bucketization_gb300/csrc/common.cuh"],
        "sha256": "efff3440144641a56f852de8f68d122acfa0cf96531f3c0882b1463378b547f9",
        "bytes_per_launch": {"prefill_fp8/sf-col-major": {"bytes": 11648640, "how": HOW}},
    },
}

# Kernels behind each stage of a step (the layout's depend on the batch size).
STAGE_KERNEL = {"permute": "permute_dyn_kernel", "permute_ranks": "permute_dyn_kernel",
                "combine": "combine_bulk_kernel or combine_kernel", "sf_col_major": "sf_col_major_kernel",
                "layout": "count_tiles + scan_columns + rank_maps, or layout_fused_kernel",
                "rank_rows": "rank_rows_kernel"}
STAGE_TRAFFIC = {"permute": "permute_dyn_kernel", "permute_ranks": "permute_dyn_kernel", "combine": "combine",
                 "sf_col_major": "sf_col_major_kernel"}
# Batches of at least this many tokens per resident CTA of the bulk combine
# (3 per SM) take that kernel; smaller ones the register kernel.
COMBINE_BULK_MIN_TOKENS_PER_CTA, COMBINE_BULK_CTAS_PER_SM = 12, 3
HBM_STAGES = ("permute", "permute_ranks", "combine", "sf_col_major")

# The other large workloads, each with a short clocked loop of its own in the
# default run: (key, workload, layout mode).
PER_CONFIG = [("decode", "decode", {}), ("skewed", "skewed", {}), ("prefill_fp8", "prefill_fp8", {}),
              ("decode/non-expand", "decode", {"non_expand": True}),
              ("prefill_fp8/sf-col-major", "prefill_fp8", {"sf_col_major": True})]


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


def traffic_of(kernel: str, key: str):
    """(bytes per launch, how it was taken) for a kernel on a workload, or (None, why not)."""
    t = TRAFFIC.get(kernel)
    if t is None:
        return None, "not an HBM-bound kernel"
    entry = t["bytes_per_launch"].get(key)
    if entry is None:
        return None, "not captured on this workload"
    if t["sha256"] != sources_sha256(t["sources"]):
        return None, "sources changed since the capture"
    return entry["bytes"], entry["how"]


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


# ----------------------------------------------------------------- clocks
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock, its maximum, power and clock-event (throttle) reasons of one
    GPU, sampled every ``period_s`` by a background thread through NVML (read
    only), with ``nvidia-smi -lms 100`` as the fallback when NVML cannot be
    loaded.  ``window(t0, t1)`` summarises the samples taken between two
    ``time.perf_counter()`` readings."""

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []            # (perf_counter, sm_mhz, sm_max_mhz, reasons mask, power W)
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        self._nvml = None
        self._handle = None
        self._index = device_index

    # -- NVML through ctypes (no Python package needed)
    def _open_nvml(self) -> bool:
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        handle = ctypes.c_void_p()
        found = False
        try:   # the CUDA device's PCI address, so that CUDA_VISIBLE_DEVICES cannot mislead the index
            p = torch.cuda.get_device_properties(self._index)
            bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
            found = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(handle)) == 0
        except (AttributeError, RuntimeError):
            found = False
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self._index), ctypes.byref(handle)) != 0:
            return False
        self._nvml, self._handle = lib, handle
        try:
            self._reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return True

    def _poll_nvml(self):
        lib, h = self._nvml, self._handle
        sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0      # NVML_CLOCK_SM
            ok = ok and lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
            ok = ok and self._reasons_fn(h, ctypes.byref(rs)) == 0
            power = pw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
            if ok:
                self.samples.append((t, float(sm.value), float(mx.value), int(rs.value), power))
            self._stop.wait(self.period)

    def start(self):
        if self._open_nvml():
            self.source = f"nvml every {self.period * 1e3:.0f} ms"
            self._thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self._thread.start()
            return self
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
        try:
            self._file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self._smi = subprocess.Popen(["nvidia-smi", f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self._index)],
                                         stdout=self._file, stderr=subprocess.DEVNULL)
            self._smi_t0 = time.perf_counter()
            self._smi_lines = 0
            self.source = "nvidia-smi every 100 ms"
            time.sleep(0.3)
        except OSError:
            self._smi = None
        return self

    def _read_smi(self):
        """nvidia-smi's complete lines so far (one every 100 ms from its start) as samples."""
        bits = (0x8, 0x40, 0x20, 0x4)
        with open(self._file.name) as f:
            lines = f.readlines()
        for i in range(self._smi_lines, len(lines)):
            if not lines[i].endswith("\n"):
                break
            self._smi_lines = i + 1
            parts = [p.strip() for p in lines[i].split(",")]
            if len(parts) < 7:
                continue
            try:
                mask = sum(b for b, fl in zip(bits, parts[3:7]) if fl == "Active")
                self.samples.append((self._smi_t0 + i * 0.1, float(parts[0]), float(parts[1]), mask,
                                     float(parts[2])))
            except ValueError:
                continue

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
            self._read_smi()
            os.unlink(self._file.name)
            self._smi = None

    def window(self, t0: float, t1: float) -> dict | None:
        """Samples taken between t0 and t1; for a region shorter than the sampling
        period, the first sample after t0 (waiting up to a few periods for it)."""
        if self.source is None:
            return None
        period = 0.1 if self._smi is not None else self.period
        deadline = time.perf_counter() + 4 * period + 0.05
        while True:
            if self._smi is not None:
                self._read_smi()
            if any(s[0] >= t0 for s in self.samples) or time.perf_counter() > deadline:
                break
            time.sleep(period / 2)
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:   # a window shorter than the period: the first sample after its start
            after = [s for s in self.samples if s[0] >= t0]
            inside = after[:1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        reasons = sorted({name for s in inside for bit, name in _REASONS.items() if s[3] & bit})
        powers = [s[4] for s in inside if s[4] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "sm_mhz_min": min(s[1] for s in inside), "reasons": reasons, "samples": len(inside),
                "power_w_max": max(powers) if powers else None, "source": self.source}


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
    """Bytes each kernel must move, from the layout of this batch.

    permute: each routed token's row (and scale row) read once, one row
    written per valid pair and per alignment-gap row, the slots and offsets
    read; combine: one expert-output row read per valid pair, slots and
    weights read, one output row written per token.  With ``sf_col_major`` the
    permute moves the rows only and the scale factors go column-major in
    their own kernel (each routed token's scale row read, every receive row's
    words written, the inverse map read)."""
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
    layout = N * K * 8 + N * K * 4 + rows * 4
    return {"permute": permute, "combine": combine, "layout": layout, "sf_col_major": sf_cm,
            "P": P, "rows": rows, "tokens_routed": n_tok}


class Case:
    """One workload resident on the device, with its stages ready to run.

    ``eo_alias`` makes the combine read the receive buffer itself instead of a
    separate stand-in expert output (same rows, same bytes; only for the small
    profiling footprint)."""

    def __init__(self, w: wl.Workload, seed: int, dev, non_expand=False, sf_col_major=False, eo_alias=False,
                 keep_inputs=False):
        from counting_sort_bucketization_gb300 import binding
        self.w, self.dev = w, dev
        self.non_expand = non_expand
        inp = wl.make(w, seed)
        self.inp = inp if keep_inputs else None
        N, H = w.num_tokens, w.hidden
        cap = wl.worst_case_rows(w)
        self.cap = cap
        self.idx_d = inp["topk_idx"].to(dev)
        self.x_d = inp["x"].to(dev)
        sf_d = inp["sf"].to(dev) if inp["sf"] is not None else None
        self.sf_d = sf_d
        self.wt_d = inp["weights"].to(dev)
        lay = binding.Layout(w, cap, device=dev)
        self.lay = lay
        self.recv = torch.empty((cap, H), dtype=self.x_d.dtype, device=dev)
        recv_sf = torch.empty((cap, sf_d.shape[1]), dtype=sf_d.dtype, device=dev) if sf_d is not None else None
        self.sf_cm = sf_col_major and sf_d is not None
        recv_sf_cm = binding.new_sf_col_major(sf_d.shape[1], cap, device=dev) if self.sf_cm else None
        perm_sf, perm_recv_sf = (None, None) if self.sf_cm else (sf_d, recv_sf)
        self.do_combine = w.row_dtype == "bf16" and not non_expand
        self.out = torch.empty((N, H), dtype=torch.bfloat16, device=dev) if self.do_combine else None
        lay.build(self.idx_d)
        lay.permute(self.x_d, self.recv, sf_d, recv_sf)
        self.eo = None
        if self.do_combine:
            if eo_alias:
                self.eo = self.recv
            else:
                # The round-trip stand-in expert applied once (harness, untimed): rows of
                # expert e scaled by 1 + e/384, in pieces to bound the temporaries.
                rows = int(lay.total_rows.item())
                self.eo = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
                off = lay.expert_offset.to(torch.int64)
                scale = inp["expert_scale"].to(dev)
                for r0 in range(0, rows, 1 << 16):
                    r1 = min(rows, r0 + (1 << 16))
                    row_e = torch.searchsorted(off[1:], torch.arange(r0, r1, device=dev), right=True)
                    self.eo[r0:r1] = (self.recv[r0:r1].float() * scale[row_e][:, None]).to(torch.bfloat16)
        assert lay.error() == 0, "device error during set-up"
        if non_expand:
            ne_cap = N * w.num_ranks
            lay.rank_rows(self.idx_d, capacity_rows=ne_cap)
            self.recv_ne = torch.empty((ne_cap, H), dtype=self.x_d.dtype, device=dev)
            self.recv_ne_sf = torch.empty((ne_cap, sf_d.shape[1]), dtype=sf_d.dtype, device=dev) \
                if sf_d is not None else None
            lay.permute_ranks(self.x_d, self.recv_ne, sf_d, self.recv_ne_sf)
            assert lay.error() == 0, "device error during set-up"
        # The step's kernels in order.
        self.stages = [("layout", lambda: lay.build(self.idx_d))]
        if non_expand:
            self.stages += [("rank_rows", lambda: lay.rank_rows(self.idx_d, capacity_rows=ne_cap)),
                            ("permute_ranks", lambda: lay.permute_ranks(self.x_d, self.recv_ne, sf_d,
                                                                        self.recv_ne_sf))]
        else:
            self.stages.append(("permute", lambda: lay.permute(self.x_d, self.recv, perm_sf, perm_recv_sf)))
            if self.sf_cm:
                self.stages.append(("sf_col_major", lambda: lay.permute_sf_col_major(sf_d, recv_sf_cm)))
            if self.do_combine:
                self.stages.append(("combine", lambda: lay.combine(self.eo, self.wt_d, self.out)))
        self.ab = algorithmic_bytes(w, lay, self.sf_cm)
        if non_expand:
            rows_ne = int(lay.rank_psum[-1].item())
            rb_all = w.row_bytes + w.sf_row_bytes
            # each routed token's row read once, one row written per (token, rank reached), the slots read
            self.ab["permute_ranks"] = self.ab["tokens_routed"] * rb_all + rows_ne * rb_all + N * w.topk * 4
            self.ab["rows_non_expand"] = rows_ne
        self.key = w.name + ("/non-expand" if non_expand else "") + ("/sf-col-major" if self.sf_cm else "")

    def run(self):
        for _, fn in self.stages:
            fn()


class Flusher:
    """Writes one 256 MiB buffer and reads another, so that the next step starts
    with a cold L2 that holds no dirty lines."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def new_events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_case(case: Case, steps: int, warmup: int, flush: Flusher, world: int, sampler: ClockSampler | None,
              breakdown_steps: int, enqueue_steps: int) -> dict:
    """Warm-up, then exactly ``steps`` timed steps (one event pair around each
    whole step, L2 flushed before it), then the per-kernel breakdown and the
    host's enqueue time per step."""
    from counting_sort_bucketization_gb300 import binding
    dev, stream = case.dev, torch.cuda.current_stream(case.dev)

    # One event before and one after the whole step: an event between two
    # kernels would stand between them in the stream and stop the next one
    # from starting during the previous one's tail (the programmatic
    # dependent launch the kernels are built for).
    def step(ev):
        ev[0].record(stream)
        case.run()
        ev[1].record(stream)

    for _ in range(warmup):
        flush()
        step(new_events(2))
    torch.cuda.synchronize(dev)
    assert case.lay.error() == 0, "device error during warm-up"
    evs = [new_events(2) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = binding.kernel_launches()
    t0 = time.perf_counter()
    for i in range(steps):
        flush()
        step(evs[i])
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    barrier(world)
    launches = binding.kernel_launches() - launches0
    assert case.lay.error() == 0, "device error in the timed region"
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    ms_per_step = reduce_max(float(step_ms.mean()), world, dev)

    # Per-kernel breakdown: separate steps with an event after every kernel.
    n_break = max(1, min(steps, breakdown_steps))
    kevs = [new_events(len(case.stages) + 1) for _ in range(n_break)]
    for i in range(n_break):
        flush()
        ev = kevs[i]
        ev[0].record(stream)
        for j, (_, fn) in enumerate(case.stages):
            fn()
            ev[j + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(case.stages))] for e in kevs])
    kern_ms = dict(zip([name for name, _ in case.stages], per.mean(axis=0).tolist()))

    # Host enqueue time: the calls of a step back to back with no flush, no
    # events and no synchronisation inside the loop.
    n_enq = max(1, min(steps, enqueue_steps))
    torch.cuda.synchronize(dev)
    e0 = time.perf_counter()
    for _ in range(n_enq):
        case.run()
    e1 = time.perf_counter()
    torch.cuda.synchronize(dev)
    assert case.lay.error() == 0, "device error in the breakdown steps"
    return {"ms_per_step": ms_per_step, "step_ms_min": float(step_ms.min()), "step_ms_max": float(step_ms.max()),
            "kernels_ms": kern_ms, "launches": launches, "wall_s": t1 - t0,
            "clocks": sampler.window(t0, t1) if sampler is not None else None,
            "breakdown_steps": n_break, "host_enqueue_us_per_step": (e1 - e0) / n_enq * 1e6,
            "host_enqueue_steps": n_enq}


def kernel_of(case: Case, stage: str) -> str:
    if stage != "combine":
        return STAGE_KERNEL[stage]
    sms = torch.cuda.get_device_properties(case.dev).multi_processor_count
    bulk = case.w.num_tokens >= COMBINE_BULK_MIN_TOKENS_PER_CTA * COMBINE_BULK_CTAS_PER_SM * sms
    return "combine_bulk_kernel" if bulk else "combine_kernel"


def roofline_of(case: Case, stage: str, kern_ms: dict, peak: dict) -> dict:
    kernel = kernel_of(case, stage)
    t_s = kern_ms[stage] / 1e3
    ab = case.ab[stage]
    achieved = ab / t_s / 1e9
    traffic, how = traffic_of(STAGE_TRAFFIC[stage], case.key)
    r = {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peak["hbm_gbs"],
         "peak_source": peak["source"], "unit": "GB/s", "frac": achieved / peak["hbm_gbs"], "traffic": traffic,
         "traffic_source": how, "algorithmic_bytes_per_launch": ab, "launch_ms": kern_ms[stage]}
    if traffic is not None:
        r["achieved_dram"] = traffic / t_s / 1e9
        r["frac_dram"] = r["achieved_dram"] / peak["hbm_gbs"]
    if stage == "sf_col_major":
        r["note"] = ("its data stays in L2: each token's scale row comes from DRAM once and then from L2 for "
                     "every further slot, and the column writes are still in L2 when it ends; the kernel moves "
                     f"{2 * case.ab['rows'] * case.w.sf_row_bytes / 1e6:.1f} MB through L2 (gathered reads + column "
                     "writes), so neither fraction measures it against its own bound")
    elif stage == "combine":
        r["note"] = ("the combine starts while the permute's last writes (up to ~60 MB) are still dirty in L2, and "
                     "their write-back runs during it; traffic, captured with caches flushed, leaves that out")
    return r


def case_summary(case: Case, t: dict, peak: dict, world: int) -> dict:
    """Throughput and per-kernel rooflines of one timed case."""
    N = case.w.num_tokens
    kern = t["kernels_ms"]
    hbm = [s for s in HBM_STAGES if s in kern]
    rl = {s: roofline_of(case, s, kern, peak) for s in hbm}
    dispatch_ms = sum(v for k, v in kern.items() if k != "combine")
    return {
        "config": config_of(case.w), "ms_per_step": t["ms_per_step"], "tokens_per_s": world * N / (t["ms_per_step"] / 1e3),
        "dispatch_tokens_per_s": world * N / (dispatch_ms / 1e3),
        **({"combine_tokens_per_s": world * N / (kern["combine"] / 1e3)} if "combine" in kern else {}),
        "kernels_ms": kern, "kernels_gbs": {s: rl[s]["achieved"] for s in hbm},
        "kernels_frac": {s: rl[s]["frac"] for s in hbm},
        "kernels_frac_dram": {s: rl[s].get("frac_dram") for s in hbm},
        "rooflines": rl,
        "layout": {"valid_pairs": case.ab["P"], "rows": case.ab["rows"], "tokens_routed": case.ab["tokens_routed"],
                   **({"rows_non_expand": case.ab["rows_non_expand"]} if case.non_expand else {})},
        "clocks": t["clocks"], "steps": None, "host_enqueue_us_per_step": t["host_enqueue_us_per_step"],
    }


def step_gaps(ends_ms) -> dict:
    """Steady state and stalls of a loop from the completion time of each step
    (ms from the loop's start): the median step, the mean, and the steps that
    took more than twice the median."""
    gaps = [b - a for a, b in zip([0.0] + ends_ms[:-1], ends_ms)][1:]   # the first step includes the ramp
    med = float(np.median(gaps))
    return {"median_ms": med, "mean_ms": float(np.mean(gaps)),
            "stalls_ms": [round(g, 1) for g in gaps if g > 2 * med]}


def link_ceiling(h2d, d2h, reps: int, dev, steps: int) -> dict:
    """Pinned host<->device copies of exactly one step's bytes: each direction
    alone (``reps`` steps), then both at once on two streams for ``steps``
    steps, as many as an end-to-end trial, with an event after each (the
    ceiling of any pipeline that moves these bytes, measured over as long a
    stretch as the trial, so that the link's own stalls count in both).
    ``h2d`` is a list of (device dst, host src), ``d2h`` of (host dst, device src)."""
    main = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(directions, n):
        # Each step forks the directions onto their streams and joins them again.
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        ends = new_events(n)
        a.record(main)
        for i in range(n):
            for s, pairs in directions:
                s.wait_stream(main)
                with torch.cuda.stream(s):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
            for s, _ in directions:
                main.wait_stream(s)
            ends[i].record(main)
        torch.cuda.synchronize(dev)
        t = [a.elapsed_time(e) for e in ends]
        return t[-1] / n / 1e3, t   # s per step, completion times (ms)

    bi = sum(d.numel() * d.element_size() for d, _ in h2d)
    bo = sum(d.numel() * d.element_size() for d, _ in d2h)
    timed([(s_in, h2d), (s_out, d2h)], reps)   # warm-up
    t_in, _ = timed([(s_in, h2d)], reps)
    t_out, _ = timed([(s_out, d2h)], reps)
    t_both, ends = timed([(s_in, h2d), (s_out, d2h)], steps)
    g = step_gaps(ends)
    return {"h2d_gbs": bi / t_in / 1e9, "d2h_gbs": bo / t_out / 1e9, "both_gbs": (bi + bo) / t_both / 1e9,
            "step_ms_both_directions": t_both * 1e3, "steady_step_ms_both_directions": g["median_ms"],
            "stalls_ms": g["stalls_ms"], "reps_one_direction": reps, "steps_both_directions": steps}


def run_e2e(case: Case, args, world: int, dev) -> dict:
    """End to end through the public API with host buffers: pinned ids, rows and
    weights in, the combined tokens back (dispatch-only workloads: the receive
    rows back).  moe_dispatch_from_host and moe_combine_to_host overlap the
    copies with the kernels, and HostPipeline keeps ``--e2e-lanes`` batches in
    flight so one batch's copy back overlaps the next one's copy in.  Every
    copy is inside the timed region; each step's working set is larger than L2."""
    from counting_sort_bucketization_gb300 import binding
    w, inp = case.w, case.inp
    N, H = w.num_tokens, w.hidden
    stream = torch.cuda.current_stream(dev)
    idx_h = inp["topk_idx"].pin_memory()
    x_h = inp["x"].pin_memory()
    sf_h = inp["sf"].pin_memory() if inp["sf"] is not None else None
    wt_h = inp["weights"].pin_memory()
    do_combine = case.do_combine
    out_shape, out_dtype = ((N, H), torch.bfloat16) if do_combine else ((case.cap, H), case.x_d.dtype)
    lanes = max(1, args.e2e_lanes)
    outs_h = [torch.empty(out_shape, dtype=out_dtype).pin_memory() for _ in range(lanes)]
    h2d = idx_h.numel() * 8 + x_h.numel() * x_h.element_size() + wt_h.numel() * 4 + \
        (sf_h.numel() * 4 if sf_h is not None else 0)
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    chunk_of = lambda n_chunks: -(-N // max(1, n_chunks))
    # Its own step count (not --steps): filling and draining the batches in
    # flight costs about one step's worth of one-way link time, so a few dozen
    # steps keep that a few per cent of the measurement.
    e2e_steps = max(3, args.e2e_steps)
    eo = case.eo
    expert = (lambda lay_, recv_, recv_sf_: eo) if do_combine else None
    sf_cols = case.sf_d.shape[1] if case.sf_d is not None else 0

    h2d_pairs = [(case.idx_d, idx_h), (case.x_d, x_h), (case.wt_d, wt_h)] + \
        ([(case.sf_d, sf_h)] if sf_h is not None else [])
    d2h_src = case.out if do_combine else case.recv

    def trials_ms(n_lanes, n_chunks, n_trials, with_link):
        """Per-step ms of each trial of e2e_steps steps on one pipeline (and, after
        each trial, the host link's ceiling for exactly one step's bytes)."""
        pipe = binding.HostPipeline(w, case.cap, H, x_dtype=case.x_d.dtype, sf_cols=sf_cols, lanes=n_lanes,
                                    chunk_tokens=chunk_of(n_chunks), device=dev)
        for i in range(2 * n_lanes):
            pipe.submit(idx_h, x_h, wt_h, outs_h[i % n_lanes], expert, sf_h)
        pipe.join(stream)
        torch.cuda.synchronize(dev)
        out = []
        for _ in range(n_trials):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ends = new_events(e2e_steps)
            a.record(stream)
            for i in range(e2e_steps):
                li = pipe.next_lane
                pipe.submit(idx_h, x_h, wt_h, outs_h[li], expert, sf_h)
                ends[i].record(pipe.lane(li)["stream"])   # batch i's result is in host memory
            pipe.join(stream)
            b.record(stream)
            torch.cuda.synchronize(dev)
            gaps = step_gaps([a.elapsed_time(e) for e in ends])
            link = link_ceiling(h2d_pairs, [(outs_h[0], d2h_src)], 5, dev, e2e_steps) if with_link else None
            out.append((a.elapsed_time(b) / e2e_steps, link, gaps))
        assert pipe.errors() == [0] * n_lanes, "device error in the end-to-end steps"
        del pipe
        torch.cuda.empty_cache()
        return out

    # The host link is shared with the rest of the machine and its rate moves
    # between runs, so the leg runs several trials, each followed by a
    # measurement of the link's own ceiling for one step's bytes; the line
    # reports the median trial and every trial with its ceiling.
    trials = trials_ms(lanes, args.e2e_chunks, max(1, args.e2e_trials), True)
    order = sorted(range(len(trials)), key=lambda i: trials[i][0])
    med_ms, link, _ = trials[order[len(order) // 2]]
    step_ms = reduce_max(med_ms, world, dev)
    # One batch in flight, its copies overlapped with the kernels in 4 chunks: the reference point.
    one_ms = reduce_max(trials_ms(1, 4, 1, False)[0][0], world, dev)
    value = world * N / (step_ms / 1e3)
    ceiling = N / (link["step_ms_both_directions"] / 1e3) * world
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "chunks": args.e2e_chunks, "batches_in_flight": lanes, "ms_per_step": step_ms,
            "value_one_batch_in_flight_4_chunks": world * N / (one_ms / 1e3),
            "link": link, "link_ceiling_tokens_per_s": ceiling, "frac_of_link": value / ceiling,
            "trials": [{"tokens_per_s": world * N / (ms / 1e3), "link_both_gbs": lk["both_gbs"],
                        "frac_of_link": lk["step_ms_both_directions"] / ms,
                        "steady_step_ms": gp["median_ms"], "stalls_ms": gp["stalls_ms"],
                        "link_steady_step_ms": lk["steady_step_ms_both_directions"],
                        "link_stalls_ms": lk["stalls_ms"]}
                       for ms, lk, gp in trials],
            "note": f"median of {len(trials)} trials of {e2e_steps} steps; link and ceiling from the link "
                    f"measurement right after that trial: {e2e_steps} steps of the same bytes in both directions "
                    "with no kernels, so that stalls of the host link (steps over twice the median) weigh on "
                    "both alike; steady_step_ms is a trial's median step",
            "api": "HostPipeline: moe_dispatch_from_host + moe_combine_to_host" if do_combine
            else "HostPipeline: moe_dispatch_from_host + receive rows copied back"}


def run_graph(case: Case, steps: int, warmup: int, flush: Flusher, world: int) -> dict:
    """The same step captured once as a CUDA graph (binding.StepGraph) and
    replayed: device time per step (events around each replay, L2 flushed
    before it) and the host's time to enqueue one replay."""
    from counting_sort_bucketization_gb300 import binding
    dev = case.dev
    eo = case.eo
    g = binding.StepGraph(case.w, case.cap, case.w.hidden, expert=(lambda lay, recv, sf: eo) if case.do_combine
                          else None, x_dtype=case.x_d.dtype, device=dev)
    g.topk_idx.copy_(case.idx_d)
    g.x.copy_(case.x_d)
    g.weights.copy_(case.wt_d)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        flush()
        g.replay()
    evs = [new_events(2) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        flush()
        evs[i][0].record(stream)
        g.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    n = max(1, min(steps, 50))
    h0 = time.perf_counter()
    for _ in range(n):
        g.replay()
    h1 = time.perf_counter()
    torch.cuda.synchronize(dev)
    assert g.error() == 0, "device error in the graph replays"
    ms = reduce_max(float(np.mean([e[0].elapsed_time(e[1]) for e in evs])), world, dev)
    res = {"ms_per_step": ms, "tokens_per_s": world * case.w.num_tokens / (ms / 1e3), "steps": steps,
           "host_us_per_replay": (h1 - h0) / n * 1e6,
           "note": "the step's kernels (and the stand-in expert's, if any) captured once with binding.StepGraph "
                   "and replayed; host_us_per_replay is the wall time of enqueueing one replay"}
    del g
    torch.cuda.empty_cache()
    return res


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
    flush = Flusher(dev)
    times = {}
    # The two-call API (count, then scan) takes int64 ids only.
    for fused in ((True,) if args.ids_int32 else (True, False)):
        evs = []
        for i in range(args.warmup + args.steps):
            flush()
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
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    if args.tokens is not None:
        w = w.replace(num_tokens=args.tokens)
    seed = wl.SEEDS[w.name] + 1000 * rank
    profile = args.profile
    sampler = ClockSampler(local).start() if (rank == 0 and not args.no_clocks and not profile) else None
    peak = measured_peaks()
    flush = Flusher(dev)
    case = Case(w, seed, dev, non_expand=args.non_expand, sf_col_major=args.sf_col_major, eo_alias=profile,
                keep_inputs=not profile)
    t = time_case(case, args.steps, args.warmup, flush, world, sampler, args.breakdown_steps, args.enqueue_steps)
    summ = case_summary(case, t, peak, world)
    kern = t["kernels_ms"]
    # The line's roofline: the HBM-bound kernel that takes the longest.
    dom = max((s for s in HBM_STAGES if s in kern), key=lambda s: kern[s])
    e2e_line = None
    if not args.non_expand and not profile and not args.no_e2e:
        e2e_line = run_e2e(case, args, world, dev)
    graph_line = None
    if not args.non_expand and case.sf_d is None and not profile and not args.no_graph:
        graph_line = run_graph(case, args.steps, args.warmup, flush, world)
    line = {
        "metric": METRIC, "value": summ["tokens_per_s"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.row_dtype == "bf16" else "fp8 rows (bytes moved)",
        "data": "synthetic", "config": config_of(w),
        "roofline": {**summ["rooflines"][dom],
                     "note": "the HBM-bound kernel with the longest time; algorithmic bytes include the "
                             "launch's last writes, still dirty in L2 when it ends (written back during the "
                             "next kernel), so frac can read a little above 1 and traffic below the "
                             "algorithmic bytes; frac_dram uses the measured DRAM bytes instead"},
        "rooflines": summ["rooflines"],
        "kernels_ms": kern, "kernels_gbs": summ["kernels_gbs"], "kernels_frac": summ["kernels_frac"],
        "kernels_frac_dram": summ["kernels_frac_dram"],
        "breakdown": {"steps": t["breakdown_steps"], "sum_of_kernels_ms": float(sum(kern.values())),
                      "note": "kernels_ms come from separate steps with an event after every kernel; those "
                              "events keep each kernel from starting during the previous one's tail, so their "
                              "sum can exceed ms_per_step, which is timed per whole step"},
        "dispatch_tokens_per_s": summ["dispatch_tokens_per_s"],
        **({"combine_tokens_per_s": summ["combine_tokens_per_s"]} if "combine_tokens_per_s" in summ else {}),
        "layout": summ["layout"],
        "host_enqueue_us_per_step": t["host_enqueue_us_per_step"],
        "graph": graph_line,
        "host_enqueue_note": f"wall time of {t['host_enqueue_steps']} steps' calls (Python binding + C ABI + "
                            "launches) enqueued back to back, divided by the steps; no synchronisation inside",
        "e2e": e2e_line,
        "gpu_launches": t["launches"],
        "wall_s_timed_region": t["wall_s"],
        "step_ms_range": [t["step_ms_min"], t["step_ms_max"]],
        "clocks": t["clocks"],
    }
    if args.non_expand:
        line["config"]["layout_mode"] = "non-expand: one row per (token, rank reached), rank-contiguous, no padding"
    if case.sf_d is not None:
        line["config"]["sf_layout"] = ("column-major, ld = capacity rounded up to 4 words (e2e leg: row-major)"
                                       if case.sf_cm else "row-major, moved by the permute")
    if profile:
        line["config"]["profile"] = "small footprint: no e2e leg, no CPU baseline, the combine reads the receive buffer"
    inp_cpu = case.inp
    del case
    torch.cuda.empty_cache()

    # The other large workloads: a clocked loop of their own each.
    if world == 1 and not profile and not args.no_per_config:
        per = {}
        only = set(args.per_config_only.split(",")) if args.per_config_only else None
        for key, name, opts in PER_CONFIG:
            if (key == line["config"]["workload"] and not opts) or (only is not None and key not in only):
                continue
            cw = wl.WORKLOADS[name]
            c = Case(cw, wl.SEEDS[name], dev, **opts)
            steps = max(args.steps, args.per_config_steps)
            ct = time_case(c, steps, max(3, args.warmup), flush, world, sampler, args.breakdown_steps,
                           args.enqueue_steps)
            s = case_summary(c, ct, peak, world)
            s["steps"], s["warmup"] = steps, max(3, args.warmup)
            s["config"] = {"workload": name, **{k: v for k, v in config_of(cw).items() if k != "l2"},
                           **({"layout_mode": "non-expand"} if opts.get("non_expand") else {}),
                           **({"sf_layout": "column-major"} if opts.get("sf_col_major") else {})}
            per[key] = s
            del c
            torch.cuda.empty_cache()
        line["per_config"] = per
    if sampler is not None:
        sampler.stop()

    if rank != 0:
        return
    if world == 1 and not args.no_cpu_baseline and not args.non_expand and not profile:
        runner = OracleRunner(w, inp_cpu)
        tps, passes = runner.time_passes(args.cpu_seconds, args.cpu_max_passes)
        line["cpu_baseline"] = {"value": tps, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{passes} full pass(es) of the {w.name} workload ({w.num_tokens} tokens): "
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
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(wl.WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per batch instead of the workload's (same recipe); for small profiling cases")
    ap.add_argument("--e2e-steps", type=int, default=60,
                    help="timed end-to-end steps (filling and draining the batches in flight is ~1 step of them)")
    ap.add_argument("--e2e-chunks", type=int, default=1, help="token chunks the host copies are split into")
    ap.add_argument("--e2e-trials", type=int, default=5, help="end-to-end trials; the line reports the median")
    ap.add_argument("--e2e-lanes", type=int, default=3, help="batches in flight in the end-to-end leg")
    ap.add_argument("--no-e2e", action="store_true", help="leave out the end-to-end leg")
    ap.add_argument("--no-graph", action="store_true", help="leave out the CUDA-graph replay of the step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-max-passes", type=int, default=20)
    ap.add_argument("--ref-seconds", type=float, default=75.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="leave out the other workloads' clocked loops")
    ap.add_argument("--per-config-only", default=None,
                    help="comma-separated keys of the other workloads' loops to run (default: all of "
                         + ", ".join(k for k, _, _ in PER_CONFIG) + ")")
    ap.add_argument("--per-config-steps", type=int, default=300,
                    help="timed steps of each other workload's loop (at least --steps)")
    ap.add_argument("--profile", action="store_true",
                    help="small device footprint for ncu: no end-to-end leg, no CPU baseline, no other "
                         "workloads, no clock sampling; the combine reads the receive buffer")
    ap.add_argument("--sf-col-major", action="store_true",
                    help="fp8 workloads: scale factors column-major (TMA-aligned) by their own kernel")
    ap.add_argument("--ids-int32", action="store_true", help="--layout-only: int32 routing ids")
    ap.add_argument("--breakdown-steps", type=int, default=300,
                    help="steps of the per-kernel breakdown loop (after the timed steps)")
    ap.add_argument("--enqueue-steps", type=int, default=50, help="steps of the host enqueue-time loop")
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
