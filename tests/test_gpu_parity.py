"""CUDA path vs. the CPU oracle, through the C ABI, on seeded inputs.

Layout, maps and permuted rows must match bit for bit.  Combine must stay
within max-abs 1e-2 and relative 4e-3 of the oracle under fp32
accumulation; both sides run the same fp32 fused multiply-add chain in
ascending k, so it is also checked to be bit-identical.

At full workload sizes the maps are compared whole; permuted rows are
compared whole where the oracle's receive buffer fits comfortably in host
memory, and otherwise (round-trip, 8 GB) through the property
recv_x[row] == x[src_idx[row]] on every row plus the oracle on sampled
tokens.  The launch configuration is the one bench.py times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
ATOL, RTOL = 1e-2, 4e-3


@pytest.fixture(scope="session", autouse=True)
def _built():
    build.build()
    binding.load_library()


# ------------------------------------------------------------------ helpers
def u8(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a (CPU or GPU) tensor, one row per leading index."""
    t = t.detach().contiguous().cpu()
    n = t.shape[0] if t.dim() else 1
    return t.view(torch.uint8).numpy().reshape(n, -1) if t.numel() else np.zeros((n, 0), np.uint8)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


SENTINEL_MAP = -9   # canary in src_idx: entries past the layout's rows must keep it


def run_gpu_layout(w, idx_cpu, cap, fused=True):
    lay = binding.Layout(w, cap, device=DEV)
    lay.src_idx.fill_(SENTINEL_MAP)
    lay.src_canary = True
    return lay.build(idx_cpu.to(DEV), fused=fused)


def assert_layout_matches(lay, ref, w, check_src=True):
    N, K = w.num_tokens, w.topk
    for key in ("expert_count", "rank_count", "expert_offset", "rank_psum"):
        np.testing.assert_array_equal(getattr(lay, key).cpu().numpy(), ref[key], err_msg=key)
    assert int(lay.total_rows.item()) == ref["total_rows"]
    np.testing.assert_array_equal(lay.dst_slot[: N * K].cpu().numpy().reshape(N, K), ref["dst_slot"])
    if check_src:
        rows = ref["total_rows"]
        src = lay.src_idx.cpu().numpy()
        np.testing.assert_array_equal(src[:rows], ref["src_idx"])
        if getattr(lay, "src_canary", False):
            assert np.all(src[rows:] == SENTINEL_MAP), "src_idx written past the layout's rows"


def scale_rows_on_gpu(recv, expert_offset, scale, rows):
    """Round-trip stand-in expert on the GPU (harness, not the method): row i of
    segment e becomes bf16(float(row) * scale[e])."""
    off = expert_offset.to(torch.int64)
    row_expert = torch.searchsorted(off[1:], torch.arange(rows, device=recv.device), right=True)
    s = scale.to(recv.device)[row_expert]
    return (recv[:rows].float() * s[:, None]).to(torch.bfloat16)


def check_combine(got_bits: np.ndarray, want_bits: np.ndarray):
    g = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (want_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs(g - r)
    assert err.max(initial=0.0) <= ATOL
    assert np.all(err <= RTOL * np.abs(r) + 1e-30) or err.max(initial=0.0) == 0
    np.testing.assert_array_equal(got_bits, want_bits)


def full_case(w: wl.Workload, seed: int, combine=True, cap=None, fused=True):
    """Everything compared whole against the oracle (sizes the host can hold twice)."""
    inp = wl.make(w, seed)
    idx = inp["topk_idx"]
    cap = cap if cap is not None else wl.worst_case_rows(w)
    ref = oracle.layout(idx.numpy(), w.num_experts, w.num_ranks, w.alignment, capacity_rows=cap)
    assert ref["status"] == oracle.OK
    lay = run_gpu_layout(w, idx, cap, fused=fused)
    rows = ref["total_rows"]
    x = inp["x"].to(DEV)
    recv = torch.full((cap, w.hidden), 0x5A, dtype=torch.uint8, device=DEV).view(x.dtype) \
        if x.element_size() == 1 else torch.full((cap, w.hidden), -7.0, dtype=x.dtype, device=DEV)
    sf = inp["sf"].to(DEV) if inp["sf"] is not None else None
    recv_sf = torch.full((cap, sf.shape[1]), -3.0, dtype=torch.float32, device=DEV) if sf is not None else None
    lay.permute(x, recv, sf, recv_sf)
    assert lay.error() == 0
    assert_layout_matches(lay, ref, w)
    _, ref_recv, ref_sf = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"],
                                         ref["expert_count"], rows,
                                         sf_bytes=u8(inp["sf"]) if sf is not None else None)
    np.testing.assert_array_equal(u8(recv[:rows]), ref_recv)
    if sf is not None:
        np.testing.assert_array_equal(u8(recv_sf[:rows]), ref_sf)
    # Canaries: receive rows past the layout's keep their fill, and the inputs are not written.
    fill = 0x5A if x.element_size() == 1 else None
    tail = u8(recv[rows:])
    assert np.all(tail == fill) if fill is not None else bool(torch.all(recv[rows:] == -7.0)), \
        "receive rows written past the layout's rows"
    if sf is not None:
        assert bool(torch.all(recv_sf[rows:] == -3.0)), "scale rows written past the layout's rows"
        np.testing.assert_array_equal(u8(sf), u8(inp["sf"]))
    np.testing.assert_array_equal(u8(x), u8(inp["x"]))
    if combine and w.row_dtype == "bf16":
        scale = inp["expert_scale"]
        eo = scale_rows_on_gpu(recv, lay.expert_offset, scale, rows)
        ref_eo = oracle.expert_scale(ref_recv.view(np.uint16).reshape(rows, w.hidden), ref["expert_offset"],
                                     scale.numpy())
        np.testing.assert_array_equal(bf16_bits(eo), ref_eo)
        # one guard row past the N output rows
        out_guard = torch.full((w.num_tokens + 1, w.hidden), 5.0, dtype=torch.bfloat16, device=DEV)
        out = out_guard[: w.num_tokens]
        lay.combine(eo, inp["weights"].to(DEV), out)
        assert lay.error() == 0
        ref_out = oracle.combine(ref_eo, ref["dst_slot"], inp["weights"].numpy())
        check_combine(bf16_bits(out), ref_out)
        assert bool(torch.all(out_guard[w.num_tokens] == 5.0)), "combine wrote past its N rows"
    return lay, recv


# ------------------------------------------------------- workload parity
@pytest.mark.parametrize("fused", [True, False], ids=["one_call", "two_calls"])
@pytest.mark.parametrize("name", ["tiny", "decode", "skewed", "prefill_fp8"])
def test_workload_full_parity(name, fused):
    w = wl.WORKLOADS[name]
    full_case(w, wl.SEEDS[name], fused=fused)


def test_roundtrip_full_size():
    """131072 tokens, 384 experts, hidden 4096: maps whole, rows by property and sampled oracle rows."""
    w = wl.WORKLOADS["roundtrip"]
    inp = wl.make(w)
    idx = inp["topk_idx"]
    cap = wl.worst_case_rows(w)
    ref = oracle.layout(idx.numpy(), w.num_experts, w.num_ranks, w.alignment, capacity_rows=cap)
    lay = run_gpu_layout(w, idx, cap)
    assert_layout_matches(lay, ref, w)
    rows = ref["total_rows"]
    x = inp["x"].to(DEV)
    recv = torch.full((cap, w.hidden), -7.0, dtype=torch.bfloat16, device=DEV)
    lay.permute(x, recv)
    assert lay.error() == 0
    x16 = x.view(torch.int16)
    r16 = recv.view(torch.int16)
    src = lay.src_idx[:rows].to(torch.int64)
    step = 1 << 16
    for lo in range(0, rows, step):
        hi = min(rows, lo + step)
        s = src[lo:hi]
        real = s >= 0
        assert torch.equal(r16[lo:hi][real], x16[s[real]]), f"rows {lo}..{hi}"
        assert int(r16[lo:hi][~real].abs().sum().item()) == 0 if (~real).any() else True
    # sampled tokens through the oracle, rows and combine
    rng = np.random.default_rng(4)
    sel = np.sort(rng.choice(w.num_tokens, size=512, replace=False))
    dst = ref["dst_slot"][sel]
    flat = dst[dst >= 0]
    np.testing.assert_array_equal(u8(recv[torch.from_numpy(flat).to(DEV).long()]),
                                  u8(inp["x"])[np.repeat(sel, (dst >= 0).sum(1))])
    eo = scale_rows_on_gpu(recv, lay.expert_offset, inp["expert_scale"], rows)
    out = torch.empty((w.num_tokens, w.hidden), dtype=torch.bfloat16, device=DEV)
    lay.combine(eo, inp["weights"].to(DEV), out)
    assert lay.error() == 0
    # compact the sampled tokens' expert rows; the oracle combines from them
    used = np.unique(flat)
    eo_sel = bf16_bits(eo[torch.from_numpy(used).to(DEV).long()])
    remap = -np.ones(rows, np.int64)
    remap[used] = np.arange(used.size)
    dst_c = np.where(dst >= 0, remap[np.maximum(dst, 0)], -1).astype(np.int32)
    # the stand-in expert's rows, recomputed on the host from x alone
    seg_e = np.searchsorted(ref["expert_offset"], used, side="right") - 1
    xf = torch.from_numpy(u8(inp["x"])[ref["src_idx"][used]].view(np.uint16).view(np.int16)).view(torch.bfloat16)
    want_eo = (xf.float() * inp["expert_scale"][torch.from_numpy(seg_e)][:, None]).to(torch.bfloat16)
    np.testing.assert_array_equal(eo_sel, bf16_bits(want_eo))
    ref_out = oracle.combine_tokens(np.arange(sel.size), eo_sel, dst_c, inp["weights"].numpy()[sel])
    check_combine(bf16_bits(out[torch.from_numpy(sel).to(DEV).long()]), ref_out)


# ------------------------------------------------------------ edge cases
def _w(N, K, E, R, A, H=64, **kw):
    return wl.Workload("edge", N, K, E, R, A, H, **kw)


EDGE = [
    _w(1000, 8, 64, 8, 16),                      # N not a multiple of the tile
    _w(777, 1, 40, 5, 7, H=128),                 # K = 1
    _w(513, 3, 37, 1, 5, H=72),                  # K does not divide 32, E not a multiple of 32
    _w(300, 32, 64, 4, 8, H=32),                 # K = 32, one token per warp chunk
    _w(2000, 6, 1024, 8, 2, H=16),               # E at the build's maximum
    _w(4096, 8, 256, 8, 1, H=8),                 # alignment 1
    _w(700, 4, 24, 6, 64, H=48, mask_prob=0.5),  # heavy masking
    _w(5000, 8, 256, 8, 128, routing="zipf", zipf_s=2.5, mask_prob=0.1, H=32),  # extreme skew
    _w(40, 2, 8, 2, 4, H=8192 * 2),              # rows wider than one 16 KiB bulk slice
    _w(129, 8, 16, 4, 4, H=384, row_dtype="fp8"),  # fp8 rows, 12-byte scale-factor rows
    _w(500, 4, 16, 4, 4096, H=16),               # alignment 4096: nearly every receive row is padding
    _w(1500, 8, 64, 8, 4, H=7168, row_dtype="fp8"),  # rows cut in 2 pieces, scale rows with the first
    _w(3000, 8, 64, 8, 16, H=5000),              # rows cut in 3 pieces, the last one shorter
    _w(40007, 3, 40, 5, 16, H=16),               # two chunks per warp, ragged last tile
    _w(70001, 1, 64, 8, 4, H=16),                # the same with K = 1
    _w(330001, 3, 40, 5, 16, H=16),              # one-call layout in the cooperative kernel, ragged last tile
    _w(1000001, 1, 64, 8, 4, H=16),              # the same with K = 1
]


@pytest.mark.parametrize("fused", [True, False], ids=["one_call", "two_calls"])
@pytest.mark.parametrize("w", EDGE, ids=lambda w: f"N{w.num_tokens}_K{w.topk}_E{w.num_experts}_A{w.alignment}")
def test_edge_parity(w, fused):
    full_case(w, seed=123, fused=fused)


def test_more_tiles_than_fit_at_once():
    """200000 tokens at top-32 make more tiles than can be resident: the one-call
    path falls back to the separate kernels and must give the same layout."""
    w = _w(200000, 32, 64, 4, 16, H=16)
    idx = wl.draw_topk_idx(w, 31)
    ref = oracle.layout(idx.numpy(), 64, 4, 16)
    rref = oracle.rank_layout(idx.numpy(), 64, 4)
    for fused in (True, False):
        lay = run_gpu_layout(w, idx, wl.worst_case_rows(w), fused=fused)
        assert lay.error() == 0
        assert_layout_matches(lay, ref, w)
        # the non-expand map reads the rank prefix this path's column scan wrote
        lay.rank_rows(idx.to(DEV), capacity_rows=rref["total_rows"])
        assert lay.error() == 0
        np.testing.assert_array_equal(lay.rank_slot.cpu().numpy().reshape(200000, 32), rref["rank_slot"])
        np.testing.assert_array_equal(lay.rank_src.cpu().numpy(), rref["rank_src"])


@pytest.mark.parametrize("w", [
    _w(5, 8, 256, 8, 128, H=16),              # one tile; ~255 experts hold only gap rows
    _w(32, 8, 256, 8, 128, H=16),             # one full tile, 32768 receive rows for 256 pairs
    _w(512, 8, 256, 8, 128, H=16),
    _w(736, 8, 256, 8, 128, H=16),
    _w(100, 6, 1024, 1024, 1, H=16),          # E = R = 1024: the largest shared-memory plan of a tile
], ids=lambda w: f"N{w.num_tokens}_E{w.num_experts}_R{w.num_ranks}_A{w.alignment}")
def test_small_batches(w):
    """Small batches at decode routing: few tiles, so each rank CTA writes the gap
    rows of many experts (one warp per expert); the non-expand map follows."""
    idx = wl.draw_topk_idx(w, 41)
    ref = oracle.layout(idx.numpy(), w.num_experts, w.num_ranks, w.alignment)
    before = binding.kernel_launches()
    lay = run_gpu_layout(w, idx, wl.worst_case_rows(w), fused=True)
    assert binding.kernel_launches() - before == 3      # count, column scan, rank
    assert lay.error() == 0
    assert_layout_matches(lay, ref, w)
    rref = oracle.rank_layout(idx.numpy(), w.num_experts, w.num_ranks)
    lay.rank_rows(idx.to(DEV), capacity_rows=rref["total_rows"])
    assert lay.error() == 0
    N, K = w.num_tokens, w.topk
    np.testing.assert_array_equal(lay.rank_slot[: N * K].cpu().numpy().reshape(N, K), rref["rank_slot"])
    np.testing.assert_array_equal(lay.rank_src.cpu().numpy(), rref["rank_src"])


def test_empty_and_all_masked():
    for N, fused in ((0, True), (0, False), (100, True), (100, False)):
        w = _w(N, 4, 16, 4, 8)
        idx = torch.full((N, 4), -1, dtype=torch.int64)
        ref = oracle.layout(idx.numpy(), 16, 4, 8)
        lay = run_gpu_layout(w, idx, 64, fused=fused)
        x = torch.randn(N, 64, device=DEV).to(torch.bfloat16)
        recv = torch.full((64, 64), 3.0, dtype=torch.bfloat16, device=DEV)
        lay.permute(x, recv)
        out = torch.full((N, 64), 5.0, dtype=torch.bfloat16, device=DEV)
        lay.combine(recv, torch.ones(N * 4, device=DEV), out)
        assert lay.error() == 0
        assert_layout_matches(lay, ref, w)
        assert int(lay.total_rows.item()) == 0
        assert torch.all(recv == 3.0), "nothing may be written when there are no rows"
        assert torch.all(out == 0)


def test_single_expert_takes_everything():
    w = _w(3000, 1, 8, 2, 128)
    idx = torch.full((3000, 1), 5, dtype=torch.int64)
    ref = oracle.layout(idx.numpy(), 8, 2, 128)
    lay = run_gpu_layout(w, idx, wl.worst_case_rows(w))
    assert_layout_matches(lay, ref, w)
    assert ref["total_rows"] == 3072


def test_capacity_error_is_reported_and_nothing_written():
    w = _w(256, 8, 32, 4, 16)
    inp = wl.make(w, 5)
    ref = oracle.layout(inp["topk_idx"].numpy(), 32, 4, 16)
    cap = ref["total_rows"] - 1
    for fused in (True, False):
        lay = binding.Layout(w, cap, device=DEV)
        lay.src_idx.fill_(-5)
        lay.build(inp["topk_idx"].to(DEV), fused=fused)
        assert lay.error() == 4
        assert torch.all(lay.dst_slot == -1) and torch.all(lay.src_idx == -5)
    assert lay.error() == 0
    assert int(lay.total_rows.item()) == ref["total_rows"]
    np.testing.assert_array_equal(lay.expert_offset.cpu().numpy(), ref["expert_offset"])
    assert torch.all(lay.dst_slot == -1) and torch.all(lay.src_idx == -5)
    recv = torch.full((cap, 64), 2.0, dtype=torch.bfloat16, device=DEV)
    lay.permute(inp["x"].to(DEV), recv)
    assert lay.error() == 4
    assert torch.all(recv == 2.0)


def test_bad_expert_id_is_reported_and_dropped():
    w = _w(64, 4, 16, 4, 4)
    idx = wl.draw_topk_idx(w, 9)
    idx[3, 1] = 16
    idx[10, 0] = 1 << 40
    ref = oracle.layout(idx.numpy(), 16, 4, 4)
    assert ref["status"] == oracle.BAD_EXPERT_ID
    for fused in (True, False):
        lay = run_gpu_layout(w, idx, wl.worst_case_rows(w), fused=fused)
        assert lay.error() == 3
        assert_layout_matches(lay, ref, w)


def test_zero_pad_off_leaves_gap_rows():
    w = _w(300, 4, 16, 4, 32, H=32)
    inp = wl.make(w, 2)
    ref = oracle.layout(inp["topk_idx"].numpy(), 16, 4, 32)
    cap = ref["total_rows"]
    lay = run_gpu_layout(w, inp["topk_idx"], cap)
    recv = torch.full((cap, 32), 9.0, dtype=torch.bfloat16, device=DEV)
    lay.permute(inp["x"].to(DEV), recv, zero_pad=False)
    assert lay.error() == 0
    pad = torch.from_numpy(ref["src_idx"] < 0).to(DEV)
    assert torch.all(recv[pad] == 9.0)
    _, ref_recv, _ = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                    cap, zero_pad=False)
    real = ref["src_idx"] >= 0
    np.testing.assert_array_equal(u8(recv)[real], ref_recv[real])


def test_deterministic_across_runs():
    w = wl.WORKLOADS["skewed"].replace(num_tokens=4096, hidden=64)
    inp = wl.make(w, 8)
    cap = wl.worst_case_rows(w)
    outs = []
    for _ in range(3):
        lay = run_gpu_layout(w, inp["topk_idx"], cap)
        recv = torch.zeros((cap, 64), dtype=torch.bfloat16, device=DEV)
        lay.permute(inp["x"].to(DEV), recv)
        out = torch.empty((4096, 64), dtype=torch.bfloat16, device=DEV)
        lay.combine(recv, inp["weights"].to(DEV), out)
        outs.append((lay.dst_slot.cpu(), recv.cpu(), out.cpu()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)


def test_combine_k32_and_out_of_range_slot():
    w = _w(200, 32, 64, 8, 4, H=64, mask_prob=0.3)
    full_case(w, seed=77)
    lay = run_gpu_layout(w, wl.draw_topk_idx(w, 77), wl.worst_case_rows(w))
    rows = int(lay.total_rows.item())
    eo = torch.randn(rows // 2, 64, device=DEV).to(torch.bfloat16)   # too few rows for some slots
    out = torch.empty((200, 64), dtype=torch.bfloat16, device=DEV)
    lay.combine(eo, torch.ones(200 * 32, device=DEV), out)
    assert lay.error() == 4


def test_kernel_launch_counter_moves():
    before = binding.kernel_launches()
    full_case(wl.WORKLOADS["tiny"], 0, fused=False)
    assert binding.kernel_launches() - before == 5     # count, column scan, rank, permute, combine
    # One-call build: the same three chained kernels until a tile holds 16 chunks per warp ...
    before = binding.kernel_launches()
    full_case(wl.WORKLOADS["tiny"], 0, fused=True)
    assert binding.kernel_launches() - before == 5
    before = binding.kernel_launches()
    full_case(_w(40007, 3, 40, 5, 16, H=16), 1, fused=True)
    assert binding.kernel_launches() - before == 5
    # ... and then the cooperative kernel
    before = binding.kernel_launches()
    full_case(_w(330001, 3, 40, 5, 16, H=16), 1, fused=True)
    assert binding.kernel_launches() - before == 3     # fused layout, permute, combine


@pytest.mark.parametrize("w", [
    _w(4096, 8, 256, 8, 128, H=64),      # the chained layout kernels
    _w(131072, 8, 256, 8, 128, H=64),    # the cooperative layout kernel
], ids=["chained", "cooperative"])
def test_back_to_back_on_one_workspace(w):
    """Three different routings through one workspace with no host synchronisation
    between them: build, permute, combine, and device-side snapshots of the maps,
    all queued on one stream.  Kernels that start before their predecessor ends
    (reads before the PDL wait, the permute's counters reset by its last CTA) must
    not mix one batch's state into the next."""
    lay = binding.Layout(w, wl.worst_case_rows(w), device=DEV)
    cap = wl.worst_case_rows(w)
    batches = []
    for seed in (61, 62, 63):
        inp = wl.make(w, seed)
        idx_d, x_d, wts_d = inp["topk_idx"].to(DEV), inp["x"].to(DEV), inp["weights"].to(DEV)
        recv = torch.empty((cap, w.hidden), dtype=x_d.dtype, device=DEV)
        out = torch.empty((w.num_tokens, w.hidden), dtype=torch.bfloat16, device=DEV)
        lay.build(idx_d)
        lay.permute(x_d, recv)
        lay.combine(recv, wts_d, out)      # the identity stands in for the experts
        snap = {k: getattr(lay, k).clone() for k in ("dst_slot", "src_idx", "expert_offset", "total_rows")}
        batches.append((inp, recv, out, snap))
    torch.cuda.synchronize()
    assert lay.error() == 0
    N, K = w.num_tokens, w.topk
    for inp, recv, out, snap in batches:
        ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment)
        rows = ref["total_rows"]
        assert int(snap["total_rows"].item()) == rows
        np.testing.assert_array_equal(snap["expert_offset"].cpu().numpy(), ref["expert_offset"])
        np.testing.assert_array_equal(snap["dst_slot"][: N * K].cpu().numpy().reshape(N, K), ref["dst_slot"])
        np.testing.assert_array_equal(snap["src_idx"][:rows].cpu().numpy(), ref["src_idx"])
        _, ref_recv, _ = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                        rows)
        np.testing.assert_array_equal(u8(recv[:rows]), ref_recv)
        ref_out = oracle.combine(ref_recv.view(np.uint16).reshape(rows, w.hidden), ref["dst_slot"],
                                 inp["weights"].numpy())
        check_combine(bf16_bits(out), ref_out)


def test_cached_dispatch_reuses_the_layout():
    """Cached mode (the page keeps the slot map and skips counting on a second
    dispatch): the same dst_slot moves a second tensor with other row bytes."""
    w = wl.WORKLOADS["skewed"].replace(num_tokens=3000, hidden=64)
    inp = wl.make(w, 12)
    cap = wl.worst_case_rows(w)
    lay = run_gpu_layout(w, inp["topk_idx"], cap)
    ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment, capacity_rows=cap)
    rows = ref["total_rows"]
    launches = binding.kernel_launches()
    for cols, dtype in ((64, torch.bfloat16), (96, torch.float32), (16, torch.uint8)):
        y = (torch.arange(3000 * cols, dtype=torch.float32).reshape(3000, cols) % 251).to(dtype)
        recv = torch.full((cap, cols), 7, dtype=dtype, device=DEV)
        lay.permute(y.to(DEV), recv)
        _, want, _ = oracle.permute(u8(y), ref["dst_slot"], ref["expert_offset"], ref["expert_count"], rows)
        np.testing.assert_array_equal(u8(recv[:rows]), want)
    assert binding.kernel_launches() - launches == 3     # permutes only, no recount
    assert lay.error() == 0


def test_cumulative_expert_stats():
    w = wl.WORKLOADS["decode"]
    cum = torch.zeros(w.num_experts, dtype=torch.int64, device=DEV)
    want = np.zeros(w.num_experts, np.int64)
    for seed in (1, 2, 3):
        idx = wl.draw_topk_idx(w, seed)
        lay = run_gpu_layout(w, idx, wl.worst_case_rows(w))
        binding.accumulate_stats(w, lay.expert_count, cum)
        want += oracle.layout(idx.numpy(), w.num_experts, w.num_ranks, w.alignment)["expert_count"]
    np.testing.assert_array_equal(cum.cpu().numpy(), want)


@pytest.mark.parametrize("name", ["decode", "skewed", "roundtrip"])
def test_int32_ids(name):
    """moe_layout_build_i32: int32 routing ids give the int64 path's layout."""
    w = wl.WORKLOADS[name]
    idx = wl.draw_topk_idx(w, 3)
    ref = oracle.layout(idx.numpy(), w.num_experts, w.num_ranks, w.alignment)
    lay = binding.Layout(w, wl.worst_case_rows(w), device=DEV).build(idx.to(torch.int32).to(DEV))
    assert lay.error() == 0
    assert_layout_matches(lay, ref, w)


def test_int32_ids_separate_kernels():
    w = _w(200000, 32, 64, 4, 16, H=16)             # more tiles than fit at once: three-kernel path
    idx = wl.draw_topk_idx(w, 32)
    ref = oracle.layout(idx.numpy(), 64, 4, 16)
    lay = binding.Layout(w, wl.worst_case_rows(w), device=DEV).build(idx.to(torch.int32).to(DEV))
    assert lay.error() == 0
    assert_layout_matches(lay, ref, w)
