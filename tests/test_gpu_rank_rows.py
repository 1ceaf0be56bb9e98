"""Non-expand (rank-contiguous) layout and permute on the GPU vs. the oracle.

The page's first scatter sends each token once to every logical rank it
reaches; rows are grouped by rank, tokens ascending, and the row goes to the
highest k of the token that reaches the rank.  Maps and rows must match the
oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.load_library()


def u8(t):
    t = t.detach().contiguous().cpu()
    return t.view(torch.uint8).numpy().reshape(t.shape[0], -1) if t.numel() else np.zeros((t.shape[0], 0), np.uint8)


def rank_case(w, seed, fused=True, cap=None, check_rows=True):
    inp = wl.make(w, seed)
    idx = inp["topk_idx"]
    N, K, E, R = w.num_tokens, w.topk, w.num_experts, w.num_ranks
    ref = oracle.rank_layout(idx.numpy(), E, R)
    assert ref["status"] == oracle.OK
    rows = ref["total_rows"]
    cap = rows if cap is None else cap
    lay = binding.Layout(w, wl.worst_case_rows(w), device=DEV).build(idx.to(DEV), fused=fused)
    lay.rank_rows(idx.to(DEV), capacity_rows=cap)
    assert lay.error() == 0
    np.testing.assert_array_equal(lay.rank_slot[: N * K].cpu().numpy().reshape(N, K), ref["rank_slot"])
    np.testing.assert_array_equal(lay.rank_src[:rows].cpu().numpy(), ref["rank_src"])
    assert int(lay.rank_psum[-1].item()) == rows
    if not check_rows:
        return lay
    x = inp["x"].to(DEV)
    recv = torch.zeros((cap, w.hidden), dtype=torch.uint8, device=DEV).view(x.dtype) if x.element_size() == 1 \
        else torch.full((cap, w.hidden), -7.0, dtype=x.dtype, device=DEV)
    sf = inp["sf"].to(DEV) if inp["sf"] is not None else None
    recv_sf = torch.full((cap, sf.shape[1]), -3.0, device=DEV) if sf is not None else None
    lay.permute_ranks(x, recv, sf, recv_sf)
    assert lay.error() == 0
    dummy = np.zeros(E + 1, np.int32)
    _, want, want_sf = oracle.permute(u8(inp["x"]), ref["rank_slot"], dummy, dummy[:E], rows,
                                      sf_bytes=u8(inp["sf"]) if sf is not None else None, zero_pad=False)
    np.testing.assert_array_equal(u8(recv[:rows]), want)
    if sf is not None:
        np.testing.assert_array_equal(u8(recv_sf[:rows]), want_sf)
    return lay


@pytest.mark.parametrize("fused", [True, False], ids=["one_call", "two_calls"])
@pytest.mark.parametrize("name", ["tiny", "decode", "skewed", "prefill_fp8"])
def test_workload_rank_rows(name, fused):
    rank_case(wl.WORKLOADS[name], wl.SEEDS[name], fused=fused)


def _w(N, K, E, R, H=64, **kw):
    return wl.Workload("edge", N, K, E, R, 1, H, **kw)


EDGE = [
    _w(1000, 8, 64, 8),
    _w(777, 1, 40, 5),
    _w(513, 3, 37, 1, H=72),
    _w(300, 32, 64, 4, H=32),
    _w(2000, 6, 1024, 1024, H=16),             # one expert per rank
    _w(700, 4, 24, 6, H=48, mask_prob=0.5),
    _w(5000, 8, 256, 8, routing="zipf", zipf_s=2.5, mask_prob=0.1, H=32),
    _w(129, 8, 16, 4, H=384, row_dtype="fp8"),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: f"N{w.num_tokens}_K{w.topk}_E{w.num_experts}_R{w.num_ranks}")
def test_edge_rank_rows(w):
    rank_case(w, seed=5)


def test_roundtrip_size_maps():
    rank_case(wl.WORKLOADS["roundtrip"], wl.SEEDS["roundtrip"], check_rows=False)


def test_rank_capacity_error():
    w = _w(256, 8, 32, 4)
    inp = wl.make(w, 6)
    ref = oracle.rank_layout(inp["topk_idx"].numpy(), 32, 4)
    lay = binding.Layout(w, wl.worst_case_rows(w), device=DEV).build(inp["topk_idx"].to(DEV))
    lay.rank_rows(inp["topk_idx"].to(DEV), capacity_rows=ref["total_rows"] - 1)
    assert lay.error() == 4
    assert torch.all(lay.rank_slot == -1)
    recv = torch.full((ref["total_rows"] - 1, 64), 2.0, dtype=torch.bfloat16, device=DEV)
    lay.permute_ranks(inp["x"].to(DEV), recv)
    assert lay.error() == 4
    assert torch.all(recv == 2.0)
