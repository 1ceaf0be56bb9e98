"""Bounded waits run out without hanging: the kernel records MOE_ERR_TIMEOUT,
finishes, and the context stays usable.

Each case arms the test hook (moe_debug_set_waits) so that one wait can never
be satisfied -- a grid-barrier target past the number of CTAs, or transaction
bytes no copy delivers -- with a 2 ms limit instead of 1 s.  Nothing faults:
the waits give up, the error word says so, and the same process then builds
and permutes correctly with the hook off.
"""
import numpy as np
import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 5          # MOE_ERR_TIMEOUT
LIMIT_NS = 2_000_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.load_library()


@pytest.fixture(autouse=True)
def _normal_waits_after():
    yield
    binding.debug_set_waits(0, 0, 0)


def u8(t):
    t = t.detach().contiguous().cpu()
    return t.view(torch.uint8).numpy().reshape(t.shape[0], -1)


def test_grid_barrier_runs_out():
    # sixteen chunks per warp: the one-call build takes the cooperative kernel with its grid barriers
    w = wl.Workload("edge", 330001, 3, 40, 5, 16, 16)
    inp = wl.make(w, 1)
    idx = inp["topk_idx"]
    cap = wl.worst_case_rows(w)
    launches = binding.kernel_launches()
    binding.debug_set_waits(LIMIT_NS, barrier_extra=1)
    lay = binding.Layout(w, cap, device=DEV).build(idx.to(DEV))
    assert binding.kernel_launches() - launches == 1        # the cooperative kernel ran
    assert lay.error() == TIMEOUT
    binding.debug_set_waits(0, 0, 0)
    # a fresh workspace (the timed-out one keeps its barrier counter set) builds exactly
    ref = oracle.layout(idx.numpy(), w.num_experts, w.num_ranks, w.alignment)
    lay2 = binding.Layout(w, cap, device=DEV).build(idx.to(DEV))
    assert lay2.error() == 0
    np.testing.assert_array_equal(lay2.dst_slot[: w.num_tokens * w.topk].cpu().numpy().reshape(w.num_tokens, -1),
                                  ref["dst_slot"])


@pytest.mark.parametrize("name", ["decode", "prefill_fp8"])
def test_permute_stage_runs_out(name):
    w = wl.WORKLOADS[name].replace(num_tokens=2048)
    inp = wl.make(w, 2)
    cap = wl.worst_case_rows(w)
    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    assert lay.error() == 0
    x = inp["x"].to(DEV)
    sf = inp["sf"].to(DEV) if inp["sf"] is not None else None
    recv = torch.zeros((cap, w.hidden), dtype=torch.uint8, device=DEV).view(x.dtype) if x.element_size() == 1 \
        else torch.zeros((cap, w.hidden), dtype=x.dtype, device=DEV)
    recv_sf = torch.zeros((cap, sf.shape[1]), device=DEV) if sf is not None else None
    binding.debug_set_waits(LIMIT_NS, extra_tx=16)
    lay.permute(x, recv, sf, recv_sf)
    assert lay.error() == TIMEOUT
    binding.debug_set_waits(0, 0, 0)
    # the same workspace (its claim counters were reset by the last CTA) permutes exactly
    lay.permute(x, recv, sf, recv_sf)
    assert lay.error() == 0
    ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment)
    rows = ref["total_rows"]
    _, want, want_sf = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                      rows, sf_bytes=u8(inp["sf"]) if sf is not None else None)
    np.testing.assert_array_equal(u8(recv[:rows]), want)
    if sf is not None:
        np.testing.assert_array_equal(u8(recv_sf[:rows]), want_sf)
