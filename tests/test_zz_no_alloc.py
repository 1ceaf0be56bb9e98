"""moe_layout_build_noalloc, the layout entry point that allocates nothing.

It serves callers that cannot allocate device memory when they build the
layout (an engine that has reserved all of HBM for its own allocator, a
plugin that must not touch its host's memory pool, a latency-critical loop
that cannot afford cudaMalloc's device synchronisation).  Its scratch is a
fixed array inside the library instead of a caller workspace.

Checked here through the C ABI: on two calls in a row, with different
inputs, its outputs equal those of moe_layout_build (the entry point that
takes a workspace) exactly, as every layout output is integer; a bad expert
id shows up in that call's device status and not in the next call's; a
problem too big for the fixed scratch is refused before any launch.

The file name makes pytest collect it last; it also runs on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

from counting_sort_bucketization_gb300 import binding, build, workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
OUTPUTS = ("expert_count", "rank_count", "expert_offset", "rank_psum", "dst_slot", "src_idx", "total_rows")


@pytest.fixture(scope="module")
def lib():
    build.build()
    lib = binding.load_library()
    p = ctypes.c_void_p
    lib.moe_layout_build_noalloc.argtypes = [ctypes.POINTER(binding._CDesc), p, p, p, p, p, p, p, ctypes.c_int64,
                                             p, p, p]
    lib.moe_layout_build_noalloc.restype = ctypes.c_int
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, w, idx_d, cap):
    """Run the no-allocation entry point into fresh output buffers."""
    N, K, E, R = w.num_tokens, w.topk, w.num_experts, w.num_ranks
    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(expert_count=torch.full((E,), -9, **i32), rank_count=torch.full((R,), -9, **i32),
               expert_offset=torch.full((E + 1,), -9, **i32), rank_psum=torch.full((R,), -9, **i32),
               dst_slot=torch.full((N * K,), -9, **i32), src_idx=torch.full((cap,), -9, **i32),
               total_rows=torch.full((1,), -9, **i32))
    dev_err = torch.full((1,), -9, **i32)
    st = lib.moe_layout_build_noalloc(
        ctypes.byref(binding._desc(w)), _ptr(idx_d), _ptr(out["expert_count"]), _ptr(out["rank_count"]),
        _ptr(out["expert_offset"]), _ptr(out["rank_psum"]), _ptr(out["dst_slot"]), _ptr(out["src_idx"]), cap,
        _ptr(out["total_rows"]), _ptr(dev_err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, int(dev_err.item()), out


def _with_workspace(w, idx_d, cap):
    """The same layout through moe_layout_build and a caller workspace."""
    lay = binding.Layout(w, cap, device=DEV)
    lay.src_idx.fill_(-9)
    lay.build(idx_d)
    return lay.error(), {k: getattr(lay, k) for k in OUTPUTS}


def test_two_calls_in_a_row_match_the_workspace_entry_point(lib):
    cases = [(wl.WORKLOADS["decode"], 1), (wl.WORKLOADS["skewed"].replace(num_tokens=8192, hidden=64), 2)]
    for w, seed in cases:
        idx_d = wl.draw_topk_idx(w, seed).to(DEV)
        cap = wl.worst_case_rows(w)
        st, dev_err, got = _noalloc(lib, w, idx_d, cap)
        assert st == 0 and dev_err == 0
        err, want = _with_workspace(w, idx_d, cap)
        assert err == 0
        rows = int(want["total_rows"].item())
        for key in OUTPUTS:
            a, b = got[key], want[key]
            if key == "src_idx":
                a, b = a[:rows], b[:rows]
            np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy(), err_msg=f"{w.name} {key}")


def test_device_status_is_per_call(lib):
    w = wl.Workload("small", 512, 4, 32, 4, 4, 64)
    idx = wl.draw_topk_idx(w, 3)
    bad = idx.clone()
    bad[7, 2] = 32                              # an id >= num_experts
    cap = wl.worst_case_rows(w)
    st, dev_err, _ = _noalloc(lib, w, bad.to(DEV), cap)
    assert st == 0 and dev_err == 3             # MOE_ERR_BAD_EXPERT_ID
    st, dev_err, got = _noalloc(lib, w, idx.to(DEV), cap)
    assert st == 0 and dev_err == 0
    _, want = _with_workspace(w, idx.to(DEV), cap)
    np.testing.assert_array_equal(got["dst_slot"].cpu().numpy(), want["dst_slot"].cpu().numpy())


def test_too_big_for_the_fixed_scratch_is_refused(lib):
    w = wl.Workload("big", 131072, 8, 1024, 8, 1, 64)   # workspace above MOE_NOALLOC_SCRATCH_BYTES
    assert binding.workspace_bytes(w) > (1 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    st = lib.moe_layout_build_noalloc(ctypes.byref(binding._desc(w)), *([_ptr(dummy)] * 7), 16, _ptr(dummy),
                                      _ptr(dummy), None)
    assert st == 6                               # MOE_ERR_UNSUPPORTED, nothing launched
