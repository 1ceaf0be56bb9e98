"""The layout at the largest problem the library accepts, against the oracle.

Slots, rows and token indices are int32 in the maps, so the host checks
refuse any problem whose worst-case row count reaches 2**31.  This test
builds a layout just under that limit: 2**31 - 2**20 (token, k) pairs at
top-1, so that the token indices written to src_idx reach the top of the
int32 range as well, on the one-call and the two-call paths (both run the
three chained kernels here: far more tiles than can be resident at once).
Every count, offset, rank sum, slot and inverse-map entry is compared with
the oracle.  About 16 GB of ids and 16 GB of maps on the device; the oracle
and the comparison hold about 50 GB of host memory.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl
from test_gpu_parity import DEV, assert_layout_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.load_library()


def test_layout_at_the_largest_accepted_problem():
    N, K, E, R, A = (1 << 31) - (1 << 20), 1, 64, 8, 1
    w = wl.Workload("largest", N, K, E, R, A, 16)
    cap = wl.worst_case_rows(w)
    assert cap < (1 << 31)
    g = torch.Generator().manual_seed(31)
    idx = torch.randint(-1, E, (N, K), generator=g, dtype=torch.int64)   # about 1 in 65 pairs masked
    ref = oracle.layout(idx.numpy(), E, R, A)
    assert ref["status"] == oracle.OK
    idx_d = idx.to(DEV)
    for fused in (True, False):
        lay = binding.Layout(w, cap, device=DEV)
        lay.build(idx_d, fused=fused)
        assert lay.error() == 0
        assert_layout_matches(lay, ref, w)
        del lay
        torch.cuda.empty_cache()
