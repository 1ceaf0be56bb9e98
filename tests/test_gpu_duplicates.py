"""Routing ids with repeats inside a token, through every layout path.

The method's precondition is that a token's top-k experts are distinct; the
pair-by-pair definition the oracle follows still gives one answer when they
are not (each repeated pair gets its own slot, in k order; the token counts
once in each rank).  The layout kernels rank a token's pairs together, so a
repeat is the case that would expose a rank taken twice: these tests draw
ids uniformly with replacement (repeats and masked entries in most tokens)
and compare counts, offsets, rank sums, both slot maps and the non-expand
maps with the oracle, bit for bit, on the three-kernel path, the cooperative
one-call kernel and the two-call API.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl
from test_gpu_parity import DEV, assert_layout_matches, run_gpu_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.load_library()


CASES = [  # (N, K, E, R, A)
    (4096, 8, 64, 8, 16),       # one chunk per warp: three chained kernels
    (131072, 8, 64, 8, 4),      # sixteen chunks per warp: the cooperative kernel
    (20000, 3, 24, 6, 5),       # K does not divide 32
    (3000, 32, 40, 4, 8),       # one token per chunk
    (50000, 2, 8, 2, 1),        # sixteen tokens per chunk, many repeats
]


@pytest.mark.parametrize("fused", [True, False], ids=["one_call", "two_calls"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "N{}_K{}_E{}_R{}_A{}".format(*c))
def test_repeated_experts_in_a_token(case, fused):
    N, K, E, R, A = case
    g = torch.Generator().manual_seed(N * 31 + K)
    idx = torch.randint(-1, E, (N, K), generator=g, dtype=torch.int64)
    assert (np.sort(idx.numpy(), axis=1)[:, 1:] == np.sort(idx.numpy(), axis=1)[:, :-1]).any(), "no repeats drawn"
    w = wl.Workload("dup", N, K, E, R, A, 16)
    ref = oracle.layout(idx.numpy(), E, R, A)
    lay = run_gpu_layout(w, idx, wl.worst_case_rows(w), fused=fused)
    assert lay.error() == 0
    assert_layout_matches(lay, ref, w)
    rref = oracle.rank_layout(idx.numpy(), E, R)
    lay.rank_rows(idx.to(DEV), capacity_rows=rref["total_rows"])
    assert lay.error() == 0
    np.testing.assert_array_equal(lay.rank_slot[: N * K].cpu().numpy().reshape(N, K), rref["rank_slot"])
    np.testing.assert_array_equal(lay.rank_src.cpu().numpy(), rref["rank_src"])
