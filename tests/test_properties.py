"""Property-based checks (hypothesis) on the CPU.

The oracle against its independent formulations on shapes hypothesis chooses
(empty batches, one expert, one expert per rank, K up to 32, large
alignments, any negative id masked, duplicate ids), and the C ABI's
descriptor checks and workspace size against a model of their rules.
"""
import ctypes

import numpy as np
import pytest

from hypothesis import HealthCheck, given, settings, strategies as st  # noqa: E402  (conftest skips the module without it)

import oracle  # noqa: E402
import oracle_checks as oc  # noqa: E402
from counting_sort_bucketization_gb300 import binding, build  # noqa: E402

SETTINGS = settings(max_examples=250, deadline=None, suppress_health_check=[HealthCheck.too_slow])


@st.composite
def routings(draw):
    R = draw(st.integers(1, 6))
    L = draw(st.integers(1, 6))
    E = R * L
    K = draw(st.integers(1, 32))
    N = draw(st.integers(0, 24))
    A = draw(st.sampled_from([1, 2, 3, 4, 7, 64, 1000]))
    ids = draw(st.lists(st.integers(-3, E - 1), min_size=N * K, max_size=N * K))
    return np.array(ids, np.int64).reshape(N, K), E, R, A


@SETTINGS
@given(routings())
def test_layout_is_the_stable_sort(case):
    idx, E, R, A = case
    got = oracle.layout(idx, E, R, A)
    assert got["status"] == oracle.OK
    oc.assert_layout_equal(got, oc.sort_formulation(idx, E, R, A), ctx=f"E={E} R={R} A={A}")


@SETTINGS
@given(routings())
def test_rank_rows_are_the_sorted_distinct_token_rank_pairs(case):
    idx, E, R, _ = case
    got = oracle.rank_layout(idx, E, R)
    assert got["status"] == oracle.OK
    want = oc.rank_sort_formulation(idx, E, R)
    assert got["total_rows"] == want["total_rows"]
    np.testing.assert_array_equal(got["rank_slot"], want["rank_slot"])
    np.testing.assert_array_equal(got["rank_src"], want["rank_src"])


# ------------------------------------------------------------ the C ABI
def model_status(N, K, E, R, A):
    """The descriptor rules of include/moe_layout.h."""
    if N < 0 or K < 1 or E < 1 or R < 1 or A < 1 or E % R != 0:
        return 1                                    # MOE_ERR_INVALID_ARG
    if K > 32 or E > 1024:
        return 6                                    # MOE_ERR_UNSUPPORTED
    if N > (1 << 31) // K or N * K + E * (A - 1) >= (1 << 31):
        return 6
    return 0


def model_workspace_bytes(N, K, E, R):
    """Error word and barrier words (256 B), then the expert and rank histograms,
    one column per tile of the tile plan, each region rounded up to 256 B."""
    tpc = 32 // K
    per_cpw = 8 * tpc
    cpw = min(max(-(-N // (per_cpw * 256)), 1), 16)
    T = -(-N // (per_cpw * cpw))
    r256 = lambda b: -(-b // 256) * 256
    return 256 + r256(E * T * 4) + r256(R * T * 4)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


int32s = st.integers(-(1 << 31), (1 << 31) - 1)


@SETTINGS
@given(st.one_of(st.integers(-5, 1 << 20), st.integers(-(1 << 62), 1 << 62)),
       st.one_of(st.integers(-2, 40), int32s), st.one_of(st.integers(-2, 1100), int32s),
       st.one_of(st.integers(-2, 40), int32s), st.one_of(st.integers(-2, 300), int32s))
def test_descriptor_checks_and_workspace_size(lib, N, K, E, R, A):
    d = binding._CDesc(N, K, E, R, A)
    n = ctypes.c_size_t(0)
    status = lib.moe_layout_workspace_bytes(ctypes.byref(d), ctypes.byref(n))
    assert status == model_status(N, K, E, R, A)
    if status == 0:
        assert n.value == model_workspace_bytes(N, K, E, R)
