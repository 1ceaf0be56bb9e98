"""Column-major, TMA-aligned scale factors on the GPU vs. the oracle.

The page "00 DeepEP Engram Architecture Deep-Dive" (§1.1-§1.2) names the
option use_tma_aligned_col_major_sf; the reading both sides follow: column
j of the receive rows' [rows, C] scale words starts at word j*ld, ld a
multiple of 4.  The output buffer starts filled with a sentinel on both
sides and must match the oracle word for word everywhere: rows written,
gap rows zeroed, and every word the method leaves alone.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = np.uint32(0xA5A5A5A5)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.load_library()


def words(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int32).numpy().view(np.uint32)


def sentinel_buffer(cols: int, ld: int) -> torch.Tensor:
    return torch.full((cols, ld), int(SENTINEL.view(np.int32)), dtype=torch.int32, device=DEV)


def _w(N, K, E, R, A, **kw):
    return wl.Workload("edge", N, K, E, R, A, 64, **kw)


def expand_case(w, seed, cols=None, extra_ld=0, zero_pad=True, fused=True, cap=None):
    inp = wl.make(w, seed)
    idx = inp["topk_idx"]
    N, E, R, A = w.num_tokens, w.num_experts, w.num_ranks, w.alignment
    sf = inp["sf"] if cols is None else wl.draw_sf_words(N, cols, seed)
    ref = oracle.layout(idx.numpy(), E, R, A)
    assert ref["status"] == oracle.OK
    rows = ref["total_rows"]
    cap = wl.worst_case_rows(w) if cap is None else cap
    lay = binding.Layout(w, cap, device=DEV).build(idx.to(DEV), fused=fused)
    ld = binding.sf_col_major_ld(cap) + extra_ld
    out = sentinel_buffer(sf.shape[1], ld)
    lay.permute_sf_col_major(sf.to(DEV), out, zero_pad=zero_pad)
    err = lay.error()
    st, want = oracle.permute_sf_col_major(words(sf), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                           rows, ld=ld, zero_pad=zero_pad)
    assert st == oracle.OK
    return err, words(out), want, lay, rows


@pytest.mark.parametrize("fused", [True, False], ids=["one_call", "two_calls"])
def test_prefill_fp8_full_size(fused):
    # 32768 tokens, 56 fp32 scale columns, ~278k receive rows: several tiles per CTA.
    w = wl.WORKLOADS["prefill_fp8"]
    err, got, want, _, _ = expand_case(w, wl.SEEDS["prefill_fp8"], fused=fused)
    assert err == 0
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("name,cols", [("tiny", 1), ("tiny", 3), ("tiny", 4), ("tiny", 64), ("tiny", 65),
                                       ("tiny", 130), ("tiny", 132), ("decode", 56), ("decode", 128),
                                       ("skewed", 7), ("skewed", 20)])
def test_workload_columns(name, cols):
    # column counts below, at and above one 64-column pass through the tile,
    # with 16-byte row loads (a multiple of 4 words) and with single words
    err, got, want, _, _ = expand_case(wl.WORKLOADS[name], wl.SEEDS[name], cols=cols)
    assert err == 0
    np.testing.assert_array_equal(got, want)


EDGE = [
    _w(1000, 3, 40, 5, 16),                                    # ragged last tile
    _w(777, 1, 40, 5, 1),
    _w(300, 32, 64, 4, 128),                                   # mostly padding
    _w(5000, 8, 256, 8, 128, routing="zipf", zipf_s=2.5, mask_prob=0.1),
    _w(129, 8, 16, 4, 2, mask_prob=0.5),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: f"N{w.num_tokens}_K{w.topk}_E{w.num_experts}_A{w.alignment}")
@pytest.mark.parametrize("cols", [5, 56])
def test_edge(w, cols):
    err, got, want, _, _ = expand_case(w, 7, cols=cols)
    assert err == 0
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_rows_wider_than_one_pass(name):
    # 200 words a row: 4 passes of 64 columns through the tile, the last one partial
    err, got, want, _, _ = expand_case(wl.WORKLOADS[name], wl.SEEDS[name], cols=200)
    assert err == 0
    np.testing.assert_array_equal(got, want)


def test_scale_rows_not_16_byte_aligned():
    # a base 4 bytes past a 16-byte boundary: single-word loads, same result
    w = wl.WORKLOADS["decode"]
    seed = wl.SEEDS["decode"]
    inp = wl.make(w, seed)
    N, C = w.num_tokens, 56
    sf = wl.draw_sf_words(N, C, seed)
    flat = torch.empty(N * C + 4, dtype=torch.int32, device=DEV)
    sf_d = flat[1: 1 + N * C].view(N, C)
    sf_d.copy_(sf.to(DEV))
    assert sf_d.data_ptr() % 16 == 4
    ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment)
    cap = wl.worst_case_rows(w)
    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    ld = binding.sf_col_major_ld(cap)
    out = sentinel_buffer(C, ld)
    lay.permute_sf_col_major(sf_d, out)
    assert lay.error() == 0
    _, want = oracle.permute_sf_col_major(words(sf), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                          ref["total_rows"], ld=ld)
    np.testing.assert_array_equal(words(out), want)


@pytest.mark.parametrize("cols", [9, 56])
def test_gap_rows_left_alone_without_zero_pad(cols):
    err, got, want, _, _ = expand_case(wl.WORKLOADS["skewed"], wl.SEEDS["skewed"], cols=cols, zero_pad=False)
    assert err == 0
    np.testing.assert_array_equal(got, want)


def test_wider_leading_dimension():
    # ld beyond the capacity: the extra words of every column stay untouched
    err, got, want, _, rows = expand_case(_w(1000, 3, 40, 5, 16), 8, cols=6, extra_ld=12)
    assert err == 0
    np.testing.assert_array_equal(got, want)
    assert np.all(got[:, rows:] == SENTINEL)


@pytest.mark.parametrize("w", [_w(0, 4, 16, 4, 8), _w(300, 4, 16, 4, 8, mask_prob=1.0)], ids=["empty", "all_masked"])
def test_no_rows(w):
    err, got, want, _, rows = expand_case(w, 9, cols=4)
    assert err == 0 and rows == 0
    assert np.all(got == SENTINEL)
    np.testing.assert_array_equal(got, want)


def test_capacity_exceeded_writes_nothing():
    w = _w(256, 8, 32, 4, 4)
    inp = wl.make(w, 6)
    ref = oracle.layout(inp["topk_idx"].numpy(), 32, 4, 4)
    cap = ref["total_rows"] - 1
    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    assert lay.error() == 4
    out = sentinel_buffer(5, binding.sf_col_major_ld(cap))
    lay.permute_sf_col_major(wl.draw_sf_words(256, 5, 6).to(DEV), out)
    assert lay.error() == 4
    assert np.all(words(out) == SENTINEL)


def test_map_entry_out_of_range_is_skipped_and_reported():
    # a corrupted inverse map: the row is skipped (never read through) and the error recorded
    w = _w(500, 4, 32, 4, 8)
    inp = wl.make(w, 10)
    ref = oracle.layout(inp["topk_idx"].numpy(), 32, 4, 8)
    cap = wl.worst_case_rows(w)
    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    assert lay.error() == 0
    bad_row = int(np.flatnonzero(ref["src_idx"] >= 0)[3])
    lay.src_idx[bad_row] = w.num_tokens + 7
    sf = wl.draw_sf_words(500, 5, 10)
    ld = binding.sf_col_major_ld(cap)
    out = sentinel_buffer(5, ld)
    lay.permute_sf_col_major(sf.to(DEV), out)
    assert lay.error() == 1
    _, want = oracle.permute_sf_col_major(words(sf), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                          ref["total_rows"], ld=ld)
    want[:, bad_row] = SENTINEL
    np.testing.assert_array_equal(words(out), want)


@pytest.mark.parametrize("name,cols", [("tiny", 3), ("prefill_fp8", None), ("skewed", 56)])
def test_rank_layout(name, cols):
    # non-expand rows (one per token and rank reached), no padding
    w = wl.WORKLOADS[name]
    inp = wl.make(w, wl.SEEDS[name])
    idx = inp["topk_idx"]
    N, E, R = w.num_tokens, w.num_experts, w.num_ranks
    sf = inp["sf"] if cols is None else wl.draw_sf_words(N, cols, wl.SEEDS[name])
    ref = oracle.rank_layout(idx.numpy(), E, R)
    rows = ref["total_rows"]
    lay = binding.Layout(w, wl.worst_case_rows(w), device=DEV).build(idx.to(DEV))
    lay.rank_rows(idx.to(DEV), capacity_rows=rows)
    ld = binding.sf_col_major_ld(lay.rank_src.numel())
    out = sentinel_buffer(sf.shape[1], ld)
    lay.permute_sf_col_major_ranks(sf.to(DEV), out)
    assert lay.error() == 0
    none = np.zeros(E + 1, np.int32)
    st, want = oracle.permute_sf_col_major(words(sf), ref["rank_slot"], none, none[:E], rows, ld=ld,
                                           zero_pad=False)
    assert st == oracle.OK
    np.testing.assert_array_equal(words(out), want)


def test_agrees_with_row_major_permute():
    # the same receive rows as the row-major scale factors the permute writes, transposed
    w = wl.WORKLOADS["prefill_fp8"].replace(num_tokens=3000)
    inp = wl.make(w, 12)
    cap = wl.worst_case_rows(w)
    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    x, sf = inp["x"].to(DEV), inp["sf"].to(DEV)
    recv = torch.empty((cap, w.hidden), dtype=x.dtype, device=DEV)
    recv_sf = torch.empty((cap, sf.shape[1]), dtype=sf.dtype, device=DEV)
    lay.permute(x, recv, sf, recv_sf)
    out = binding.new_sf_col_major(sf.shape[1], cap, device=DEV)
    lay.permute_sf_col_major(sf, out)
    assert lay.error() == 0
    rows = int(lay.total_rows.item())
    np.testing.assert_array_equal(words(out)[:, :rows], words(recv_sf)[:rows].T)
