"""The combine's bulk-copy kernel against the oracle, through the C ABI.

Batches of at least 12 tokens per resident CTA of that kernel (about 5500
tokens on a 152-SM GB300) take it; smaller ones take the register kernel,
which the decode, tiny and edge-case tests cover.  The shapes here are all
above the threshold and vary what the bulk kernel's plan depends on: the
number of row pieces (hidden not a multiple of the 1024-column piece, a last
piece shorter than the others), narrow pieces for large top-k, odd top-k,
masked pairs (fewer rows in a stage, whole tokens with none) and slots past
the expert-output rows.  Results must be bit-identical to the oracle's fp32
fma chain (and so within max-abs 1e-2, relative 4e-3).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from counting_sort_bucketization_gb300 import binding, build, workloads as wl
from test_gpu_parity import DEV, bf16_bits, check_combine, full_case, run_gpu_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.load_library()


def _w(N, K, E, R, A, H, **kw):
    return wl.Workload("bulk", N, K, E, R, A, H, **kw)


BULK = [
    _w(8192, 8, 64, 8, 4, 5000),                  # 5 pieces, the last 904 columns
    _w(9000, 3, 40, 5, 16, 72),                   # odd top-k, one narrow piece
    _w(6000, 32, 64, 4, 8, 512, mask_prob=0.3),   # top-32: 256-column pieces
    _w(10000, 1, 16, 4, 1, 16),                   # top-1, the smallest row
    _w(8000, 8, 64, 8, 4, 2048, mask_prob=0.6),   # heavy masking: many stages with few rows
    _w(7000, 5, 100, 10, 8, 4096),                # top-5, 4 pieces
    _w(12000, 8, 256, 8, 128, 1024, routing="zipf", mask_prob=0.1),   # skewed routing
]


@pytest.mark.parametrize("w", BULK, ids=lambda w: f"N{w.num_tokens}_K{w.topk}_H{w.hidden}_m{w.mask_prob}")
def test_bulk_combine_matches_the_oracle(w):
    full_case(w, seed=2024)


def test_bulk_combine_all_masked_gives_zeros():
    N, K, H = 8000, 8, 256
    w = _w(N, K, 16, 4, 8, H)
    idx = torch.full((N, K), -1, dtype=torch.int64)
    lay = run_gpu_layout(w, idx, 64)
    eo = torch.randn(64, H, device=DEV).to(torch.bfloat16)
    out = torch.full((N, H), 5.0, dtype=torch.bfloat16, device=DEV)
    lay.combine(eo, torch.ones(N * K, device=DEV), out)
    assert lay.error() == 0
    assert torch.all(out == 0)


def test_bulk_combine_skips_and_reports_slots_past_the_rows():
    """Slots at or past expert_out_rows are skipped (MOE_ERR_CAPACITY); every
    other term is still summed, as in the oracle given the same slots masked."""
    N, K, H = 8000, 8, 64
    w = _w(N, K, 64, 8, 4, H)
    inp = wl.make(w, 99)
    lay = run_gpu_layout(w, inp["topk_idx"], wl.worst_case_rows(w))
    rows = int(lay.total_rows.item())
    keep = rows // 2
    eo = torch.randn(keep, H, device=DEV).to(torch.bfloat16)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=DEV)
    lay.combine(eo, inp["weights"].to(DEV), out)
    assert lay.error() == 4                       # MOE_ERR_CAPACITY
    dst = lay.dst_slot[: N * K].cpu().numpy().reshape(N, K).copy()
    dst[dst >= keep] = -1
    ref = oracle.combine(bf16_bits(eo), dst, inp["weights"].numpy())
    check_combine(bf16_bits(out), ref)


def test_roundtrip_whole_rows_and_combine():
    """The round-trip workload at full size (131072 tokens, hidden 4096), in the
    launch configuration bench.py times: every receive row and every combined
    token compared with the oracle's, bit for bit.  The oracle runs its own
    layout, permute and stand-in expert on the host (about 17 GB of host memory)."""
    from test_gpu_parity import scale_rows_on_gpu, u8

    w = wl.WORKLOADS["roundtrip"]
    inp = wl.make(w)
    cap = wl.worst_case_rows(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment, capacity_rows=cap)
    rows = ref["total_rows"]
    _, ref_recv, _ = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"], rows)
    ref_eo = oracle.expert_scale(ref_recv.view(np.uint16).reshape(rows, H), ref["expert_offset"],
                                 inp["expert_scale"].numpy())
    ref_out = oracle.combine(ref_eo, ref["dst_slot"], inp["weights"].numpy())

    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    recv = torch.empty((cap, H), dtype=torch.bfloat16, device=DEV)
    lay.permute(inp["x"].to(DEV), recv)
    eo = scale_rows_on_gpu(recv, lay.expert_offset, inp["expert_scale"], rows)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=DEV)
    lay.combine(eo, inp["weights"].to(DEV), out)
    assert lay.error() == 0
    np.testing.assert_array_equal(lay.dst_slot.cpu().numpy().reshape(N, K), ref["dst_slot"])
    step = 1 << 16
    for lo in range(0, rows, step):
        hi = min(rows, lo + step)
        np.testing.assert_array_equal(u8(recv[lo:hi]), ref_recv[lo:hi], err_msg=f"receive rows {lo}..{hi}")
    del recv, eo
    for lo in range(0, N, step):
        hi = min(N, lo + step)
        check_combine(bf16_bits(out[lo:hi]), ref_out[lo:hi])
