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


def test_permute_and_combine_at_the_largest_accepted_problem():
    """The permute and the combine at the same size (2**31 - 2**20 tokens,
    top-1, alignment 2, 16-byte bf16 rows), checked through properties that
    hold at any size, in chunks on the device: every receive row equals
    x[src_idx[row]] and every gap row is zero; every combined token is
    bf16(w * x) for its one expert output (the stand-in expert is the
    identity) and zero when masked.  Rows and weights are drawn so that no
    product is zero or below the normal range, where a fused multiply-add
    from +0 and a plain product could differ in the sign of a zero.  About
    136 GB of device memory."""
    N, K, E, R, A, H = (1 << 31) - (1 << 20), 1, 64, 8, 2, 8
    w = wl.Workload("largest", N, K, E, R, A, H)
    cap = wl.worst_case_rows(w)
    assert cap < (1 << 31)
    g = torch.Generator(device=DEV).manual_seed(37)
    idx = torch.randint(-1, E, (N, K), generator=g, dtype=torch.int64, device=DEV)
    # bf16 bit patterns with exponents 0x78..0x87 (about 2**-7 .. 2**8) and a random sign
    x = torch.empty((N, H), dtype=torch.int16, device=DEV)
    step = 1 << 27
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        mag = torch.randint(0x3C00, 0x4400, (r1 - r0, H), generator=g, dtype=torch.int16, device=DEV)
        neg = torch.randint(0, 2, (r1 - r0, H), generator=g, dtype=torch.int16, device=DEV) * -32768
        x[r0:r1] = mag | neg
    x = x.view(torch.bfloat16)
    wt = torch.rand((N, K), generator=g, device=DEV) * 0.75 + 0.25

    lay = binding.Layout(w, cap, device=DEV).build(idx)
    recv = torch.empty((cap, H), dtype=torch.bfloat16, device=DEV)
    lay.permute(x, recv)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=DEV)
    lay.combine(recv, wt, out)
    assert lay.error() == 0
    rows = int(lay.total_rows.item())
    assert rows > N * 0.98

    xi, ri, oi = x.view(torch.int16), recv.view(torch.int16), out.view(torch.int16)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        src = lay.src_idx[r0:r1].long()
        gap = src < 0
        want = xi[src.clamp(min=0)]
        want[gap] = 0
        assert torch.equal(ri[r0:r1], want), f"receive rows {r0}..{r1}"
        del src, gap, want
    for t0 in range(0, N, step):
        t1 = min(N, t0 + step)
        slot = lay.dst_slot[t0:t1].long()
        valid = slot >= 0
        want = (wt[t0:t1] * x[t0:t1].float()).to(torch.bfloat16).view(torch.int16)
        want[~valid] = 0
        assert torch.equal(oi[t0:t1], want), f"combined tokens {t0}..{t1}"
        del slot, valid, want
    del lay, recv, out, x, idx, wt
    torch.cuda.empty_cache()
