"""Dispatch from host memory and combine to host memory, with the copies
overlapped with the kernels in chunks: results must equal the oracle's for
any chunk size (one chunk, ragged chunks, one token per chunk)."""
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


def pipeline_case(w, seed, chunk):
    inp = wl.make(w, seed)
    N, K, H = w.num_tokens, w.topk, w.hidden
    cap = wl.worst_case_rows(w)
    idx_h = inp["topk_idx"].pin_memory()
    x_h = inp["x"].pin_memory()
    wt_h = inp["weights"].pin_memory()
    sf_h = inp["sf"].pin_memory() if inp["sf"] is not None else None
    idx_d = torch.empty_like(inp["topk_idx"], device=DEV)
    x_d = torch.empty_like(inp["x"], device=DEV)
    wt_d = torch.empty_like(inp["weights"], device=DEV)
    sf_d = torch.empty_like(inp["sf"], device=DEV) if sf_h is not None else None
    recv = torch.zeros((cap, H), dtype=torch.uint8, device=DEV).view(x_d.dtype) if x_d.element_size() == 1 \
        else torch.full((cap, H), -7.0, dtype=x_d.dtype, device=DEV)
    recv_sf = torch.full((cap, sf_d.shape[1]), -3.0, device=DEV) if sf_d is not None else None
    lay = binding.Layout(w, cap, device=DEV)
    copy = torch.cuda.Stream()
    binding.dispatch_from_host(lay, idx_h, x_h, idx_d, x_d, recv, weights_host=wt_h, weights=wt_d, sf_host=sf_h,
                               sf=sf_d, recv_sf=recv_sf, chunk_tokens=chunk, copy_stream=copy)
    torch.cuda.synchronize()
    assert lay.error() == 0
    ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment, capacity_rows=cap)
    rows = ref["total_rows"]
    np.testing.assert_array_equal(lay.dst_slot[: N * K].cpu().numpy().reshape(N, K), ref["dst_slot"])
    _, ref_recv, ref_sf = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                         rows, sf_bytes=u8(inp["sf"]) if sf_h is not None else None)
    np.testing.assert_array_equal(u8(recv[:rows]), ref_recv)
    if sf_h is not None:
        np.testing.assert_array_equal(u8(recv_sf[:rows]), ref_sf)
        return
    np.testing.assert_array_equal(wt_d.cpu().numpy(), inp["weights"].numpy())
    eo = recv[:rows].contiguous()
    out = torch.empty((N, H), dtype=torch.bfloat16, device=DEV)
    out_h = torch.full((N, H), 3.0, dtype=torch.bfloat16).pin_memory()
    binding.combine_to_host(lay, eo, wt_d, out, out_h, chunk_tokens=chunk, copy_stream=copy)
    torch.cuda.current_stream().synchronize()
    assert lay.error() == 0
    ref_out = oracle.combine(ref_recv.view(np.uint16).reshape(rows, H), ref["dst_slot"], inp["weights"].numpy())
    np.testing.assert_array_equal(out_h.view(torch.int16).numpy().view(np.uint16), ref_out)


@pytest.mark.parametrize("chunk", [0, 100, 1])
def test_tiny(chunk):
    pipeline_case(wl.WORKLOADS["tiny"], 0, chunk)


@pytest.mark.parametrize("chunk", [0, 1000])
def test_decode(chunk):
    pipeline_case(wl.WORKLOADS["decode"], 1, chunk)


def test_fp8_rows_with_scale_factors():
    pipeline_case(wl.WORKLOADS["prefill_fp8"].replace(num_tokens=3000), 3, 512)


def test_masked_and_ragged():
    pipeline_case(wl.Workload("edge", 777, 4, 24, 6, 8, 64, mask_prob=0.3), 7, 100)


def stand_in_expert(scale_d):
    """Rows of expert e's segment scaled by scale[e] (fp32 product, one bf16 rounding); gap rows stay 0."""
    def expert(lay, recv, recv_sf):
        rows = recv.shape[0]
        off = lay.expert_offset.to(torch.int64)
        row_e = torch.searchsorted(off[1:], torch.arange(rows, device=recv.device), right=True)
        row_e = row_e.clamp(max=scale_d.shape[0] - 1)
        return (recv.float() * scale_d[row_e][:, None]).to(torch.bfloat16)
    return expert


def oracle_batch(inp, w):
    ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment)
    rows = ref["total_rows"]
    _, recv, _ = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"], rows)
    eo = oracle.expert_scale(recv.view(np.uint16).reshape(rows, w.hidden), ref["expert_offset"],
                             inp["expert_scale"].numpy())
    return oracle.combine(eo, ref["dst_slot"], inp["weights"].numpy())


@pytest.mark.parametrize("lanes", [1, 2, 3])
@pytest.mark.parametrize("name,chunk", [("tiny", 100), ("decode", 1024)])
def test_pipelined_batches(name, chunk, lanes):
    # five different batches, several in flight at once; each result equals the oracle's
    w = wl.WORKLOADS[name]
    if name == "decode":
        w = w.replace(num_tokens=1536)
    cap = wl.worst_case_rows(w)
    pipe = binding.HostPipeline(w, cap, w.hidden, lanes=lanes, chunk_tokens=chunk, device=DEV)
    expert = stand_in_expert(wl.expert_scale(w).to(DEV))
    batches = [wl.make(w, 20 + b) for b in range(5)]
    host = [(b["topk_idx"].pin_memory(), b["x"].pin_memory(), b["weights"].pin_memory()) for b in batches]
    outs = [torch.full((w.num_tokens, w.hidden), 5.0, dtype=torch.bfloat16).pin_memory() for _ in batches]
    done = [pipe.submit(i, x, wt, o, expert) for (i, x, wt), o in zip(host, outs)]
    for ev in done:
        ev.synchronize()
    assert pipe.errors() == [0] * lanes
    for b, o in zip(batches, outs):
        np.testing.assert_array_equal(o.view(torch.int16).numpy().view(np.uint16), oracle_batch(b, w))


@pytest.mark.parametrize("chunk", [0, 6000])
def test_pipelined_batches_through_the_bulk_combine(chunk):
    # round-trip routing, 12000 tokens per batch (and 6000-token chunks): every
    # combine launch is large enough for the bulk-copy combine kernel
    w = wl.WORKLOADS["roundtrip"].replace(num_tokens=12000, hidden=512)
    cap = wl.worst_case_rows(w)
    pipe = binding.HostPipeline(w, cap, w.hidden, lanes=3, chunk_tokens=chunk, device=DEV)
    expert = stand_in_expert(wl.expert_scale(w).to(DEV))
    batches = [wl.make(w, 40 + b) for b in range(4)]
    host = [(b["topk_idx"].pin_memory(), b["x"].pin_memory(), b["weights"].pin_memory()) for b in batches]
    outs = [torch.full((w.num_tokens, w.hidden), 5.0, dtype=torch.bfloat16).pin_memory() for _ in batches]
    done = [pipe.submit(i, x, wt, o, expert) for (i, x, wt), o in zip(host, outs)]
    for ev in done:
        ev.synchronize()
    assert pipe.errors() == [0] * 3
    for b, o in zip(batches, outs):
        np.testing.assert_array_equal(o.view(torch.int16).numpy().view(np.uint16), oracle_batch(b, w))


def test_pipelined_dispatch_only_fp8():
    # expert=None: the receive rows come back to host memory; fp8 rows with scale factors
    w = wl.WORKLOADS["prefill_fp8"].replace(num_tokens=2000)
    cap = wl.worst_case_rows(w)
    pipe = binding.HostPipeline(w, cap, w.hidden, x_dtype=torch.float8_e4m3fn, sf_cols=w.hidden // w.sf_block,
                                lanes=2, chunk_tokens=700, device=DEV)
    batches = [wl.make(w, 40 + b) for b in range(3)]
    outs = [torch.zeros((cap, w.hidden), dtype=torch.uint8).pin_memory().view(torch.float8_e4m3fn) for _ in batches]
    done = []
    for b, o in zip(batches, outs):
        done.append(pipe.submit(b["topk_idx"].pin_memory(), b["x"].pin_memory(), b["weights"].pin_memory(), o, None,
                                sf_host=b["sf"].pin_memory()))
    for ev in done:
        ev.synchronize()
    assert pipe.errors() == [0, 0]
    for i, (b, o) in enumerate(zip(batches, outs)):
        ref = oracle.layout(b["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment)
        rows = ref["total_rows"]
        _, want, want_sf = oracle.permute(u8(b["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                          rows, sf_bytes=u8(b["sf"]))
        np.testing.assert_array_equal(u8(o[:rows]), want)
        if i == len(batches) - 1:   # the lane of the last batch still holds its scale rows
            lane = pipe.lane(i % pipe.lanes)
            np.testing.assert_array_equal(u8(lane["recv_sf"][:rows]), want_sf)


def test_short_buffers_are_refused_before_anything_runs():
    # host or device buffers smaller than N rows: the binding raises, nothing is copied or launched
    w = wl.WORKLOADS["tiny"]
    cap = wl.worst_case_rows(w)
    inp = wl.make(w, 31)
    N, H = w.num_tokens, w.hidden
    lay = binding.Layout(w, cap, device=DEV).build(inp["topk_idx"].to(DEV))
    x = inp["x"].to(DEV)
    recv = torch.empty((cap, H), dtype=x.dtype, device=DEV)
    launches = binding.kernel_launches()
    with pytest.raises(ValueError, match="x needs at least"):
        lay.permute(x[: N - 1], recv)
    pipe = binding.HostPipeline(w, cap, H, lanes=1, device=DEV)
    idx_h, x_h, w_h = inp["topk_idx"].pin_memory(), inp["x"].pin_memory(), inp["weights"].pin_memory()
    out_h = torch.empty((N, H), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError, match="x_host needs at least"):
        pipe.submit(idx_h, x_h[: N - 1], w_h, out_h, expert=None)
    with pytest.raises(ValueError, match="topk_idx_host needs at least"):
        pipe.submit(idx_h[: N - 1], x_h, w_h, out_h, expert=None)
    assert binding.kernel_launches() == launches
    torch.cuda.synchronize()
    assert lay.error() == 0
