"""A whole step (layout, permute, stand-in expert, combine) captured as one
CUDA graph and replayed on new batches copied into the captured inputs: every
replay's layout, receive rows and combined tokens equal the oracle's, on the
chained layout kernels (decode) and on the cooperative layout kernel with the
bulk-copy combine (round-trip routing, 131072 tokens)."""
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
    return t.view(torch.uint8).numpy().reshape(t.shape[0], -1)


def expert_for(w):
    scale_d = wl.expert_scale(w).to(DEV)

    def expert(lay, recv, recv_sf):
        # rows of expert e's segment scaled by scale[e], gap rows 0 (harness, not the method)
        rows = recv.shape[0]
        off = lay.expert_offset.to(torch.int64)
        row_e = torch.searchsorted(off[1:], torch.arange(rows, device=recv.device), right=True)
        row_e = row_e.clamp(max=scale_d.shape[0] - 1)
        return (recv.float() * scale_d[row_e][:, None]).to(torch.bfloat16)
    return expert


@pytest.mark.parametrize("w", [wl.WORKLOADS["decode"], wl.WORKLOADS["roundtrip"].replace(hidden=256)],
                         ids=["decode", "roundtrip_h256"])
def test_graph_replays_match_the_oracle(w):
    N, K, H = w.num_tokens, w.topk, w.hidden
    cap = wl.worst_case_rows(w)
    g = binding.StepGraph(w, cap, H, expert=expert_for(w))
    assert g.error() == 0
    launches = binding.kernel_launches()
    for seed in (11, 12, 13):
        inp = wl.make(w, seed)
        g.topk_idx.copy_(inp["topk_idx"])
        g.x.copy_(inp["x"])
        g.weights.copy_(inp["weights"])
        g.replay()
        torch.cuda.synchronize()
        assert g.error() == 0
        ref = oracle.layout(inp["topk_idx"].numpy(), w.num_experts, w.num_ranks, w.alignment, capacity_rows=cap)
        rows = ref["total_rows"]
        np.testing.assert_array_equal(g.layout.dst_slot.cpu().numpy().reshape(N, K), ref["dst_slot"])
        np.testing.assert_array_equal(g.layout.src_idx[:rows].cpu().numpy(), ref["src_idx"])
        _, ref_recv, _ = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"],
                                        rows)
        np.testing.assert_array_equal(u8(g.recv_x[:rows]), ref_recv)
        eo = oracle.expert_scale(ref_recv.view(np.uint16).reshape(rows, H), ref["expert_offset"],
                                 inp["expert_scale"].numpy())
        ref_out = oracle.combine(eo, ref["dst_slot"], inp["weights"].numpy())
        np.testing.assert_array_equal(g.out.view(torch.int16).cpu().numpy().view(np.uint16), ref_out)
    # replays run the captured kernels: nothing was launched through the library's host code
    assert binding.kernel_launches() == launches
