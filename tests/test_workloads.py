"""The seeded generators: deterministic, and shaped like the workloads they stand for."""
import numpy as np
import pytest
import torch

from counting_sort_bucketization_gb300 import workloads as wl


def test_deterministic_and_seed_sensitive():
    a, b = wl.make("tiny"), wl.make("tiny")
    for key in ("topk_idx", "x", "weights", "expert_scale"):
        assert torch.equal(a[key], b[key])
    c = wl.make("tiny", seed=99)
    assert not torch.equal(a["topk_idx"], c["topk_idx"])


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_routing_shape(name):
    w = wl.WORKLOADS[name]
    idx = wl.draw_topk_idx(w, wl.SEEDS[name]).numpy()
    assert idx.shape == (w.num_tokens, w.topk) and idx.dtype == np.int64
    assert idx.max() < w.num_experts and idx.min() >= -1
    masked = (idx < 0).mean()
    assert abs(masked - w.mask_prob) < 0.01
    srt = np.sort(np.where(idx < 0, -np.arange(1, w.topk + 1)[None, :], idx), axis=1)
    assert np.all(np.diff(srt, axis=1) != 0), "experts within a token must be distinct"
    counts = np.bincount(idx[idx >= 0], minlength=w.num_experts)
    if w.routing == "zipf":
        assert counts.max() > 50 * max(counts.min(), 1)
    else:
        assert counts.min() > 0.5 * counts.mean()


def test_fp8_rows_and_scales():
    w = wl.WORKLOADS["prefill_fp8"].replace(num_tokens=64)
    x, sf = wl.draw_x(w, 3)
    assert x.dtype == torch.float8_e4m3fn and x.shape == (64, 7168)
    assert sf.dtype == torch.float32 and sf.shape == (64, 56)
    assert float(sf.min()) >= 0.01 and float(sf.max()) <= 1.0
    assert w.row_bytes == 7168 and w.sf_row_bytes == 224


def test_weights_and_scale():
    w = wl.WORKLOADS["tiny"]
    wt = wl.draw_weights(w, 0)
    assert torch.allclose(wt.sum(1), torch.ones(w.num_tokens), atol=1e-6)
    s = wl.expert_scale(wl.WORKLOADS["roundtrip"])
    assert s.dtype == torch.float32 and float(s[0]) == 1.0 and abs(float(s[383]) - (1 + 383 / 384)) < 1e-6
