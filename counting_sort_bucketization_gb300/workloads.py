"""Seeded synthetic workloads for the MoE dispatch layout.

This module only draws inputs: routing ids, masks, activations, scale factors,
top-k weights and the per-expert scale of the round-trip stand-in expert.  It
does none of the counting, prefix sums, scatter or combine, so both the CUDA
path and the CPU oracle can take their inputs from it.

Everything is drawn on the host with a CPU ``torch.Generator`` seeded per
call, so a (config, seed) pair always gives the same bytes on any machine.

The five workloads (routing, masking and value distributions as the method's
MoE dispatch setting describes them):

=========== ======= == === == === ===== ============ ===================== ======
name        N       K  E   R  A   H     row dtype    routing               mask
=========== ======= == === == === ===== ============ ===================== ======
tiny        256     2  8   2  1   256   bf16 U[-1,1] uniform distinct      none
decode      4096    8  256 8  128 7168  bf16 N(0,1)  uniform distinct      none
skewed      16384   8  256 8  128 7168  bf16 N(0,1)  Zipf(1.2) w/o replace 10%
prefill_fp8 32768   8  256 32 128 7168  fp8 e4m3+sf  uniform distinct      none
roundtrip   131072  8  384 16 64  4096  bf16 N(0,1)  uniform distinct      5%
=========== ======= == === == === ===== ============ ===================== ======
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_tokens: int
    topk: int
    num_experts: int
    num_ranks: int
    alignment: int
    hidden: int
    row_dtype: str = "bf16"        # "bf16" or "fp8" (fp8 rows carry fp32 scale factors)
    routing: str = "uniform"       # "uniform" or "zipf"
    zipf_s: float = 1.2
    mask_prob: float = 0.0
    x_dist: str = "normal"         # "normal" N(0,1) or "uniform" U[-1,1]
    sf_block: int = 128            # columns per fp8 scale factor

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.num_ranks

    @property
    def row_bytes(self) -> int:
        return self.hidden * (2 if self.row_dtype == "bf16" else 1)

    @property
    def sf_row_bytes(self) -> int:
        return 4 * (self.hidden // self.sf_block) if self.row_dtype == "fp8" else 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 256, 2, 8, 2, 1, 256, x_dist="uniform"),
    "decode": Workload("decode", 4096, 8, 256, 8, 128, 7168),
    "skewed": Workload("skewed", 16384, 8, 256, 8, 128, 7168, routing="zipf", mask_prob=0.10),
    "prefill_fp8": Workload("prefill_fp8", 32768, 8, 256, 32, 128, 7168, row_dtype="fp8"),
    "roundtrip": Workload("roundtrip", 131072, 8, 384, 16, 64, 4096, mask_prob=0.05),
}
# Seeds: the workload's position in the table above.
SEEDS = {name: i for i, name in enumerate(WORKLOADS)}


def get(name_or_workload) -> Workload:
    if isinstance(name_or_workload, Workload):
        return name_or_workload
    return WORKLOADS[name_or_workload]


def _gen(seed: int, stream: int) -> torch.Generator:
    # One generator per drawn quantity, so that changing one draw (say the
    # routing) leaves the others' bytes unchanged.
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + stream)
    return g


def draw_topk_idx(w: Workload, seed: int) -> torch.Tensor:
    """int64 [N, K]: K distinct experts per token in random order, then masks."""
    N, K, E = w.num_tokens, w.topk, w.num_experts
    if N == 0:
        return torch.empty((0, K), dtype=torch.int64)
    g = _gen(seed, 1)
    if w.routing == "uniform":
        # The K largest of E i.i.d. uniform keys: a uniformly random K-subset,
        # listed in the (random) order of its keys.
        keys = torch.rand((N, E), generator=g)
        idx = keys.topk(K, dim=1).indices
    elif w.routing == "zipf":
        # Popularity p_i ~ (i+1)^-s over a seeded permutation of the experts,
        # K draws per token without replacement.
        perm = torch.randperm(E, generator=g)
        pop = torch.arange(1, E + 1, dtype=torch.float64).pow(-w.zipf_s)
        p = torch.empty(E, dtype=torch.float64)
        p[perm] = pop
        idx = torch.multinomial(p.to(torch.float32).expand(N, E), K, replacement=False, generator=g)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    idx = idx.to(torch.int64)
    if w.mask_prob > 0:
        gm = _gen(seed, 2)
        drop = torch.rand((N, K), generator=gm) < w.mask_prob
        idx = idx.masked_fill(drop, -1)
    return idx.contiguous()


def draw_x(w: Workload, seed: int) -> tuple[torch.Tensor, torch.Tensor | None]:
    """Token rows: bf16 [N, H]; or fp8 e4m3 [N, H] plus fp32 scale factors [N, H/128]."""
    N, H = w.num_tokens, w.hidden
    g = _gen(seed, 3)
    if w.x_dist == "uniform":
        v = torch.rand((N, H), generator=g) * 2.0 - 1.0
    else:
        v = torch.randn((N, H), generator=g)
    if w.row_dtype == "bf16":
        return v.to(torch.bfloat16).contiguous(), None
    # fp8: scale factors uniform in [0.01, 1] per (token, 128-column block);
    # the stored value is v / sf, clamped to the e4m3 range and cast.
    gs = _gen(seed, 4)
    nb = H // w.sf_block
    sf = torch.rand((N, nb), generator=gs) * 0.99 + 0.01
    q = (v.view(N, nb, w.sf_block) / sf.unsqueeze(-1)).clamp(-448.0, 448.0)
    return q.view(N, H).to(torch.float8_e4m3fn).contiguous(), sf.to(torch.float32).contiguous()


def draw_sf_words(num_tokens: int, cols: int, seed: int) -> torch.Tensor:
    """int32 [N, cols]: arbitrary 32-bit scale words (any bit pattern: the layouts move them verbatim)."""
    g = _gen(seed, 6)
    return torch.randint(-(2 ** 31), 2 ** 31, (num_tokens, cols), dtype=torch.int64, generator=g).to(
        torch.int32).contiguous()


def draw_weights(w: Workload, seed: int) -> torch.Tensor:
    """fp32 [N, K]: softmax over the K slots of N(0,1) logits (masked slots keep their weight; combine skips them)."""
    g = _gen(seed, 5)
    logits = torch.randn((w.num_tokens, w.topk), generator=g)
    return torch.softmax(logits, dim=1).to(torch.float32).contiguous()


def expert_scale(w: Workload) -> torch.Tensor:
    """fp32 [E]: the round-trip stand-in expert multiplies expert e's rows by 1 + e/384."""
    e = torch.arange(w.num_experts, dtype=torch.float32)
    return (1.0 + e / 384.0).to(torch.float32)


def make(name_or_workload, seed: int | None = None) -> dict:
    """All inputs of one workload as CPU tensors."""
    w = get(name_or_workload)
    if seed is None:
        seed = SEEDS.get(w.name, 0)
    x, sf = draw_x(w, seed)
    return dict(workload=w, seed=seed, topk_idx=draw_topk_idx(w, seed), x=x, sf=sf,
                weights=draw_weights(w, seed), expert_scale=expert_scale(w))


def worst_case_rows(w: Workload) -> int:
    """Receive-buffer rows that always suffice: every pair valid plus A-1 pad rows per expert."""
    return w.num_tokens * w.topk + w.num_experts * (w.alignment - 1)
