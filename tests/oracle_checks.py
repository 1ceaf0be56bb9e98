"""Pins for the CPU oracle: each check ties it to something other than itself.

Every ``check_*`` takes a loaded oracle library (``oracle.load(path)``) so the
same checks run against the real oracle (tests/test_oracle_pins.py) and
against copies of it with a planted mistake (tests/test_oracle_mutations.py),
which must fail at least one check.

What pins what (page: "07 DeepEP Counting Sort / Bucketization", sections):
  handworked     -- a layout derived by hand from the definitions (§4.2,
                    §5.5, §6.4, §7.2, §7.3) and the expand-mode handle
                    properties of §10.3; golden file in tests/golden/.
  padding        -- the page's own worked example in §7.3 (50 tokens,
                    alignment 64 -> 64 slots, 14 zero rows).
  sort           -- a second formulation: a stable library sort of the valid
                    pairs by expert id, np.bincount / np.unique for counts.
  bruteforce     -- every topk_idx over tiny shapes (duplicates included),
                    checked against the per-pair definition by enumeration.
  invariants     -- counts sum to the valid pairs, offsets monotone and
                    aligned, scatter a bijection onto non-pad rows, etc.
  permute        -- rows land where src_idx says (numpy fancy indexing),
                    pads are zero, scale-factor rows follow.
  combine_closed -- unit weights on dispatched rows give n_valid * x exactly.
  combine_bound  -- exact fp64 sum within the fp32-accumulation + bf16 bound.
  combine_exact  -- exact rational emulation of the fp32 fused multiply-add
                    chain and round-to-nearest-even (IEEE 754 definitions).
  roundtrip      -- dispatch, stand-in expert, combine vs. a direct formula
                    from x that never builds the receive buffer.
  bf16           -- fp32 -> bf16 rounding vs. torch's CPU cast.
  errors         -- bad expert ids and too-small capacity are reported.
  rank_sort      -- the non-expand (rank-contiguous) rows as a library sort of the
                    distinct (token, rank) pairs; master lane = highest k (§6.2);
                    also part of handworked and bruteforce.
  sf_col_major   -- column-major scale factors (option named on the page "00
                    DeepEP Engram Architecture Deep-Dive", §1.1-§1.2): columns
                    derived by hand (golden file), a gather through src_idx,
                    the transpose of the row-major scatter, untouched words past
                    the rows, and the leading-dimension rule.
"""
from __future__ import annotations

import itertools
import json
import os
import sys
from fractions import Fraction

import numpy as np
import torch

_REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _REPO not in sys.path:
    sys.path.insert(0, _REPO)

import oracle  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- helpers
def align(v, a):
    return -(-np.asarray(v) // a) * a


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def random_idx(rng: np.random.Generator, N, K, E, mask_prob=0.0, skew=False):
    """K distinct experts per token (optionally skewed), some masked with -1."""
    if N == 0:
        return np.empty((0, K), np.int64)
    if skew:
        p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
        p = p[rng.permutation(E)]
        p /= p.sum()
        idx = np.stack([rng.choice(E, size=K, replace=False, p=p) for _ in range(N)])
    else:
        idx = np.argsort(rng.random((N, E)), axis=1)[:, :K]
    idx = idx.astype(np.int64)
    if mask_prob > 0:
        idx[rng.random((N, K)) < mask_prob] = -1
    return idx


def sort_formulation(idx: np.ndarray, E: int, R: int, A: int) -> dict:
    """The layout as a stable sort of the valid (t, k) pairs by expert id."""
    N, K = idx.shape
    flat = idx.reshape(-1)
    pairs = np.nonzero(flat >= 0)[0]
    keys = flat[pairs]
    order = np.argsort(keys, kind="stable")
    spairs, skeys = pairs[order], keys[order]
    counts = np.bincount(keys, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(align(counts, A))])
    group_start = np.concatenate([[0], np.cumsum(counts)])[:-1]
    within = np.arange(spairs.size) - group_start[skeys]
    dst = np.full(N * K, -1, np.int64)
    dst[spairs] = offsets[skeys] + within
    src = np.full(int(offsets[-1]), -1, np.int64)
    src[dst[spairs]] = spairs // K
    L = E // R
    tok_rank = np.unique((pairs // K) * R + keys // L)
    rank_count = np.bincount(tok_rank % R, minlength=R)
    return dict(expert_count=counts, rank_count=rank_count, expert_offset=offsets,
                rank_psum=np.cumsum(rank_count), dst_slot=dst.reshape(N, K), src_idx=src,
                total_rows=int(offsets[-1]))


def rank_sort_formulation(idx: np.ndarray, E: int, R: int) -> dict:
    """Non-expand rows as a sort of the distinct (token, rank) pairs by (rank, token);
    the row goes to the highest k of the token that reaches the rank."""
    N, K = idx.shape
    L = E // R
    flat = idx.reshape(-1)
    pairs = np.nonzero(flat >= 0)[0]
    t_of, r_of, k_of = pairs // K, flat[pairs] // L, pairs % K
    key = t_of * R + r_of
    uniq = np.unique(key)                                  # (t, r) pairs, t-major
    ut, ur = uniq // R, uniq % R
    order = np.lexsort((ut, ur))                           # by rank, then token
    row_of = np.empty(uniq.size, np.int64)
    row_of[order] = np.arange(uniq.size)
    master_k = np.full(uniq.size, -1)
    np.maximum.at(master_k, np.searchsorted(uniq, key), k_of)
    slot = np.full((N, K), -1, np.int64)
    slot[ut, master_k] = row_of
    src = np.empty(uniq.size, np.int64)
    src[row_of] = ut
    return dict(rank_slot=slot, rank_src=src, total_rows=int(uniq.size))


def assert_layout_equal(got: dict, want: dict, ctx=""):
    for key in ("expert_count", "rank_count", "expert_offset", "rank_psum", "dst_slot", "src_idx"):
        np.testing.assert_array_equal(np.asarray(got[key]), np.asarray(want[key]), err_msg=f"{key} {ctx}")
    assert int(got["total_rows"]) == int(want["total_rows"]), ctx


def check_layout_invariants(idx: np.ndarray, E: int, R: int, A: int, r: dict):
    N, K = idx.shape
    valid = idx >= 0
    P = int(valid.sum())
    cnt, off, rc = r["expert_count"], r["expert_offset"].astype(np.int64), r["rank_count"]
    dst, src, rows = r["dst_slot"], r["src_idx"], r["total_rows"]
    assert int(cnt.sum()) == P
    assert int(rc.sum()) <= P
    if K == 1:
        assert int(rc.sum()) == P
    assert off[0] == 0 and np.all(np.diff(off) >= 0) and np.all(off % A == 0)
    np.testing.assert_array_equal(np.diff(off), align(cnt, A))
    assert rows == off[-1]
    # rank_psum[R-1] = number of distinct (token, rank) pairs
    L = E // R
    distinct = sum(len({int(e) // L for e in row if e >= 0}) for row in idx)
    assert int(r["rank_psum"][-1]) == distinct
    d = dst[valid]
    assert np.all(dst[~valid] == -1)
    assert np.unique(d).size == d.size, "dst_slot not injective"
    # image of dst_slot plus the pad rows tiles [0, rows) exactly
    is_pad = np.ones(rows, bool)
    is_pad[d] = False
    for e in range(E):
        seg = np.arange(off[e], off[e + 1])
        np.testing.assert_array_equal(is_pad[seg], np.arange(seg.size) >= cnt[e])
        s = src[off[e]:off[e] + cnt[e]]
        assert np.all(np.diff(s) >= 0), "segment not token-ascending"
    assert np.all(src[is_pad] == -1)
    t_of = np.repeat(np.arange(N), K).reshape(N, K)
    np.testing.assert_array_equal(src[d], t_of[valid])
    # expand-mode handle value (aligned start + real count) and its two properties
    handle = off[:-1] + cnt
    for i in range(1, E):
        assert handle[i] - align(handle[i - 1], A) == cnt[i]
        assert align(handle[i - 1], A) == off[i]


# ------------------------------------------------------------------ checks
def check_handworked(lib):
    g = json.load(open(os.path.join(GOLDEN, "handworked_n4_k2_e4_r2_a2.json")))
    idx = np.array(g["topk_idx"], np.int64)
    E, R, A = g["num_experts"], g["num_ranks"], g["alignment"]
    r = oracle.layout(idx, E, R, A, lib=lib)
    assert r["status"] == oracle.OK
    assert_layout_equal(r, g, "handworked")
    np.testing.assert_array_equal(r["expert_offset"][:-1] + r["expert_count"], g["handle_psum"])
    rr = oracle.rank_layout(idx, E, R, lib=lib)
    assert rr["status"] == oracle.OK and rr["total_rows"] == sum(g["rank_count"])
    np.testing.assert_array_equal(rr["rank_slot"], g["rank_slot"])
    np.testing.assert_array_equal(rr["rank_src"], g["rank_src"])
    # rows: token t's row is bf16 values (t+1)/8 .. so n * x is exact
    H = 8
    x = np.zeros((4, H), np.float32)
    for t in range(4):
        x[t] = (t + 1) / 8.0 + np.arange(H) / 64.0
    xb = torch_bf16_bits(x)
    st, recv, _ = oracle.permute(xb.view(np.uint8).reshape(4, 2 * H), r["dst_slot"],
                                 r["expert_offset"], r["expert_count"], 8, lib=lib)
    assert st == oracle.OK
    recv16 = recv.view(np.uint16).reshape(8, H)
    for i, s in enumerate(g["src_idx"]):
        if s < 0:
            assert np.all(recv16[i] == 0), f"pad row {i} not zero"
        else:
            np.testing.assert_array_equal(recv16[i], xb[s])
    out = oracle.combine(recv16, r["dst_slot"], np.ones((4, 2), np.float32), lib=lib)
    want = torch_bf16_bits(np.array(g["unit_weight_combine_multiplier"], np.float32)[:, None]
                           * bf16_bits_to_f32(xb))
    np.testing.assert_array_equal(out, want)


def check_padding_example(lib):
    g = json.load(open(os.path.join(GOLDEN, "padding_example_50_tokens_a64.json")))
    A, n = g["alignment"], g["tokens_for_expert"]
    # 3 experts, K=1: 7 tokens to expert 0, 50 to expert 1 (the page's case), 70 to expert 2,
    # interleaved so that the segment is built from scattered tokens.
    rng = np.random.default_rng(7)
    ids = np.array([0] * 7 + [1] * n + [2] * 70, np.int64)
    rng.shuffle(ids)
    idx = ids[:, None]
    r = oracle.layout(idx, 3, 1, A, lib=lib)
    assert r["status"] == oracle.OK
    off = r["expert_offset"]
    assert off[2] - off[1] == g["segment_slots"]
    seg = r["src_idx"][off[1]:off[2]]
    assert int((seg >= 0).sum()) == g["real_rows"]
    assert np.all(seg[:g["real_rows"]] >= 0) and np.all(seg[g["real_rows"]:] == -1)
    assert int((seg < 0).sum()) == g["pad_rows"]
    x = rng.integers(1, 255, size=(ids.size, 16), dtype=np.uint8)
    st, recv, _ = oracle.permute(x, r["dst_slot"], off, r["expert_count"], r["total_rows"], lib=lib)
    assert st == oracle.OK
    assert np.all(recv[off[1] + g["real_rows"]:off[2]] == 0)
    assert np.all(recv[off[1]:off[1] + g["real_rows"]] != 0)


SORT_CASES = [
    # N, K, E, R, A, mask, skew
    (1, 1, 1, 1, 1, 0.0, False),
    (37, 2, 8, 2, 1, 0.0, False),
    (300, 8, 64, 8, 16, 0.1, False),
    (513, 8, 256, 8, 128, 0.0, False),
    (400, 6, 48, 4, 3, 0.2, True),
    (200, 32, 40, 5, 7, 0.05, False),
    (90, 3, 9, 3, 5, 0.5, True),
    (64, 8, 16, 16, 4, 1.0, False),   # everything masked
]


def check_sort_formulation(lib, cases=SORT_CASES, seed=11):
    rng = np.random.default_rng(seed)
    for case in cases:
        N, K, E, R, A, mask, skew = case
        idx = random_idx(rng, N, K, E, mask, skew)
        r = oracle.layout(idx, E, R, A, lib=lib)
        assert r["status"] == oracle.OK
        assert_layout_equal(r, sort_formulation(idx, E, R, A), f"case {case}")


def check_rank_sort_formulation(lib, cases=SORT_CASES, seed=21):
    rng = np.random.default_rng(seed)
    for case in cases:
        N, K, E, R, A, mask, skew = case
        idx = random_idx(rng, N, K, E, mask, skew)
        r = oracle.rank_layout(idx, E, R, lib=lib)
        want = rank_sort_formulation(idx, E, R)
        assert r["status"] == oracle.OK and r["total_rows"] == want["total_rows"], case
        np.testing.assert_array_equal(r["rank_slot"], want["rank_slot"], err_msg=str(case))
        np.testing.assert_array_equal(r["rank_src"], want["rank_src"], err_msg=str(case))
        # rank blocks have the expand layout's rank counts, in rank order
        lay = oracle.layout(idx, E, R, A, lib=lib)
        starts = np.concatenate([[0], lay["rank_psum"][:-1]])
        for rr_ in range(R):
            blk = r["rank_src"][starts[rr_]:lay["rank_psum"][rr_]]
            assert blk.size == lay["rank_count"][rr_] and np.all(np.diff(blk) > 0)


def check_invariants(lib, seed=12):
    rng = np.random.default_rng(seed)
    for case in SORT_CASES:
        N, K, E, R, A, mask, skew = case
        idx = random_idx(rng, N, K, E, mask, skew)
        r = oracle.layout(idx, E, R, A, lib=lib)
        check_layout_invariants(idx, E, R, A, r)
    # single expert takes everything (K=1)
    idx = np.full((50, 1), 3, np.int64)
    r = oracle.layout(idx, 4, 2, 8, lib=lib)
    check_layout_invariants(idx, 4, 2, 8, r)
    assert r["total_rows"] == 56


def _definition_by_enumeration(idx, E, R, A):
    """The layout written pair by pair from its definition (tiny inputs only)."""
    N, K = idx.shape
    L = E // R
    cnt = [sum(1 for t in range(N) for k in range(K) if idx[t, k] == e) for e in range(E)]
    rc = [sum(1 for t in range(N) if any(idx[t, k] >= 0 and idx[t, k] // L == r for k in range(K)))
          for r in range(R)]
    off = [sum(-(-cnt[j] // A) * A for j in range(e)) for e in range(E + 1)]
    dst = np.full((N, K), -1, np.int64)
    src = np.full(off[E], -1, np.int64)
    for t in range(N):
        for k in range(K):
            e = idx[t, k]
            if e < 0:
                continue
            before = sum(1 for t2 in range(N) for k2 in range(K)
                         if (t2, k2) < (t, k) and idx[t2, k2] == e)
            dst[t, k] = off[e] + before
            src[off[e] + before] = t
    # non-expand rows: (t, r) pairs by rank then token; the highest k reaching r takes the row
    rstart = [sum(rc[:r]) for r in range(R)]
    rslot = np.full((N, K), -1, np.int64)
    rsrc = np.full(sum(rc), -1, np.int64)
    for t in range(N):
        for r in range(R):
            ks = [k for k in range(K) if idx[t, k] >= 0 and idx[t, k] // L == r]
            if not ks:
                continue
            row = rstart[r] + sum(1 for t2 in range(t) if any(idx[t2, k] >= 0 and idx[t2, k] // L == r
                                                              for k in range(K)))
            rslot[t, max(ks)] = row
            rsrc[row] = t
    return dict(expert_count=cnt, rank_count=rc, expert_offset=off,
                rank_psum=np.cumsum(rc), dst_slot=dst, src_idx=src, total_rows=off[E],
                rank_slot=rslot, rank_src=rsrc)


BRUTE_SHAPES = [(1, 1, 3), (2, 2, 3), (3, 2, 2), (1, 3, 4), (2, 1, 4)]


def check_bruteforce(lib, shapes=BRUTE_SHAPES, alignments=(1, 2, 3)):
    for N, K, E in shapes:
        ranks = [r for r in range(1, E + 1) if E % r == 0]
        for combo in itertools.product(range(-1, E), repeat=N * K):
            idx = np.array(combo, np.int64).reshape(N, K)
            for R in ranks:
                for A in alignments:
                    r = oracle.layout(idx, E, R, A, lib=lib)
                    assert r["status"] == oracle.OK
                    want = _definition_by_enumeration(idx, E, R, A)
                    assert_layout_equal(r, want, f"idx={combo} E={E} R={R} A={A}")
                    if A == 1:
                        rr = oracle.rank_layout(idx, E, R, lib=lib)
                        np.testing.assert_array_equal(rr["rank_slot"], want["rank_slot"])
                        np.testing.assert_array_equal(rr["rank_src"], want["rank_src"])


def check_permute(lib, seed=13):
    rng = np.random.default_rng(seed)
    N, K, E, R, A = 300, 8, 32, 4, 16
    idx = random_idx(rng, N, K, E, 0.15)
    r = oracle.layout(idx, E, R, A, lib=lib)
    rows = r["total_rows"]
    x = rng.integers(0, 256, size=(N, 48), dtype=np.uint8)
    sf = rng.integers(0, 256, size=(N, 12), dtype=np.uint8)
    st, recv, recv_sf = oracle.permute(x, r["dst_slot"], r["expert_offset"], r["expert_count"],
                                       rows, sf_bytes=sf, lib=lib)
    assert st == oracle.OK
    src = r["src_idx"]
    real = src >= 0
    np.testing.assert_array_equal(recv[real], x[src[real]])
    np.testing.assert_array_equal(recv_sf[real], sf[src[real]])
    assert np.all(recv[~real] == 0) and np.all(recv_sf[~real] == 0)
    # without zero padding the pad rows are left as they were
    st, recv2, _ = oracle.permute(x, r["dst_slot"], r["expert_offset"], r["expert_count"], rows,
                                  zero_pad=False, lib=lib)
    np.testing.assert_array_equal(recv2[real], x[src[real]])
    assert np.all(recv2[~real] == 0xA5)


def _dispatch_bf16(lib, idx, E, R, A, x_f32):
    r = oracle.layout(idx, E, R, A, lib=lib)
    xb = torch_bf16_bits(x_f32)
    N, H = xb.shape
    st, recv, _ = oracle.permute(xb.view(np.uint8).reshape(N, 2 * H), r["dst_slot"],
                                 r["expert_offset"], r["expert_count"], r["total_rows"], lib=lib)
    assert st == oracle.OK
    return r, xb, recv.view(np.uint16).reshape(r["total_rows"], H)


def check_combine_closed_form(lib, seed=14):
    """Unit weights, expert output = dispatched rows: out[t] = bf16(n_valid(t) * x[t])."""
    rng = np.random.default_rng(seed)
    N, K, E, R, A, H = 180, 8, 16, 4, 4, 40
    idx = random_idx(rng, N, K, E)
    n_valid = np.arange(N) % (K + 1)           # 0..8 valid slots, in random positions
    for t in range(N):
        drop = rng.permutation(K)[: K - n_valid[t]]
        idx[t, drop] = -1
    x = rng.standard_normal((N, H)).astype(np.float32)
    r, xb, recv = _dispatch_bf16(lib, idx, E, R, A, x)
    out = oracle.combine(recv, r["dst_slot"], np.ones((N, K), np.float32), lib=lib)
    # n * x is exact in fp32 (<= 11 significant bits); torch rounds it to bf16.
    want = torch_bf16_bits(n_valid[:, None].astype(np.float32) * bf16_bits_to_f32(xb))
    want[n_valid == 0] = 0                     # an empty sum is +0, not 0 * x
    np.testing.assert_array_equal(out, want)
    pow2 = np.isin(n_valid, [1, 2, 4, 8])
    np.testing.assert_array_equal(bf16_bits_to_f32(out[pow2]),
                                  n_valid[pow2, None] * bf16_bits_to_f32(xb[pow2]))
    assert np.all(out[n_valid == 0] == 0)


def check_combine_bound(lib, seed=15):
    rng = np.random.default_rng(seed)
    N, K, E, R, A, H = 150, 8, 24, 6, 8, 64
    idx = random_idx(rng, N, K, E, 0.2)
    r = oracle.layout(idx, E, R, A, lib=lib)
    rows = r["total_rows"]
    eo = torch_bf16_bits(rng.standard_normal((rows, H)).astype(np.float32) * 3)
    w = torch.softmax(torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)), 1).numpy()
    w = w * rng.choice([-1.0, 1.0], size=(N, K)).astype(np.float32)   # signs matter too
    out = oracle.combine(eo, r["dst_slot"], w, lib=lib)
    eo64 = bf16_bits_to_f32(eo).astype(np.float64)
    dst = r["dst_slot"]
    exact = np.zeros((N, H))
    absum = np.zeros((N, H))
    for t in range(N):
        for k in range(K):
            if dst[t, k] >= 0:
                term = float(w[t, k]) * eo64[dst[t, k]]
                exact[t] += term
                absum[t] += np.abs(term)
    got = bf16_bits_to_f32(out).astype(np.float64)
    # fp32 fma chain: <= K * 2^-24 * sum|w x|; bf16 rounding: <= 2^-8 |result| (8 significant bits)
    bound = K * 2.0 ** -24 * absum + 2.0 ** -8 * np.abs(got) + 1e-30
    err = np.abs(got - exact)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound)}"
    # all-masked tokens give exact zeros
    none = (dst < 0).all(axis=1)
    assert np.all(out[none] == 0)
    # tokens_subset agrees with the full combine
    sel = np.array([0, 7, N - 1, 42], np.int64)
    np.testing.assert_array_equal(oracle.combine_tokens(sel, eo, dst, w, lib=lib), out[sel])


def _round_f32(q: Fraction) -> Fraction:
    """IEEE binary32 round-to-nearest-even of an exact rational (normal and subnormal)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum_exp = max(e - 23, -149)
    scaled = a / Fraction(2) ** quantum_exp
    n, rem = divmod(scaled.numerator, scaled.denominator)
    rem = Fraction(rem, scaled.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * Fraction(2) ** quantum_exp


def _round_bf16_bits(q: Fraction) -> int:
    """binary32 value (exact rational) -> bf16 bits, round to nearest even (8-bit significand)."""
    if q == 0:
        return 0
    sign = 1 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum_exp = max(e - 7, -133)
    scaled = a / Fraction(2) ** quantum_exp
    n, rem = divmod(scaled.numerator, scaled.denominator)
    rem = Fraction(rem, scaled.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    f = np.float32(float(n * Fraction(2) ** quantum_exp))
    bits = int(np.array([f], np.float32).view(np.uint32)[0] >> 16)
    return bits | (sign << 15)


def check_combine_exact(lib, seed=16):
    """Bit-exact against an exact-rational emulation of the fp32 fma chain (k ascending)."""
    rng = np.random.default_rng(seed)
    N, K, E, R, A, H = 24, 8, 12, 3, 2, 12
    idx = random_idx(rng, N, K, E, 0.25)
    r = oracle.layout(idx, E, R, A, lib=lib)
    rows = r["total_rows"]
    eo = torch_bf16_bits(rng.standard_normal((rows, H)).astype(np.float32) * 7)
    w = (rng.standard_normal((N, K)) / 3).astype(np.float32)
    out = oracle.combine(eo, r["dst_slot"], w, lib=lib)
    eof = bf16_bits_to_f32(eo)
    dst = r["dst_slot"]
    for t in range(N):
        for h in range(H):
            acc = Fraction(0)
            for k in range(K):
                s = dst[t, k]
                if s < 0:
                    continue
                acc = _round_f32(Fraction(float(w[t, k])) * Fraction(float(eof[s, h])) + acc)
            assert int(out[t, h]) == _round_bf16_bits(acc), (t, h)
    # A cancellation case where one rounding and two roundings differ after
    # the bf16 cast: with r = fp32(w1 * x1), the terms r * (-1) then w1 * x1
    # leave exactly the product's rounding error under a fused multiply-add
    # (here 2^-30 * c) but 0 under multiply-then-add.  Reversing k also gives 0.
    H2 = 4
    c = np.array([1.0, -2.0, 0.5, 8.0], np.float32)
    x1 = np.float32(1.0 + 2.0 ** -7)                        # exact in bf16
    w1 = np.float32(1.0 + 2.0 ** -23)
    r_ = np.float32(w1 * x1)                                # fp32 product, 2^-30 dropped
    eo2 = torch_bf16_bits(np.stack([-c, x1 * c]).astype(np.float32))   # both rows exact in bf16
    dst2 = np.array([[0, 1]], np.int32)
    out2 = oracle.combine(eo2, dst2, np.array([[r_, w1]], np.float32), lib=lib)
    want2 = torch_bf16_bits((c * np.float32(2.0 ** -30)).astype(np.float32))[None]
    for h in range(H2):
        acc = _round_f32(Fraction(float(r_)) * Fraction(float(-c[h])))
        acc = _round_f32(Fraction(float(w1)) * Fraction(float(x1 * c[h])) + acc)
        assert _round_bf16_bits(acc) == int(want2[0, h])
    np.testing.assert_array_equal(out2, want2)


def check_roundtrip_direct(lib, seed=17):
    """dispatch -> stand-in expert (x * s_e) -> combine, against a formula from x alone."""
    rng = np.random.default_rng(seed)
    N, K, E, R, A, H = 256, 8, 24, 4, 8, 32
    idx = random_idx(rng, N, K, E, 0.05)
    x = rng.standard_normal((N, H)).astype(np.float32)
    r, xb, recv = _dispatch_bf16(lib, idx, E, R, A, x)
    s = (1.0 + np.arange(E, dtype=np.float32) / np.float32(384.0)).astype(np.float32)
    eo = oracle.expert_scale(recv, r["expert_offset"], s, lib=lib)
    w = torch.softmax(torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)), 1).numpy()
    out = oracle.combine(eo, r["dst_slot"], w, lib=lib)
    xf = bf16_bits_to_f32(xb)
    exact = np.zeros((N, H))
    absum = np.zeros((N, H))
    for t in range(N):
        for k in range(K):
            e = idx[t, k]
            if e < 0:
                continue
            # the expert's output row, rounded by torch, never via recv_x
            y = bf16_bits_to_f32(torch_bf16_bits(xf[t] * s[e])).astype(np.float64)
            exact[t] += float(w[t, k]) * y
            absum[t] += np.abs(float(w[t, k]) * y)
    got = bf16_bits_to_f32(out).astype(np.float64)
    bound = K * 2.0 ** -24 * absum + 2.0 ** -8 * np.abs(got) + 1e-30
    assert np.all(np.abs(got - exact) <= bound)
    # the stand-in expert itself vs torch on every real row
    src = r["src_idx"]
    seg_e = np.searchsorted(r["expert_offset"], np.arange(r["total_rows"]), side="right") - 1
    real = src >= 0
    np.testing.assert_array_equal(eo[real], torch_bf16_bits(xf[src[real]] * s[seg_e[real], None]))
    assert np.all(eo[~real] == 0)


def check_bf16(lib, seed=18):
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    # make a quarter of them exact ties, and avoid NaN payload comparisons
    u[::4] = (u[::4] & 0xFFFF0000) | 0x8000
    f = u.view(np.float32)
    f = f[~np.isnan(f)]
    np.testing.assert_array_equal(oracle.f32_to_bf16(f, lib=lib), torch_bf16_bits(f))


def check_errors(lib):
    idx = np.array([[0, 5], [1, -1], [4, 2]], np.int64)   # 5 and 4 are >= E=4
    r = oracle.layout(idx, 4, 2, 2, lib=lib)
    assert r["status"] == oracle.BAD_EXPERT_ID
    np.testing.assert_array_equal(r["expert_count"], [1, 1, 1, 0])
    np.testing.assert_array_equal(r["dst_slot"], [[0, -1], [2, -1], [-1, 4]])
    rr = oracle.rank_layout(idx, 4, 2, lib=lib)
    assert rr["status"] == oracle.BAD_EXPERT_ID
    np.testing.assert_array_equal(rr["rank_slot"], [[0, -1], [1, -1], [-1, 2]])
    idx = np.array([[0], [0], [0]], np.int64)
    r = oracle.layout(idx, 2, 1, 4, capacity_rows=3, lib=lib)
    assert r["status"] == oracle.CAPACITY and r["total_rows"] == 4
    rr = oracle.rank_layout(idx, 2, 1, capacity_rows=2, lib=lib)
    assert rr["status"] == oracle.CAPACITY and rr["total_rows"] == 3


def check_sf_col_major(lib, seed=19):
    g = json.load(open(os.path.join(GOLDEN, "handworked_n4_k2_e4_r2_a2.json")))
    sfw = np.array(g["sf_words"], np.uint32)
    st, out = oracle.permute_sf_col_major(sfw, g["dst_slot"], g["expert_offset"], g["expert_count"],
                                          g["total_rows"], lib=lib)
    assert st == oracle.OK and out.shape == (3, 8)
    np.testing.assert_array_equal(out, g["sf_col_major"])
    # a wider leading dimension: words past the rows are not written
    st, out = oracle.permute_sf_col_major(sfw, g["dst_slot"], g["expert_offset"], g["expert_count"],
                                          g["total_rows"], ld=12, lib=lib)
    assert st == oracle.OK
    np.testing.assert_array_equal(out[:, :8], g["sf_col_major"])
    assert np.all(out[:, 8:] == 0xA5A5A5A5)
    # leading dimension must cover the rows and be a multiple of 4 words (16 bytes)
    for ld in (6, 10):
        st, _ = oracle.permute_sf_col_major(sfw, g["dst_slot"], g["expert_offset"], g["expert_count"],
                                            g["total_rows"], ld=ld, lib=lib)
        assert st == oracle.BAD_ARG, ld

    rng = np.random.default_rng(seed)
    N, K, E, R, A, C = 300, 8, 32, 4, 16, 7
    idx = random_idx(rng, N, K, E, 0.15)
    r = oracle.layout(idx, E, R, A, lib=lib)
    rows = r["total_rows"]
    sf = rng.integers(0, 2**32, size=(N, C), dtype=np.uint32)
    src = r["src_idx"]
    real = src >= 0
    ld = (rows + 3) // 4 * 4 + 4
    st, out = oracle.permute_sf_col_major(sf, r["dst_slot"], r["expert_offset"], r["expert_count"], rows,
                                          ld=ld, lib=lib)
    assert st == oracle.OK
    # gather formulation: column j of row i is word j of token src_idx[i]
    np.testing.assert_array_equal(out[:, :rows][:, real], sf[src[real]].T)
    assert np.all(out[:, :rows][:, ~real] == 0)
    assert np.all(out[:, rows:] == 0xA5A5A5A5)
    # the transpose of the row-major scatter of the same words
    _, _, recv_sf = oracle.permute(np.zeros((N, 16), np.uint8), r["dst_slot"], r["expert_offset"],
                                   r["expert_count"], rows, sf_bytes=sf.view(np.uint8).reshape(N, 4 * C), lib=lib)
    np.testing.assert_array_equal(out[:, :rows], recv_sf.view(np.uint32).reshape(rows, C).T)
    # without zero padding the gap rows keep what was there
    st, out2 = oracle.permute_sf_col_major(sf, r["dst_slot"], r["expert_offset"], r["expert_count"], rows,
                                           zero_pad=False, lib=lib)
    np.testing.assert_array_equal(out2[:, :rows][:, real], sf[src[real]].T)
    assert np.all(out2[:, :rows][:, ~real] == 0xA5A5A5A5)


ALL_CHECKS = [
    check_handworked, check_padding_example, check_sort_formulation, check_rank_sort_formulation,
    check_invariants,
    check_bruteforce, check_permute, check_combine_closed_form, check_combine_bound,
    check_combine_exact, check_roundtrip_direct, check_bf16, check_errors, check_sf_col_major,
]


def main(argv):
    """Run every check against the oracle library at argv[1]; exit 1 on the first failure."""
    lib = oracle.load(argv[1])
    for chk in ALL_CHECKS:
        try:
            chk(lib)
        except AssertionError as exc:
            print(f"FAILED {chk.__name__}: {str(exc)[:300]}")
            return 1
    print("all checks passed")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
