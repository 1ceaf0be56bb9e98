"""Each plausible mistake planted in a copy of the oracle must fail a pin.

The mistakes are planted on the CPU only, in a temporary copy of oracle.c;
the real oracle is never modified.  A mutant that still passes every check
in tests/oracle_checks.py would mean the pins cannot tell that mistake from
the method, so the test fails.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = open(os.path.join(os.path.dirname(HERE), "oracle", "oracle.c")).read()

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("no_alignment", "run += align_up(expert_count[e], A);", "run += expert_count[e];"),
    ("align_rounds_down", "return ((x + a - 1) / a) * a;", "return (x / a) * a;"),
    ("align_one_too_many", "return ((x + a - 1) / a) * a;", "return ((x + a) / a) * a;"),
    ("no_rank_dedup", "if (last_token[r] != t) {\n        last_token[r] = t;", "if (1) {\n        last_token[r] = t;"),
    ("rank_is_e_mod_R", "expert_count[e] += 1;\n      int32_t r = (int32_t)(e / L);",
     "expert_count[e] += 1;\n      int32_t r = (int32_t)(e % R);"),
    ("rank_psum_exclusive", "rrun += rank_count[r];\n    rank_psum[r] = (int32_t)rrun;",
     "rank_psum[r] = (int32_t)rrun;\n    rrun += rank_count[r];"),
    ("expert_zero_dropped", "if (e < 0) continue;\n      if (e >= E) { status = ORACLE_BAD_EXPERT_ID; continue; }\n      expert_count",
     "if (e <= 0) continue;\n      if (e >= E) { status = ORACLE_BAD_EXPERT_ID; continue; }\n      expert_count"),
    ("pads_first_in_segment", "cursor[e] = expert_offset[e];",
     "cursor[e] = expert_offset[e + 1] - expert_count[e];"),
    ("token_order_reversed",
     "for (int64_t t = 0; t < N; ++t) {\n    for (int32_t k = 0; k < K; ++k) {\n      int64_t e = topk_idx[t * K + k];\n      if (e < 0 || e >= E) {",
     "for (int64_t t = N - 1; t >= 0; --t) {\n    for (int32_t k = 0; k < K; ++k) {\n      int64_t e = topk_idx[t * K + k];\n      if (e < 0 || e >= E) {"),
    ("src_idx_off_by_one", "src_idx[s] = (int32_t)t;", "src_idx[s] = (int32_t)t + 1;"),
    ("no_zero_pad", "memset(recv_x + i * row_bytes, 0, (size_t)row_bytes);", "(void)0;"),
    ("pad_range_from_segment_start", "int64_t lo = (int64_t)expert_offset[e] + expert_count[e];",
     "int64_t lo = (int64_t)expert_offset[e] + expert_count[e] / 2;"),
    ("sf_row_not_followed", "memcpy(recv_sf + s * sf_row_bytes, sf + t * sf_row_bytes,",
     "memcpy(recv_sf + s * sf_row_bytes, sf,"),
    ("combine_weights_reversed", "acc = fmaf(w[t * K + k],", "acc = fmaf(w[t * K + (K - 1 - k)],"),
    ("combine_masked_not_skipped", "if (s < 0) continue;\n      acc", "if (s < 0) s = 0;\n      acc"),
    ("combine_mul_then_add", "acc = fmaf(w[t * K + k], bf16_to_f32(eo[s * H + h]), acc);",
     "{ volatile float p_ = w[t * K + k] * bf16_to_f32(eo[s * H + h]); acc = p_ + acc; }"),
    ("bf16_truncates", "u += 0x7fffu + keep_lsb;", "u += 0u * keep_lsb;"),
    ("bf16_ties_away", "u += 0x7fffu + keep_lsb;", "u += 0x8000u + 0u * keep_lsb;"),
    ("expert_scale_wrong_expert", "* scale[e]);", "* scale[e == 0 ? 0 : e - 1]);"),
    ("rank_rows_to_lowest_lane", "for (int32_t k2 = k + 1; k2 < K; ++k2) {", "for (int32_t k2 = 0; k2 < k; ++k2) {"),
    ("rank_rows_dedup_ignored_in_count", "if (last_token[r] != t) { last_token[r] = t; count[r] += 1; }",
     "count[r] += 1;"),
    ("rank_rows_no_dedup", "if (taken) continue;", "(void)taken;"),
    ("rank_block_start_inclusive", "cursor[r] = run; run += count[r];", "run += count[r]; cursor[r] = run - 1;"),
    ("sf_col_major_stored_row_major", "for (int64_t j = 0; j < C; ++j) out[j * ld + s] = sf[t * C + j];",
     "for (int64_t j = 0; j < C; ++j) out[s * C + j] = sf[t * C + j];"),
    ("sf_col_major_columns_reversed", "for (int64_t j = 0; j < C; ++j) out[j * ld + s] = sf[t * C + j];",
     "for (int64_t j = 0; j < C; ++j) out[j * ld + s] = sf[t * C + (C - 1 - j)];"),
    ("sf_col_major_no_zero_pad", "for (int64_t j = 0; j < C; ++j) out[j * ld + i] = 0;", "(void)0;"),
    ("sf_col_major_ld_not_checked", "ld < rows || ld % 4 != 0", "ld < 0"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    assert SRC.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = tmp_path / f"liboracle_{name}.so"
    oracle.build(str(src), str(lib))
    proc = subprocess.run([sys.executable, os.path.join(HERE, "oracle_checks.py"), str(lib)],
                          capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"mutant {name} passed every pin:\n{proc.stdout}\n{proc.stderr}"
