"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer.

Every parity claim rests on oracle/oracle.c, so it is also built with
-fsanitize=address,undefined and run, in a child process with the sanitizer
runtimes preloaded, through every pin of tests/oracle_checks.py and one
decode-sized pass of each entry point (layout, permute with scale rows,
combine, the non-expand rows, the column-major scale factors).  Any
out-of-bounds access, use of freed memory, signed overflow or other undefined
behaviour aborts the child and fails the test.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import os, sys
repo, lib_path = sys.argv[1], sys.argv[2]
sys.path[:0] = [repo, os.path.join(repo, "tests")]
import numpy as np
import torch
import oracle
oracle._LIB_PATH = lib_path
import oracle_checks as oc
from counting_sort_bucketization_gb300 import workloads as wl

lib = oracle.load(lib_path)
for check in oc.ALL_CHECKS:
    check(lib)

def u8(t):
    t = t.contiguous()
    return t.view(torch.uint8).numpy().reshape(t.shape[0], -1)

w = wl.WORKLOADS["decode"]
inp = wl.make(w, wl.SEEDS["decode"])
idx = inp["topk_idx"].numpy()
ref = oracle.layout(idx, w.num_experts, w.num_ranks, w.alignment)
rows = ref["total_rows"]
st, recv, _ = oracle.permute(u8(inp["x"]), ref["dst_slot"], ref["expert_offset"], ref["expert_count"], rows)
assert st == oracle.OK
oracle.combine(recv.view(np.uint16).reshape(rows, w.hidden), ref["dst_slot"], inp["weights"].numpy())
oracle.rank_layout(idx, w.num_experts, w.num_ranks)
sfw = wl.draw_sf_words(w.num_tokens, 56, 1).numpy().view(np.uint32)
st, _ = oracle.permute_sf_col_major(sfw, ref["dst_slot"], ref["expert_offset"], ref["expert_count"], rows)
assert st == oracle.OK
wf = wl.WORKLOADS["prefill_fp8"].replace(num_tokens=2048)
inpf = wl.make(wf, 3)
reff = oracle.layout(inpf["topk_idx"].numpy(), wf.num_experts, wf.num_ranks, wf.alignment)
st, _, _ = oracle.permute(u8(inpf["x"]), reff["dst_slot"], reff["expert_offset"], reff["expert_count"],
                          reff["total_rows"], sf_bytes=u8(inpf["sf"]))
assert st == oracle.OK
print("clean")
'''


def _runtime(name: str):
    path = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_is_clean_under_sanitizers(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not installed")
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc's sanitizer runtimes are not installed")
    lib = str(tmp_path / "liboracle_sanitized.so")
    oracle.build(out=lib, extra_flags=["-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
                                       "-fno-sanitize-recover=undefined"])
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}", ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    proc = subprocess.run([sys.executable, "-c", CHILD, REPO, lib], env=env, capture_output=True, text=True,
                          timeout=900)
    assert proc.returncode == 0 and proc.stdout.strip().endswith("clean"), proc.stderr[-4000:]
