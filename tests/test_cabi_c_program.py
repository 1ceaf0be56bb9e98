"""The C ABI from C: include/moe_layout.h compiles as C99 and as C++17 with
warnings as errors, and a C program links against libmoe_layout.so and gets
the host-side answers (workspace size, argument checks, status strings)
without a GPU."""
import os
import shutil
import subprocess

import pytest

from counting_sort_bucketization_gb300 import binding, build

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(REPO, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe_layout.h"

int main(void) {
  moe_layout_desc d;
  size_t bytes = 0, bytes_more = 0;
  memset(&d, 0, sizeof d);
  d.num_tokens = 4096; d.topk = 8; d.num_experts = 256; d.num_ranks = 8; d.alignment = 128;
  if (moe_layout_workspace_bytes(&d, &bytes) != MOE_OK || bytes == 0 || bytes % 256 != 0) return 1;
  d.num_tokens = 131072;
  if (moe_layout_workspace_bytes(&d, &bytes_more) != MOE_OK || bytes_more <= bytes) return 2;
  d.num_tokens = 4096;
  if (moe_layout_workspace_bytes(NULL, &bytes) != MOE_ERR_INVALID_ARG) return 3;
  d.topk = MOE_MAX_TOPK + 1;
  if (moe_layout_workspace_bytes(&d, &bytes) != MOE_ERR_UNSUPPORTED) return 4;
  d.topk = 8;
  d.num_ranks = 7;                                   /* R must divide E */
  if (moe_layout_workspace_bytes(&d, &bytes) != MOE_ERR_INVALID_ARG) return 5;
  d.num_ranks = 8;
  /* rejected on the host before any CUDA call: no workspace */
  if (moe_layout_count(&d, (const int64_t*)0, (int32_t*)0, (int32_t*)0, (void*)0, bytes, (void*)0) !=
      MOE_ERR_INVALID_ARG) return 6;
  if (moe_strerror(MOE_ERR_CAPACITY) == NULL || strlen(moe_strerror(MOE_ERR_CAPACITY)) == 0) return 7;
  printf("ok %lu %lu\n", (unsigned long)bytes, (unsigned long)bytes_more);
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    build.build()
    return binding.library_path()


def test_header_compiles_as_c_and_cxx(tmp_path):
    if shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("gcc/g++ not installed")
    src = tmp_path / "only_header.c"
    src.write_text('#include "moe_layout.h"\nint moe_test_unused;\n')
    for cmd in (["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic"],
                ["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-x", "c++"]):
        proc = subprocess.run([*cmd, f"-I{INCLUDE}", "-fsyntax-only", str(src)], capture_output=True, text=True)
        assert proc.returncode == 0, proc.stderr


def test_c_program_links_and_runs(tmp_path, lib_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not installed")
    src = tmp_path / "use_moe_layout.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_moe_layout"
    libdir = os.path.dirname(lib_path)
    name = os.path.basename(lib_path)
    proc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{INCLUDE}", str(src), "-o", str(exe),
                           f"-L{libdir}", f"-l:{name}", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert proc.returncode == 0, proc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, f"exit {run.returncode}: {run.stdout} {run.stderr}"
    assert run.stdout.startswith("ok ")
