"""GPU parity through the C ABI from a C program (tests/c/layout_parity.c):
the library driven with device memory from the CUDA runtime and the legacy
default stream, no Python on the data path, every output compared bit for bit
with the C oracle linked into the same program."""
import os
import shutil
import subprocess

import pytest

from counting_sort_bucketization_gb300 import binding, build

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_matches_the_oracle(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not installed")
    build.build()
    lib = binding.library_path()
    libdir, name = os.path.dirname(lib), os.path.basename(lib)
    cudalib = next((p for p in (os.path.join(CUDA_HOME, "lib64"), os.path.join(CUDA_HOME, "lib"))
                    if os.path.isdir(p)), None)
    exe = tmp_path / "layout_parity"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Werror",
           f"-I{os.path.join(REPO, 'include')}", f"-I{os.path.join(CUDA_HOME, 'include')}",
           os.path.join(REPO, "tests", "c", "layout_parity.c"), os.path.join(REPO, "oracle", "oracle.c"),
           "-o", str(exe), f"-L{libdir}", f"-l:{name}", f"-Wl,-rpath,{libdir}",
           f"-L{cudalib}", "-lcudart", f"-Wl,-rpath,{cudalib}", "-lm"]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    assert proc.returncode == 0, proc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert run.returncode == 0, f"exit {run.returncode}\n{run.stdout}\n{run.stderr}"
    assert "all cases match" in run.stdout
