"""The C ABI without a GPU: the library loads, exports every declared entry
point, and its host-side checks reject bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from counting_sort_bucketization_gb300 import binding, build

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(REPO, "include", "moe_layout.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_four_steps():
    names = declared_functions()
    for fn in ("moe_layout_count", "moe_layout_scan", "moe_dispatch_permute", "moe_combine_unpermute"):
        assert fn in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(lib):
    for fn in declared_functions():
        assert hasattr(lib, fn), f"{fn} declared in moe_layout.h but not exported"


def _desc(N=64, K=8, E=16, R=4, A=4):
    return binding._CDesc(N, K, E, R, A)


def test_workspace_bytes_and_desc_checks(lib):
    n = ctypes.c_size_t(0)
    assert lib.moe_layout_workspace_bytes(ctypes.byref(_desc()), ctypes.byref(n)) == 0
    assert n.value >= 256 and n.value % 256 == 0
    bad = [_desc(N=-1), _desc(K=0), _desc(E=0), _desc(R=0), _desc(A=0), _desc(E=10, R=4)]
    for d in bad:
        assert lib.moe_layout_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == 1
    for d in (_desc(K=33), _desc(E=2048, R=1), _desc(N=1 << 28, K=16)):
        assert lib.moe_layout_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == 6
    assert lib.moe_layout_workspace_bytes(None, ctypes.byref(n)) == 1
    assert lib.moe_layout_workspace_bytes(ctypes.byref(_desc()), None) == 1


def test_workspace_grows_with_tiles_and_experts(lib):
    sizes = []
    for N, E in ((4096, 256), (131072, 384), (16, 8)):
        n = ctypes.c_size_t(0)
        assert lib.moe_layout_workspace_bytes(ctypes.byref(_desc(N=N, E=E, R=8)), ctypes.byref(n)) == 0
        sizes.append(n.value)
    assert sizes[1] > sizes[0] > sizes[2]


def test_host_checks_reject_before_launch(lib):
    d = ctypes.byref(_desc())
    n = ctypes.c_size_t(0)
    lib.moe_layout_workspace_bytes(d, ctypes.byref(n))
    fake = ctypes.c_void_p(1 << 20)         # never dereferenced: every call below fails its checks
    misaligned_ws = ctypes.c_void_p((1 << 20) + 8)
    # workspace missing, misaligned or too small
    assert lib.moe_layout_count(d, fake, fake, fake, None, n.value, None) == 1
    assert lib.moe_layout_count(d, fake, fake, fake, misaligned_ws, n.value, None) == 1
    assert lib.moe_layout_count(d, fake, fake, fake, fake, n.value - 1, None) == 1
    # null outputs
    assert lib.moe_layout_count(d, None, fake, fake, fake, n.value, None) == 1
    assert lib.moe_layout_scan(d, fake, fake, fake, fake, n.value, fake, fake, None, fake, 100, fake, None) == 1
    assert lib.moe_layout_scan(d, fake, fake, fake, fake, n.value, fake, fake, fake, None, 100, fake, None) == 1
    assert lib.moe_layout_scan(d, fake, fake, fake, fake, n.value, fake, fake, fake, fake, -1, fake, None) == 1
    # permute: row bytes not a multiple of 16, misaligned rows, bad scale-factor rows
    args = lambda rb, x, sf, srb, rsf: (d, x, rb, sf, srb, fake, fake, fake, fake, rsf, 100, 1, fake, n.value, None)
    assert lib.moe_dispatch_permute(*args(24, fake, None, 0, None)) == 1
    assert lib.moe_dispatch_permute(*args(0, fake, None, 0, None)) == 1
    assert lib.moe_dispatch_permute(*args(32, ctypes.c_void_p((1 << 20) + 4), None, 0, None)) == 1
    assert lib.moe_dispatch_permute(*args(32, fake, fake, 6, fake)) == 1
    assert lib.moe_dispatch_permute(*args(32, fake, fake, 8, None)) == 1
    # combine: hidden not a multiple of 8, null weights
    assert lib.moe_combine_unpermute(d, fake, 10, 12, fake, fake, fake, fake, n.value, None) == 1
    assert lib.moe_combine_unpermute(d, fake, 10, 16, fake, None, fake, fake, n.value, None) == 1
    # column-major scale factors: ld not a multiple of 4 or below capacity, no columns,
    # output not 16-byte aligned, missing total or map
    sfa = lambda C, src, tot, out, ld: (d, fake, C, src, tot, out, ld, 100, 1, fake, n.value, None)
    assert lib.moe_dispatch_sf_col_major(*sfa(56, fake, fake, fake, 102)) == 1
    assert lib.moe_dispatch_sf_col_major(*sfa(56, fake, fake, fake, 96)) == 1
    assert lib.moe_dispatch_sf_col_major(*sfa(0, fake, fake, fake, 100)) == 1
    assert lib.moe_dispatch_sf_col_major(*sfa(56, fake, fake, ctypes.c_void_p((1 << 20) + 4), 100)) == 1
    assert lib.moe_dispatch_sf_col_major(*sfa(56, fake, None, fake, 100)) == 1
    assert lib.moe_dispatch_sf_col_major(*sfa(56, None, fake, fake, 100)) == 1
    assert lib.moe_layout_get_error(None, None, None) == 1


def test_oversized_rows_are_refused_before_launch(lib):
    """Rows past MOE_MAX_ROW_BYTES (2^30) return MOE_ERR_UNSUPPORTED (6): every
    byte offset stays well inside int64."""
    d = ctypes.byref(_desc())
    n = ctypes.c_size_t(0)
    lib.moe_layout_workspace_bytes(d, ctypes.byref(n))
    fake = ctypes.c_void_p(1 << 20)         # never dereferenced
    big = (1 << 30) + 16
    args = lambda rb, sf, srb: (d, fake, rb, sf, srb, fake, fake, fake, fake, fake if sf else None, 100, 1, fake,
                                n.value, None)
    assert lib.moe_dispatch_permute(*args(big, None, 0)) == 6
    assert lib.moe_dispatch_permute(*args(32, fake, big)) == 6
    ranks = lambda rb: (d, fake, rb, None, 0, fake, fake, fake, None, 100, fake, n.value, None)
    assert lib.moe_dispatch_permute_ranks(*ranks(big)) == 6
    assert lib.moe_combine_unpermute(d, fake, 10, (1 << 29) + 8, fake, fake, fake, fake, n.value, None) == 6
    sfa = lambda C, ld: (d, fake, C, fake, fake, fake, ld, 100, 1, fake, n.value, None)
    assert lib.moe_dispatch_sf_col_major(*sfa((1 << 28) + 1, 100)) == 6
    assert lib.moe_dispatch_sf_col_major(*sfa(56, (1 << 32) + 4)) == 6


def test_last_cuda_error_is_readable_without_a_gpu(lib):
    lib.moe_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
    lib.moe_last_cuda_error.restype = ctypes.c_int
    msg = ctypes.c_char_p()
    assert lib.moe_last_cuda_error(ctypes.byref(msg)) == 0      # no CUDA call has failed in this thread
    assert msg.value
    assert lib.moe_last_cuda_error(None) == 0


def test_wait_test_hook_checks_its_arguments(lib):
    lib.moe_debug_set_waits.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
    lib.moe_debug_set_waits.restype = ctypes.c_int
    assert lib.moe_debug_set_waits(2_000_000_000, 0, 0) == 1   # longer than the 1 s bound
    assert lib.moe_debug_set_waits(1_000_000, 0, 8) == 1       # bytes not a multiple of 16
    assert lib.moe_debug_set_waits(1_000_000, 1, 16) == 0
    assert lib.moe_debug_set_waits(0, 0, 0) == 0                # back to normal operation


def test_strerror_and_launch_counter(lib):
    for code, name in binding.ERROR_NAMES.items():
        assert lib.moe_strerror(code)
    assert lib.moe_strerror(99) == b"unknown status"
    assert lib.moe_kernel_launches() >= 0
