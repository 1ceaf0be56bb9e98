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


def _no_cuda_device() -> bool:
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return True


@pytest.mark.skipif(not _no_cuda_device(), reason="needs a machine without a CUDA device (fake pointers below)")
def test_every_cuda_failure_is_recorded_for_last_cuda_error(lib):
    """On a machine with no CUDA device the first CUDA call of each entry point
    fails; every one of them must return MOE_ERR_CUDA (2) and leave the CUDA
    error behind it for moe_last_cuda_error, in the calling thread.  The
    pointers are never dereferenced: each path fails at its first CUDA call,
    which cannot reach a device."""
    import threading

    import numpy as np

    lib.moe_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
    lib.moe_last_cuda_error.restype = ctypes.c_int
    p, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.moe_layout_build_noalloc.argtypes = [ctypes.POINTER(binding._CDesc), p, p, p, p, p, p, p, i64, p, p, p]
    lib.moe_layout_build_noalloc.restype = ctypes.c_int
    N, K, E, R, A, H = 64, 8, 16, 4, 4, 16
    d = ctypes.byref(_desc(N, K, E, R, A))
    n = ctypes.c_size_t(0)
    assert lib.moe_layout_workspace_bytes(d, ctypes.byref(n)) == 0
    fake = ctypes.c_void_p(1 << 20)
    ids = np.zeros((N, K), np.int64)
    x = np.zeros((N, H), np.uint16)
    w = np.zeros((N, K), np.float32)
    host = lambda a: ctypes.c_void_p(a.ctypes.data)
    calls = {
        "moe_dispatch_from_host": lambda: lib.moe_dispatch_from_host(
            d, host(ids), host(x), 2 * H, None, 0, host(w), fake, fake, None, fake, fake, fake, fake, fake, fake,
            fake, fake, fake, None, 1024, fake, n.value, 0, None, fake),
        "moe_combine_to_host": lambda: lib.moe_combine_to_host(
            d, fake, 1024, H, fake, fake, fake, host(x), fake, n.value, 0, None, fake),
        "moe_layout_build_noalloc": lambda: lib.moe_layout_build_noalloc(
            d, fake, fake, fake, fake, fake, fake, fake, 1024, fake, fake, None),
        "moe_layout_build": lambda: lib.moe_layout_build(
            d, fake, fake, fake, fake, n.value, fake, fake, fake, fake, 1024, fake, None),
        "moe_layout_get_error": lambda: lib.moe_layout_get_error(fake, ctypes.byref(ctypes.c_int32()), None),
    }
    results = {}

    def run():
        for name, call in calls.items():
            st = call()
            results[name] = (st, lib.moe_last_cuda_error(None))

    t = threading.Thread(target=run)
    t.start()
    t.join()
    for name, (st, code) in results.items():
        assert st == 2, f"{name} returned {st}"
        assert code != 0, f"{name}: moe_last_cuda_error() is 0 after MOE_ERR_CUDA"
    # The record is per thread: this thread has had no failing CUDA call.
    assert lib.moe_last_cuda_error(None) == 0
