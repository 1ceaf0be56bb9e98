"""CPU oracle for the MoE dispatch layout and combine -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never calls
it, and it never imports the library: the two share nothing but the seeded
input generators.

The arithmetic lives in ``oracle.c`` (plain single-threaded C; each function
there cites the section of the page "07 DeepEP Counting Sort /
Bucketization" it follows).  This module only builds that file with gcc and
marshals numpy arrays into it.  Parity status of each function: pinned, see
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

# Error codes returned by oracle.c.
OK = 0
BAD_ARG = 1
BAD_EXPERT_ID = 2
CAPACITY = 3

# Plain optimisation, no fast-math, no contraction: fmaf is called explicitly.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib_cache: dict[str, ctypes.CDLL] = {}


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags: list[str] | None = None) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc; returns ``out``."""
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _needs_build(src: str, out: str) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if missing or stale) the oracle library at ``path``."""
    path = path or _LIB_PATH
    with _lock:
        if path in _lib_cache:
            return _lib_cache[path]
        if path == _LIB_PATH and _needs_build(_SRC, _LIB_PATH):
            build()
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib_cache[path] = lib
        return lib


def _declare(lib: ctypes.CDLL) -> None:
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.oracle_layout.restype = ctypes.c_int
    lib.oracle_layout.argtypes = [i64, i32, i32, i32, i32, p, p, p, p, p, p, p, i64, p]
    lib.oracle_rank_layout.restype = ctypes.c_int
    lib.oracle_rank_layout.argtypes = [i64, i32, i32, i32, p, p, p, i64, p]
    lib.oracle_permute.restype = ctypes.c_int
    lib.oracle_permute.argtypes = [i64, i32, p, p, i64, p, i64, i32, p, p, p, p, i64, i32]
    lib.oracle_f32_to_bf16.restype = None
    lib.oracle_permute_sf_col_major.argtypes = [i64, i32, p, p, i64, i32, p, p, p, i64, i64, i32]
    lib.oracle_permute_sf_col_major.restype = ctypes.c_int
    lib.oracle_f32_to_bf16.argtypes = [i64, p, p]
    lib.oracle_expert_scale.restype = None
    lib.oracle_expert_scale.argtypes = [i64, i64, p, i32, p, p, p]
    lib.oracle_combine.restype = None
    lib.oracle_combine.argtypes = [i64, i32, p, p, p, i64, p]
    lib.oracle_combine_tokens.restype = None
    lib.oracle_combine_tokens.argtypes = [i64, p, i32, p, p, p, i64, p]


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _as(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def layout(topk_idx, num_experts: int, num_ranks: int, alignment: int,
           capacity_rows: int | None = None, lib: ctypes.CDLL | None = None) -> dict:
    """Count, prefix sums and slot maps.  ``topk_idx`` is int64 [N, K].

    Returns a dict with ``status``, ``expert_count`` [E], ``rank_count`` [R],
    ``expert_offset`` [E+1], ``rank_psum`` [R], ``dst_slot`` [N, K],
    ``src_idx`` [rows] and ``total_rows``.
    """
    lib = lib or load()
    idx = _as(topk_idx, np.int64)
    N, K = idx.shape
    E, R, A = int(num_experts), int(num_ranks), int(alignment)
    ec = np.zeros(E, np.int32)
    rc = np.zeros(R, np.int32)
    off = np.zeros(E + 1, np.int32)
    rps = np.zeros(R, np.int32)
    dst = np.full((N, K), -1, np.int32)
    if capacity_rows is None:
        capacity_rows = N * K + E * (A - 1)
    src = np.full(max(int(capacity_rows), 0), -1, np.int32)
    total = ctypes.c_int64(0)
    st = lib.oracle_layout(N, K, E, R, A, _ptr(idx), _ptr(ec), _ptr(rc), _ptr(off), _ptr(rps),
                           _ptr(dst), _ptr(src), int(capacity_rows), ctypes.addressof(total))
    rows = int(total.value)
    return dict(status=int(st), expert_count=ec, rank_count=rc, expert_offset=off, rank_psum=rps,
                dst_slot=dst, src_idx=src[:rows] if st != CAPACITY else src, total_rows=rows)


def rank_layout(topk_idx, num_experts: int, num_ranks: int, capacity_rows: int | None = None,
                lib: ctypes.CDLL | None = None) -> dict:
    """Non-expand (rank-contiguous) slot map: ``status``, ``rank_slot`` [N, K],
    ``rank_src`` [rows], ``total_rows``."""
    lib = lib or load()
    idx = _as(topk_idx, np.int64)
    N, K = idx.shape
    if capacity_rows is None:
        capacity_rows = N * num_ranks
    slot = np.full((N, K), -1, np.int32)
    src = np.full(max(int(capacity_rows), 0), -1, np.int32)
    total = ctypes.c_int64(0)
    st = lib.oracle_rank_layout(N, K, int(num_experts), int(num_ranks), _ptr(idx), _ptr(slot), _ptr(src),
                                int(capacity_rows), ctypes.addressof(total))
    rows = int(total.value)
    return dict(status=int(st), rank_slot=slot, rank_src=src[:rows] if st != CAPACITY else src, total_rows=rows)


def permute(x_bytes: np.ndarray, dst_slot, expert_offset, expert_count, rows: int,
            sf_bytes: np.ndarray | None = None, zero_pad: bool = True,
            lib: ctypes.CDLL | None = None, out: np.ndarray | None = None,
            out_sf: np.ndarray | None = None):
    """Expand-mode row scatter.  ``x_bytes`` is uint8 [N, row_bytes]
    (any row dtype viewed as bytes); returns ``(status, recv_x, recv_sf)``.
    Without ``out`` the receive buffer is new and filled with 0xA5 bytes, so
    rows the oracle leaves alone stay visible."""
    lib = lib or load()
    x = _as(x_bytes, np.uint8)
    dst = _as(dst_slot, np.int32)
    off = _as(expert_offset, np.int32)
    cnt = _as(expert_count, np.int32)
    N, rb = x.shape
    K = dst.shape[1] if dst.ndim == 2 else (dst.size // max(N, 1) if N else 1)
    E = cnt.shape[0]
    if out is None:
        recv = np.full((rows, rb), 0xA5, np.uint8)
    else:
        recv = out
        assert recv.dtype == np.uint8 and recv.shape[1] == rb and recv.shape[0] >= rows
    sf = srb = recv_sf = None
    if sf_bytes is not None:
        sf = _as(sf_bytes, np.uint8)
        srb = sf.shape[1]
        recv_sf = np.full((rows, srb), 0xA5, np.uint8) if out_sf is None else out_sf
    st = lib.oracle_permute(N, K, _ptr(dst), _ptr(x), rb, _ptr(sf), srb or 0, E, _ptr(off),
                            _ptr(cnt), _ptr(recv), _ptr(recv_sf), rows, 1 if zero_pad else 0)
    return int(st), recv, recv_sf


def permute_sf_col_major(sf_words: np.ndarray, dst_slot, expert_offset, expert_count, rows: int,
                         ld: int | None = None, zero_pad: bool = True, lib: ctypes.CDLL | None = None):
    """Scale factors of the receive buffer, column-major: ``sf_words`` is
    uint32 [N, C] (fp32 scales viewed as words); returns ``(status, out)``,
    out uint32 [C, ld] with column j of the receive rows in out[j, :rows].
    ``ld`` defaults to ``rows`` rounded up to a multiple of 4.  A new ``out``
    is filled with 0xA5A5A5A5 so words the oracle leaves alone stay visible."""
    lib = lib or load()
    sf = _as(sf_words, np.uint32)
    dst = _as(dst_slot, np.int32)
    off = _as(expert_offset, np.int32)
    cnt = _as(expert_count, np.int32)
    N, C = sf.shape
    K = dst.shape[1] if dst.ndim == 2 else (dst.size // max(N, 1) if N else 1)
    ld = (rows + 3) // 4 * 4 if ld is None else ld
    out = np.full((C, max(ld, 0)), 0xA5A5A5A5, np.uint32)
    st = lib.oracle_permute_sf_col_major(N, K, _ptr(dst), _ptr(sf), C, cnt.shape[0], _ptr(off), _ptr(cnt),
                                         _ptr(out), ld, rows, 1 if zero_pad else 0)
    return int(st), out


def f32_to_bf16(a, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """fp32 -> bf16 bits (uint16), round to nearest even."""
    lib = lib or load()
    a = _as(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib.oracle_f32_to_bf16(a.size, _ptr(a), _ptr(out))
    return out


def expert_scale(recv_x_bf16: np.ndarray, expert_offset, scale,
                 lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Round-trip stand-in expert: segment e scaled by ``scale[e]`` (bf16 bits in and out)."""
    lib = lib or load()
    rx = _as(recv_x_bf16, np.uint16)
    off = _as(expert_offset, np.int32)
    s = _as(scale, np.float32)
    rows, H = rx.shape
    eo = np.zeros_like(rx)
    lib.oracle_expert_scale(rows, H, _ptr(rx), s.shape[0], _ptr(off), _ptr(s), _ptr(eo))
    return eo


def combine(expert_out_bf16: np.ndarray, dst_slot, weights, lib: ctypes.CDLL | None = None,
            out: np.ndarray | None = None) -> np.ndarray:
    """Weighted top-k combine; bf16 bits [rows, H] in, bf16 bits [N, H] out."""
    lib = lib or load()
    eo = _as(expert_out_bf16, np.uint16)
    dst = _as(dst_slot, np.int32)
    w = _as(weights, np.float32)
    N, K = dst.shape
    H = eo.shape[1]
    if out is None:
        out = np.empty((N, H), np.uint16)
    assert out.dtype == np.uint16 and out.shape == (N, H) and out.flags["C_CONTIGUOUS"]
    lib.oracle_combine(N, K, _ptr(dst), _ptr(w), _ptr(eo), H, _ptr(out))
    return out


def combine_tokens(tokens, expert_out_bf16: np.ndarray, dst_slot, weights,
                   lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Combine for the listed tokens only; returns bf16 bits [len(tokens), H]."""
    lib = lib or load()
    tok = _as(tokens, np.int64)
    eo = _as(expert_out_bf16, np.uint16)
    dst = _as(dst_slot, np.int32)
    w = _as(weights, np.float32)
    K = dst.shape[1]
    H = eo.shape[1]
    out = np.empty((tok.size, H), np.uint16)
    lib.oracle_combine_tokens(tok.size, _ptr(tok), K, _ptr(dst), _ptr(w), _ptr(eo), H, _ptr(out))
    return out
