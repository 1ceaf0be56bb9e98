"""Python binding of libmoe_layout.so (include/moe_layout.h), via ctypes.

Argument marshalling only: each function checks that the torch tensors it is
given have the dtype, device and layout the C ABI expects, passes their data
pointers and the current CUDA stream, and raises ``LayoutError`` on a
non-zero status.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback.  If the library has not been built, the first
call raises.

A description (``desc``) is any object with the attributes ``num_tokens``,
``topk``, ``num_experts``, ``num_ranks`` and ``alignment`` (for instance a
``workloads.Workload``, or ``LayoutDesc``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import torch

from . import build as _build

ERROR_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_CUDA", 3: "MOE_ERR_BAD_EXPERT_ID",
    4: "MOE_ERR_CAPACITY", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_UNSUPPORTED",
}


class LayoutError(RuntimeError):
    def __init__(self, what: str, status: int):
        text = f"{what}: {ERROR_NAMES.get(status, status)} ({strerror(status)})"
        if status == 2:   # MOE_ERR_CUDA: add the CUDA error behind it
            msg = ctypes.c_char_p()
            code = load_library().moe_last_cuda_error(ctypes.byref(msg))
            text += f"; CUDA error {code}: {msg.value.decode() if msg.value else '?'}"
        super().__init__(text)
        self.status = status


@dataclasses.dataclass(frozen=True)
class LayoutDesc:
    num_tokens: int
    topk: int
    num_experts: int
    num_ranks: int
    alignment: int


class _CDesc(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int64), ("topk", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("num_ranks", ctypes.c_int32), ("alignment", ctypes.c_int32)]


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def library_path() -> str:
    """The in-tree build, unless MOE_LAYOUT_LIBRARY names another build of the same library."""
    return os.environ.get("MOE_LAYOUT_LIBRARY") or _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Open libmoe_layout.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run counting_sort_bucketization_gb300.build.build()")
        lib = ctypes.CDLL(path)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        dp = ctypes.POINTER(_CDesc)
        lib.moe_layout_workspace_bytes.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        lib.moe_layout_count.argtypes = [dp, p, p, p, p, sz, p]
        lib.moe_layout_scan.argtypes = [dp, p, p, p, p, sz, p, p, p, p, i64, p, p]
        lib.moe_layout_build.argtypes = [dp, p, p, p, p, sz, p, p, p, p, i64, p, p]
        lib.moe_layout_build_i32.argtypes = [dp, p, p, p, p, sz, p, p, p, p, i64, p, p]
        lib.moe_dispatch_permute.argtypes = [dp, p, i64, p, i64, p, p, p, p, p, i64, ctypes.c_int, p, sz, p]
        lib.moe_layout_rank_rows.argtypes = [dp, p, p, p, sz, p, p, i64, p]
        lib.moe_layout_accumulate_stats.argtypes = [dp, p, p, p]
        lib.moe_dispatch_from_host.argtypes = [dp, p, p, i64, p, i64, p, p, p, p, p, p, p, p, p, p, p, p, p, p,
                                               i64, p, sz, i64, p, p]
        lib.moe_combine_to_host.argtypes = [dp, p, i64, i64, p, p, p, p, p, sz, i64, p, p]
        lib.moe_dispatch_permute_ranks.argtypes = [dp, p, i64, p, i64, p, p, p, p, i64, p, sz, p]
        lib.moe_combine_unpermute.argtypes = [dp, p, i64, i64, p, p, p, p, sz, p]
        lib.moe_dispatch_sf_col_major.argtypes = [dp, p, i64, p, p, p, i64, i64, ctypes.c_int, p, sz, p]
        lib.moe_layout_get_error.argtypes = [p, ctypes.POINTER(i32), p]
        lib.moe_strerror.argtypes = [ctypes.c_int]
        lib.moe_strerror.restype = ctypes.c_char_p
        lib.moe_kernel_launches.argtypes = []
        lib.moe_kernel_launches.restype = ctypes.c_uint64
        lib.moe_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
        lib.moe_last_cuda_error.restype = ctypes.c_int
        lib.moe_debug_set_waits.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        lib.moe_debug_set_waits.restype = ctypes.c_int
        for name in ("moe_layout_workspace_bytes", "moe_layout_count", "moe_layout_scan", "moe_layout_build",
                     "moe_layout_build_i32",
                     "moe_layout_rank_rows", "moe_dispatch_permute_ranks", "moe_dispatch_from_host",
                     "moe_combine_to_host", "moe_layout_accumulate_stats",
                     "moe_dispatch_permute", "moe_combine_unpermute", "moe_layout_get_error",
                     "moe_dispatch_sf_col_major"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def strerror(status: int) -> str:
    return load_library().moe_strerror(int(status)).decode()


def debug_set_waits(limit_ns: int = 0, barrier_extra: int = 0, extra_tx: int = 0) -> None:
    """Test hook for the bounded waits (see moe_debug_set_waits); (0, 0, 0) restores normal operation."""
    _check(load_library().moe_debug_set_waits(int(limit_ns), int(barrier_extra), int(extra_tx)),
           "moe_debug_set_waits")


def kernel_launches() -> int:
    """Kernels the library has launched in this process."""
    return int(load_library().moe_kernel_launches())


def _desc(d) -> _CDesc:
    return _CDesc(int(d.num_tokens), int(d.topk), int(d.num_experts), int(d.num_ranks), int(d.alignment))


def _check(status: int, what: str) -> None:
    if status != 0:
        raise LayoutError(what, status)


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _dev(t: torch.Tensor | None, name: str, dtype=None, numel=None, allow_none=False, nbytes=None):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} needs at least {numel} elements, has {t.numel()}")
    if nbytes is not None and _nbytes(t) < nbytes:
        raise ValueError(f"{name} needs at least {nbytes} bytes, has {_nbytes(t)}")
    return ctypes.c_void_p(t.data_ptr())


def workspace_bytes(desc) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().moe_layout_workspace_bytes(ctypes.byref(_desc(desc)), ctypes.byref(n)),
           "moe_layout_workspace_bytes")
    return int(n.value)


def new_workspace(desc, device="cuda") -> torch.Tensor:
    """Zero-filled workspace for ``desc`` (torch's allocations are 256-byte aligned)."""
    return torch.zeros(max(workspace_bytes(desc), 256), dtype=torch.uint8, device=device)


def layout_count(desc, topk_idx, expert_count, rank_count, workspace, stream=None) -> None:
    N, K, E, R = int(desc.num_tokens), int(desc.topk), int(desc.num_experts), int(desc.num_ranks)
    st = load_library().moe_layout_count(
        ctypes.byref(_desc(desc)), _dev(topk_idx, "topk_idx", torch.int64, N * K),
        _dev(expert_count, "expert_count", torch.int32, E), _dev(rank_count, "rank_count", torch.int32, R),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_layout_count")


def layout_scan(desc, topk_idx, expert_count, rank_count, workspace, expert_offset, rank_psum, dst_slot,
                src_idx, total_rows, stream=None) -> None:
    N, K, E, R = int(desc.num_tokens), int(desc.topk), int(desc.num_experts), int(desc.num_ranks)
    st = load_library().moe_layout_scan(
        ctypes.byref(_desc(desc)), _dev(topk_idx, "topk_idx", torch.int64, N * K),
        _dev(expert_count, "expert_count", torch.int32, E), _dev(rank_count, "rank_count", torch.int32, R),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _dev(expert_offset, "expert_offset", torch.int32, E + 1), _dev(rank_psum, "rank_psum", torch.int32, R),
        _dev(dst_slot, "dst_slot", torch.int32, N * K), _dev(src_idx, "src_idx", torch.int32),
        src_idx.numel(), _dev(total_rows, "total_rows", torch.int32, 1), _stream(stream))
    _check(st, "moe_layout_scan")


def layout_build(desc, topk_idx, expert_count, rank_count, workspace, expert_offset, rank_psum, dst_slot,
                 src_idx, total_rows, stream=None) -> None:
    """layout_count + layout_scan in one call (one cooperative kernel when it fits).
    ``topk_idx`` may be int64 or int32."""
    N, K, E, R = int(desc.num_tokens), int(desc.topk), int(desc.num_experts), int(desc.num_ranks)
    lib = load_library()
    fn = lib.moe_layout_build_i32 if topk_idx.dtype == torch.int32 else lib.moe_layout_build
    st = fn(
        ctypes.byref(_desc(desc)), _dev(topk_idx, "topk_idx", topk_idx.dtype if topk_idx.dtype == torch.int32
                                        else torch.int64, N * K),
        _dev(expert_count, "expert_count", torch.int32, E), _dev(rank_count, "rank_count", torch.int32, R),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _dev(expert_offset, "expert_offset", torch.int32, E + 1), _dev(rank_psum, "rank_psum", torch.int32, R),
        _dev(dst_slot, "dst_slot", torch.int32, N * K), _dev(src_idx, "src_idx", torch.int32),
        src_idx.numel(), _dev(total_rows, "total_rows", torch.int32, 1), _stream(stream))
    _check(st, "moe_layout_build")


def _row_bytes(t: torch.Tensor, rows: int) -> int:
    if rows == 0:
        return t.shape[-1] * t.element_size() if t.dim() >= 2 else 0
    return t.numel() * t.element_size() // rows


def dispatch_permute(desc, x, dst_slot, expert_offset, expert_count, recv_x, workspace, sf=None,
                     recv_sf=None, zero_pad=True, stream=None) -> None:
    """recv_x[dst_slot[t,k]] = x[t] (bytes); gap rows zeroed.  x [N, ...], recv_x [capacity, ...]."""
    N, K, E = int(desc.num_tokens), int(desc.topk), int(desc.num_experts)
    cap = recv_x.shape[0]
    rb = x.shape[1] * x.element_size() if x.dim() == 2 else _row_bytes(x, N)
    if recv_x.numel() * recv_x.element_size() != cap * rb:
        raise ValueError("recv_x rows must have the same byte size as x rows")
    srb = 0
    if sf is not None:
        srb = sf.shape[1] * sf.element_size()
        if recv_sf is None or recv_sf.shape[0] != cap or recv_sf.numel() * recv_sf.element_size() != cap * srb:
            raise ValueError("recv_sf must be [capacity, sf row] when sf is given")
    st = load_library().moe_dispatch_permute(
        ctypes.byref(_desc(desc)), _dev(x, "x", nbytes=N * rb), rb, _dev(sf, "sf", allow_none=True, nbytes=N * srb),
        srb,
        _dev(dst_slot, "dst_slot", torch.int32, N * K), _dev(expert_offset, "expert_offset", torch.int32, E + 1),
        _dev(expert_count, "expert_count", torch.int32, E), _dev(recv_x, "recv_x"),
        _dev(recv_sf, "recv_sf", allow_none=True), cap, 1 if zero_pad else 0,
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_dispatch_permute")


def layout_rank_rows(desc, topk_idx, rank_count, workspace, rank_slot, rank_src, stream=None) -> None:
    """Non-expand slot map (one row per token and rank); follows a layout build on ``workspace``."""
    N, K, R = int(desc.num_tokens), int(desc.topk), int(desc.num_ranks)
    st = load_library().moe_layout_rank_rows(
        ctypes.byref(_desc(desc)), _dev(topk_idx, "topk_idx", torch.int64, N * K),
        _dev(rank_count, "rank_count", torch.int32, R), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _dev(rank_slot, "rank_slot", torch.int32, N * K), _dev(rank_src, "rank_src", torch.int32),
        rank_src.numel(), _stream(stream))
    _check(st, "moe_layout_rank_rows")


def dispatch_permute_ranks(desc, x, rank_slot, rank_psum, recv, workspace, sf=None, recv_sf=None,
                           stream=None) -> None:
    """recv[rank_slot[t,k]] = x[t] (bytes) for the slots that hold a row; no padding."""
    N, K, R = int(desc.num_tokens), int(desc.topk), int(desc.num_ranks)
    cap = recv.shape[0]
    rb = x.shape[1] * x.element_size()
    if recv.numel() * recv.element_size() != cap * rb:
        raise ValueError("recv rows must have the same byte size as x rows")
    srb = 0
    if sf is not None:
        srb = sf.shape[1] * sf.element_size()
        if recv_sf is None or recv_sf.shape[0] != cap or recv_sf.numel() * recv_sf.element_size() != cap * srb:
            raise ValueError("recv_sf must be [capacity, sf row] when sf is given")
    st = load_library().moe_dispatch_permute_ranks(
        ctypes.byref(_desc(desc)), _dev(x, "x", nbytes=N * rb), rb, _dev(sf, "sf", allow_none=True, nbytes=N * srb),
        srb,
        _dev(rank_slot, "rank_slot", torch.int32, N * K), _dev(rank_psum, "rank_psum", torch.int32, R),
        _dev(recv, "recv"), _dev(recv_sf, "recv_sf", allow_none=True), cap,
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_dispatch_permute_ranks")


def sf_col_major_ld(capacity_rows: int) -> int:
    """Leading dimension of a column-major scale buffer: rows rounded up to 4 words (16 bytes)."""
    return (int(capacity_rows) + 3) // 4 * 4


def new_sf_col_major(cols: int, capacity_rows: int, dtype=torch.float32, device="cuda") -> torch.Tensor:
    """Storage [cols, ld] for column-major scale factors; ``.t()[:capacity_rows]`` is the [rows, cols] view."""
    return torch.empty((int(cols), sf_col_major_ld(capacity_rows)), dtype=dtype, device=device)


def dispatch_sf_col_major(desc, sf, src, total_rows, recv_sf_cm, capacity_rows, workspace, zero_pad=True,
                          stream=None) -> None:
    """recv_sf_cm[j, i] = sf[src[i], j] for the receive rows i (column-major, ld = recv_sf_cm.shape[1])."""
    N = int(desc.num_tokens)
    if sf.element_size() != 4 or recv_sf_cm.element_size() != 4:
        raise ValueError("sf and recv_sf_cm must have 4-byte elements")
    if sf.dim() != 2 or sf.shape[0] != N or recv_sf_cm.dim() != 2 or recv_sf_cm.shape[0] != sf.shape[1]:
        raise ValueError("sf must be [N, C] and recv_sf_cm [C, ld]")
    st = load_library().moe_dispatch_sf_col_major(
        ctypes.byref(_desc(desc)), _dev(sf, "sf"), sf.shape[1], _dev(src, "src", torch.int32, capacity_rows),
        _dev(total_rows, "total_rows", torch.int32, 1), _dev(recv_sf_cm, "recv_sf_cm"), recv_sf_cm.shape[1],
        int(capacity_rows), 1 if zero_pad else 0, _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(st, "moe_dispatch_sf_col_major")


def combine_unpermute(desc, expert_out, dst_slot, weights, out, workspace, stream=None) -> None:
    """out[t] = bf16(sum_k w[t,k] * expert_out[dst_slot[t,k]]) with an fp32 fma chain."""
    N, K = int(desc.num_tokens), int(desc.topk)
    if expert_out.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("expert_out and out must be bfloat16")
    H = expert_out.shape[1]
    if out.shape != (N, H):
        raise ValueError(f"out must be [{N}, {H}]")
    st = load_library().moe_combine_unpermute(
        ctypes.byref(_desc(desc)), _dev(expert_out, "expert_out"), expert_out.shape[0], H,
        _dev(dst_slot, "dst_slot", torch.int32, N * K), _dev(weights, "weights", torch.float32, N * K),
        _dev(out, "out"), _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_combine_unpermute")


def accumulate_stats(desc, expert_count, cumulative, stream=None) -> None:
    """cumulative[e] += expert_count[e] on the device (int64 running totals)."""
    E = int(desc.num_experts)
    st = load_library().moe_layout_accumulate_stats(
        ctypes.byref(_desc(desc)), _dev(expert_count, "expert_count", torch.int32, E),
        _dev(cumulative, "cumulative", torch.int64, E), _stream(stream))
    _check(st, "moe_layout_accumulate_stats")


def _host(t: torch.Tensor | None, name: str, allow_none=False, nbytes=None):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor (page-locked for overlap)")
    if nbytes is not None and _nbytes(t) < nbytes:
        raise ValueError(f"{name} needs at least {nbytes} bytes, has {_nbytes(t)}")
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(s) -> ctypes.c_void_p:
    return ctypes.c_void_p(s.cuda_stream)


def dispatch_from_host(lay: "Layout", topk_idx_host, x_host, topk_idx, x, recv_x, weights_host=None, weights=None,
                       sf_host=None, sf=None, recv_sf=None, chunk_tokens=0, stream=None, copy_stream=None) -> None:
    """Host ids/rows in, layout + permuted rows on the device; copies overlapped with the permute.

    Asynchronous: the host tensors must stay alive and unwritten until
    ``stream`` reaches this point (the copies run outside torch's caching)."""
    d = lay.desc
    N, K = int(d.num_tokens), int(d.topk)
    s = stream if stream is not None else torch.cuda.current_stream()
    if copy_stream is None:
        raise ValueError("copy_stream is required (a stream other than `stream`)")
    rb = x_host.shape[1] * x_host.element_size()
    srb = sf_host.shape[1] * sf_host.element_size() if sf_host is not None else 0
    st = load_library().moe_dispatch_from_host(
        ctypes.byref(_desc(d)), _host(topk_idx_host, "topk_idx_host", nbytes=8 * N * K),
        _host(x_host, "x_host", nbytes=N * rb), rb, _host(sf_host, "sf_host", True, nbytes=N * srb), srb,
        _host(weights_host, "weights_host", True, nbytes=4 * N * K),
        _dev(topk_idx, "topk_idx", torch.int64, N * K), _dev(x, "x", nbytes=N * rb),
        _dev(sf, "sf", allow_none=True, nbytes=N * srb),
        _dev(weights, "weights", torch.float32, N * K, allow_none=True),
        _dev(lay.expert_count, "expert_count"), _dev(lay.rank_count, "rank_count"),
        _dev(lay.expert_offset, "expert_offset"), _dev(lay.rank_psum, "rank_psum"), _dev(lay.dst_slot, "dst_slot"),
        _dev(lay.src_idx, "src_idx"), _dev(lay.total_rows, "total_rows"),
        _dev(recv_x, "recv_x", nbytes=recv_x.shape[0] * rb),
        _dev(recv_sf, "recv_sf", allow_none=True, nbytes=recv_x.shape[0] * srb), recv_x.shape[0],
        _dev(lay.workspace, "workspace"),
        lay.workspace.numel(), int(chunk_tokens), _stream_ptr(s), _stream_ptr(copy_stream))
    _check(st, "moe_dispatch_from_host")


def combine_to_host(lay: "Layout", expert_out, weights, out, out_host, chunk_tokens=0, stream=None,
                    copy_stream=None) -> None:
    """Combine on the device with each chunk's result copied to ``out_host`` while the next is combined.

    Asynchronous: ``out_host`` must stay alive and unread until ``stream`` reaches this point."""
    d = lay.desc
    N, K = int(d.num_tokens), int(d.topk)
    s = stream if stream is not None else torch.cuda.current_stream()
    if copy_stream is None:
        raise ValueError("copy_stream is required (a stream other than `stream`)")
    if expert_out.dtype != torch.bfloat16 or out.dtype != torch.bfloat16 or out_host.dtype != torch.bfloat16:
        raise ValueError("expert_out, out and out_host must be bfloat16")
    st = load_library().moe_combine_to_host(
        ctypes.byref(_desc(d)), _dev(expert_out, "expert_out"), expert_out.shape[0], expert_out.shape[1],
        _dev(lay.dst_slot, "dst_slot", torch.int32, N * K), _dev(weights, "weights", torch.float32, N * K),
        _dev(out, "out", nbytes=2 * N * expert_out.shape[1]),
        _host(out_host, "out_host", nbytes=2 * N * expert_out.shape[1]), _dev(lay.workspace, "workspace"),
        lay.workspace.numel(),
        int(chunk_tokens), _stream_ptr(s), _stream_ptr(copy_stream))
    _check(st, "moe_combine_to_host")


def get_error(workspace, stream=None) -> int:
    """Synchronise, read and clear the workspace's sticky device error (0 = none)."""
    v = ctypes.c_int32(0)
    _check(load_library().moe_layout_get_error(_dev(workspace, "workspace", torch.uint8), ctypes.byref(v),
                                               _stream(stream)), "moe_layout_get_error")
    return int(v.value)


class Layout:
    """Device buffers of one dispatch layout (counts, offsets, maps) plus its workspace."""

    def __init__(self, desc, capacity_rows: int, device="cuda"):
        self.desc = desc
        self.capacity = int(capacity_rows)
        N, K, E, R = int(desc.num_tokens), int(desc.topk), int(desc.num_experts), int(desc.num_ranks)
        i32 = dict(dtype=torch.int32, device=device)
        self.workspace = new_workspace(desc, device)
        self.expert_count = torch.zeros(E, **i32)
        self.rank_count = torch.zeros(R, **i32)
        self.expert_offset = torch.zeros(E + 1, **i32)
        self.rank_psum = torch.zeros(R, **i32)
        self.dst_slot = torch.empty(max(N * K, 1), **i32)
        self.src_idx = torch.empty(max(self.capacity, 1), **i32)[: self.capacity]
        self.total_rows = torch.zeros(1, **i32)

    def count(self, topk_idx, stream=None):
        layout_count(self.desc, topk_idx, self.expert_count, self.rank_count, self.workspace, stream)

    def scan(self, topk_idx, stream=None):
        layout_scan(self.desc, topk_idx, self.expert_count, self.rank_count, self.workspace, self.expert_offset,
                    self.rank_psum, self.dst_slot, self.src_idx, self.total_rows, stream)

    def build(self, topk_idx, stream=None, fused=True):
        """The whole layout; ``fused=False`` runs the two-call path (count, then scan)."""
        if fused:
            layout_build(self.desc, topk_idx, self.expert_count, self.rank_count, self.workspace,
                         self.expert_offset, self.rank_psum, self.dst_slot, self.src_idx, self.total_rows, stream)
        else:
            self.count(topk_idx, stream)
            self.scan(topk_idx, stream)
        return self

    def permute(self, x, recv_x, sf=None, recv_sf=None, zero_pad=True, stream=None):
        dispatch_permute(self.desc, x, self.dst_slot, self.expert_offset, self.expert_count, recv_x,
                         self.workspace, sf, recv_sf, zero_pad, stream)

    def permute_sf_col_major(self, sf, recv_sf_cm, zero_pad=True, stream=None):
        """Scale factors of the expand layout, column-major into ``recv_sf_cm`` [C, ld]."""
        dispatch_sf_col_major(self.desc, sf, self.src_idx, self.total_rows, recv_sf_cm, self.capacity,
                              self.workspace, zero_pad, stream)

    def rank_rows(self, topk_idx, capacity_rows=None, stream=None):
        """Non-expand slot map after ``build``: sets ``rank_slot`` [N*K] and ``rank_src`` [capacity]."""
        N, K, R = int(self.desc.num_tokens), int(self.desc.topk), int(self.desc.num_ranks)
        cap = N * R if capacity_rows is None else int(capacity_rows)
        dev = self.dst_slot.device
        if getattr(self, "rank_src", None) is None or self.rank_src.numel() != cap:   # reuse across calls
            self.rank_slot = torch.empty(max(N * K, 1), dtype=torch.int32, device=dev)
            self.rank_src = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)[:cap]
        layout_rank_rows(self.desc, topk_idx, self.rank_count, self.workspace, self.rank_slot, self.rank_src,
                         stream)
        return self

    def permute_ranks(self, x, recv, sf=None, recv_sf=None, stream=None):
        dispatch_permute_ranks(self.desc, x, self.rank_slot, self.rank_psum, recv, self.workspace, sf, recv_sf,
                               stream)

    def permute_sf_col_major_ranks(self, sf, recv_sf_cm, stream=None):
        """Scale factors of the non-expand layout (after ``rank_rows``), column-major."""
        R = int(self.desc.num_ranks)
        dispatch_sf_col_major(self.desc, sf, self.rank_src, self.rank_psum[R - 1:], recv_sf_cm,
                              self.rank_src.numel(), self.workspace, False, stream)

    def combine(self, expert_out, weights, out, stream=None):
        combine_unpermute(self.desc, expert_out, self.dst_slot, weights, out, self.workspace, stream)

    def error(self, stream=None) -> int:
        return get_error(self.workspace, stream)


class HostPipeline:
    """Batches from host memory through dispatch, an expert step and combine
    back to host memory, with ``lanes`` batches in flight.

    Each lane owns a layout (with its workspace), device buffers and a pair
    of streams.  Batch i runs on lane i % lanes: ``dispatch_from_host``, then
    ``expert(layout, recv_x, recv_sf)`` (called on the lane's stream; it
    returns the bf16 expert outputs in receive-row order), then
    ``combine_to_host``; with ``expert=None`` the batch is a dispatch only and
    its receive rows come back to ``out_host`` instead (same shape and dtype
    as the lane's receive buffer).  Batches on different lanes are independent, so one
    batch's copy back to the host overlaps the next batch's copy in: the host
    link carries both directions at once.  ``submit`` returns an event that
    completes when the batch's result is in ``out_host``; until then the
    batch's host buffers must not be written.  The pipeline keeps a reference
    to them until then, so temporaries (``x.pin_memory()`` passed inline) are
    safe: the copies run outside torch, which would otherwise hand a freed
    page-locked block to the next allocation while a copy still reads it.  A
    lane is reused only after its previous batch, by stream order.
    """

    def __init__(self, desc, capacity_rows: int, hidden: int, x_dtype=torch.bfloat16, sf_cols: int = 0,
                 lanes: int = 2, chunk_tokens: int = 0, device="cuda"):
        if lanes < 1:
            raise ValueError("lanes must be >= 1")
        N, K = int(desc.num_tokens), int(desc.topk)
        self.desc, self.chunk_tokens, self.device = desc, int(chunk_tokens), torch.device(device)
        self._lanes = []
        for _ in range(lanes):
            lane = {
                "layout": Layout(desc, capacity_rows, device=device),
                "topk_idx": torch.empty((N, K), dtype=torch.int64, device=device),
                "x": torch.empty((N, hidden), dtype=x_dtype, device=device),
                "recv": torch.empty((int(capacity_rows), hidden), dtype=x_dtype, device=device),
                "weights": torch.empty((N, K), dtype=torch.float32, device=device),
                "sf": torch.empty((N, sf_cols), dtype=torch.float32, device=device) if sf_cols else None,
                "recv_sf": torch.empty((int(capacity_rows), sf_cols), dtype=torch.float32, device=device)
                if sf_cols else None,
                "out": None,
                "stream": torch.cuda.Stream(device),
                "copy": torch.cuda.Stream(device),
            }
            self._lanes.append(lane)
        self._next = 0
        self._in_flight = []   # (event, host tensors) of batches not known to be done

    @property
    def lanes(self) -> int:
        return len(self._lanes)

    def lane(self, i: int) -> dict:
        return self._lanes[i]

    @property
    def next_lane(self) -> int:
        """Index of the lane the next ``submit`` uses."""
        return self._next

    def submit(self, topk_idx_host, x_host, weights_host, out_host, expert, sf_host=None) -> torch.cuda.Event:
        lane = self._lanes[self._next]
        self._next = (self._next + 1) % len(self._lanes)
        s, cs, lay = lane["stream"], lane["copy"], lane["layout"]
        # The lane's stream starts after whatever the caller enqueued so far.
        s.wait_stream(torch.cuda.current_stream(self.device))
        dispatch_from_host(lay, topk_idx_host, x_host, lane["topk_idx"], lane["x"], lane["recv"],
                           weights_host=weights_host, weights=lane["weights"], sf_host=sf_host, sf=lane["sf"],
                           recv_sf=lane["recv_sf"], chunk_tokens=self.chunk_tokens, stream=s, copy_stream=cs)
        if expert is None:
            cs.wait_stream(s)
            with torch.cuda.stream(cs):
                out_host.copy_(lane["recv"], non_blocking=True)
            s.wait_stream(cs)
        else:
            with torch.cuda.stream(s):
                eo = expert(lay, lane["recv"], lane["recv_sf"])
                if lane["out"] is None or lane["out"].shape != out_host.shape:
                    lane["out"] = torch.empty(out_host.shape, dtype=torch.bfloat16, device=self.device)
            combine_to_host(lay, eo, lane["weights"], lane["out"], out_host, chunk_tokens=self.chunk_tokens,
                            stream=s, copy_stream=cs)
        done = torch.cuda.Event()
        done.record(s)
        self._in_flight = [(ev, refs) for ev, refs in self._in_flight if not ev.query()]
        self._in_flight.append((done, (topk_idx_host, x_host, weights_host, out_host, sf_host)))
        return done

    def join(self, stream=None) -> None:
        """Make ``stream`` (default: the current one) wait for every submitted batch."""
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        for lane in self._lanes:
            st.wait_stream(lane["stream"])

    def errors(self) -> list[int]:
        """Each lane's sticky device error (synchronises the lanes)."""
        return [lane["layout"].error(lane["stream"]) for lane in self._lanes]


class StepGraph:
    """One dispatch -> expert -> combine step captured once as a CUDA graph and
    replayed, for serving loops where launching the step's kernels one by one
    from the host costs as much as running them.

    The step's device tensors are fixed at capture: copy each batch into
    ``topk_idx`` [N, K], ``x`` [N, H] and ``weights`` [N, K] (owned by this
    object), call ``replay()``, and read ``recv_x`` (the receive buffer) and
    ``out`` (the combined tokens).  ``expert(layout, recv_x, None)`` is captured
    with the step and must return the bf16 expert outputs in receive-row order;
    with ``expert=None`` the step is a dispatch only.  The library's kernels go
    into the graph with their programmatic-dependent-launch edges, and the
    step is run once outside capture first so that every one-time host lookup
    (shared-memory limits, occupancies) is done before it.  ``error()`` reads
    and clears the device error word (it synchronises; call it between replays).
    """

    def __init__(self, desc, capacity_rows: int, hidden: int, expert=None, x_dtype=torch.bfloat16, device="cuda"):
        N, K = int(desc.num_tokens), int(desc.topk)
        self.device = torch.device(device)
        self.layout = Layout(desc, capacity_rows, device=self.device)
        self.topk_idx = torch.full((N, K), -1, dtype=torch.int64, device=self.device)
        self.x = torch.zeros((N, hidden), dtype=x_dtype, device=self.device)
        self.weights = torch.zeros((N, K), dtype=torch.float32, device=self.device)
        self.recv_x = torch.empty((int(capacity_rows), hidden), dtype=x_dtype, device=self.device)
        self.out = torch.empty((N, hidden), dtype=torch.bfloat16, device=self.device) if expert is not None else None
        self._expert = expert

        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self._step()
        torch.cuda.current_stream(self.device).wait_stream(side)
        torch.cuda.synchronize(self.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._step()

    def _step(self):
        self.layout.build(self.topk_idx)
        self.layout.permute(self.x, self.recv_x)
        if self._expert is not None:
            eo = self._expert(self.layout, self.recv_x, None)
            self.layout.combine(eo, self.weights, self.out)

    def replay(self) -> None:
        """Run the captured step on the current stream."""
        self.graph.replay()

    def error(self) -> int:
        return self.layout.error()


def dispatch(topk_idx, x, num_experts, num_ranks, alignment, sf=None, capacity_rows=None, stream=None):
    """Count, scan and permute in one call; returns ``(layout, recv_x, recv_sf)``.

    With ``capacity_rows`` None the receive buffers get the bound that never
    overflows (N*K + E*(A-1) rows), so no host synchronisation is needed.
    """
    N, K = topk_idx.shape
    desc = LayoutDesc(N, K, num_experts, num_ranks, alignment)
    cap = capacity_rows if capacity_rows is not None else N * K + num_experts * (alignment - 1)
    lay = Layout(desc, cap, device=topk_idx.device).build(topk_idx, stream)
    recv_x = torch.empty((cap,) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
    recv_sf = None
    if sf is not None:
        recv_sf = torch.empty((cap,) + tuple(sf.shape[1:]), dtype=sf.dtype, device=sf.device)
    lay.permute(x, recv_x, sf, recv_sf, stream=stream)
    return lay, recv_x, recv_sf
