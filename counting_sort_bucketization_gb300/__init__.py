"""GB300-native MoE dispatch layout: counting sort / bucketization on one GPU.

The compute path is the C-ABI library ``libmoe_layout.so`` (declared in
``include/moe_layout.h``; sm_103a CUDA kernels in ``csrc/``).  This package
holds the thin Python binding over it (``binding``: argument marshalling
only, torch tensors in, device pointers out) and the seeded synthetic
workloads (``workloads``).

Importing the package loads nothing; the library is opened on first use of a
binding function and the call fails loudly when it is missing.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = (
    "Layout", "LayoutDesc", "LayoutError", "workspace_bytes", "new_workspace", "layout_count", "layout_scan",
    "layout_build", "layout_rank_rows", "dispatch_permute_ranks", "dispatch_from_host", "combine_to_host",
    "accumulate_stats", "dispatch_sf_col_major", "new_sf_col_major", "sf_col_major_ld",
    "dispatch_permute", "combine_unpermute", "get_error", "kernel_launches", "strerror",
    "library_path", "load_library", "dispatch", "ERROR_NAMES", "HostPipeline",
)

__all__ = list(_BINDING_NAMES) + ["workloads"]


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(__name__ + ".binding"), name)
    if name in ("workloads", "binding"):
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
