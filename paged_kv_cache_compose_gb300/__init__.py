"""GB300-native paged-KV compose of a context-parallel prefill.

The compute path is the CUDA library ``libcpkv.so`` (C ABI in
include/cpkv.h); ``cpkv`` is its thin ctypes binding and ``runtime`` holds the
per-batch / per-layer drivers.  Importing this package does not load the
library; the first call does, and fails loudly if it has not been built.
"""
from . import cpkv  # noqa: F401
from .cpkv import (  # noqa: F401
    CpkvError,
    cpkv_compose_fused,
    cpkv_compose_fused_planes,
    cpkv_compose_gather,
    cpkv_compose_gather_kinds,
    cpkv_compose_layer,
    cpkv_compose_layer_planes,
    cpkv_fill_current,
    cpkv_fill_current_planes,
    cpkv_plan_build,
    cpkv_plan_sizes,
    cpkv_plan_workspace_bytes,
    cpkv_ragged_plan_build,
    cpkv_ragged_plan_sizes,
    cpkv_version,
    cpkv_writer_token_counts,
    plan_buffers,
    ragged_buffers,
)

__all__ = [
    "cpkv", "CpkvError", "cpkv_compose_fused", "cpkv_compose_fused_planes", "cpkv_compose_gather", "cpkv_compose_gather_kinds", "cpkv_compose_layer", "cpkv_compose_layer_planes", "cpkv_fill_current", "cpkv_fill_current_planes", "cpkv_plan_build", "cpkv_plan_sizes",
    "cpkv_plan_workspace_bytes",    "cpkv_ragged_plan_build", "cpkv_ragged_plan_sizes", "cpkv_version", "cpkv_writer_token_counts",
    "plan_buffers", "ragged_buffers",
]
