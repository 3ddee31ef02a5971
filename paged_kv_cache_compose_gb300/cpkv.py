"""Thin Python binding of ``libcpkv.so`` (the C ABI declared in include/cpkv.h).

Argument marshalling only: torch tensors become device pointers, Python
sequences become host arrays, the current torch stream becomes the CUDA
stream.  Every computation runs in the library's kernels; there is no CPU or
PyTorch fallback — if the library is missing or a call fails, a
``CpkvError`` is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpkv.so")

CPKV_OK = 0
CPKV_ERR_ARG = -1
CPKV_ERR_UNALIGNED_PREFIX = -2
CPKV_ERR_CAPACITY = -3
CPKV_ERR_LIMIT = -4
CPKV_ERR_CUDA = -5

STATUS_PAGE_OOB = 1
STATUS_WRITER_OOB = 2
STATUS_DUP_CURRENT_PAGE = 4
STATUS_CURRENT_IN_PREFIX = 8
STATUS_DESC_OOB = 16
STATUS_ROW_OOB = 32
STATUS_CHUNK_OOB = 64
STATUS_OUT_CAPACITY = 128
STATUS_TIMEOUT = 256

GATHER_POOL = 1
GATHER_STAGING = 2
GATHER_ZERO = 4
GATHER_ALL = 7
GATHER_CONSUME_STAGING = 8  # flag: staging bytes are undefined after the gather (L2 lines dropped)
GATHER_EARLY_INPUTS = 16  # flag: launched early behind the fill (its contract is the caller's)
FLAG_CONSUME_STAGING = 1    # layer compose: the stagings are consumed
FLAG_EARLY_INPUTS = 2       # layer / fused compose: inputs complete before the previous kernel started
FILL_PAGE_RUNS = 4          # fill: the index arrays are a plan of cpkv_plan_build (pages move as runs)


def compose_flags(consume_staging=False, early_inputs=False) -> int:
    return (FLAG_CONSUME_STAGING if consume_staging else 0) | (FLAG_EARLY_INPUTS if early_inputs else 0)

MAX_CP = 64
MAX_BATCH = 1024

EXPORTED = (
    "cpkv_plan_sizes", "cpkv_writer_token_counts", "cpkv_plan_build", "cpkv_plan_workspace_bytes",
    "cpkv_plan_build_noalloc",
    "cpkv_fill_current",
    "cpkv_fill_current_planes",
    "cpkv_compose_gather", "cpkv_compose_gather_kinds", "cpkv_compose_layer", "cpkv_compose_layer_planes",
    "cpkv_compose_fused", "cpkv_compose_fused_planes", "cpkv_selftest_ring_timeout", "cpkv_ragged_plan_sizes",
    "cpkv_ragged_plan_build", "cpkv_error_string", "cpkv_version",
)


class CpkvError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str = ""):
        super().__init__(f"{fn} failed: {msg or code}")
        self.code = code


class _Sizes(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("C", ctypes.c_int64), ("D", ctypes.c_int64)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_lib = None


def _declare(lib):
    lib.cpkv_plan_sizes.argtypes = [_I, _I, _P, _P, ctypes.POINTER(_Sizes)]
    lib.cpkv_writer_token_counts.argtypes = [_I, _I, _I, _P, _P, _L, _P]
    lib.cpkv_plan_build.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _P, _L] + [_P] * 10 + [_L, _P, _P]
    lib.cpkv_plan_workspace_bytes.argtypes = [_I, _I, _I, _P, _P]
    lib.cpkv_plan_build_noalloc.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _P, _L] + [_P] * 11
    lib.cpkv_fill_current.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _L, _P, _P, _P, _L, _I, _P, _P]
    lib.cpkv_compose_gather.argtypes = [_I, _I, _L, _P, _P, _P, _P, _L, _P, _P, _P]
    lib.cpkv_fill_current_planes.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _L, _P, _P, _P, _L, _I, _P, _P]
    lib.cpkv_compose_gather_kinds.argtypes = [_I, _I, _L, _P, _P, _P, _P, _L, _I, _P, _P, _P]
    lib.cpkv_compose_layer.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _P, _P, _P, _P, _L, _P, _I, _P, _P]
    lib.cpkv_compose_layer_planes.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _L, _P, _I, _P,
                                              _P]
    lib.cpkv_compose_fused.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _P, _P, _P, _P, _L, _P, _I, _P, _P]
    lib.cpkv_selftest_ring_timeout.argtypes = [_P, _P, _P]
    lib.cpkv_compose_fused_planes.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _L, _P, _I, _P,
                                              _P]
    lib.cpkv_ragged_plan_sizes.argtypes = [_I, _I, _P, _P, _L, _P, _P]
    lib.cpkv_ragged_plan_build.argtypes = [_I, _I, _I, _I, _P, _P, _P, _L, _P, _L] + [_P] * 7 + [_L, _P, _P, _P]
    for name in EXPORTED:
        getattr(lib, name).restype = _I
    lib.cpkv_error_string.argtypes = [_I]
    lib.cpkv_error_string.restype = ctypes.c_char_p
    lib.cpkv_version.argtypes = []
    return lib


def load(path: str = LIB_PATH):
    """Load the CUDA library (built by ``paged_kv_cache_compose_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise CpkvError("load", -100, f"{path} is missing: build the CUDA library first "
                                          "(python -m paged_kv_cache_compose_gb300.build)")
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def _check(fn: str, rc: int):
    if rc != CPKV_OK:
        raise CpkvError(fn, rc, load().cpkv_error_string(rc).decode())


def _host_i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _host_i64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _hp(a: np.ndarray):
    return _P(a.ctypes.data) if a.size else None


def _dp(t):
    """Device pointer of a torch tensor (None for None/empty)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise CpkvError("marshal", CPKV_ERR_ARG, "expected a CUDA tensor")
    if not t.is_contiguous():
        raise CpkvError("marshal", CPKV_ERR_ARG, "expected a contiguous tensor")
    return _P(t.data_ptr()) if t.numel() else None


def _ptr_array(ptrs: Sequence) -> ctypes.Array:
    vals = []
    for p in ptrs:
        if p is None:
            vals.append(None)
        elif isinstance(p, int):
            vals.append(p)
        else:
            vals.append(p.data_ptr() if p.numel() else None)
    return (ctypes.c_void_p * len(vals))(*vals)


def _stream(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return _P(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ---------------------------------------------------------------------------
# host-only entry points
# ---------------------------------------------------------------------------

def cpkv_plan_sizes(prefix_lens, cur_lens, page_size: int):
    """(T, C, D) of a batch."""
    pl, cl = _host_i32(prefix_lens), _host_i32(cur_lens)
    out = _Sizes()
    _check("cpkv_plan_sizes", load().cpkv_plan_sizes(len(pl), page_size, _hp(pl), _hp(cl), ctypes.byref(out)))
    return out.T, out.C, out.D


def cpkv_writer_token_counts(cur_lens, writer, page_size: int, cp_size: int) -> np.ndarray:
    cl, wr = _host_i32(cur_lens), _host_i32(writer)
    out = np.zeros(cp_size, np.int64)
    _check("cpkv_writer_token_counts",
           load().cpkv_writer_token_counts(len(cl), page_size, cp_size, _hp(cl), _hp(wr), len(wr), _hp(out)))
    return out


def cpkv_ragged_plan_sizes(q_lens, cp_index, chunk: int):
    ql, ci = _host_i32(q_lens), _host_i32(cp_index)
    S, Q = ctypes.c_int64(), ctypes.c_int64()
    _check("cpkv_ragged_plan_sizes", load().cpkv_ragged_plan_sizes(len(ql), chunk, _hp(ql), _hp(ci), len(ci),
                                                                   ctypes.byref(S), ctypes.byref(Q)))
    return S.value, Q.value


# ---------------------------------------------------------------------------
# device entry points (stream-ordered, asynchronous)
# ---------------------------------------------------------------------------

def cpkv_plan_workspace_bytes(cur_lens, page_size: int, cp_size: int) -> int:
    """Device workspace bytes that ``cpkv_plan_build`` needs for this batch."""
    cl = _host_i32(cur_lens)
    out = ctypes.c_int64(0)
    _check("cpkv_plan_workspace_bytes",
           load().cpkv_plan_workspace_bytes(len(cl), page_size, cp_size, _hp(cl), ctypes.byref(out)))
    return int(out.value)


def cpkv_plan_build(prefix_lens, cur_lens, d_prefix_pages, d_cur_pages, d_writer, *, page_size, cp_size,
                    num_pool_pages, dense_cap_pages, out, d_status, stream=None):
    """Build the compose plan into the tensors of ``out`` (see ``plan_buffers``;
    ``out["workspace"]`` is the call's device workspace)."""
    pl, cl = _host_i32(prefix_lens), _host_i32(cur_lens)
    ws = out["workspace"]
    rc = load().cpkv_plan_build(
        len(pl), page_size, cp_size, num_pool_pages, _hp(pl), _hp(cl), _dp(d_prefix_pages), _dp(d_cur_pages),
        _dp(d_writer), dense_cap_pages, _dp(out["prefix_spans"]), _dp(out["cur_spans"]), _dp(out["owner"]),
        _dp(out["src"]), _dp(out["page_inverse"]), _dp(out["staging_page_inverse"]), _dp(out["mixed_locs"]),
        _dp(out["staging_rows"]), _dp(out["token_writer_row"]), _dp(ws), ws.numel() * ws.element_size(),
        _dp(d_status), _stream(stream))
    _check("cpkv_plan_build", rc)


def cpkv_plan_build_noalloc(prefix_lens, cur_lens, d_prefix_pages, d_cur_pages, d_writer, *, page_size, cp_size,
                            num_pool_pages, dense_cap_pages, out, d_status, stream=None):
    """``cpkv_plan_build`` without a caller workspace: the library's fixed
    device array serves instead (for callers that cannot allocate; see
    include/cpkv.h for its size limit and sharing rules).  ``out`` as for
    ``cpkv_plan_build``; its "workspace" entry, if any, is not used."""
    pl, cl = _host_i32(prefix_lens), _host_i32(cur_lens)
    rc = load().cpkv_plan_build_noalloc(
        len(pl), page_size, cp_size, num_pool_pages, _hp(pl), _hp(cl), _dp(d_prefix_pages), _dp(d_cur_pages),
        _dp(d_writer), dense_cap_pages, _dp(out["prefix_spans"]), _dp(out["cur_spans"]), _dp(out["owner"]),
        _dp(out["src"]), _dp(out["page_inverse"]), _dp(out["staging_page_inverse"]), _dp(out["mixed_locs"]),
        _dp(out["staging_rows"]), _dp(out["token_writer_row"]), _dp(d_status), _stream(stream))
    _check("cpkv_plan_build_noalloc", rc)


def cpkv_fill_current(cur_lens, cur_rows: Sequence, staging: Sequence, *, page_size, cp_size, row_bytes,
                      staging_cap_pages, d_staging_rows, d_token_writer_row, d_writer, num_cur_pages,
                      d_status, cur_rows_cap=None, early_inputs=False, page_runs=False, stream=None):
    """Per-layer fill.  ``cur_rows[w]`` / ``staging[w]``: uint8 CUDA tensors (or raw pointers with
    ``cur_rows_cap`` given).  ``early_inputs``: FLAG_EARLY_INPUTS; ``page_runs``: FILL_PAGE_RUNS (the
    index arrays are a plan of cpkv_plan_build for this batch); both contracts are the caller's."""
    cl = _host_i32(cur_lens)
    if cur_rows_cap is None:
        cur_rows_cap = [t.numel() // row_bytes for t in cur_rows]
    caps = _host_i64(cur_rows_cap)
    rows_arr = _ptr_array(cur_rows)
    stg_arr = _ptr_array(staging)
    rc = load().cpkv_fill_current(
        len(cl), page_size, cp_size, row_bytes, _hp(cl), ctypes.cast(rows_arr, _P), _hp(caps),
        ctypes.cast(stg_arr, _P), staging_cap_pages, _dp(d_staging_rows), _dp(d_token_writer_row),
        _dp(d_writer), num_cur_pages, compose_flags(early_inputs=early_inputs) | (FILL_PAGE_RUNS if page_runs else 0),
        _dp(d_status), _stream(stream))
    _check("cpkv_fill_current", rc)


def cpkv_fill_current_planes(cur_lens, cur_planes: Sequence, staging: Sequence, *, page_size, cp_size, plane_bytes,
                             staging_cap_pages, d_staging_rows, d_token_writer_row, d_writer, num_cur_pages,
                             d_status, cur_rows_cap=None, early_inputs=False, page_runs=False, stream=None):
    """Planar-page fill.  ``cur_planes[p][w]``: writer w's rows of plane p (uint8 CUDA tensors).
    ``early_inputs``: FLAG_EARLY_INPUTS; ``page_runs``: FILL_PAGE_RUNS; both contracts are the caller's."""
    cl, pb = _host_i32(cur_lens), _host_i32(plane_bytes)
    n_planes = len(pb)
    if cur_rows_cap is None:
        cur_rows_cap = [cur_planes[0][w].numel() // int(pb[0]) for w in range(cp_size)]
    caps = _host_i64(cur_rows_cap)
    flat = _ptr_array([cur_planes[p][w] for p in range(n_planes) for w in range(cp_size)])
    stg = _ptr_array(staging)
    rc = load().cpkv_fill_current_planes(len(cl), page_size, cp_size, n_planes, _hp(pb), _hp(cl),
                                         ctypes.cast(flat, _P), _hp(caps), ctypes.cast(stg, _P), staging_cap_pages,
                                         _dp(d_staging_rows), _dp(d_token_writer_row), _dp(d_writer), num_cur_pages,
                                         compose_flags(early_inputs=early_inputs) | (FILL_PAGE_RUNS if page_runs else 0), _dp(d_status), _stream(stream))
    _check("cpkv_fill_current_planes", rc)


def cpkv_compose_gather(src_table: Sequence, src_cap_pages, d_owner, d_src, d_dense, *, page_size, cp_size,
                        row_bytes, dense_cap_pages, d_status, stream=None):
    """Slot-dense page gather over the 2*cp table [pools | stagings]."""
    caps = _host_i64(src_cap_pages)
    tbl = _ptr_array(src_table)
    rc = load().cpkv_compose_gather(page_size, cp_size, row_bytes, ctypes.cast(tbl, _P), _hp(caps),
                                    _dp(d_owner), _dp(d_src), dense_cap_pages, _dp(d_dense), _dp(d_status),
                                    _stream(stream))
    _check("cpkv_compose_gather", rc)


def cpkv_compose_gather_kinds(src_table: Sequence, src_cap_pages, d_owner, d_src, d_dense, *, page_size, cp_size,
                              row_bytes, dense_cap_pages, kinds, d_status, stream=None):
    """The gather restricted to slot kinds (GATHER_POOL | GATHER_STAGING | GATHER_ZERO)."""
    caps = _host_i64(src_cap_pages)
    tbl = _ptr_array(src_table)
    rc = load().cpkv_compose_gather_kinds(page_size, cp_size, row_bytes, ctypes.cast(tbl, _P), _hp(caps),
                                          _dp(d_owner), _dp(d_src), dense_cap_pages, kinds, _dp(d_dense),
                                          _dp(d_status), _stream(stream))
    _check("cpkv_compose_gather_kinds", rc)


def cpkv_compose_layer(cur_lens, cur_rows: Sequence, src_table: Sequence, src_cap_pages, d_owner, d_src,
                       d_token_writer_row, d_dense, *, page_size, cp_size, row_bytes, dense_cap_pages, d_status,
                       cur_rows_cap=None, consume_staging=False, early_inputs=False, stream=None):
    """Fill + slot-dense gather of one layer in a single launch (``consume_staging``:
    the staging bytes are undefined afterwards; ``early_inputs``: see
    CPKV_FLAG_EARLY_INPUTS)."""
    cl = _host_i32(cur_lens)
    if cur_rows_cap is None:
        cur_rows_cap = [t.numel() // row_bytes for t in cur_rows]
    rcaps, tcaps = _host_i64(cur_rows_cap), _host_i64(src_cap_pages)
    rarr, tarr = _ptr_array(cur_rows), _ptr_array(src_table)
    rc = load().cpkv_compose_layer(len(cl), page_size, cp_size, row_bytes, _hp(cl), ctypes.cast(rarr, _P), _hp(rcaps),
                                   ctypes.cast(tarr, _P), _hp(tcaps), _dp(d_owner), _dp(d_src),
                                   _dp(d_token_writer_row), dense_cap_pages, _dp(d_dense),
                                   compose_flags(consume_staging, early_inputs), _dp(d_status), _stream(stream))
    _check("cpkv_compose_layer", rc)


def cpkv_compose_layer_planes(cur_lens, cur_planes: Sequence, src_table: Sequence, src_cap_pages, d_owner, d_src,
                              d_token_writer_row, d_dense, *, page_size, cp_size, plane_bytes, dense_cap_pages,
                              d_status, cur_rows_cap=None, consume_staging=False, early_inputs=False, stream=None):
    """Fill + gather of one layer of planar pages in a single launch
    (``cur_planes[p][w]``: writer w's rows of plane p)."""
    cl, pb = _host_i32(cur_lens), _host_i32(plane_bytes)
    n_planes = len(pb)
    if cur_rows_cap is None:
        cur_rows_cap = [cur_planes[0][w].numel() // int(pb[0]) for w in range(cp_size)]
    rcaps, tcaps = _host_i64(cur_rows_cap), _host_i64(src_cap_pages)
    flat = _ptr_array([cur_planes[p][w] for p in range(n_planes) for w in range(cp_size)])
    tarr = _ptr_array(src_table)
    rc = load().cpkv_compose_layer_planes(len(cl), page_size, cp_size, n_planes, _hp(pb), _hp(cl),
                                          ctypes.cast(flat, _P), _hp(rcaps), ctypes.cast(tarr, _P), _hp(tcaps),
                                          _dp(d_owner), _dp(d_src), _dp(d_token_writer_row), dense_cap_pages,
                                          _dp(d_dense), compose_flags(consume_staging, early_inputs), _dp(d_status),
                                          _stream(stream))
    _check("cpkv_compose_layer_planes", rc)


def cpkv_compose_fused(cur_lens, pools: Sequence, cur_rows: Sequence, d_owner, d_src, d_token_writer_row, d_dense,
                       *, page_size, cp_size, row_bytes, dense_cap_pages, d_status, pool_cap_pages=None,
                       cur_rows_cap=None, early_inputs=False, stream=None):
    """Single-GPU compose of one layer without staging (pools + writers' current rows -> dense)."""
    cl = _host_i32(cur_lens)
    if pool_cap_pages is None:
        pool_cap_pages = [t.shape[0] for t in pools]
    if cur_rows_cap is None:
        cur_rows_cap = [t.numel() // row_bytes for t in cur_rows]
    pcaps, rcaps = _host_i64(pool_cap_pages), _host_i64(cur_rows_cap)
    parr, rarr = _ptr_array(pools), _ptr_array(cur_rows)
    rc = load().cpkv_compose_fused(len(cl), page_size, cp_size, row_bytes, _hp(cl), ctypes.cast(parr, _P), _hp(pcaps),
                                   ctypes.cast(rarr, _P), _hp(rcaps), _dp(d_owner), _dp(d_src),
                                   _dp(d_token_writer_row), dense_cap_pages, _dp(d_dense),
                                   compose_flags(early_inputs=early_inputs), _dp(d_status),
                                   _stream(stream))
    _check("cpkv_compose_fused", rc)


def cpkv_compose_fused_planes(cur_lens, pools: Sequence, cur_planes: Sequence, d_owner, d_src, d_token_writer_row,
                              d_dense, *, page_size, cp_size, plane_bytes, dense_cap_pages, d_status,
                              pool_cap_pages=None, cur_rows_cap=None, early_inputs=False, stream=None):
    """Single-GPU compose of one layer of planar pages without staging
    (``cur_planes[p][w]``: writer w's rows of plane p)."""
    cl, pb = _host_i32(cur_lens), _host_i32(plane_bytes)
    n_planes = len(pb)
    if pool_cap_pages is None:
        pool_cap_pages = [t.shape[0] for t in pools]
    if cur_rows_cap is None:
        cur_rows_cap = [cur_planes[0][w].numel() // int(pb[0]) for w in range(cp_size)]
    pcaps, rcaps = _host_i64(pool_cap_pages), _host_i64(cur_rows_cap)
    parr = _ptr_array(pools)
    flat = _ptr_array([cur_planes[p][w] for p in range(n_planes) for w in range(cp_size)])
    rc = load().cpkv_compose_fused_planes(len(cl), page_size, cp_size, n_planes, _hp(pb), _hp(cl),
                                          ctypes.cast(parr, _P), _hp(pcaps), ctypes.cast(flat, _P), _hp(rcaps),
                                          _dp(d_owner), _dp(d_src), _dp(d_token_writer_row), dense_cap_pages,
                                          _dp(d_dense), compose_flags(early_inputs=early_inputs), _dp(d_status),
                                          _stream(stream))
    _check("cpkv_compose_fused_planes", rc)


def cpkv_selftest_ring_timeout(d_dst16, d_status, stream=None):
    """Diagnostics: the bulk ring's bounded wait on a load that never arrives
    (raises STATUS_TIMEOUT on the device, writes nothing to ``d_dst16``)."""
    _check("cpkv_selftest_ring_timeout",
           load().cpkv_selftest_ring_timeout(_dp(d_dst16), _dp(d_status), _stream(stream)))


def cpkv_ragged_plan_build(prefix_lens, q_lens, d_cp_index, n_owned: int, *, chunk, k_align, topk, out, d_counts,
                           d_status, stream=None):
    """Ragged index plan of one rank into the tensors of ``out`` (see ``ragged_buffers``);
    ``topk``: the indexer's keys per query (validated > 0)."""
    pl, ql = _host_i32(prefix_lens), _host_i32(q_lens)
    rc = load().cpkv_ragged_plan_build(
        len(pl), chunk, k_align, topk, _hp(pl), _hp(ql), _dp(d_cp_index), n_owned, _dp(out["topk_offsets"]),
        out["topk_offsets"].numel(), _dp(out["seg_req"]), _dp(out["kv_lens"]), _dp(out["q_starts"]),
        _dp(out["q_lens"]), _dp(out["k_bases"]), _dp(out["q_bases"]), _dp(out["current_bases"]),
        out["seg_req"].numel(), _dp(d_counts), _dp(d_status), _stream(stream))
    _check("cpkv_ragged_plan_build", rc)


def cpkv_version() -> int:
    return load().cpkv_version()


# ---------------------------------------------------------------------------
# allocation helpers (torch device memory; no computation)
# ---------------------------------------------------------------------------

def plan_buffers(B: int, T: int, dense_cap_pages: int, num_pool_pages: int, device="cuda",
                 workspace_bytes: int = 0) -> dict:
    import torch

    i32, i64 = torch.int32, torch.int64
    return {
        "workspace": torch.empty(-(-workspace_bytes // 4), dtype=i32, device=device),
        "prefix_spans": torch.empty((B, 2), dtype=i32, device=device),
        "cur_spans": torch.empty((B, 2), dtype=i32, device=device),
        "owner": torch.empty(dense_cap_pages, dtype=i32, device=device),
        "src": torch.empty(dense_cap_pages, dtype=i32, device=device),
        "page_inverse": torch.empty(num_pool_pages, dtype=i32, device=device),
        "staging_page_inverse": torch.empty(num_pool_pages, dtype=i32, device=device),
        "mixed_locs": torch.empty(T, dtype=i64, device=device),
        "staging_rows": torch.empty(T, dtype=i64, device=device),
        "token_writer_row": torch.empty(T, dtype=i32, device=device),
    }


def ragged_buffers(seg_cap: int, topk_cap: int, device="cuda") -> dict:
    import torch

    out = {k: torch.empty(seg_cap, dtype=torch.int32, device=device)
           for k in ("seg_req", "kv_lens", "q_starts", "q_lens", "k_bases", "q_bases", "current_bases")}
    out["topk_offsets"] = torch.empty(topk_cap, dtype=torch.int32, device=device)
    return out
