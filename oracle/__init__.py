"""CPU oracle of the paged-KV compose (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does, and this package imports nothing from it.

The arithmetic lives in ``cpkv_oracle.c`` (plain C, one walk over requests,
``memcpy``/``memset`` per row).  This module compiles it with gcc, loads it
with ctypes and offers numpy-shaped wrappers.  See the C file's header for the
passages of the pages each function follows and the readings taken where the
pages are silent.

Parity status of each function (what pins it, see tests/test_oracle_pins.py):
  oracle_compose_plan   pinned: brute-force inversion, loc identities, writer
                        counting, hand-worked golden example
  oracle_compose_dense  pinned: token-level logical-loc formulation, cp=1
                        reduction to index_select + cat, golden example
  oracle_staging        pinned: golden example, round trip through the gather
  oracle_gather         pinned: per-slot brute force, -1 sentinel, golden
  oracle_fill_index_copy pinned: equals oracle_staging on plan-built indices;
                        a hand-worked permuted case
  oracle_fill_planes, oracle_compose_dense_planes
                        pinned: one plane equals the row functions; a
                        hand-worked two-plane page; plane-by-plane reduction
                        to the row definition
  oracle_ragged_plan    pinned: cumsum / repeat closed forms, tiling of every
                        request across ranks, cp=1 special case, golden
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcpkv_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_ARG = -1
UNALIGNED_PREFIX = -2
CAPACITY = -3

PAGE_OOB = 1
WRITER_OOB = 2
DUP_CURRENT_PAGE = 4
CURRENT_IN_PREFIX = 8
DESC_OOB = 16
ROW_OOB = 32
CHUNK_OOB = 64


class OracleError(RuntimeError):
    pass


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C file into a shared library (gcc -O2)."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", *extra_flags, "-o", out, src]
    subprocess.run(cmd, check=True)
    return out


def _foreign_elf(path: str) -> bool:
    """True when ``path`` is a shared object built for another CPU than this
    host's (ELF e_machine: 62 x86-64, 183 AArch64)."""
    import platform

    want = {"x86_64": 62, "aarch64": 183}.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return True
    return want is not None and (head[:4] != b"\x7fELF" or int.from_bytes(head[18:20], "little") != want)


def build() -> str:
    with _lock:
        if (not os.path.exists(_LIB_PATH)) or _foreign_elf(_LIB_PATH) or \
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            compile_oracle(out=tmp)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64


def _declare(lib):
    lib.oracle_sizes.argtypes = [_I, _I, _P, _P, _P, _P, _P]
    lib.oracle_compose_plan.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _P, _L] + [_P] * 10
    lib.oracle_compose_dense.argtypes = [_I, _I, _I, _L, _L, _P, _P, _P, _P, _P, _L, _P]
    lib.oracle_staging.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _L]
    lib.oracle_gather.argtypes = [_I, _I, _L, _P, _P, _P, _P, _L, _P, _P]
    lib.oracle_fill_index_copy.argtypes = [_I, _I, _I, _L, _P, _P, _P, _P, _L, _P, _P, _P, _L, _P]
    lib.oracle_ragged_plan.argtypes = [_I, _I, _I, _P, _P, _P, _L] + [_P] * 11
    lib.oracle_fill_planes.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _L, _P, _P, _P, _L, _P]
    lib.oracle_compose_dense_planes.argtypes = [_I, _I, _I, _I, _P, _L, _P, _P, _P, _P, _P, _L, _P]
    for f in ("oracle_sizes", "oracle_compose_plan", "oracle_compose_dense",
              "oracle_staging", "oracle_gather", "oracle_ragged_plan", "oracle_fill_index_copy",
              "oracle_fill_planes", "oracle_compose_dense_planes"):
        getattr(lib, f).restype = _I
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first if needed).  ``path`` loads
    another build of the same source (used by the planted-mistake tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what} returned {rc}")


def sizes(prefix_lens, cur_lens, page_size, lib=None):
    lib = lib or load()
    pl, cl = _i32(prefix_lens), _i32(cur_lens)
    out = np.zeros(3, dtype=np.int64)
    rc = lib.oracle_sizes(len(pl), page_size, _ptr(pl), _ptr(cl),
                          _P(out.ctypes.data), _P(out.ctypes.data + 8), _P(out.ctypes.data + 16))
    _check(rc, "oracle_sizes")
    return int(out[0]), int(out[1]), int(out[2])


def compose_plan(prefix_lens, cur_lens, prefix_pages, cur_pages, writer, *, page_size, cp_size,
                 num_pool_pages, dense_cap=None, lib=None) -> dict:
    """Plan arrays of one batch (see ``oracle_compose_plan`` in the C file)."""
    lib = lib or load()
    pl, cl = _i32(prefix_lens), _i32(cur_lens)
    pp, cpg, wr = _i32(prefix_pages), _i32(cur_pages), _i32(writer)
    B = len(pl)
    T, C, D = sizes(pl, cl, page_size, lib)
    cap = D if dense_cap is None else int(dense_cap)
    out = {
        "prefix_spans": np.zeros((B, 2), np.int32),
        "cur_spans": np.zeros((B, 2), np.int32),
        "owner": np.zeros(max(cap, 1), np.int32)[:cap],
        "src": np.zeros(max(cap, 1), np.int32)[:cap],
        "page_inverse": np.zeros(num_pool_pages, np.int32),
        "staging_page_inverse": np.zeros(num_pool_pages, np.int32),
        "mixed_locs": np.zeros(max(T, 1), np.int64)[:T],
        "staging_rows": np.zeros(max(T, 1), np.int64)[:T],
        "token_writer_row": np.zeros(max(T, 1), np.int32)[:T],
    }
    status = np.zeros(1, np.int32)
    rc = lib.oracle_compose_plan(
        B, page_size, cp_size, num_pool_pages, _ptr(pl), _ptr(cl), _ptr(pp), _ptr(cpg), _ptr(wr), cap,
        *[_ptr(out[k]) for k in ("prefix_spans", "cur_spans", "owner", "src", "page_inverse",
                                 "staging_page_inverse", "mixed_locs", "staging_rows",
                                 "token_writer_row")],
        _ptr(status))
    _check(rc, "oracle_compose_plan")
    out["status"] = int(status[0])
    out["T"], out["C"], out["D"] = T, C, D
    return out


def compose_dense(prefix_lens, cur_lens, prefix_pages, pool_slabs, cur_rows, *, page_size, cp_size,
                  dense_cap=None, lib=None) -> np.ndarray:
    """Dense KV [dense_cap * ps, R] by the plain definition (prefix || current || 0)."""
    lib = lib or load()
    pl, cl, pp = _i32(prefix_lens), _i32(cur_lens), _i32(prefix_pages)
    slabs = [np.ascontiguousarray(s, dtype=np.uint8) for s in pool_slabs]
    assert len(slabs) == cp_size
    slab_pages = slabs[0].shape[0]
    R = slabs[0].shape[-1]
    rows = np.ascontiguousarray(cur_rows, dtype=np.uint8)
    T, C, D = sizes(pl, cl, page_size, lib)
    cap = D if dense_cap is None else int(dense_cap)
    table = (ctypes.c_void_p * cp_size)(*[s.ctypes.data for s in slabs])
    dense = np.empty((cap * page_size, R), np.uint8)
    rc = lib.oracle_compose_dense(len(pl), page_size, cp_size, R, slab_pages, _ptr(pl), _ptr(cl),
                                  _ptr(pp), ctypes.cast(table, ctypes.c_void_p),
                                  _ptr(rows) if rows.size else None, cap, _ptr(dense))
    _check(rc, "oracle_compose_dense")
    return dense


def staging(cur_lens, writer, cur_rows, staging_bufs, *, page_size, cp_size, lib=None):
    """Write the defined pages of each writer's staging (in place)."""
    lib = lib or load()
    cl, wr = _i32(cur_lens), _i32(writer)
    rows = np.ascontiguousarray(cur_rows, dtype=np.uint8)
    R = rows.shape[-1] if rows.ndim == 2 else staging_bufs[0].shape[-1]
    for s in staging_bufs:
        assert s.flags.c_contiguous and s.dtype == np.uint8
    cap_pages = staging_bufs[0].shape[0] // page_size
    table = (ctypes.c_void_p * cp_size)(*[s.ctypes.data for s in staging_bufs])
    rc = lib.oracle_staging(len(cl), page_size, cp_size, R, _ptr(cl), _ptr(wr),
                            _ptr(rows) if rows.size else None,
                            ctypes.cast(table, ctypes.c_void_p), cap_pages)
    _check(rc, "oracle_staging")


def fill_index_copy(cur_lens, staging_rows, token_writer_row, writer, cur_rows_per_writer, staging_bufs, *,
                    page_size, cp_size, row_bytes, lib=None) -> int:
    """The fill as an index copy for arbitrary row indices (in place on
    ``staging_bufs``).  Returns the status bits."""
    lib = lib or load()
    cl, wr = _i32(cur_lens), _i32(writer)
    sr = np.ascontiguousarray(np.asarray(staging_rows, dtype=np.int64))
    tw = _i32(token_writer_row)
    rows = [np.ascontiguousarray(r, dtype=np.uint8) for r in cur_rows_per_writer]
    caps = np.array([r.shape[0] if r.ndim == 2 else 0 for r in rows], np.int64)
    for st in staging_bufs:
        assert st.flags.c_contiguous and st.dtype == np.uint8
    cap_pages = staging_bufs[0].shape[0] // page_size
    rt = (ctypes.c_void_p * cp_size)(*[r.ctypes.data if r.size else None for r in rows])
    stt = (ctypes.c_void_p * cp_size)(*[st.ctypes.data for st in staging_bufs])
    status = np.zeros(1, np.int32)
    rc = lib.oracle_fill_index_copy(len(cl), page_size, cp_size, row_bytes, _ptr(cl), _ptr(sr), _ptr(tw), _ptr(wr),
                                    len(wr), ctypes.cast(rt, ctypes.c_void_p), _ptr(caps),
                                    ctypes.cast(stt, ctypes.c_void_p), cap_pages, _ptr(status))
    _check(rc, "oracle_fill_index_copy")
    return int(status[0])


def fill_planes(cur_lens, staging_rows, token_writer_row, writer, cur_planes, staging_bufs, *, page_size, cp_size,
                plane_bytes, lib=None) -> int:
    """Planar fill as an index copy (in place on ``staging_bufs``, each
    [staging_cap_pages, page_bytes] uint8).  ``cur_planes[p][w]`` is writer
    w's plane-p rows [rows_w, plane_bytes[p]].  Returns the status bits."""
    lib = lib or load()
    cl, wr, pb = _i32(cur_lens), _i32(writer), _i32(plane_bytes)
    sr = np.ascontiguousarray(np.asarray(staging_rows, dtype=np.int64))
    tw = _i32(token_writer_row)
    n_planes = len(pb)
    flat = [np.ascontiguousarray(cur_planes[p][w], dtype=np.uint8) for p in range(n_planes) for w in range(cp_size)]
    caps = np.array([flat[w].shape[0] for w in range(cp_size)], np.int64)
    pt = (ctypes.c_void_p * len(flat))(*[a.ctypes.data if a.size else None for a in flat])
    stt = (ctypes.c_void_p * cp_size)(*[s.ctypes.data for s in staging_bufs])
    cap_pages = staging_bufs[0].shape[0]
    status = np.zeros(1, np.int32)
    rc = lib.oracle_fill_planes(len(cl), page_size, cp_size, n_planes, _ptr(pb), _ptr(cl), _ptr(sr), _ptr(tw),
                                _ptr(wr), len(wr), ctypes.cast(pt, ctypes.c_void_p), _ptr(caps),
                                ctypes.cast(stt, ctypes.c_void_p), cap_pages, _ptr(status))
    _check(rc, "oracle_fill_planes")
    return int(status[0])


def compose_dense_planes(prefix_lens, cur_lens, prefix_pages, pool_slabs, cur_planes, *, page_size, cp_size,
                         plane_bytes, dense_cap=None, lib=None) -> np.ndarray:
    """Dense planar KV [dense_cap, page_bytes] by the plain definition.
    ``pool_slabs[r]``: [slab_pages, page_bytes]; ``cur_planes[p]``: [T, plane_bytes[p]] batch order."""
    lib = lib or load()
    pl, cl, pp, pb = _i32(prefix_lens), _i32(cur_lens), _i32(prefix_pages), _i32(plane_bytes)
    slabs = [np.ascontiguousarray(s, dtype=np.uint8) for s in pool_slabs]
    planes = [np.ascontiguousarray(c, dtype=np.uint8) for c in cur_planes]
    page_bytes = int(page_size * pb.sum())
    T, C, D = sizes(pl, cl, page_size, lib)
    cap = D if dense_cap is None else int(dense_cap)
    st = (ctypes.c_void_p * cp_size)(*[s.ctypes.data for s in slabs])
    ct = (ctypes.c_void_p * len(planes))(*[c.ctypes.data if c.size else None for c in planes])
    dense = np.empty((cap, page_bytes), np.uint8)
    rc = lib.oracle_compose_dense_planes(len(pl), page_size, cp_size, len(pb), _ptr(pb), slabs[0].shape[0], _ptr(pl),
                                         _ptr(cl), _ptr(pp), ctypes.cast(st, ctypes.c_void_p),
                                         ctypes.cast(ct, ctypes.c_void_p), cap, _ptr(dense))
    _check(rc, "oracle_compose_dense_planes")
    return dense


def gather(table_bufs, cap_pages, owner, src, *, page_size, row_bytes, dense_cap, lib=None):
    """Slot-dense page gather, descriptor by descriptor.  Returns (dense, status)."""
    lib = lib or load()
    bufs = [np.ascontiguousarray(b, dtype=np.uint8) for b in table_bufs]
    ow, sr = _i32(owner), _i32(src)
    caps = np.ascontiguousarray(np.asarray(cap_pages, dtype=np.int64))
    table = (ctypes.c_void_p * len(bufs))(*[b.ctypes.data for b in bufs])
    dense = np.empty((dense_cap * page_size, row_bytes), np.uint8)
    status = np.zeros(1, np.int32)
    rc = lib.oracle_gather(page_size, len(bufs), row_bytes, ctypes.cast(table, ctypes.c_void_p),
                           _ptr(caps), _ptr(ow), _ptr(sr), dense_cap, _ptr(dense), _ptr(status))
    _check(rc, "oracle_gather")
    return dense, int(status[0])


def ragged_plan(prefix_lens, q_lens, cp_index, *, chunk, k_align=1, lib=None) -> dict:
    """Ragged index plan of one rank (see ``oracle_ragged_plan``)."""
    lib = lib or load()
    pl, ql, ci = _i32(prefix_lens), _i32(q_lens), _i32(cp_index)
    n = len(ci)
    segs = {k: np.zeros(max(n, 1), np.int32) for k in
            ("seg_req", "kv_lens", "q_starts", "q_lens", "k_bases", "q_bases", "current_bases")}
    topk = np.zeros(max(n * chunk, 1), np.int32)
    S = np.zeros(1, np.int64)
    Q = np.zeros(1, np.int64)
    status = np.zeros(1, np.int32)
    rc = lib.oracle_ragged_plan(
        len(pl), chunk, k_align, _ptr(pl), _ptr(ql), _ptr(ci), n, _ptr(topk),
        *[_ptr(segs[k]) for k in ("seg_req", "kv_lens", "q_starts", "q_lens", "k_bases", "q_bases",
                                  "current_bases")],
        _ptr(S), _ptr(Q), _ptr(status))
    _check(rc, "oracle_ragged_plan")
    s, q = int(S[0]), int(Q[0])
    out = {k: v[:s].copy() for k, v in segs.items()}
    out["topk_offsets"] = topk[:q].copy()
    out["S"], out["Q"], out["status"] = s, q, int(status[0])
    return out


__all__ = [
    "build", "load", "compile_oracle", "sizes", "compose_plan", "compose_dense", "staging", "fill_index_copy",
    "fill_planes", "compose_dense_planes",
    "gather", "ragged_plan", "OracleError",
]
