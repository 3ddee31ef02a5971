"""CPU-only checks of the C ABI: the library loads, exports every function
declared in include/cpkv.h, and its host-side sizing and argument checks
agree with the oracle.  Nothing here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import oracle_pins as pins
import workloads as wl
from paged_kv_cache_compose_gb300 import build as cuda_build
from paged_kv_cache_compose_gb300 import cpkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return cpkv.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^(?:const\s+char\s*\*|int)\s*(cpkv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("cpkv_plan_build", "cpkv_fill_current", "cpkv_compose_gather", "cpkv_ragged_plan_build"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in cpkv.EXPORTED, n
    assert lib.cpkv_version() == 1


def test_library_targets_sm103a_only():
    so = cpkv.LIB_PATH
    assert os.path.exists(so)
    assert cuda_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("batch", pins.edge_batches() + [wl.traced_batch(), wl.fp8_nsa_batch()],
                         ids=lambda b: b.name)
def test_sizes_match_oracle(lib, batch):
    assert cpkv.cpkv_plan_sizes(batch.prefix_lens, batch.cur_lens, batch.page_size) == \
        oracle.sizes(batch.prefix_lens, batch.cur_lens, batch.page_size)
    counts = cpkv.cpkv_writer_token_counts(batch.cur_lens, batch.writer, batch.page_size, batch.cp_size)
    tw = wl.token_writer(batch)
    assert counts.tolist() == [int((tw == w).sum()) for w in range(batch.cp_size)]


@pytest.mark.parametrize("rb", pins.ragged_edge_batches() + [wl.ragged_batch()], ids=lambda r: r.name)
def test_ragged_sizes_match_oracle(lib, rb):
    for r in range(rb.cp_size):
        want = oracle.ragged_plan(rb.prefix_lens, rb.q_lens, rb.cp_index(r), chunk=rb.chunk, k_align=rb.k_align)
        assert cpkv.cpkv_ragged_plan_sizes(rb.q_lens, rb.cp_index(r), rb.chunk) == (want["S"], want["Q"])


def test_host_errors_before_any_launch(lib):
    pl = np.array([3], np.int32)
    cl = np.array([4], np.int32)
    null = None
    rc = lib.cpkv_plan_build(1, 2, 1, 8, pl.ctypes.data, cl.ctypes.data, *([null] * 3), 10, *([null] * 10), 0, null, null)
    assert rc == cpkv.CPKV_ERR_UNALIGNED_PREFIX
    pl = np.array([2], np.int32)
    rc = lib.cpkv_plan_build(1, 2, 1, 8, pl.ctypes.data, cl.ctypes.data, *([null] * 3), 2, *([null] * 10), 0, null, null)
    assert rc == cpkv.CPKV_ERR_CAPACITY
    rc = lib.cpkv_plan_build(1, 2, 65, 8, pl.ctypes.data, cl.ctypes.data, *([null] * 3), 10, *([null] * 10), 0, null, null)
    assert rc == cpkv.CPKV_ERR_ARG
    big = np.zeros(1025, np.int32)
    rc = lib.cpkv_plan_build(1025, 2, 1, 8, big.ctypes.data, big.ctypes.data, *([null] * 3), 10, *([null] * 10), 0, null, null)
    assert rc == cpkv.CPKV_ERR_LIMIT
    # missing output pointers are reported, not dereferenced
    rc = lib.cpkv_plan_build(1, 2, 1, 8, pl.ctypes.data, cl.ctypes.data, *([null] * 3), 10, *([null] * 10), 0, null, null)
    assert rc == cpkv.CPKV_ERR_ARG
    # fill: row width must be a multiple of 16
    rc = lib.cpkv_fill_current(1, 2, 1, 100, cl.ctypes.data, *([null] * 3), 5, *([null] * 3), 2, 0, null, null)
    assert rc == cpkv.CPKV_ERR_ARG
    # gather kinds: with no dense pages the call returns before any launch, so only the mask decides
    tbl2 = (ctypes.c_void_p * 2)(16, 32)
    caps2 = np.zeros(2, np.int64)
    for kinds, want in ((cpkv.GATHER_ALL, cpkv.CPKV_OK), (cpkv.GATHER_ALL | cpkv.GATHER_EARLY_INPUTS, cpkv.CPKV_OK),
                        (cpkv.GATHER_ALL | cpkv.GATHER_CONSUME_STAGING | cpkv.GATHER_EARLY_INPUTS, cpkv.CPKV_OK),
                        (32, cpkv.CPKV_ERR_ARG), (cpkv.GATHER_ALL | 32, cpkv.CPKV_ERR_ARG), (-1, cpkv.CPKV_ERR_ARG)):
        rc = lib.cpkv_compose_gather_kinds(16, 1, 64, ctypes.cast(tbl2, ctypes.c_void_p), caps2.ctypes.data, null,
                                           null, 0, kinds, null, 64, null)
        assert rc == want, kinds
    # fill flags: an empty batch returns before any launch, so only the flag word decides
    empty = np.zeros(1, np.int32)
    fake = (ctypes.c_void_p * 1)(16)  # never dereferenced: nothing to copy
    zero_cap = np.zeros(1, np.int64)
    pb = np.array([16], np.int32)
    for flags, want in ((0, cpkv.CPKV_OK), (cpkv.FLAG_EARLY_INPUTS, cpkv.CPKV_OK), (cpkv.FLAG_CONSUME_STAGING, cpkv.CPKV_ERR_ARG),
                        (cpkv.FILL_PAGE_RUNS, cpkv.CPKV_OK), (cpkv.FILL_PAGE_RUNS | cpkv.FLAG_EARLY_INPUTS, cpkv.CPKV_OK),
                        (8, cpkv.CPKV_ERR_ARG), (-1, cpkv.CPKV_ERR_ARG)):
        rc = lib.cpkv_fill_current(1, 2, 1, 64, empty.ctypes.data, ctypes.cast(fake, ctypes.c_void_p),
                                   zero_cap.ctypes.data, ctypes.cast(fake, ctypes.c_void_p), 1, null, null, null, 0,
                                   flags, 64, null)
        assert rc == want, ("fill", flags)
    for flags, want in ((0, cpkv.CPKV_OK), (cpkv.FLAG_EARLY_INPUTS, cpkv.CPKV_OK), (cpkv.FLAG_CONSUME_STAGING, cpkv.CPKV_ERR_ARG),
                        (cpkv.FILL_PAGE_RUNS, cpkv.CPKV_OK), (8, cpkv.CPKV_ERR_ARG), (-1, cpkv.CPKV_ERR_ARG)):
        rc = lib.cpkv_fill_current_planes(1, 2, 1, 1, pb.ctypes.data, empty.ctypes.data,
                                          ctypes.cast(fake, ctypes.c_void_p), zero_cap.ctypes.data,
                                          ctypes.cast(fake, ctypes.c_void_p), 1, null, null, null, 0, flags, 64, null)
        assert rc == want, ("fill_planes", flags)
    # gather: unaligned dense pointer
    tbl = (ctypes.c_void_p * 2)(16, 32)
    caps = np.array([1, 1], np.int64)
    rc = lib.cpkv_compose_gather(2, 1, 64, ctypes.cast(tbl, ctypes.c_void_p), caps.ctypes.data, 64, 64, 1, 8, 64, null)
    assert rc == cpkv.CPKV_ERR_ARG
    # one-launch layer compose: a staging without room for slots 1..C, then a row width not a multiple of 16
    rows = (ctypes.c_void_p * 1)(16)
    rcap = np.array([4], np.int64)
    tcaps = np.array([8, 1], np.int64)
    rc = lib.cpkv_compose_layer(1, 2, 1, 64, cl.ctypes.data, ctypes.cast(rows, ctypes.c_void_p), rcap.ctypes.data,
                                ctypes.cast(tbl, ctypes.c_void_p), tcaps.ctypes.data, 64, 64, 64, 4, 64, 0, 64, null)
    assert rc == cpkv.CPKV_ERR_CAPACITY
    tcaps = np.array([8, 3], np.int64)
    rc = lib.cpkv_compose_layer(1, 2, 1, 40, cl.ctypes.data, ctypes.cast(rows, ctypes.c_void_p), rcap.ctypes.data,
                                ctypes.cast(tbl, ctypes.c_void_p), tcaps.ctypes.data, 64, 64, 64, 4, 64, 0, 64, null)
    assert rc == cpkv.CPKV_ERR_ARG
    # planar layer compose: plane counts, widths and page sizes outside the contract
    for n_planes, pb, ps in ((0, [16], 2), (5, [16] * 5, 2), (2, [128, 2], 2), (2, [128, 4], 3)):
        pba = np.array(pb, np.int32)
        rc = lib.cpkv_compose_layer_planes(1, ps, 1, n_planes, pba.ctypes.data, cl.ctypes.data,
                                           ctypes.cast(rows, ctypes.c_void_p), rcap.ctypes.data,
                                           ctypes.cast(tbl, ctypes.c_void_p), tcaps.ctypes.data, 64, 64, 64, 4, 64, 0,
                                           64, null)
        assert rc == cpkv.CPKV_ERR_ARG, (n_planes, pb, ps)
    # planar fused compose: the same plane checks
    for n_planes, pb, ps in ((0, [16], 2), (5, [16] * 5, 2), (2, [128, 2], 2), (2, [128, 4], 3)):
        pba = np.array(pb, np.int32)
        rc = lib.cpkv_compose_fused_planes(1, ps, 1, n_planes, pba.ctypes.data, cl.ctypes.data,
                                           ctypes.cast(tbl, ctypes.c_void_p), tcaps.ctypes.data,
                                           ctypes.cast(rows, ctypes.c_void_p), rcap.ctypes.data, 64, 64, 64, 4, 64, 0,
                                           64, null)
        assert rc == cpkv.CPKV_ERR_ARG, (n_planes, pb, ps)
    # unknown flag bits (and consuming, for the fused forms) are argument errors
    tcaps = np.array([8, 3], np.int64)
    for flags in (4, 8, -1):
        rc = lib.cpkv_compose_layer(1, 2, 1, 64, cl.ctypes.data, ctypes.cast(rows, ctypes.c_void_p), rcap.ctypes.data,
                                    ctypes.cast(tbl, ctypes.c_void_p), tcaps.ctypes.data, 64, 64, 64, 4, 64, flags,
                                    64, null)
        assert rc == cpkv.CPKV_ERR_ARG, flags
    for flags in (cpkv.FLAG_CONSUME_STAGING, 4):
        rc = lib.cpkv_compose_fused(1, 2, 1, 64, cl.ctypes.data, ctypes.cast(tbl, ctypes.c_void_p), tcaps.ctypes.data,
                                    ctypes.cast(rows, ctypes.c_void_p), rcap.ctypes.data, 64, 64, 64, 4, 64, flags,
                                    64, null)
        assert rc == cpkv.CPKV_ERR_ARG, flags
    # ragged: bad chunk / k_align
    rc = lib.cpkv_ragged_plan_build(1, 0, 1, 2048, pl.ctypes.data, cl.ctypes.data, null, 0, null, 0,
                                    *([null] * 7), 0, null, null, null)
    assert rc == cpkv.CPKV_ERR_ARG
    # ragged: a topk that is not positive, every other argument well formed
    fake = ctypes.c_void_p(256)
    for topk in (0, -2048):
        rc = lib.cpkv_ragged_plan_build(1, 4, 1, topk, pl.ctypes.data, cl.ctypes.data, fake, 1, fake, 8,
                                        *([fake] * 7), 2, fake, fake, null)
        assert rc == cpkv.CPKV_ERR_ARG, topk


def test_unaligned_prefix_raises_in_binding(lib):
    with pytest.raises(cpkv.CpkvError) as e:
        cpkv.cpkv_plan_sizes([5], [3], 4)
    assert e.value.code == cpkv.CPKV_ERR_UNALIGNED_PREFIX


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.cpkv_error_string(code).startswith(b"CPKV_")


def test_missing_library_fails_loudly(tmp_path):
    saved = cpkv._lib
    cpkv._lib = None
    try:
        with pytest.raises(cpkv.CpkvError):
            cpkv.load(str(tmp_path / "absent.so"))
    finally:
        cpkv._lib = saved


def test_build_rebuilds_a_library_compiled_for_another_cpu(tmp_path, lib):
    import platform

    from paged_kv_cache_compose_gb300 import build as cuda_build

    mine = cuda_build._ELF_MACHINE.get(platform.machine())
    if mine is None:
        pytest.skip("host CPU not in the ELF table")
    other = 183 if mine == 62 else 62
    for machine, foreign in ((mine, False), (other, True)):
        f = tmp_path / f"lib{machine}.so"
        f.write_bytes(b"\x7fELF" + bytes(14) + machine.to_bytes(2, "little") + bytes(44))
        assert cuda_build._built_for_other_machine(str(f)) is foreign
    junk = tmp_path / "junk.so"
    junk.write_bytes(b"not an elf file at all")
    assert cuda_build._built_for_other_machine(str(junk))
    assert not cuda_build._built_for_other_machine(cuda_build.LIB_PATH)
