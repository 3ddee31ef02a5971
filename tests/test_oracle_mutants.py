"""Planted mistakes in the oracle must be caught by the pins.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong index, a transposed operand), compiles the copy into a
temporary library and runs every pin against it in a child process.  The
case passes only if at least one pin fails.  CPU only; nothing here touches
the CUDA library.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "cpkv_oracle.c")

MUTANTS = [
    ("owner_src_transposed", "owner[d] = lp % cp;\n      src[d] = lp / cp;",
     "owner[d] = lp / cp;\n      src[d] = lp % cp;"),
    ("staging_slot_not_reserved", "src[d] = (int32_t)(i + 1);", "src[d] = (int32_t)(i);"),
    ("current_owner_missing_cp", "owner[d] = cp + w;", "owner[d] = w;"),
    ("mixed_locs_dropped_prefix", "mixed_locs[t] = (dense + npp + k / ps) * ps + off;",
     "mixed_locs[t] = (dense + k / ps) * ps + off;"),
    ("staging_rows_off_by_one_page", "staging_rows[t] = (i + 1) * ps + off;", "staging_rows[t] = i * ps + off;"),
    ("writer_row_single_counter", "(int32_t)(writer_count[w]++)", "(int32_t)(writer_count[0]++)"),
    ("page_inverse_keeps_last", "if (page_inverse[lp] == -1) page_inverse[lp] = (int32_t)d;\n    }\n    for",
     "page_inverse[lp] = (int32_t)d;\n    }\n    for"),
    ("cur_span_start", "cur_spans[2 * b] = (int32_t)(dense + npp);", "cur_spans[2 * b] = (int32_t)(dense);"),
    ("staging_inverse_zero_based", "staging_page_inverse[lp] = (int32_t)(i + 1);",
     "staging_page_inverse[lp] = (int32_t)(i);"),
    ("dense_no_page_pad", "while (row % ps != 0) {", "while (0) {"),
    ("dense_pool_row_offset_dropped", "pool_slabs[owner] + (local * ps + off) * R",
     "pool_slabs[owner] + (local * ps) * R"),
    ("dense_current_before_prefix_skip", "memcpy(dense_out + row * R, cur_rows + (tok + k) * R, (size_t)R);",
     "memcpy(dense_out + row * R, cur_rows + (k) * R, (size_t)R);"),
    ("staging_pad_not_zeroed", "else memset(page + r * R, 0, (size_t)R);", "else (void)0;"),
    ("gather_sentinel_wrong", "if (o == -1) { memset(dst, 0, (size_t)page_bytes); continue; }",
     "if (o == -2) { memset(dst, 0, (size_t)page_bytes); continue; }"),
    ("fill_pad_overwrites_last_row", "for (int64_t row = sr + 1; row < (slot + 1) * ps; ++row)",
     "for (int64_t row = sr; row < (slot + 1) * ps; ++row)"),
    ("fill_writer_of_wrong_slot", "    int32_t w = writer[slot - 1];\n    if (w < 0 || w >= cp) { *status |= ORC_WRITER_OOB; continue; }\n    int32_t r",
     "    int32_t w = writer[slot % C];\n    if (w < 0 || w >= cp) { *status |= ORC_WRITER_OOB; continue; }\n    int32_t r"),
    ("planes_offset_ignores_plane_start",
     "memcpy(staging[w] + slot * page_bytes + plane_start + off * wp, cur_planes[p * cp + w] + r * wp,",
     "memcpy(staging[w] + slot * page_bytes + off * wp, cur_planes[p * cp + w] + r * wp,"),
    ("planes_dense_pool_offset_dropped",
     "memcpy(dst, pool_slabs[owner] + local * page_bytes + plane_start + (k % ps) * wp, (size_t)wp);",
     "memcpy(dst, pool_slabs[owner] + local * page_bytes + (k % ps) * wp, (size_t)wp);"),
    ("planes_pad_from_wrong_row", "for (int64_t off = sr % ps + 1; off < ps; ++off)",
     "for (int64_t off = sr % ps + 2; off < ps; ++off)"),
    ("ragged_kbase_unaligned", "kbase[b + 1] = kbase[b] + ceil_div64(kv, k_align) * k_align;",
     "kbase[b + 1] = kbase[b] + kv;"),
    ("ragged_kv_dropped_prefix", "int64_t kv = (int64_t)prefix_lens[b] + q_lens[b];", "int64_t kv = q_lens[b];"),
    ("ragged_kv_lens_dropped_qstart", "kv_lens[S - 1] = prefix_lens[b] + q_starts[S - 1] + q_lens_out[S - 1];",
     "kv_lens[S - 1] = prefix_lens[b] + q_lens_out[S - 1];"),
    ("ragged_never_merge", "if (!(b == prev_req && id == prev_id + 1)) {", "if (1) {"),
    ("ragged_merge_across_requests", "if (!(b == prev_req && id == prev_id + 1)) {", "if (!(id == prev_id + 1)) {"),
    ("ragged_current_base_no_prefix", "current_bases[S] = (int32_t)(kbase[b] + prefix_lens[b]);",
     "current_bases[S] = (int32_t)(kbase[b]);"),
    ("ragged_q_bases_segment_count", "q_bases[S] = (int32_t)Q;", "q_bases[S] = (int32_t)S;"),
    ("ragged_offset_global_chunk", "int64_t off = (id - chunk_start[b]) * chunk;", "int64_t off = id * chunk;"),
]

RUNNER = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import oracle, oracle_pins
    lib = oracle.load({lib!r})
    failed = []
    for name, check in oracle_pins.ALL_PINS:
        try:
            check(lib)
        except Exception as e:
            failed.append(name)
    print("FAILED_PINS", failed)
    sys.exit(1 if failed else 0)
""")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation target not found: {name}"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mut.c"
    c_path.write_text(mutated)
    so = str(tmp_path / "libmut.so")
    oracle.compile_oracle(src=str(c_path), out=so)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"planted mistake {name} survived every pin:\n{r.stdout}\n{r.stderr}"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness on an unmodified copy passes every pin."""
    so = str(tmp_path / "libcopy.so")
    oracle.compile_oracle(out=so)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
