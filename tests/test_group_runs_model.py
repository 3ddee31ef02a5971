"""CPU model of the grouped small-page gather's run decomposition.

The grouped gather (gather_groups_kernel) cuts the dense pages into groups
of G = 8 KB / page bytes (at most 32); within a group, lane j's page
continues page j - 1 when both are copies from one table entry with
consecutive source pages, a run starts at every copy page that does not
continue, and its length is the count of continuing pages right after it,
plus one (taken from a 32-bit ballot by a find-first-zero).  This model
replays exactly that arithmetic on random descriptor tables (with runs,
zero slots and invalid descriptors) and checks that the runs stay inside
the stage and the source entry, never mix pools with stagings, cover every
copy page once, and reproduce a page-by-page gather byte for byte.
"""
import numpy as np
import pytest

GROUP_BYTES = 8 * 1024


def _ffs64(x):
    x &= (1 << 64) - 1
    return (x & -x).bit_length()


def _model(owner, src, caps, n_pool, pb, dense_cap, table):
    n_table = len(caps)
    G = min(32, GROUP_BYTES // pb)
    dense = np.full(dense_cap * pb, 0xCD, np.uint8)
    oob = 0
    for u in range(-(-dense_cap // G)):
        d0 = u * G
        n = min(G, dense_cap - d0)
        kind, o, s = [0] * 32, [-1] * 32, [0] * 32
        for j in range(n):
            o[j], s[j] = int(owner[d0 + j]), int(src[d0 + j])
            if o[j] == -1:
                kind[j] = 1
            elif o[j] < -1 or o[j] >= n_table or s[j] < 0 or s[j] >= caps[o[j]]:
                kind[j] = 1
                oob += 1
            else:
                kind[j] = 2
        cont = [j > 0 and kind[j] == 2 and kind[j - 1] == 2 and o[j] == o[j - 1] and s[j] == s[j - 1] + 1
                for j in range(32)]
        cont_mask = sum(1 << j for j in range(32) if cont[j])
        stage = np.full(G * pb, 0x77, np.uint8)
        covered = 0
        for j in range(32):
            if kind[j] == 1:
                stage[j * pb:(j + 1) * pb] = 0
            if kind[j] != 2 or cont[j]:
                continue
            run = _ffs64(~(cont_mask >> (j + 1)))
            assert 1 <= run <= n - j
            assert all(o[j + k] == o[j] and s[j + k] == s[j] + k for k in range(run))
            assert s[j] + run <= caps[o[j]]
            assert len({o[j + k] >= n_pool for k in range(run)}) == 1
            stage[j * pb:(j + run) * pb] = table[o[j]][s[j] * pb:(s[j] + run) * pb]
            covered += run
        assert covered == sum(1 for j in range(32) if kind[j] == 2)
        dense[d0 * pb:(d0 + n) * pb] = stage[:n * pb]
    return dense, oob


def _direct(owner, src, caps, pb, dense_cap, table):
    out = np.zeros(dense_cap * pb, np.uint8)
    oob = 0
    for d in range(dense_cap):
        o, s = int(owner[d]), int(src[d])
        if o == -1:
            continue
        if o < -1 or o >= len(caps) or s < 0 or s >= caps[o]:
            oob += 1
            continue
        out[d * pb:(d + 1) * pb] = table[o][s * pb:(s + 1) * pb]
    return out, oob


@pytest.mark.parametrize("seed", range(12))
def test_group_run_model_matches_a_page_by_page_gather(seed):
    rng = np.random.default_rng(seed)
    for _ in range(25):
        cp = int(rng.integers(1, 9))
        pb = 16 * int(rng.integers(1, GROUP_BYTES // 32 + 1))  # up to 4 KB: the grouped range
        caps = [int(rng.integers(0, 40)) for _ in range(2 * cp)]
        table = [rng.integers(0, 256, size=c * pb, dtype=np.uint8) for c in caps]
        dense_cap = int(rng.integers(1, 150))
        owner = np.empty(dense_cap, np.int64)
        src = np.empty(dense_cap, np.int64)
        for d in range(dense_cap):
            r = rng.random()
            if r < 0.5 and d > 0 and owner[d - 1] >= 0:
                owner[d], src[d] = owner[d - 1], src[d - 1] + 1  # a run (possibly past the capacity)
            elif r < 0.75:
                k = int(rng.integers(0, 2 * cp))
                owner[d], src[d] = k, int(rng.integers(0, max(1, caps[k])))
            elif r < 0.9:
                owner[d], src[d] = -1, 0
            else:
                owner[d], src[d] = int(rng.integers(-3, 2 * cp + 3)), int(rng.integers(-2, 50))
        got, got_oob = _model(owner, src, caps, cp, pb, dense_cap, table)
        want, want_oob = _direct(owner, src, caps, pb, dense_cap, table)
        assert np.array_equal(got, want) and got_oob == want_oob
