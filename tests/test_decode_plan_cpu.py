"""The decode plan (host logic, no GPU): how fia_decode deals the 128-key
stages of every unit (batch, kv head) to its CTAs.  The kernels rely on its
structure: each unit's stages covered once, in order, by segments whose part
numbers are consecutive; at most one segment of a unit per CTA (the CTA that
completes a unit merges it, and a CTA's last segment is merged by its own
compute warps); a CTA's shared pieces ahead of its whole units."""
import numpy as np
import pytest

from attention_fia_prefill_gb300 import _binding as B
from attention_fia_prefill_gb300 import build as fia_build

import fia_inputs


@pytest.fixture(scope="module")
def lib():
    fia_build.build()
    return B.load_library()


def check_plan(kv_len, n2, n_cta_max):
    cta_seg, segs, parts = B.debug_plan_decode(kv_len, n2, n_cta_max)
    n_cta = len(cta_seg) - 1
    nst = [-(-int(L) // 128) for L in kv_len for _ in range(n2)]
    total = sum(nst)
    assert n_cta <= min(n_cta_max, max(total, 0)) or (total == 0 and n_cta == 0)
    assert cta_seg[0] == 0 and cta_seg[-1] == len(segs)
    assert all(a <= b for a, b in zip(cta_seg, cta_seg[1:]))
    assert all(cta_seg[c + 1] > cta_seg[c] for c in range(n_cta)), "a CTA without work"
    # every segment is non-empty; its part number indexes the creation order
    assert sorted(s[3] for s in segs) == list(range(len(segs)))
    assert all(s[2] > s[1] for s in segs)
    by_part = {s[3]: s for s in segs}
    for u, (first, count) in enumerate(parts):
        if nst[u] == 0:
            assert count == 0
            continue
        assert count >= 1
        pieces = [by_part[first + k] for k in range(count)]
        assert all(p[0] == u for p in pieces)
        # consecutive parts cover [0, nst) in order
        assert pieces[0][1] == 0 and pieces[-1][2] == nst[u]
        assert all(a[2] == b[1] for a, b in zip(pieces, pieces[1:]))
    assert sum(s[2] - s[1] for s in segs) == total
    for c in range(n_cta):
        mine = segs[cta_seg[c]:cta_seg[c + 1]]
        units = [s[0] for s in mine]
        assert len(units) == len(set(units)), "two pieces of one unit in a CTA"
        shared = [parts[s[0]][1] > 1 for s in mine]
        assert shared == sorted(shared, reverse=True), "a whole unit ahead of a shared piece"
    return n_cta, segs


@pytest.mark.parametrize("n_cta_max", [1, 7, 151, 152, 256])
def test_plan_headline_lengths(lib, n_cta_max):
    """The paged decode workload's lengths (B=16, U[1,4096]) over 8 kv heads."""
    lens = fia_inputs.workload_paged_gqa_decode().kv_lens
    n_cta, segs = check_plan(lens, 8, n_cta_max)
    assert n_cta >= min(n_cta_max, 128) * 0.9


@pytest.mark.parametrize("lens,n2", [([0, 0, 0], 4), ([1], 1), ([16384] * 8, 8), ([256] * 300, 1),
                                     ([0, 1, 127, 128, 129, 700, 2049, 3], 2), ([100000, 1, 1], 1)])
def test_plan_edge_lengths(lib, lens, n2):
    """Empty sequences, one key, long sequences split over many CTAs, many
    short ones, one very long sequence beside tiny ones."""
    for n_cta_max in (1, 3, 151):
        check_plan(lens, n2, n_cta_max)


def test_plan_random_lengths(lib):
    rng = np.random.default_rng(11)
    for _ in range(40):
        B = int(rng.integers(1, 40))
        lens = [int(x) for x in rng.integers(0, 9000, B)]
        n2 = int(rng.choice([1, 2, 4, 8]))
        check_plan(lens, n2, int(rng.integers(1, 257)))


def test_plan_hook_checks_capacity(lib):
    import ctypes
    lens = (ctypes.c_int32 * 2)(500, 700)
    small = (ctypes.c_int32 * 1)()
    n_cta, n_segs = ctypes.c_int(0), ctypes.c_int(0)
    big = (ctypes.c_int32 * 64)()
    assert lib.fia_debug_plan_decode(lens, 2, 1, 4, small, 1, big, 64, big, 64, ctypes.byref(n_cta),
                                     ctypes.byref(n_segs)) == 3
    assert lib.fia_debug_plan_decode(None, 2, 1, 4, big, 64, big, 64, big, 64, ctypes.byref(n_cta),
                                     ctypes.byref(n_segs)) == 1
