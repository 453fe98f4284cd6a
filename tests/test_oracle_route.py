"""Pins for the oracle's routing metadata (histogram, offsets, stable
permutation, inverse map, padded offsets, tile-count bound).

Each check ties the oracle to something other than itself: numpy's stable sort
and bincount, exhaustive enumeration on tiny cases, and the worked example of
the ragged-dw layout printed on the matmul_ogs.py page."""
import itertools
import os

import numpy as np
import pytest

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals = [int(x) for x in v.split(",")]
            out[k] = vals[0] if len(vals) == 1 else np.array(vals, np.int32)
    return out


@pytest.mark.parametrize("T,topk,E,seed", [(1, 1, 1, 0), (7, 2, 3, 1), (64, 2, 4, 2),
                                           (50, 8, 16, 3), (33, 4, 64, 4), (200, 3, 5, 5)])
def test_route_matches_library_stable_sort(T, topk, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    r = orc.route(ids, T, topk, E, pad_block=8)
    flat = ids.reshape(-1)
    np.testing.assert_array_equal(r["m_sizes"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(r["offsets"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    # stable sort by expert id == ascending slot index within each expert
    np.testing.assert_array_equal(r["gather_idx"], np.argsort(flat, kind="stable"))
    # inverse map
    np.testing.assert_array_equal(r["row_id_map"], np.argsort(r["gather_idx"], kind="stable"))


def test_route_invariants_skewed():
    rng = np.random.default_rng(11)
    T, topk, E = 300, 4, 12
    p = np.arange(1, E + 1, dtype=float) ** -1.5
    p[[3, 7]] = 0.0  # two empty experts
    p /= p.sum()
    ids = rng.choice(E, size=(T, topk), p=p).astype(np.int32)
    r = orc.route(ids, T, topk, E)
    m, off, g, rim = r["m_sizes"], r["offsets"], r["gather_idx"], r["row_id_map"]
    R = T * topk
    assert m.sum() == R and off[-1] == R
    assert m[3] == 0 and m[7] == 0
    assert sorted(g.tolist()) == list(range(R))            # a permutation
    assert (rim[g] == np.arange(R)).all()                  # inverse on one side
    assert (g[rim] == np.arange(R)).all()                  # and the other
    flat = ids.reshape(-1)
    for e in range(E):
        seg = g[off[e]:off[e + 1]]
        assert (flat[seg] == e).all()                      # rows belong to their expert
        assert (np.diff(seg) > 0).all()                    # ascending slot order


def test_route_brute_force_tiny_exhaustive():
    # every assignment of R=4 slots (T=2, topk=2) to E=3 experts
    T, topk, E = 2, 2, 3
    for combo in itertools.product(range(E), repeat=T * topk):
        ids = np.array(combo, np.int32).reshape(T, topk)
        r = orc.route(ids, T, topk, E)
        # brute force: walk the experts, then the slots in order
        expect = [f for e in range(E) for f in range(T * topk) if combo[f] == e]
        assert r["gather_idx"].tolist() == expect
        counts = [sum(1 for c in combo if c == e) for e in range(E)]
        assert r["m_sizes"].tolist() == counts


def test_route_rejects_out_of_range_ids():
    ids = np.array([[0, 1], [2, 3]], np.int32)
    with pytest.raises(ValueError):
        orc.route(ids, 2, 2, 3)
    with pytest.raises(ValueError):
        orc.route(np.array([[0, -1]], np.int32), 1, 2, 3)


def test_padded_layout_worked_example():
    g = _read_golden("ragged_k_padded_example.txt")
    hist, bk = g["expt_hist"], g["block_k"]
    np.testing.assert_array_equal(orc.ragged_k_starts(hist, bk, padded=False), g["unpadded_starts"])
    np.testing.assert_array_equal(orc.ragged_k_starts(hist, bk, padded=True), g["padded_starts"])
    # the route's padded offsets agree when the histogram comes from routing
    ids = np.repeat(np.arange(5, dtype=np.int32), hist)
    rng = np.random.default_rng(0)
    ids = ids[rng.permutation(ids.size)]
    r = orc.route(ids.reshape(-1, 1), ids.size, 1, 5, pad_block=bk)
    np.testing.assert_array_equal(r["m_sizes"], hist)
    np.testing.assert_array_equal(r["offsets"], g["unpadded_starts"])
    np.testing.assert_array_equal(r["padded_offsets"], g["padded_starts"])


def _compositions(n, k):
    """All ways to write n as an ordered sum of k non-negative integers."""
    if k == 1:
        yield (n,)
        return
    for first in range(n + 1):
        for rest in _compositions(n - first, k - 1):
            yield (first,) + rest


@pytest.mark.parametrize("E,block_m", [(1, 4), (2, 3), (3, 4), (4, 2), (5, 8)])
def test_n_blocks_is_the_exact_worst_case(E, block_m):
    # exhaustive over every split of n rows into E experts
    for n in range(0, 14):
        worst = max(sum(-(-m // block_m) for m in comp) for comp in _compositions(n, E))
        assert orc.n_blocks(n, E, block_m) == worst, (n, E, block_m)
