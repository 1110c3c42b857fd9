"""Pins of the oracle's tile scheduler against what the pages and arithmetic fix.

- the worked example printed in "Hy3 Preview AI Infra 推理优化精读笔记", §3.1
  (tests/golden/worked_example.txt);
- the balance property of "大模型推理性能优化新范式：Hy3架构下的全栈优化技术拆解" §二.1
  (budgets base or base+1, remainder to the first CTAs);
- brute force over every contiguous partition on tiny inputs;
- coverage and ordering invariants on seeded random batches.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from oracle import scheduler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        vals[k] = [int(x) for x in v]
    return vals


def _owner_from_segments(p):
    """Stream tile -> CTA, rebuilt from the segment table alone."""
    owner = -np.ones(p["T"], dtype=np.int64)
    for r, lo, hi, c in p["segs"]:
        for i in range(lo, hi):
            t = p["cu_tiles"][r] + i
            assert owner[t] == -1, "tile assigned twice"
            owner[t] = c
    return owner


def _check_invariants(p, lens, tile, C):
    counts = [(int(L) + tile - 1) // tile for L in lens]
    assert list(p["counts"]) == counts
    assert p["cu_tiles"][0] == 0 and list(np.diff(p["cu_tiles"])) == counts
    T = sum(counts)
    assert p["T"] == T
    loads = np.diff(p["cta_begin"])
    assert loads.sum() == T and loads.min() >= 0
    assert loads.max() - loads.min() <= 1
    owner = _owner_from_segments(p)
    assert (owner >= 0).all(), "tile left unassigned"
    # owners are non-decreasing along the stream (contiguous CTA ranges, in order)
    assert (np.diff(owner) >= 0).all()
    for c in range(C):
        idx = np.nonzero(owner == c)[0]
        assert len(idx) == loads[c]
        if len(idx):
            assert idx[0] == p["cta_begin"][c] and idx[-1] == p["cta_begin"][c + 1] - 1
    # segment table: ordered, non-empty, within requests, bounded count
    S = p["S"]
    assert S == len(p["segs"]) <= len(lens) + C - 1
    for a, b in zip(p["segs"][:-1], p["segs"][1:]):
        assert (a[0], a[1]) < (b[0], b[1])
    for r, lo, hi, c in p["segs"]:
        assert 0 <= lo < hi <= counts[r]
    assert p["seg_off"][0] == 0 and p["seg_off"][-1] == S
    for r in range(len(lens)):
        for s in range(p["seg_off"][r], p["seg_off"][r + 1]):
            assert p["segs"][s][0] == r
    assert p["cta_seg"][0] == 0 and p["cta_seg"][-1] == S
    for c in range(C):
        for s in range(p["cta_seg"][c], p["cta_seg"][c + 1]):
            assert p["segs"][s][3] == c


def test_worked_example_golden():
    g = _golden()
    p = oracle.plan(g["seq_lens"], g["tile"][0], g["num_ctas"][0])
    assert list(p["counts"]) == g["tiles"]
    assert list(scheduler.cta_loads(p)) == g["cta_loads"]
    r = g["spanning_request"][0]
    ctas = {int(c) for rr, _, _, c in p["segs"] if rr == r}
    assert len(ctas) > 1
    _check_invariants(p, g["seq_lens"], 512, 4)


def test_worked_example_segments():
    # The segment table follows from the printed loads: CTA0 takes request 0's
    # two tiles and request 1's first two, CTA1 and CTA2 four tiles each of
    # request 1, CTA3 all of request 2.
    p = oracle.plan([1024, 5120, 2048], 512, 4)
    assert p["segs"].tolist() == [[0, 0, 2, 0], [1, 0, 2, 0], [1, 2, 6, 1], [1, 6, 10, 2],
                                  [2, 0, 4, 3]]
    assert p["seg_off"].tolist() == [0, 1, 4, 5]
    assert p["cta_seg"].tolist() == [0, 2, 3, 4, 5]
    assert (p["base"], p["rem"]) == (4, 0)


@pytest.mark.parametrize("L,n", [(1, 1), (511, 1), (512, 1), (513, 2), (1024, 2), (1025, 3),
                                 (196608, 384)])
def test_tile_count_is_ceiling(L, n):
    assert scheduler.tile_counts([L], 512) == [n]


def test_remainder_goes_to_first_ctas():
    p = oracle.plan([512 * 7], 512, 3)          # 7 tiles over 3 CTAs: 3, 2, 2
    assert list(scheduler.cta_loads(p)) == [3, 2, 2]
    assert (p["base"], p["rem"]) == (2, 1)


def test_more_ctas_than_tiles():
    p = oracle.plan([100, 600], 512, 7)         # 3 tiles, 7 CTAs
    assert list(scheduler.cta_loads(p)) == [1, 1, 1, 0, 0, 0, 0]
    assert p["cta_seg"].tolist() == [0, 1, 2, 3, 3, 3, 3, 3]
    _check_invariants(p, [100, 600], 512, 7)


def _compositions(T, C):
    """All ways to cut T ordered tiles into C contiguous (possibly empty) ranges."""
    for cuts in itertools.combinations_with_replacement(range(T + 1), C - 1):
        edges = (0,) + cuts + (T,)
        yield [edges[i + 1] - edges[i] for i in range(C)]


@pytest.mark.parametrize("T", range(1, 13))
@pytest.mark.parametrize("C", range(1, 6))
def test_brute_force_balance(T, C):
    p = oracle.plan([512] * T, 512, C)          # T single-tile requests
    loads = list(scheduler.cta_loads(p))
    comps = list(_compositions(T, C))
    best_max = min(max(x) for x in comps)
    best_min = max(min(x) for x in comps)
    assert max(loads) == best_max == -(-T // C)
    assert min(loads) == best_min
    # among optimal partitions, ours is the one giving the extra tile to the first CTAs
    optimal = [x for x in comps if max(x) == best_max and min(x) == best_min]
    front_loaded = [x for x in optimal if x == sorted(x, reverse=True)]
    assert front_loaded == [loads]


@pytest.mark.parametrize("seed", range(20))
def test_random_invariants(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    lens = rng.integers(1, 20000, size=B)
    tile = int(rng.choice([64, 128, 256, 512, 1024]))
    C = int(rng.integers(1, 80))
    p = oracle.plan(lens, tile, C)
    _check_invariants(p, lens, tile, C)


def test_invalid_inputs():
    with pytest.raises(ValueError):
        oracle.plan([0, 5], 512, 4)
    with pytest.raises(ValueError):
        oracle.plan([5], 512, 0)
    with pytest.raises(ValueError):
        oracle.plan_static([5], 512, 0)


@pytest.mark.parametrize("seed", range(10))
def test_static_plan(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 20))
    lens = rng.integers(1, 40000, size=B)
    S = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    p = oracle.plan_static(lens, 512, S)
    assert p["C"] == B * S
    owner = _owner_from_segments(p)
    assert (owner >= 0).all()
    assert (np.diff(p["cta_seg"]) <= 1).all()        # at most one chunk per CTA
    for r, L in enumerate(lens):
        n = (int(L) + 511) // 512
        k = min(S, n)
        sizes = [hi - lo for rr, lo, hi, _ in p["segs"] if rr == r]
        assert len(sizes) == k and sum(sizes) == n
        assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    assert (np.diff(p["cta_begin"]) >= 0).all()
    assert p["cta_begin"][-1] == p["T"]


def test_static_one_split_is_one_segment_per_request():
    p = oracle.plan_static([1024, 5120, 2048], 512, 1)
    assert p["segs"].tolist() == [[0, 0, 2, 0], [1, 0, 10, 1], [2, 0, 4, 2]]


# ----------------------------------------------------------------------------- token-weighted
def _key_loads(p, lens, tile):
    loads = np.zeros(p["C"], dtype=np.int64)
    for r, lo, hi, c in p["segs"]:
        loads[c] += min(int(hi) * tile, int(lens[r])) - int(lo) * tile
    return loads


@pytest.mark.parametrize("seed", range(20))
def test_weighted_plan_invariants(seed):
    rng = np.random.default_rng(500 + seed)
    B = int(rng.integers(1, 30))
    lens = rng.integers(1, 30000, size=B)
    tile = int(rng.choice([64, 256, 512]))
    C = int(rng.integers(1, 60))
    p = oracle.plan_weighted(lens, tile, C)
    assert p["kind"] == 2
    owner = _owner_from_segments(p)
    assert (owner >= 0).all() and (np.diff(owner) >= 0).all()
    assert p["S"] <= B + C - 1
    K = int(np.sum(lens))
    loads = _key_loads(p, lens, tile)
    assert loads.sum() == K
    # every partition is within one tile of the equal share K / C
    assert (np.abs(loads - K / C) <= tile).all()


def test_weighted_plan_counts_a_partial_tile_by_its_fill():
    # 4 requests of 513 keys: 8 tiles, four of them hold a single key.  By tiles,
    # 2 partitions take 4 tiles each; by keys, each takes about 1026 keys.
    lens = [513] * 4
    pt = oracle.plan(lens, 512, 2)
    pw = oracle.plan_weighted(lens, 512, 2)
    assert list(_key_loads(pt, lens, 512)) == [1026, 1026]
    assert list(_key_loads(pw, lens, 512)) == [1026, 1026]
    lens = [1024 + 1, 1]                       # tiles of 512, 512, 1 and 1 keys
    pt = oracle.plan(lens, 512, 2)             # 2 tiles each: 1024 vs 2 keys
    pw = oracle.plan_weighted(lens, 512, 2)    # the key shares: 512 vs 514
    assert list(_key_loads(pt, lens, 512)) == [1024, 2]
    assert list(_key_loads(pw, lens, 512)) == [512, 514]


@pytest.mark.parametrize("T,C", [(7, 3), (8, 3), (10, 4), (12, 5), (1, 4), (100, 7)])
def test_weighted_equals_tile_budgets_when_tiles_are_full(T, C):
    lens = [512] * T
    lt = sorted(scheduler.cta_loads(oracle.plan(lens, 512, C)))
    lw = sorted(scheduler.cta_loads(oracle.plan_weighted(lens, 512, C)))
    assert lt == lw                            # the same multiset of loads, max - min <= 1
