"""Pins of the oracle's FBS / VBS partitions (CPU only).

FreeScale (arXiv 2604.24073) §4.1 "Partitioning Algorithms".  Every check here
comes from the pages or from mathematics, not from re-running the oracle's own
formula: hand-worked examples, the pages' index-list form of the zig-zag,
library sorts for the degenerate cases, counting invariants and the VBS
weight bound.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ FBS

@pytest.mark.parametrize("case", _load("fbs_hand_examples.json")["cases"])
def test_fbs_hand_examples(case):
    perm, ro = oracle.balance_fbs(np.array(case["L"]), case["n"])
    assert perm.tolist() == case["perm"]
    assert ro.tolist() == case["rank_offsets"]
    if "rank_len_sums" in case:
        L = np.array(case["L"])
        sums = [int(L[perm[ro[r]:ro[r + 1]]].sum()) for r in range(case["n"])]
        assert sums == case["rank_len_sums"]


def _pages_index_list(n, S):
    """Rank i (1-based) gets sorted positions i, 2n+1-i, 2n+i, 4n+1-i, ... (1-based).

    This is the §4.1 list [i, 2n-i, 2n+i, 4n-i, ...] with its off-by-one repaired;
    returned 0-based, per rank.
    """
    out = []
    for i in range(1, n + 1):
        lst, m = [], 0
        while True:
            a = 2 * m * n + i              # i, 2n+i, 4n+i, ...
            b = 2 * (m + 1) * n + 1 - i    # 2n+1-i, 4n+1-i, ...
            if a <= S:
                lst.append(a - 1)
            if b <= S:
                lst.append(b - 1)
            if a > S and b > S:
                break
            m += 1
        out.append(lst)
    return out


@pytest.mark.parametrize("n,S", [(1, 7), (2, 8), (3, 12), (4, 64), (8, 512), (5, 23), (16, 16), (7, 3)])
def test_fbs_matches_pages_index_list(n, S):
    rng = np.random.default_rng(n * 1000 + S)
    L = rng.integers(1, 50, S).astype(np.int32)
    perm, ro = oracle.balance_fbs(L, n)
    order = np.argsort(L, kind="stable")            # library stable sort: (L, g)
    for r, plist in enumerate(_pages_index_list(n, S)):
        assert perm[ro[r]:ro[r + 1]].tolist() == order[plist].tolist()


def test_fbs_brute_force_tiny():
    """All S <= 6 with all orderings of distinct lengths, n in {1, 2, 3}."""
    for S in range(0, 7):
        for n in (1, 2, 3):
            for Lp in itertools.permutations(range(1, S + 1)):
                L = np.array(Lp, np.int32)
                perm, ro = oracle.balance_fbs(L, n)
                assert sorted(perm.tolist()) == list(range(S))              # each sample once
                counts = np.diff(ro)
                assert counts.max() - counts.min() <= 1                      # equal counts
                if S % n == 0:
                    assert (counts == S // n).all()
                rank_of = np.empty(S, np.int64)
                for r in range(n):
                    rank_of[perm[ro[r]:ro[r + 1]]] = r
                    seq = L[perm[ro[r]:ro[r + 1]]]
                    assert (np.diff(seq) > 0).all()                          # round order = ascending L
                sorted_g = np.argsort(L, kind="stable")
                for rho in range(0, (S + n - 1) // n):
                    block = sorted_g[rho * n:(rho + 1) * n]
                    ranks = rank_of[block].tolist()
                    expect = list(range(len(block))) if rho % 2 == 0 else list(range(n - 1, n - 1 - len(block), -1))
                    assert ranks == expect                                   # snake direction per round


@pytest.mark.parametrize("seed", range(6))
def test_fbs_invariants_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    B = int(rng.integers(1, 30))
    S = n * B
    L = np.clip(np.round(rng.lognormal(5, 1.2, S)), 1, 2048).astype(np.int32)
    perm, ro = oracle.balance_fbs(L, n)
    assert np.array_equal(np.sort(perm), np.arange(S))
    assert np.array_equal(ro, np.arange(n + 1) * B)
    sums = np.array([L[perm[ro[r]:ro[r + 1]]].astype(np.int64).sum() for r in range(n)])
    # one sample per rank per round over consecutive sorted blocks: the spread of
    # the per-rank sums is at most the sum of the per-round spreads <= max L - min L
    assert sums.max() - sums.min() <= int(L.max()) - int(L.min())


def test_fbs_degenerate_cases():
    L = np.array([5, 3, 5, 1, 9, 3], np.int32)
    order = np.argsort(L, kind="stable")
    perm, ro = oracle.balance_fbs(L, 1)                 # n = 1: the stable sort itself
    assert perm.tolist() == order.tolist() and ro.tolist() == [0, 6]
    perm, ro = oracle.balance_fbs(L, 6)                 # n = S: rank r gets sorted position r
    assert perm.tolist() == order.tolist() and ro.tolist() == list(range(7))
    perm, ro = oracle.balance_fbs(L, 3)                 # S = 2n: rank r gets r and 2n-1-r
    assert [perm[ro[r]:ro[r + 1]].tolist() for r in range(3)] == [[order[r], order[5 - r]] for r in range(3)]
    perm, ro = oracle.balance_fbs(np.zeros(0, np.int32), 4)   # empty batch
    assert perm.size == 0 and ro.tolist() == [0] * 5


# ------------------------------------------------------------------ VBS

def _exact_q15(L):
    """round(256 * L^1.5) from exact integer arithmetic (L^1.5 = sqrt(L^3))."""
    # 256 * L^1.5 = sqrt(65536 * L^3); nearest integer of sqrt(N):
    N = 65536 * L ** 3
    r = math.isqrt(N)
    # r <= sqrt(N) < r + 1; nearest is r+1 iff sqrt(N) >= r + 1/2 iff 4N >= (2r+1)^2
    return r + 1 if 4 * N >= (2 * r + 1) ** 2 else r


def test_vbs_weight_perfect_squares():
    for m in range(1, 129):
        assert oracle.vbs_weight(m * m, 1.5) == 256 * m ** 3
    assert oracle.vbs_weight(1, 1.5) == 256
    assert oracle.vbs_weight(2, 1.5) == 724          # 256 * 2.828427... = 724.077
    assert oracle.vbs_weight(0, 1.5) == 0
    assert oracle.vbs_weight(16384, 1.5) == 256 * 128 ** 3


def test_vbs_weight_alpha15_exact_for_all_lengths():
    """q(L^1.5) equals the exactly rounded real value for every L in [1, 16384]."""
    bad = [L for L in range(1, 16385) if oracle.vbs_weight(L, 1.5) != _exact_q15(L)]
    assert bad == []


def test_vbs_weight_other_alphas():
    for L in (1, 2, 3, 17, 1000, 16384):
        assert oracle.vbs_weight(L, 1.0) == 256 * L
        assert oracle.vbs_weight(L, 2.0) == 256 * L * L
        assert oracle.vbs_weight(L, 3.0) == 256 * L ** 3
    # general alpha (pow): within one unit of 256 * L^alpha
    for L in (2, 3, 10, 999, 16384):
        assert abs(oracle.vbs_weight(L, 1.3) - 256 * L ** 1.3) <= 1


@pytest.mark.parametrize("case", _load("vbs_hand_examples.json")["cases"])
def test_vbs_hand_examples(case):
    perm, ro, sw = oracle.balance_vbs(np.array(case["L"]), case["n"], case["alpha"], case["sort_by_len"])
    if "w" in case:
        assert [oracle.vbs_weight(l, case["alpha"]) for l in case["L"]] == case["w"]
    assert perm.tolist() == case["perm"]
    assert ro.tolist() == case["rank_offsets"]
    assert sw.tolist() == case["seg_weight"]


@pytest.mark.parametrize("seed,sort_by_len", [(s, b) for s in range(5) for b in (0, 1)])
def test_vbs_invariants_random(seed, sort_by_len):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 64))
    S = int(rng.integers(1, 3000))
    L = np.clip(np.round(rng.lognormal(6, 1.4, S)), 1, 4096).astype(np.int32)
    perm, ro, sw = oracle.balance_vbs(L, n, 1.5, sort_by_len)
    assert np.array_equal(np.sort(perm), np.arange(S))                 # each sample once
    assert ro[0] == 0 and ro[-1] == S and (np.diff(ro) >= 0).all()     # contiguous segments
    order = np.argsort(L, kind="stable") if sort_by_len else np.arange(S)
    assert np.array_equal(perm, order)
    w = np.array([oracle.vbs_weight(int(l), 1.5) for l in L[perm]], dtype=object)
    W = int(sum(w))
    for r in range(n):
        assert int(sw[r]) == int(sum(w[ro[r]:ro[r + 1]]))
    assert sum(int(x) for x in sw) == W
    # bound from the cut rule: heaviest segment <= W/n + heaviest single weight
    assert n * max(int(x) for x in sw) <= W + n * int(max(w))


def test_vbs_degenerate_cases():
    L = np.array([7, 1, 30, 2, 2], np.int32)
    perm, ro, sw = oracle.balance_vbs(L, 1, 1.5, 0)
    assert perm.tolist() == [0, 1, 2, 3, 4] and ro.tolist() == [0, 5]
    # equal lengths, S = n*B -> exactly B per rank
    perm, ro, sw = oracle.balance_vbs(np.full(12, 37, np.int32), 4, 1.5, 1)
    assert ro.tolist() == [0, 3, 6, 9, 12]
    # all weights zero -> equal counts
    perm, ro, sw = oracle.balance_vbs(np.zeros(6, np.int32), 3, 1.5, 0)
    assert ro.tolist() == [0, 2, 4, 6] and sw.tolist() == [0, 0, 0]
    # empty
    perm, ro, sw = oracle.balance_vbs(np.zeros(0, np.int32), 3, 1.5, 1)
    assert ro.tolist() == [0, 0, 0, 0]
