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


# ------------------------------------------------------------------ VBS AutoTune

_AT = _load("vbs_autotune_hand_examples.json")


@pytest.mark.parametrize("case", _AT["update_cases"])
def test_autotune_update_hand_examples(case):
    out = oracle.vbs_autotune(np.array(case["t"]), np.array(case["delta_in"]), case["step"], case["tol_ppm"])
    assert out.tolist() == case["delta_out"]


@pytest.mark.parametrize("case", _AT["tuned_cases"])
def test_vbs_tuned_hand_examples(case):
    perm, ro, sw = oracle.balance_vbs_tuned(np.array(case["L"]), case["n"], case["alpha"], case["sort_by_len"],
                                            np.array(case["delta"]))
    assert perm.tolist() == case["perm"]
    assert ro.tolist() == case["rank_offsets"]
    assert sw.tolist() == case["seg_weight"]


@pytest.mark.parametrize("case", _AT["bad_tuned_cases"])
def test_vbs_tuned_rejects_bad_corrections(case):
    with pytest.raises(oracle.OracleError):
        oracle.balance_vbs_tuned(np.array(case["L"]), case["n"], 1.0, 0, np.array(case["delta"]))


def test_autotune_update_rejects_bad_arguments():
    for t, step, tol in (([-1, 2], 1, 0), ([1 << 53, 2], 1, 0), ([1, 2], -1, 0), ([1, 2], 1, 1000001),
                         ([1, 2], 1, -1)):
        with pytest.raises(oracle.OracleError):
            oracle.vbs_autotune(np.array(t), np.zeros(2, np.int64), step, tol)


@pytest.mark.parametrize("seed", range(6))
def test_autotune_update_invariants_random(seed):
    """What the page's rule fixes whatever the times: the global batch stays
    put, each rank moves by 0 or one step, only ranks above the average give
    samples and only ranks below it take them, in equal numbers, and those
    chosen are the most extreme ones (checked with exact fractions)."""
    from fractions import Fraction
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(1, 80))
    t = rng.integers(0, 1000 if seed % 2 else 10**12, n)
    if seed == 3:
        t = rng.integers(5, 8, n)                     # many ties
    d0 = rng.integers(-50, 50, n)
    d0[-1] -= d0.sum()
    step = int(rng.integers(1, 5))
    tol = [0, 0, 20000, 0, 100000, 0][seed]
    d1 = oracle.vbs_autotune(t, d0, step, tol)
    ch = d1 - d0
    assert d1.sum() == d0.sum()
    assert set(ch.tolist()) <= {-step, 0, step}
    mean = Fraction(int(t.sum()), n)
    slow = [r for r in range(n) if Fraction(int(t[r])) > mean * Fraction(10**6 + tol, 10**6)]
    fast = [r for r in range(n) if Fraction(int(t[r])) < mean * Fraction(10**6 - tol, 10**6)]
    lost = [r for r in range(n) if ch[r] < 0]
    gained = [r for r in range(n) if ch[r] > 0]
    assert set(lost) <= set(slow) and set(gained) <= set(fast)
    assert len(lost) == len(gained) == min(len(slow), len(fast))
    for r in set(slow) - set(lost):      # every slow rank left alone is no slower than those chosen
        assert all(t[r] < t[q] or (t[r] == t[q] and r > q) for q in lost)
    for r in set(fast) - set(gained):
        assert all(t[r] > t[q] or (t[r] == t[q] and r > q) for q in gained)


@pytest.mark.parametrize("seed,sort_by_len", [(s, b) for s in range(4) for b in (0, 1)])
def test_vbs_tuned_invariants_random(seed, sort_by_len):
    rng = np.random.default_rng(400 + seed)
    n = int(rng.integers(1, 40))
    S = int(rng.integers(1, 2000))
    L = np.clip(np.round(rng.lognormal(6, 1.4, S)), 1, 4096).astype(np.int32)
    perm0, ro0, _ = oracle.balance_vbs(L, n, 1.5, sort_by_len)
    # a zero correction is the plain cut
    perm, ro, sw = oracle.balance_vbs_tuned(L, n, 1.5, sort_by_len, np.zeros(n, np.int64))
    assert np.array_equal(perm, perm0) and np.array_equal(ro, ro0)
    # a small correction changes every count by exactly its entry
    c = np.diff(ro0)
    d = np.zeros(n, np.int64)
    for _ in range(3 * n):
        a, b = rng.integers(0, n, 2)
        if c[a] + d[a] > 0:
            d[a] -= 1
            d[b] += 1
    perm, ro, sw = oracle.balance_vbs_tuned(L, n, 1.5, sort_by_len, d)
    assert np.array_equal(perm, perm0)
    assert np.array_equal(np.diff(ro), c + d)
    w = np.array([oracle.vbs_weight(int(l), 1.5) for l in L[perm]], dtype=object)
    assert [int(x) for x in sw] == [int(sum(w[ro[r]:ro[r + 1]])) for r in range(n)]
    # a large one: contiguous, non-negative counts, every sample once
    d = rng.integers(-S, S + 1, n)
    d[-1] = 0
    d[-1] = -d.sum()
    if abs(d[-1]) <= S:
        perm, ro, sw = oracle.balance_vbs_tuned(L, n, 1.5, sort_by_len, d)
        assert ro[0] == 0 and ro[-1] == S and (np.diff(ro) >= 0).all()
        assert sum(int(x) for x in sw) == int(sum(w))


def test_autotune_balances_heterogeneous_ranks():
    """The point of AutoTune: when the weights miss a per-rank cost (here four
    ranks run 1.5x slower), repeated updates move samples off the slow ranks
    until every rank's time is close to the average."""
    from jagged_embedding_gb300 import synthetic
    n, B = 16, 128
    rng = np.random.default_rng(7)
    L = np.clip(np.round(rng.lognormal(6, 1.4, n * B)), 1, 4096).astype(np.int32)
    speed = np.where(np.arange(n) % 4 == 0, 1.5, 1.0)
    d = np.zeros(n, np.int64)

    def spread(d):
        perm, ro, _ = oracle.balance_vbs_tuned(L, n, 1.5, 0, d)
        t = synthetic.rank_times(L, perm, ro, speed, 1.5)
        return t, t.max() / t.mean()

    t, first = spread(d)
    for _ in range(120):
        d = oracle.vbs_autotune(t, d, 1, 0)
        t, last = spread(d)
    assert d.sum() == 0 and (d[::4] < 0).all()
    assert first > 1.3 and last < 1.1
