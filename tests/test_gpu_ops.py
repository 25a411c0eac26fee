"""Parity of every C-ABI call with the CPU oracle, element by element (GPU).

Bit-exact for partitions, permutations, bucketize, collision lists / masks and
gathers; toleranced (see helpers.assert_table_close) for updated embeddings.
Inputs are seeded and synthetic; sizes span several tiles plus a ragged tail.
"""
import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from jagged_embedding_gb300 import synthetic
from tests.helpers import assert_state_close, assert_table_close, to_np, update_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(err):
    B.check(err)


def _lens(rng, S, mu=5.0, sigma=1.2, lmax=2048):
    return np.clip(np.round(rng.lognormal(mu, sigma, S)), 1, lmax).astype(np.int32)


# ------------------------------------------------------------------ balance

@pytest.mark.parametrize("n,S", [(8, 512), (64, 16384), (256, 131072), (3, 12), (5, 23), (1, 100), (7, 3), (4, 0),
                                 (512, 32768), (13, 4097)])
def test_fbs_matches_oracle(n, S):
    rng = np.random.default_rng(n * 7 + S)
    L = _lens(rng, S, 6.8, 1.5, 16384)
    perm, ro, err = B.fs_balance_fbs(torch.from_numpy(L).to(DEV), n)
    _check(err)
    p_ref, ro_ref = oracle.balance_fbs(L, n)
    assert np.array_equal(to_np(perm), p_ref)
    assert np.array_equal(to_np(ro), ro_ref)


def test_fbs_ties_and_extremes():
    L = np.array([5] * 1000 + [0] * 50 + [2 ** 31 - 1] * 3 + [7] * 4000, np.int32)
    perm, ro, err = B.fs_balance_fbs(torch.from_numpy(L).to(DEV), 6)
    _check(err)
    p_ref, ro_ref = oracle.balance_fbs(L, 6)
    assert np.array_equal(to_np(perm), p_ref) and np.array_equal(to_np(ro), ro_ref)


def test_fbs_negative_length_sets_error():
    L = torch.tensor([3, -1, 4], dtype=torch.int32, device=DEV)
    _, _, err = B.fs_balance_fbs(L, 2)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 1


@pytest.mark.parametrize("n,S,sort_by_len", [(16, 2048, 0), (512, 32768, 1), (16, 2048, 1), (3, 7, 1), (1, 50, 0),
                                             (64, 20000, 0), (7, 0, 1)])
def test_vbs_matches_oracle(n, S, sort_by_len):
    rng = np.random.default_rng(n + S + sort_by_len)
    L = _lens(rng, S, 7.0, 1.6, 16384)
    perm, ro, sw, err = B.fs_balance_vbs(torch.from_numpy(L).to(DEV), n, 1.5, sort_by_len)
    _check(err)
    p_ref, ro_ref, sw_ref = oracle.balance_vbs(L, n, 1.5, sort_by_len)
    assert np.array_equal(to_np(perm), p_ref)
    assert np.array_equal(to_np(ro), ro_ref)
    assert np.array_equal(to_np(sw).astype(np.uint64), sw_ref)


@pytest.mark.parametrize("alpha", [1.5, 1.0, 2.0, 0.5, 2.5, 3.0])
def test_vbs_weight_table_exact(alpha):
    """Every L in [1, 16384] (4096 for alpha = 3), shuffled, one rank per sample: the cut and every
    segment weight (a sum of fixed-point weights) equal the oracle's bit for bit."""
    lmax = 4096 if alpha >= 3.0 else 16384            # S * max weight must stay below 2^62
    L = np.random.default_rng(1).permutation(np.arange(1, lmax + 1, dtype=np.int32))
    S = L.size
    perm, ro, sw, err = B.fs_balance_vbs(torch.from_numpy(L).to(DEV), S, alpha, 0)
    _check(err)
    p_ref, ro_ref, sw_ref = oracle.balance_vbs(L, S, alpha, 0)
    assert np.array_equal(to_np(ro), ro_ref)
    assert np.array_equal(to_np(sw).astype(np.uint64), sw_ref)


def test_vbs_general_alpha_total():
    """alpha = 1.3 goes through pow(); device and host pow may differ by an ulp, which the
    fixed-point rounding absorbs except next to a half-integer: totals within 16 units."""
    L = np.arange(1, 16385, dtype=np.int32)
    _, _, sw, err = B.fs_balance_vbs(torch.from_numpy(L).to(DEV), 1, 1.3, 0)
    _check(err)
    ref = sum(oracle.vbs_weight(int(l), 1.3) for l in L)
    assert abs(int(to_np(sw)[0]) - ref) <= 16


# ------------------------------------------------------------------ VBS AutoTune

def _autotune_gold():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "vbs_autotune_hand_examples.json")) as f:
        return json.load(f)


def test_autotune_hand_examples():
    gold = _autotune_gold()
    for c in gold["update_cases"]:
        d = torch.tensor(c["delta_in"], dtype=torch.int64, device=DEV)
        _, err = B.fs_vbs_autotune(torch.tensor(c["t"], dtype=torch.int64, device=DEV), d, c["step"], c["tol_ppm"])
        _check(err)
        assert d.tolist() == c["delta_out"], c["note"]
    for c in gold["tuned_cases"]:
        perm, ro, sw, err = B.fs_balance_vbs_tuned(torch.tensor(c["L"], dtype=torch.int32, device=DEV), c["n"],
                                                   c["alpha"], c["sort_by_len"],
                                                   torch.tensor(c["delta"], dtype=torch.int64, device=DEV))
        _check(err)
        assert to_np(perm).tolist() == c["perm"] and to_np(ro).tolist() == c["rank_offsets"], c["note"]
        assert to_np(sw).tolist() == c["seg_weight"]


@pytest.mark.parametrize("n,kind,step,tol", [(1, "wide", 1, 0), (4, "ties", 1, 0), (16, "wide", 3, 0),
                                             (512, "wide", 1, 20000), (512, "ties", 2, 0), (4097, "wide", 1, 0),
                                             (65536, "ties", 1, 5000), (65536, "wide", 7, 0)])
def test_autotune_update_matches_oracle(n, kind, step, tol):
    rng = np.random.default_rng(n + step)
    t = rng.integers(0, 2 ** 53, n) if kind == "wide" else rng.integers(1000, 1004, n)
    d0 = rng.integers(-100, 100, n)
    d0[-1] -= d0.sum()
    d = torch.from_numpy(d0).to(DEV)
    _, err = B.fs_vbs_autotune(torch.from_numpy(t).to(DEV), d, step, tol)
    _check(err)
    assert np.array_equal(to_np(d), oracle.vbs_autotune(t, d0, step, tol))


def test_autotune_bad_time_sets_error_and_keeps_delta():
    d = torch.tensor([1, -1, 0], dtype=torch.int64, device=DEV)
    for bad in (-5, 2 ** 53):
        _, err = B.fs_vbs_autotune(torch.tensor([3, bad, 4], dtype=torch.int64, device=DEV), d)
        with pytest.raises(B.FsError) as e:
            _check(err)
        assert e.value.code == 1
        assert d.tolist() == [1, -1, 0]


def _zero_sum(rng, n, lim):
    """Random corrections in [-lim, lim] that sum to 0 (entries visited in random
    order absorb the excess; their room, n * lim + |sum|, always suffices)."""
    d = rng.integers(-lim, lim + 1, n)
    s = int(d.sum())
    for i in rng.permutation(n):
        if s == 0:
            break
        c = int(np.clip(-s, -lim - d[i], lim - d[i]))
        d[i] += c
        s += c
    return d


@pytest.mark.parametrize("n,S,sort_by_len,lim", [(16, 2048, 0, 3), (16, 2048, 1, 500), (512, 32768, 1, 20),
                                                 (512, 32768, 0, 32768), (3000, 20000, 0, 4),
                                                 (3000, 20000, 1, 20000), (2048, 2048, 0, 1), (1, 50, 0, 0),
                                                 (7, 0, 1, 0)])
def test_vbs_tuned_matches_oracle(n, S, sort_by_len, lim):
    """Small corrections (each count moves by its entry) and large ones (the clamp
    and the running maximum act); n > 1024 crosses the adjustment's chunks."""
    rng = np.random.default_rng(n + S + lim)
    L = _lens(rng, S, 7.0, 1.6, 16384)
    d = _zero_sum(rng, n, lim)
    perm, ro, sw, err = B.fs_balance_vbs_tuned(torch.from_numpy(L).to(DEV), n, 1.5, sort_by_len,
                                               torch.from_numpy(d).to(DEV))
    _check(err)
    p_ref, ro_ref, sw_ref = oracle.balance_vbs_tuned(L, n, 1.5, sort_by_len, d)
    assert np.array_equal(to_np(perm), p_ref)
    assert np.array_equal(to_np(ro), ro_ref)
    assert np.array_equal(to_np(sw).astype(np.uint64), sw_ref)


def test_vbs_tuned_bad_correction_sets_error_and_keeps_cut():
    rng = np.random.default_rng(5)
    L = _lens(rng, 100)
    _, ro_plain, _ = oracle.balance_vbs(L, 4, 1.5, 0)
    for d in ([1, 0, 0, 0], [101, -101, 0, 0]):
        _, ro, _, err = B.fs_balance_vbs_tuned(torch.from_numpy(L).to(DEV), 4, 1.5, 0,
                                               torch.tensor(d, dtype=torch.int64, device=DEV))
        with pytest.raises(B.FsError) as e:
            _check(err)
        assert e.value.code == 1
        assert np.array_equal(to_np(ro), ro_plain)


@pytest.mark.parametrize("n,B_,sort_by_len", [(16, 128, 0), (512, 64, 1)])
def test_autotune_loop_matches_oracle(n, B_, sort_by_len):
    """The whole feedback loop: tuned cut -> simulated rank times -> update, on the
    device and in the oracle, iteration by iteration, a fresh batch each time."""
    rng = np.random.default_rng(n)
    speed = np.where(np.arange(n) % 4 == 0, 1.5, 1.0)
    d_dev = torch.zeros(n, dtype=torch.int64, device=DEV)
    d_ref = np.zeros(n, np.int64)
    for it in range(25):
        L = _lens(rng, n * B_, 7.0, 1.6, 16384)
        perm, ro, _, err = B.fs_balance_vbs_tuned(torch.from_numpy(L).to(DEV), n, 1.5, sort_by_len, d_dev)
        _check(err)
        p_ref, ro_ref, _ = oracle.balance_vbs_tuned(L, n, 1.5, sort_by_len, d_ref)
        assert np.array_equal(to_np(perm), p_ref) and np.array_equal(to_np(ro), ro_ref), it
        t = synthetic.rank_times(L, p_ref, ro_ref, speed, 1.5)
        _, err = B.fs_vbs_autotune(torch.from_numpy(t).to(DEV), d_dev, 1, 0)
        _check(err)
        d_ref = oracle.vbs_autotune(t, d_ref, 1, 0)
        assert np.array_equal(to_np(d_dev), d_ref), it
    if not sort_by_len:
        assert (d_ref[::4] < 0).all()             # the slow ranks have given samples away


# ------------------------------------------------------------------ permute

def _jagged(rng, S, R, mu=5.0, sigma=1.2, lmax=2048):
    lens = _lens(rng, S, mu, sigma, lmax).astype(np.int64)
    off = np.zeros(S + 1, np.int64)
    off[1:] = np.cumsum(lens)
    ids = rng.integers(0, R, int(off[-1])).astype(np.int64)
    return off, ids


@pytest.mark.parametrize("S", [1, 7, 512, 4096, 16384, 40000])
def test_permute_matches_oracle(S):
    rng = np.random.default_rng(S)
    off, ids = _jagged(rng, S, 10 ** 6)
    perm = rng.permutation(S).astype(np.int32)
    n = max(1, S // 64)
    cuts = np.sort(rng.integers(0, S + 1, n - 1))
    ro = np.concatenate([[0], cuts, [S]]).astype(np.int64)
    o2, v2, rio, err = B.fs_permute_jagged(torch.from_numpy(off).to(DEV), torch.from_numpy(ids).to(DEV),
                                           torch.from_numpy(perm).to(DEV), rank_offsets=torch.from_numpy(ro).to(DEV))
    _check(err)
    o_ref, v_ref = oracle.permute_jagged(off, ids, perm)
    assert np.array_equal(to_np(o2), o_ref) and np.array_equal(to_np(v2), v_ref)
    assert np.array_equal(to_np(rio), o_ref[ro])


def test_permute_with_empty_samples_and_long_samples():
    rng = np.random.default_rng(3)
    S = 3000
    lens = rng.integers(0, 3, S).astype(np.int64)
    lens[rng.integers(0, S, 20)] = 16384          # a few very long samples span many copy tiles
    lens[:100] = 0
    off = np.zeros(S + 1, np.int64)
    off[1:] = np.cumsum(lens)
    ids = rng.integers(0, 1 << 40, int(off[-1])).astype(np.int64)
    perm = rng.permutation(S).astype(np.int32)
    o2, v2, _, err = B.fs_permute_jagged(torch.from_numpy(off).to(DEV), torch.from_numpy(ids).to(DEV),
                                         torch.from_numpy(perm).to(DEV))
    _check(err)
    o_ref, v_ref = oracle.permute_jagged(off, ids, perm)
    assert np.array_equal(to_np(o2), o_ref) and np.array_equal(to_np(v2), v_ref)


def test_permute_many_short_samples_per_tile_with_rank_offsets():
    """Tiles covering many short samples (and runs of empty ones) next to long samples, through the
    ID-balanced copy (rank offsets requested)."""
    rng = np.random.default_rng(17)
    S = 60000
    lens = rng.integers(0, 7, S).astype(np.int64)
    lens[rng.integers(0, S, 30)] = 9000
    off = np.zeros(S + 1, np.int64)
    off[1:] = np.cumsum(lens)
    ids = rng.integers(0, 1 << 40, int(off[-1])).astype(np.int64)
    perm = np.argsort(lens, kind="stable").astype(np.int32)       # short samples first, as a sorted VBS order
    ro = np.linspace(0, S, 9).round().astype(np.int64)
    o2, v2, rio, err = B.fs_permute_jagged(torch.from_numpy(off).to(DEV), torch.from_numpy(ids).to(DEV),
                                           torch.from_numpy(perm).to(DEV), rank_offsets=torch.from_numpy(ro).to(DEV))
    _check(err)
    o_ref, v_ref = oracle.permute_jagged(off, ids, perm)
    assert np.array_equal(to_np(o2), o_ref) and np.array_equal(to_np(v2), v_ref)
    assert np.array_equal(to_np(rio), o_ref[ro])


def test_permute_errors():
    off = torch.tensor([0, 2, 5], dtype=torch.int64, device=DEV)
    val = torch.arange(5, dtype=torch.int64, device=DEV)
    _, _, _, err = B.fs_permute_jagged(off, val, torch.tensor([0, 2], dtype=torch.int32, device=DEV))
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 3
    _, _, _, err = B.fs_permute_jagged(off, val, torch.tensor([1, 0], dtype=torch.int32, device=DEV), capacity=4)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 4


def test_permute_empty_batch():
    off = torch.zeros(1, dtype=torch.int64, device=DEV)
    o2, v2, rio, err = B.fs_permute_jagged(off, torch.zeros(0, dtype=torch.int64, device=DEV),
                                           torch.zeros(0, dtype=torch.int32, device=DEV),
                                           rank_offsets=torch.zeros(4, dtype=torch.int64, device=DEV))
    _check(err)
    assert to_np(o2).tolist() == [0] and to_np(rio).tolist() == [0, 0, 0, 0]


# ------------------------------------------------------------------ keyed transpose

@pytest.mark.parametrize("F,nb,maxlen,base", [(3, 1000, 40, False), (26, 4096, 12, True), (1, 5000, 30, True),
                                               (8, 1, 20000, False), (64, 700, 3, True), (5, 0, 1, False)])
def test_keyed_transpose_matches_oracle(F, nb, maxlen, base):
    """F features x nb samples."""
    rng = np.random.default_rng(F * 7919 + nb)
    lens = rng.integers(0, maxlen + 1, F * nb)
    off = np.zeros(F * nb + 1, np.int64)
    off[1:] = np.cumsum(lens)
    val = rng.integers(0, 1 << 40, int(off[-1])).astype(np.int64)
    rb = rng.integers(0, 1 << 20, F).astype(np.int64) if base else None
    o2, v2, err = B.fs_keyed_transpose(torch.from_numpy(off).to(DEV), torch.from_numpy(val).to(DEV), F, nb,
                                       row_base=None if rb is None else torch.from_numpy(rb).to(DEV))
    _check(err)
    o_ref, v_ref = oracle.keyed_transpose(off, val, F, nb, rb)
    assert np.array_equal(to_np(o2), o_ref) and np.array_equal(to_np(v2), v_ref)


def test_keyed_transpose_errors():
    off = torch.tensor([0, 2, 1, 3], dtype=torch.int64, device=DEV)          # decreasing: bad offsets
    val = torch.arange(3, dtype=torch.int64, device=DEV)
    _, _, err = B.fs_keyed_transpose(off, val, 3, 1)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 3
    off = torch.tensor([0, 2, 5], dtype=torch.int64, device=DEV)
    _, _, err = B.fs_keyed_transpose(off, torch.arange(5, dtype=torch.int64, device=DEV), 2, 1, capacity=4)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 4


# ------------------------------------------------------------------ bucketize

@pytest.mark.parametrize("n,R,T", [(8, 100_000, 150_000), (64, 10_000_000, 500_000), (512, 50_000_000, 300_001),
                                   (256, 100_000_000, 70_000), (1, 1000, 5000), (13, 12, 4097), (7, 100, 0)])
def test_bucketize_matches_oracle(n, R, T):
    rng = np.random.default_rng(n + T)
    ids = rng.integers(0, R, T).astype(np.int64)
    cuts = np.sort(rng.integers(0, T + 1, n - 1))
    rio = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    sm, pos, splits, so, err = B.fs_bucketize_rowwise(torch.from_numpy(ids).to(DEV), torch.from_numpy(rio).to(DEV), R)
    _check(err)
    sm_ref, pos_ref, splits_ref, so_ref = oracle.bucketize_rowwise(ids, rio, n, R)
    assert np.array_equal(to_np(sm), sm_ref)
    assert np.array_equal(to_np(pos), pos_ref)
    assert np.array_equal(to_np(splits), splits_ref)
    assert np.array_equal(to_np(so), so_ref)


def test_bucketize_zipf_hot_rows():
    w = synthetic.WORKLOADS["mid-full-step"]
    rng = torch.Generator(device="cpu").manual_seed(5)
    ids = synthetic.zipf_rows(w.R, w.zipf_s, 400_000, rng, "cpu")
    n = w.n
    rio = np.linspace(0, ids.numel(), n + 1).astype(np.int64)
    sm, pos, splits, so, err = B.fs_bucketize_rowwise(ids.to(DEV), torch.from_numpy(rio).to(DEV), w.R)
    _check(err)
    sm_ref, pos_ref, splits_ref, so_ref = oracle.bucketize_rowwise(ids.numpy(), rio, n, w.R)
    assert np.array_equal(to_np(sm), sm_ref) and np.array_equal(to_np(pos), pos_ref)
    assert np.array_equal(to_np(splits), splits_ref)


def test_bucketize_id_out_of_range():
    ids = torch.tensor([1, 5, 100], dtype=torch.int64, device=DEV)
    rio = torch.tensor([0, 3], dtype=torch.int64, device=DEV)
    *_, err = B.fs_bucketize_rowwise(ids, rio, 50)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 2


# ------------------------------------------------------------------ collision

@pytest.mark.parametrize("R,n,Tt,Tn", [(100_000, 8, 70_000, 80_000), (20, 4, 6, 6), (10_000_000, 64, 300_000, 250_000),
                                       (100_000_000, 256, 200_000, 200_000), (50_000_000, 512, 0, 1000),
                                       (33, 5, 1000, 0), (1_000_003, 7, 123_457, 98_765)])
def test_collision_matches_oracle(R, n, Tt, Tn):
    rng = np.random.default_rng(R + Tt)
    a = rng.integers(0, R, Tt).astype(np.int64)
    b = rng.integers(0, R, Tn).astype(np.int64)
    if Tt and Tn:
        b[: Tn // 2] = a[rng.integers(0, Tt, Tn // 2)]      # plenty of collisions
    out, err = B.fs_collision_split(torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV), R, n)
    _check(err)
    ref = oracle.collision_split(a, b, R, n)
    counts = to_np(out["counts"])
    assert counts.tolist() == [ref["co"].size, ref["ex_t"].size, ref["ex_next"].size]
    for k, c in (("co", 0), ("ex_t", 1), ("ex_next", 2)):
        assert np.array_equal(to_np(out[k])[: counts[c]], ref[k]), k
        assert np.array_equal(to_np(out[k + "_off"]), ref[k + "_off"]), k
    assert np.array_equal(to_np(out["is_co_t"]), ref["is_co_t"])
    assert np.array_equal(to_np(out["is_co_next"]), ref["is_co_next"])


@pytest.mark.parametrize("R,n,Tt,Tn", [(100_000, 8, 70_000, 80_000), (50_000_000, 512, 300_000, 0),
                                       (1_000_003, 7, 123_457, 98_765)])
def test_collision_from_bitmaps_matches_oracle(R, n, Tt, Tn):
    rng = np.random.default_rng(R + Tn)
    a = rng.integers(0, R, Tt).astype(np.int64)
    b = rng.integers(0, R, Tn).astype(np.int64)
    if Tt and Tn:
        b[: Tn // 2] = a[rng.integers(0, Tt, Tn // 2)]
    ad, bd = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    bm_a, err = B.fs_row_bitmap(ad, R)
    bm_b, _ = B.fs_row_bitmap(bd, R, err=err)
    _check(err)
    # bitmap = the set of rows, bit r % 32 of word r / 32
    words = to_np(bm_a).view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:R]
    assert np.array_equal(np.flatnonzero(bits), np.unique(a))
    cap = Tt + Tn
    out = {k: torch.empty(cap, dtype=torch.int64, device=DEV) for k in ("co", "ex_t", "ex_next")}
    out.update({"counts": torch.empty(3, dtype=torch.int64, device=DEV),
                "co_off": torch.empty(n + 1, dtype=torch.int64, device=DEV),
                "ex_t_off": torch.empty(n + 1, dtype=torch.int64, device=DEV),
                "ex_next_off": torch.empty(n + 1, dtype=torch.int64, device=DEV),
                "is_co_t": torch.empty(Tt, dtype=torch.uint8, device=DEV),
                "is_co_next": torch.empty(Tn, dtype=torch.uint8, device=DEV)})
    B.fs_collision_split_bitmaps(ad, bm_a, bd, bm_b, R, n, out, cap, err=err)
    _check(err)
    ref = oracle.collision_split(a, b, R, n)
    counts = to_np(out["counts"])
    for k, c in (("co", 0), ("ex_t", 1), ("ex_next", 2)):
        assert np.array_equal(to_np(out[k])[: counts[c]], ref[k]), k
        assert np.array_equal(to_np(out[k + "_off"]), ref[k + "_off"]), k
    assert np.array_equal(to_np(out["is_co_t"]), ref["is_co_t"])
    assert np.array_equal(to_np(out["is_co_next"]), ref["is_co_next"])


def test_collision_single_mask():
    """Either mask may be omitted; the other one is unchanged."""
    rng = np.random.default_rng(77)
    R = 500_000
    a = rng.integers(0, R, 200_000).astype(np.int64)
    b = rng.integers(0, R, 150_000).astype(np.int64)
    ref = oracle.collision_split(a, b, R, 16)
    out, err = B.fs_collision_split(torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV), R, 16,
                                    want_next_mask=False)
    _check(err)
    assert np.array_equal(to_np(out["is_co_t"]), ref["is_co_t"])
    assert np.array_equal(to_np(out["co"])[: to_np(out["counts"])[0]], ref["co"])


def test_collision_capacity_error():
    a = torch.arange(100, dtype=torch.int64, device=DEV)
    out, err = B.fs_collision_split(a, a.flip(0).contiguous(), 1000, 4, cap_rows=10)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 4


# ------------------------------------------------------------------ gather

@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 128), ("f32", 128), ("f32", 3), ("bf16", 6), ("f32", 20),
                                     ("bf16", 8), ("f32", 512), ("f32", 1024), ("bf16", 32)])
def test_gather_bit_exact(dtype, D):
    rng = np.random.default_rng(D)
    R, T = 5000, 77_777
    tt = torch.float32 if dtype == "f32" else torch.bfloat16
    table = torch.randn(R, D, generator=torch.Generator().manual_seed(1)).to(tt)
    ids = rng.integers(0, R, T).astype(np.int64)
    out, err = B.fs_emb_gather(table.to(DEV), torch.from_numpy(ids).to(DEV))
    _check(err)
    ref = oracle.emb_gather(to_np(table), ids)
    assert np.array_equal(to_np(out), ref)


def test_gather_masked_merge():
    rng = np.random.default_rng(9)
    R, D, T = 3000, 64, 50_000
    table = torch.randn(R, D, generator=torch.Generator().manual_seed(2))
    ids = rng.integers(0, R, T).astype(np.int64)
    mask = rng.integers(0, 2, T).astype(np.uint8)
    out = torch.full((T, D), -3.5, device=DEV)
    tdev, idev, mdev = table.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(mask).to(DEV)
    _, err = B.fs_emb_gather(tdev, idev, out=out, mask=mdev, sel=0)
    _check(err)
    got = to_np(out)
    assert np.array_equal(got[mask == 0], to_np(table)[ids[mask == 0]])
    assert (got[mask == 1] == -3.5).all()
    B.fs_emb_gather(tdev, idev, out=out, mask=mdev, sel=1, err=err)
    _check(err)
    assert np.array_equal(to_np(out), to_np(table)[ids])


def test_gather_bad_id():
    _, err = B.fs_emb_gather(torch.zeros(10, 64, device=DEV), torch.tensor([3, 10], dtype=torch.int64, device=DEV))
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 2


# ------------------------------------------------------------------ backward

def _bwd_case(seed, R, D, T, dtype, s=1.1):
    g = torch.Generator().manual_seed(seed)
    ids = synthetic.zipf_rows(R, s, T, g, "cpu")
    tt = torch.float32 if dtype == "f32" else torch.bfloat16
    W = (torch.randn(R, D, generator=g) * 0.01).to(tt)
    G = torch.randn(T, D, generator=g).to(tt)
    return ids, W, G


@pytest.mark.parametrize("dtype,D,optim,T,R", [
    ("f32", 64, "sgd", 150_000, 100_000),
    ("f32", 64, "adagrad", 300_000, 1_000_000),
    ("bf16", 128, "adagrad", 200_000, 10_000_000),
    ("f32", 32, "adagrad", 50_000, 3000),
    ("f32", 128, "sgd", 40_000, 100),
    ("bf16", 64, "sgd", 60_000, 70_000),
    ("bf16", 256, "adagrad", 20_000, 5000),
    ("f32", 64, "adagrad", 5, 10),
])
def test_backward_matches_oracle(dtype, D, optim, T, R):
    ids, W, G = _bwd_case(T + D, R, D, T, dtype)
    state = torch.rand(R, generator=torch.Generator().manual_seed(3)) if optim == "adagrad" else None
    Wd = W.to(DEV)
    sd = state.to(DEV) if state is not None else None
    err = B.fs_emb_backward_adagrad(Wd, sd, ids.to(DEV), G.to(DEV), optim, 0.01, 1e-8)
    _check(err)
    W_ref = to_np(W)
    s_ref = state.numpy().copy() if state is not None else None
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), optim, 0.01, 1e-8)
    scale = update_scale(ids.numpy(), to_np(G), R, optim, 0.01, 1e-8, s_ref)
    assert_table_close(to_np(Wd), W_ref, dtype, 0.01, scale=scale)
    if state is not None:
        assert_state_close(to_np(sd), s_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_phases_and_determinism(dtype):
    R, D, T = 200_000, 64 if dtype == "f32" else 128, 250_000
    ids, W, G = _bwd_case(11, R, D, T, dtype, s=1.05)
    rng = np.random.default_rng(4)
    nxt = synthetic.zipf_rows(R, 1.05, 200_000, torch.Generator().manual_seed(12), "cpu").numpy()
    is_co = np.isin(ids.numpy(), nxt).astype(np.uint8)
    results = []
    for _ in range(2):
        Wd, sd = W.to(DEV), torch.zeros(R, device=DEV)
        idd, Gd, md = ids.to(DEV), G.to(DEV), torch.from_numpy(is_co).to(DEV)
        err = B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8, is_co=md, phase=B.PHASE_COLLISION)
        B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8, is_co=md, phase=B.PHASE_EXCLUSIVE, err=err)
        _check(err)
        results.append((to_np(Wd), to_np(sd)))
    assert np.array_equal(results[0][0], results[1][0]) and np.array_equal(results[0][1], results[1][1])
    W_ref, s_ref = to_np(W), np.zeros(R, np.float32)
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), "adagrad", 0.01, 1e-8, is_co=is_co, phase=1)
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), "adagrad", 0.01, 1e-8, is_co=is_co, phase=2)
    assert_table_close(results[0][0], W_ref, dtype, 0.01)
    assert_state_close(results[0][1], s_ref)


@pytest.mark.parametrize("dtype,R", [("f32", 200_000), ("bf16", 3_000_000), ("f32", 100_000_000)])
def test_backward_both_phases_in_one_call_equals_two_calls(dtype, R):
    """COLLISION_THEN_EXCLUSIVE (one sort, phase in the key's top bit) gives the same
    bits as a COLLISION call followed by an EXCLUSIVE call."""
    D, T = (64 if dtype == "f32" else 128), 300_000
    g = torch.Generator().manual_seed(31)
    ids = synthetic.zipf_rows(R, 1.05, T, g, "cpu")
    tt = torch.float32 if dtype == "f32" else torch.bfloat16
    rows = torch.unique(ids)
    W0 = (torch.randn(R, D, generator=g) * 0.01).to(tt)
    G = torch.randn(T, D, generator=g).to(tt)
    is_co = (torch.rand(rows.numel(), generator=g) < 0.5).to(torch.uint8)
    mask = is_co[torch.searchsorted(rows, ids)].contiguous()
    outs = []
    for mode in ("one", "two"):
        Wd, sd = W0.to(DEV), torch.zeros(R, device=DEV)
        idd, Gd, md = ids.to(DEV), G.to(DEV), mask.to(DEV)
        if mode == "one":
            err = B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8, is_co=md,
                                            phase=B.PHASE_COLLISION_THEN_EXCLUSIVE)
        else:
            err = B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8, is_co=md, phase=B.PHASE_COLLISION)
            B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8, is_co=md, phase=B.PHASE_EXCLUSIVE,
                                      err=err)
        _check(err)
        outs.append((Wd[rows.to(DEV)].cpu(), sd[rows.to(DEV)].cpu()))
    assert torch.equal(outs[0][0].view(torch.int16) if dtype == "bf16" else outs[0][0],
                       outs[1][0].view(torch.int16) if dtype == "bf16" else outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("dtype,D", [("f32", 32), ("bf16", 64)])
def test_backward_rows_not_16_byte_aligned(dtype, D):
    """Gradient rows that start 4 bytes past a 16-byte boundary take the
    narrow-load reduce (the wide one needs 16-byte rows); same result bar."""
    R, T = 40_000, 120_000
    ids, W, G = _bwd_case(5, R, D, T, dtype)
    state = torch.rand(R, generator=torch.Generator().manual_seed(8))
    Wd, sd = W.to(DEV), state.to(DEV)
    shift = 4 // G.element_size()
    flat = torch.empty(T * D + shift, dtype=G.dtype, device=DEV)
    Gd = flat[shift:].view(T, D)
    Gd.copy_(G.to(DEV))
    assert Gd.data_ptr() % 16 == 4
    err = B.fs_emb_backward_adagrad(Wd, sd, ids.to(DEV), Gd, "adagrad", 0.01, 1e-8)
    _check(err)
    W_ref, s_ref = to_np(W), state.numpy().copy()
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), "adagrad", 0.01, 1e-8)
    scale = update_scale(ids.numpy(), to_np(G), R, "adagrad", 0.01, 1e-8, s_ref)
    assert_table_close(to_np(Wd), W_ref, dtype, 0.01, scale=scale)
    assert_state_close(to_np(sd), s_ref)


@pytest.mark.parametrize("dtype,phase", [("f32", 3), ("bf16", 3), ("f32", 1), ("f32", 2)])
def test_backward_phase_from_row_bitmap_equals_mask(dtype, phase):
    """Collision flags read per row from a bitmap give the same bits as the per-position mask."""
    R, D, T = 500_000, (64 if dtype == "f32" else 128), 400_000
    g = torch.Generator().manual_seed(41)
    ids = synthetic.zipf_rows(R, 1.05, T, g, "cpu")
    nxt = synthetic.zipf_rows(R, 1.05, 300_000, g, "cpu")
    tt = torch.float32 if dtype == "f32" else torch.bfloat16
    W0 = (torch.randn(R, D, generator=g) * 0.01).to(tt)
    G = torch.randn(T, D, generator=g).to(tt)
    bm, err = B.fs_row_bitmap(nxt.to(DEV), R)                      # rows of the next batch
    _check(err)
    mask = torch.from_numpy(np.isin(ids.numpy(), nxt.numpy()).astype(np.uint8))
    outs = []
    for kw in ({"is_co": mask.to(DEV)}, {"co_rows": bm}):
        Wd, sd = W0.to(DEV), torch.zeros(R, device=DEV)
        err = B.fs_emb_backward_adagrad(Wd, sd, ids.to(DEV), G.to(DEV), "adagrad", 0.01, 1e-8, phase=phase, **kw)
        _check(err)
        outs.append((Wd.cpu(), sd.cpu()))
    view = (lambda x: x.view(torch.int16)) if dtype == "bf16" else (lambda x: x)
    assert torch.equal(view(outs[0][0]), view(outs[1][0]))
    assert torch.equal(outs[0][1], outs[1][1])


def test_backward_single_hot_row_spans_many_tiles():
    """One row owns most positions: its sum crosses hundreds of reduce tiles (carry chain)."""
    R, D, T = 1000, 64, 1_000_000
    g = torch.Generator().manual_seed(21)
    ids = torch.where(torch.rand(T, generator=g) < 0.9, torch.tensor(7), torch.randint(0, R, (T,), generator=g))
    W = torch.randn(R, D, generator=g) * 0.01
    G = torch.randn(T, D, generator=g)
    s = torch.zeros(R)
    Wd, sd = W.to(DEV), s.to(DEV)
    err = B.fs_emb_backward_adagrad(Wd, sd, ids.to(DEV), G.to(DEV), "adagrad", 0.01, 1e-8)
    _check(err)
    W_ref, s_ref = W.numpy().copy(), s.numpy().copy()
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), G.numpy(), "adagrad", 0.01, 1e-8)
    assert_table_close(to_np(Wd), W_ref, "f32", 0.01)
    assert_state_close(to_np(sd), s_ref)


def test_backward_rejects_unsupported_dim():
    with pytest.raises(B.FsError):
        B.fs_emb_backward_adagrad(torch.zeros(10, 48, device=DEV), torch.zeros(10, device=DEV),
                                  torch.zeros(4, dtype=torch.int64, device=DEV), torch.zeros(4, 48, device=DEV),
                                  "adagrad", 0.01, 1e-8)


# ------------------------------------------------------------------ bounded waits

def test_lookback_wait_gives_up_with_timeout_status():
    """A scan tile that never publishes: later tiles stop waiting and report FS_ERR_TIMEOUT."""
    rng = np.random.default_rng(0)
    S = 40_000                                             # 20 scan tiles of 2048
    L = _lens(rng, S)
    B.set_spin_limit(1 << 14)
    B.debug_skip_publish(3)
    try:
        _, _, _, err = B.fs_balance_vbs(torch.from_numpy(L).to(DEV), 16, 1.5, 0)
        with pytest.raises(B.FsError) as e:
            _check(err)
        assert e.value.code == 6
    finally:
        B.debug_skip_publish(-1)
        B.set_spin_limit(1 << 22)
    # the context is still usable
    _, _, _, err = B.fs_balance_vbs(torch.from_numpy(L).to(DEV), 16, 1.5, 0)
    _check(err)


def test_gradient_copy_wait_gives_up_with_timeout_status():
    """A gradient stage that is never copied: the update's wait for it runs out,
    the call reports FS_ERR_TIMEOUT, and the context stays usable."""
    R, D, T = 5000, 64, 40_000                              # 20 sorted tiles of 2048
    ids, W, G = _bwd_case(9, R, D, T, "f32")
    Wd, sd, idd, Gd = W.to(DEV), torch.zeros(R, device=DEV), ids.to(DEV), G.to(DEV)
    assert Gd.data_ptr() % 16 == 0                         # the bulk-copy path
    B.set_spin_limit(1 << 14)
    B.debug_skip_publish(2)
    try:
        err = B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8)
        with pytest.raises(B.FsError) as e:
            _check(err)
        assert e.value.code == 6
    finally:
        B.debug_skip_publish(-1)
        B.set_spin_limit(1 << 22)
    Wd, sd = W.to(DEV), torch.zeros(R, device=DEV)
    err = B.fs_emb_backward_adagrad(Wd, sd, idd, Gd, "adagrad", 0.01, 1e-8)
    _check(err)
    W_ref, s_ref = to_np(W), np.zeros(R, np.float32)
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), "adagrad", 0.01, 1e-8)
    assert_table_close(to_np(Wd), W_ref, "f32", 0.01)


# ------------------------------------------------------------------ row-sorted path

def _sorted_ws(W, T):
    R, D = W.shape
    return B.workspace(B.backward_workspace_size(T, R, D, B.dtype_code(W)), W.device)


@pytest.mark.parametrize("dtype,D,T,R,phase", [
    ("f32", 64, 300_000, 1_000_000, "all"), ("f32", 64, 250_000, 200_000, "mask"),
    ("bf16", 128, 200_000, 10_000_000, "mask"), ("bf16", 128, 70_001, 5000, "bitmap"),
    ("f32", 32, 50_000, 3000, "all"), ("f32", 128, 40_000, 100, "mask"), ("bf16", 64, 60_000, 70_000, "all"),
    ("bf16", 256, 20_000, 5000, "bitmap"), ("f32", 64, 5, 10, "mask"), ("bf16", 32, 1, 1, "all"),
])
def test_gather_sorted_matches_oracle(dtype, D, T, R, phase):
    """out[p] = W[ids[p]] from the update's sorted entries, bit for bit, for every row size the update
    takes, with the phase bit in the keys or not; several tiles and a ragged tail."""
    ids, W, _ = _bwd_case(T + 7 * D, R, D, T, dtype)
    nxt = synthetic.zipf_rows(R, 1.1, max(T // 2, 1), torch.Generator().manual_seed(T), "cpu").numpy()
    is_co = np.isin(ids.numpy(), nxt).astype(np.uint8)
    Wd, idd = W.to(DEV), ids.to(DEV)
    ws = _sorted_ws(Wd, T)
    kw = {}
    ph = B.PHASE_ALL
    if phase == "mask":
        kw, ph = {"is_co": torch.from_numpy(is_co).to(DEV)}, B.PHASE_COLLISION_THEN_EXCLUSIVE
    elif phase == "bitmap":
        bm = np.zeros((R + 31) // 32, np.uint32)
        np.bitwise_or.at(bm, nxt >> 5, (np.uint32(1) << (nxt & 31).astype(np.uint32)))
        kw, ph = {"co_rows": torch.from_numpy(bm.view(np.int32)).to(DEV)}, B.PHASE_COLLISION_THEN_EXCLUSIVE
    err = B.fs_emb_sort_rows(Wd, idd, ws, phase=ph, **kw)
    out, _ = B.fs_emb_gather_sorted(Wd, T, ws, phase=ph, err=err)
    _check(err)
    assert np.array_equal(to_np(out), oracle.emb_gather(to_np(W), ids.numpy()))


@pytest.mark.parametrize("dtype,D,optim,T,R,phase", [
    ("f32", 64, "adagrad", 300_000, 1_000_000, "mask"), ("bf16", 128, "adagrad", 200_000, 10_000_000, "bitmap"),
    ("f32", 32, "sgd", 50_000, 3000, "all"), ("bf16", 256, "adagrad", 20_000, 5000, "mask"),
])
def test_update_sorted_equals_one_call_update(dtype, D, optim, T, R, phase):
    """sort + gather + update from the sorted entries leaves table and state bit-identical to the one-call
    update (same sort, same reduce order), and within tolerance of the oracle."""
    ids, W, G = _bwd_case(T + D, R, D, T, dtype, s=1.05)
    nxt = synthetic.zipf_rows(R, 1.05, T, torch.Generator().manual_seed(D), "cpu").numpy()
    is_co = np.isin(ids.numpy(), nxt).astype(np.uint8)
    kw, ph = {}, B.PHASE_ALL
    if phase == "mask":
        kw, ph = {"is_co": torch.from_numpy(is_co).to(DEV)}, B.PHASE_COLLISION_THEN_EXCLUSIVE
    elif phase == "bitmap":
        bm = np.zeros((R + 31) // 32, np.uint32)
        np.bitwise_or.at(bm, nxt >> 5, (np.uint32(1) << (nxt & 31).astype(np.uint32)))
        kw, ph = {"co_rows": torch.from_numpy(bm.view(np.int32)).to(DEV)}, B.PHASE_COLLISION_THEN_EXCLUSIVE
    state = torch.rand(R, generator=torch.Generator().manual_seed(3)) if optim == "adagrad" else None
    idd, Gd = ids.to(DEV), G.to(DEV)
    W1, s1 = W.to(DEV), (state.to(DEV) if state is not None else None)
    W2, s2 = W.to(DEV), (state.to(DEV) if state is not None else None)
    err = B.fs_emb_backward_adagrad(W1, s1, idd, Gd, optim, 0.01, 1e-8, phase=ph, **kw)
    ws = _sorted_ws(W2, T)
    B.fs_emb_sort_rows(W2, idd, ws, phase=ph, err=err, **kw)
    out, _ = B.fs_emb_gather_sorted(W2, T, ws, phase=ph, err=err)
    B.fs_emb_update_sorted(W2, s2, Gd, T, ws, optim, 0.01, 1e-8, phase=ph, err=err)
    _check(err)
    assert np.array_equal(to_np(out), to_np(W)[ids.numpy()])        # the gather saw the table before the update
    assert np.array_equal(to_np(W1), to_np(W2))
    if state is not None:
        assert np.array_equal(to_np(s1), to_np(s2))
    W_ref = to_np(W)
    s_ref = state.numpy().copy() if state is not None else None
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), optim, 0.01, 1e-8)
    scale = update_scale(ids.numpy(), to_np(G), R, optim, 0.01, 1e-8, s_ref)
    assert_table_close(to_np(W2), W_ref, dtype, 0.01, scale=scale)


def test_gather_sorted_skips_unsorted_positions():
    """A position the sort drops (an ID out of range: FS_ERR_ID_RANGE; a flag byte above 1) keeps its
    output row; every other position gets its table row."""
    R, D, T = 1000, 64, 5000
    ids, W, _ = _bwd_case(9, R, D, T, "f32")
    ids = ids.clone()
    ids[17] = R + 5
    m = torch.zeros(T, dtype=torch.uint8)
    m[::3] = 1
    m[100] = 2
    Wd = W.to(DEV)
    ws = _sorted_ws(Wd, T)
    out = torch.full((T, D), -7.0, device=DEV)
    err = B.fs_emb_sort_rows(Wd, ids.to(DEV), ws, phase=B.PHASE_COLLISION_THEN_EXCLUSIVE, is_co=m.to(DEV))
    B.fs_emb_gather_sorted(Wd, T, ws, out=out, phase=B.PHASE_COLLISION_THEN_EXCLUSIVE, err=err)
    with pytest.raises(B.FsError) as e:
        _check(err)
    assert e.value.code == 2
    o = to_np(out)
    keep = np.ones(T, bool)
    keep[[17, 100]] = False
    assert (o[~keep] == -7.0).all()
    assert np.array_equal(o[keep], to_np(W)[ids.numpy()[keep]])


def test_sorted_calls_refuse_partial_phases_and_misalignment():
    R, D, T = 100, 64, 10
    ids, W, G = _bwd_case(1, R, D, T, "f32")
    Wd, idd = W.to(DEV), ids.to(DEV)
    ws = _sorted_ws(Wd, T)
    m = torch.zeros(T, dtype=torch.uint8, device=DEV)
    for ph in (B.PHASE_COLLISION, B.PHASE_EXCLUSIVE):
        with pytest.raises(B.FsError) as e:
            B.fs_emb_sort_rows(Wd, idd, ws, phase=ph, is_co=m)
        assert e.value.code == 1
    B.fs_emb_sort_rows(Wd, idd, ws)
    out = torch.empty(T * D + 1, device=DEV)[1:].view(T, D)               # 4-byte aligned only
    with pytest.raises(B.FsError) as e:
        B.fs_emb_gather_sorted(Wd, T, ws, out=out)
    assert e.value.code == 8
    with pytest.raises(B.FsError) as e:                                    # workspace too small
        B.fs_emb_gather_sorted(Wd, T, ws[:16])
    assert e.value.code == 5


@pytest.mark.parametrize("n,R,T", [(256, (1 << 33) + 12_345, 300_000), (7, (1 << 32) + 1, 50_001)])
def test_bucketize_tables_of_2_32_rows_or_more(n, R, T):
    """Tables of 2^32 rows or more keep the 64-bit staging (rows do not fit 32 bits); same parity."""
    rng = np.random.default_rng(n + 11)
    ids = rng.integers(0, R, T).astype(np.int64)
    ids[: T // 10] = rng.integers((1 << 32) - 5, min(R, (1 << 32) + 5), T // 10)   # rows around 2^32
    cuts = np.sort(rng.integers(0, T + 1, n - 1))
    rio = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    sm, pos, splits, so, err = B.fs_bucketize_rowwise(torch.from_numpy(ids).to(DEV), torch.from_numpy(rio).to(DEV), R)
    _check(err)
    sm_ref, pos_ref, splits_ref, so_ref = oracle.bucketize_rowwise(ids, rio, n, R)
    assert np.array_equal(to_np(sm), sm_ref)
    assert np.array_equal(to_np(pos), pos_ref)
    assert np.array_equal(to_np(splits), splits_ref)
    assert np.array_equal(to_np(so), so_ref)
