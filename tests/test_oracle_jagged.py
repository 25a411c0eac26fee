"""Pins of the oracle's jagged permute, row-wise bucketize and collision split (CPU only).

FreeScale (arXiv 2604.24073): §3.1 Algorithm 1 Stage III (sample shuffle),
§3.2 (batch-major / shard-major forms), Algorithm 2 lines 8 and 10, §4.2
(indexed permute, ranged dispatch).  Checks: hand-worked fixtures, library
stable sorts, Python set brute force and counting identities.
"""
import bisect
import json
import os

import numpy as np
import pytest

import oracle
from jagged_embedding_gb300 import synthetic

GOLD = os.path.join(os.path.dirname(__file__), "golden")
with open(os.path.join(GOLD, "jagged_hand_examples.json")) as f:
    HAND = json.load(f)


def _rand_jagged(rng, S, R, maxlen=40):
    lens = rng.integers(0, maxlen, S)
    off = np.zeros(S + 1, np.int64)
    off[1:] = np.cumsum(lens)
    ids = rng.integers(0, R, int(off[-1])).astype(np.int64)
    return off, ids


# ------------------------------------------------------------------ permute

def test_permute_hand_example():
    h = HAND["permute"]
    off, val = oracle.permute_jagged(np.array(h["offsets"]), np.array(h["values"]), np.array(h["perm"]))
    assert off.tolist() == h["out_offsets"] and val.tolist() == h["out_values"]


@pytest.mark.parametrize("seed", range(4))
def test_permute_sample_contents(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 300))
    off, ids = _rand_jagged(rng, S, 1000)
    perm = rng.permutation(S).astype(np.int32)
    o2, v2 = oracle.permute_jagged(off, ids, perm)
    assert o2[-1] == off[-1]
    for k in range(S):
        g = perm[k]
        assert np.array_equal(v2[o2[k]:o2[k + 1]], ids[off[g]:off[g + 1]])
    assert np.array_equal(np.sort(v2), np.sort(ids))          # same multiset
    o3, v3 = oracle.permute_jagged(off, ids, np.arange(S, dtype=np.int32))
    assert np.array_equal(o3, off) and np.array_equal(v3, ids)  # identity


def test_permute_rejects_bad_perm():
    off = np.array([0, 1, 2], np.int64)
    with pytest.raises(oracle.OracleError):
        oracle.permute_jagged(off, np.array([5, 6]), np.array([0, 2], np.int32))


# ------------------------------------------------------------------ bucketize

def test_bucketize_hand_example():
    h = HAND["bucketize"]
    sm, pos, splits, so = oracle.bucketize_rowwise(np.array(h["ids"]), np.array(h["rank_id_offsets"]), h["n"], h["R"])
    assert sm.tolist() == h["sm_ids"] and pos.tolist() == h["pos"]
    assert so.tolist() == h["shard_offsets"] and splits.tolist() == h["splits"]


@pytest.mark.parametrize("n,R", [(1, 100), (7, 1000), (64, 10_000), (512, 50_000), (13, 12)])
def test_bucketize_is_stable_sort_by_shard(n, R):
    rng = np.random.default_rng(n + R)
    T = 5000
    ids = rng.integers(0, R, T).astype(np.int64)
    cuts = np.sort(rng.integers(0, T + 1, n - 1))
    rio = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    sm, pos, splits, so = oracle.bucketize_rowwise(ids, rio, n, R)
    block = -(-R // n)
    shard = ids // block
    order = np.argsort(shard, kind="stable")                   # library stable sort
    assert np.array_equal(pos, order) and np.array_equal(sm, ids[order])
    assert np.array_equal(so, np.concatenate([[0], np.cumsum(np.bincount(shard, minlength=n))]))
    assert splits.sum() == T
    assert np.array_equal(splits.sum(axis=1), np.diff(rio))     # per source rank
    assert np.array_equal(splits.sum(axis=0), np.diff(so))      # per shard
    src = np.searchsorted(rio, pos, side="right") - 1
    for s in range(n):
        seg = slice(so[s], so[s + 1])
        assert (sm[seg] // block == s).all()
        assert (np.diff(pos[seg]) > 0).all()                    # source-rank, position order
        assert np.array_equal(np.bincount(src[seg], minlength=n), splits[:, s])
    if n == 1:
        assert np.array_equal(sm, ids)


def test_bucketize_rejects_out_of_range():
    with pytest.raises(oracle.OracleError):
        oracle.bucketize_rowwise(np.array([0, 10]), np.array([0, 2]), 1, 10)
    with pytest.raises(oracle.OracleError):
        oracle.bucketize_rowwise(np.array([0, -1]), np.array([0, 2]), 1, 10)


def test_bucketize_empty():
    sm, pos, splits, so = oracle.bucketize_rowwise(np.zeros(0, np.int64), np.zeros(4, np.int64), 3, 10)
    assert sm.size == 0 and splits.sum() == 0 and so.tolist() == [0, 0, 0, 0]


# ------------------------------------------------------------------ collision

def test_collision_hand_example():
    h = HAND["collision"]
    c = oracle.collision_split(np.array(h["ids_t"]), np.array(h["ids_next"]), h["R"], h["n"])
    for k in ("co", "ex_t", "ex_next", "co_off", "ex_t_off", "ex_next_off", "is_co_t", "is_co_next"):
        assert c[k].tolist() == h[k], k


@pytest.mark.parametrize("seed", range(6))
def test_collision_brute_force_sets(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 200))
    n = int(rng.integers(1, 20))
    a = rng.integers(0, R, int(rng.integers(0, 150))).astype(np.int64)
    b = rng.integers(0, R, int(rng.integers(0, 150))).astype(np.int64)
    c = oracle.collision_split(a, b, R, n)
    A, B = set(a.tolist()), set(b.tolist())
    assert c["co"].tolist() == sorted(A & B)
    assert c["ex_t"].tolist() == sorted(A - B)
    assert c["ex_next"].tolist() == sorted(B - A)
    assert len(c["co"]) + len(c["ex_t"]) == len(A) and len(c["co"]) + len(c["ex_next"]) == len(B)
    assert c["is_co_t"].tolist() == [int(x in B) for x in a.tolist()]
    assert c["is_co_next"].tolist() == [int(x in A) for x in b.tolist()]
    block = -(-R // n)
    for key in ("co", "ex_t", "ex_next"):
        lst = c[key].tolist()
        assert c[key + "_off"].tolist() == [bisect.bisect_left(lst, k * block) for k in range(n + 1)]


def test_collision_special_cases():
    a = np.array([4, 1, 4, 9], np.int64)
    c = oracle.collision_split(a, a[::-1].copy(), 10, 3)      # same rows: nothing exclusive
    assert c["co"].tolist() == [1, 4, 9] and c["ex_t"].size == 0 and c["ex_next"].size == 0
    assert c["is_co_t"].tolist() == [1, 1, 1, 1]
    c = oracle.collision_split(a, np.array([0, 2, 3], np.int64), 10, 3)   # disjoint: no collision
    assert c["co"].size == 0 and c["ex_t"].tolist() == [1, 4, 9] and c["ex_next"].tolist() == [0, 2, 3]
    c = oracle.collision_split(np.zeros(0, np.int64), np.zeros(0, np.int64), 10, 3)
    assert c["co"].size == 0 and c["co_off"].tolist() == [0, 0, 0, 0]


def test_collision_on_synthetic_batches_is_order_free():
    """Row sets do not depend on batch- or shard-major order (FreeScale §3.2)."""
    w = synthetic.WORKLOADS["tiny-fbs-sgd"]
    b0 = {k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in synthetic.batch(w, 0).items()}
    b1 = {k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in synthetic.batch(w, 1).items()}
    p0, p1 = oracle.prepare(w, b0), oracle.prepare(w, b1)
    c_bm = oracle.collision_split(p0["ids"], p1["ids"], w.R, w.n)
    c_sm = oracle.collision_split(p0["sm_ids"], p1["sm_ids"], w.R, w.n)
    for k in ("co", "ex_t", "ex_next", "co_off"):
        assert np.array_equal(c_bm[k], c_sm[k])
    # shard-major mask, moved to batch-major through pos, equals the batch-major mask
    m = np.empty_like(c_sm["is_co_t"])
    m[p0["pos"]] = c_sm["is_co_t"]
    assert np.array_equal(m, c_bm["is_co_t"])


# ------------------------------------------------------------------ keyed transpose

with open(os.path.join(GOLD, "keyed_transpose_hand_examples.json")) as f:
    KT = json.load(f)


@pytest.mark.parametrize("case", KT["cases"], ids=lambda c: f"F{c['F']}B{c['B']}{'_base' if c['row_base'] else ''}")
def test_keyed_transpose_hand_examples(case):
    off, val = oracle.keyed_transpose(np.array(case["offsets"]), np.array(case["values"]), case["F"], case["B"],
                                      None if case["row_base"] is None else np.array(case["row_base"]))
    assert off.tolist() == case["out_offsets"] and val.tolist() == case["out_values"]


def _nested(off, val, F, B):
    """Feature-major arrays as nested lists: seg[f][b] = list of IDs."""
    return [[val[off[f * B + b]:off[f * B + b + 1]].tolist() for b in range(B)] for f in range(F)]


@pytest.mark.parametrize("F,B,seed", [(1, 7, 0), (5, 1, 1), (4, 9, 2), (13, 6, 3), (3, 0, 4)])
def test_keyed_transpose_against_nested_lists(F, B, seed):
    rng = np.random.default_rng(seed)
    off, val = _rand_jagged(rng, F * B, 10 ** 6, maxlen=12)
    base = rng.integers(0, 10 ** 9, F).astype(np.int64)
    o2, v2 = oracle.keyed_transpose(off, val, F, B, base)
    seg = _nested(off, val, F, B)
    flat, lens = [], []
    for b in range(B):                       # batch-major: sample, then feature
        for f in range(F):
            flat += [x + int(base[f]) for x in seg[f][b]]
            lens.append(len(seg[f][b]))
    assert v2.tolist() == flat
    expected = [0] + np.cumsum(lens).tolist() if lens else [0]
    assert o2.tolist() == expected


@pytest.mark.parametrize("F,B", [(4, 9), (1, 5), (6, 1), (7, 3)])
def test_keyed_transpose_twice_with_roles_swapped_is_identity(F, B):
    """Batch-major output read as feature-major with B features of F samples transposes back."""
    rng = np.random.default_rng(F * 10 + B)
    off, val = _rand_jagged(rng, F * B, 1000)
    o2, v2 = oracle.keyed_transpose(off, val, F, B)
    o3, v3 = oracle.keyed_transpose(o2, v2, B, F)
    assert np.array_equal(o3, off) and np.array_equal(v3, val)
    if F == 1 or B == 1:                     # one feature or one sample: nothing moves
        assert np.array_equal(o2, off) and np.array_equal(v2, val)


def test_keyed_transpose_rejects_bad_offsets():
    with pytest.raises(oracle.OracleError):
        oracle.keyed_transpose(np.array([0, 3, 2]), np.array([1, 2, 3]), 1, 2)


# ------------------------------------------------------------------ composite candidates

def test_composite_candidate_lengths_move_with_their_samples():
    """Algorithm 1 Stage II: with multi-ID candidates, each output sample's row is its UIH IDs plus
    the IDs of its candidates, and its candidate lengths are the source sample's, in order."""
    w = synthetic.WORKLOADS["composite-cand"]
    b = {k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in synthetic.batch(w, 0).items()}
    # the recipe itself: row length = UIH + sum of the candidate lengths
    co, cl = b["cand_offsets"], b["cand_lens"]
    per = np.array([cl[co[g]:co[g + 1]].sum() for g in range(w.S)])
    assert np.array_equal(np.diff(b["offsets"]), b["uih_len"].astype(np.int64) + per)
    assert np.array_equal(np.diff(co), b["num_cand"])
    p = oracle.prepare(w, b)
    perm = p["perm"]
    for k in range(w.S):
        g = perm[k]
        assert p["cand_lens"][p["cand_offsets"][k]:p["cand_offsets"][k + 1]].tolist() == cl[co[g]:co[g + 1]].tolist()
        row = p["ids"][p["offsets"][k]:p["offsets"][k + 1]]
        assert row.tolist() == b["ids"][b["offsets"][g]:b["offsets"][g + 1]].tolist()
