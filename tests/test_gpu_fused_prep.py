"""Fused jagged permute + row-wise bucketize (fs_permute_bucketize), and the gather
from its output in shard-major order (fs_emb_gather_shard_major) (GPU).

Its outputs must equal, bit for bit, the oracle's permute followed by its
bucketize (FreeScale Algorithm 1 Stage III and §4.2; Algorithm 2 line 8) and
the two separate GPU calls: permuted offsets and IDs, rank ID ranges,
shard-major IDs, positions, send splits and shard offsets.  Cases: FBS and
VBS permutations, long samples (several tiles each), many short samples per
tile, empty samples, one rank, 1024 ranks, a ragged tail, no samples, an ID
out of range and a capacity too small.
"""
import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from tests.helpers import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _batch(seed, S, mu, sigma, lmax, R, empty_frac=0.0):
    rng = np.random.default_rng(seed)
    L = np.clip(np.round(rng.lognormal(mu, sigma, S)), 1, lmax).astype(np.int64)
    if empty_frac:
        L[rng.random(S) < empty_frac] = 0
    off = np.zeros(S + 1, np.int64)
    np.cumsum(L, out=off[1:])
    ids = (rng.zipf(1.2, off[-1]) * 2654435761 % R).astype(np.int64)
    return L.astype(np.int32), off, ids


def _perm(L, n, kind):
    if kind == "fbs":
        return oracle.balance_fbs(L, n)
    p, ro, _ = oracle.balance_vbs(L, n, 1.5, 1)
    return p, ro


@pytest.mark.parametrize("S,n,R,mu,sigma,lmax,kind,empty", [
    (4096, 64, 1_000_000, 6.5, 1.5, 8192, "fbs", 0.0),       # long samples
    (32768, 512, 5_000_000, 3.0, 1.0, 200, "vbs", 0.0),     # length-sorted short samples: many per tile
    (2000, 8, 100_000, 5.0, 1.2, 2048, "fbs", 0.1),          # some empty samples
    (777, 1, 50_000, 4.0, 1.0, 1000, "fbs", 0.0),            # one rank, ragged tail
    (4096, 1024, 3_000_000, 4.0, 1.5, 4096, "fbs", 0.0),     # the most shards
    (1024, 64, (1 << 33) + 7, 5.0, 1.2, 2048, "fbs", 0.0),    # rows beyond 2^32: 64-bit staging
    (16, 4, 1000, 1.0, 0.5, 10, "vbs", 0.0),                 # a few IDs
])
def test_fused_prep_matches_oracle_and_two_calls(S, n, R, mu, sigma, lmax, kind, empty):
    L, off, ids = _batch(S + n, S, mu, sigma, lmax, R, empty)
    perm, ro = _perm(L, n, kind)
    T = int(off[-1])
    off2, ids2 = oracle.permute_jagged(off, ids, perm)
    rio = off2[ro]
    sm, pos, splits, so = oracle.bucketize_rowwise(ids2, rio, n, R)
    d = {k: torch.from_numpy(v).to(DEV) for k, v in dict(off=off, ids=ids, perm=perm, ro=ro).items()}
    cap = T + 100
    g = B.fs_permute_bucketize(d["off"], d["ids"], d["perm"], d["ro"], R, capacity=cap)
    B.check(g[-1])
    o_off, o_ids, o_rio, o_sm, o_pos, o_splits, o_so = (to_np(x) for x in g[:7])
    assert np.array_equal(o_off, off2) and np.array_equal(o_ids[:T], ids2)
    assert np.array_equal(o_rio, rio)
    assert np.array_equal(o_sm[:T], sm) and np.array_equal(o_pos[:T], pos)
    assert np.array_equal(o_splits, splits) and np.array_equal(o_so, so)
    # the two separate calls give the same bytes
    p_off, p_ids, p_rio, err = B.fs_permute_jagged(d["off"], d["ids"], d["perm"], capacity=cap, rank_offsets=d["ro"])
    b_sm, b_pos, b_splits, b_so, err2 = B.fs_bucketize_rowwise(p_ids, p_rio, R, T=T)
    B.check(err)
    B.check(err2)
    assert np.array_equal(to_np(b_sm)[:T], o_sm[:T]) and np.array_equal(to_np(b_pos)[:T], o_pos[:T])
    assert np.array_equal(to_np(b_splits), o_splits) and np.array_equal(to_np(b_so), o_so)


def test_fused_prep_no_samples():
    z = torch.zeros(1, dtype=torch.int64, device=DEV)
    ro = torch.zeros(5, dtype=torch.int64, device=DEV)
    g = B.fs_permute_bucketize(z, torch.zeros(0, dtype=torch.int64, device=DEV),
                               torch.zeros(0, dtype=torch.int32, device=DEV), ro, 100, capacity=0)
    B.check(g[-1])
    assert to_np(g[0]).tolist() == [0] and to_np(g[2]).tolist() == [0] * 5
    assert (to_np(g[5]) == 0).all() and to_np(g[6]).tolist() == [0] * 5


def test_fused_prep_reports_bad_ids_and_capacity():
    L, off, ids = _batch(5, 300, 4.0, 1.0, 500, 10_000)
    perm, ro = _perm(L, 4, "fbs")
    d = {k: torch.from_numpy(v).to(DEV) for k, v in dict(off=off, ids=ids, perm=perm, ro=ro).items()}
    bad = d["ids"].clone()
    bad[7] = 10_000
    g = B.fs_permute_bucketize(d["off"], bad, d["perm"], d["ro"], 10_000, capacity=int(off[-1]))
    with pytest.raises(B.FsError) as e:
        B.check(g[-1])
    assert e.value.code == 2
    T = int(off[-1])
    g = B.fs_permute_bucketize(d["off"], d["ids"], d["perm"], d["ro"], 10_000, capacity=T - 5)
    with pytest.raises(B.FsError) as e:
        B.check(g[-1])
    assert e.value.code == 4
    # the first capacity IDs are written and bucketized
    off2, ids2 = oracle.permute_jagged(off, ids, perm)
    assert np.array_equal(to_np(g[1]), ids2[: T - 5])
    assert to_np(g[6])[-1] == T - 5


@pytest.mark.parametrize("dtype,D,n,R", [("bf16", 128, 512, 5_000_000), ("f32", 64, 16, 1_000_000),
                                         ("f32", 24, 8, 100_000), ("bf16", 256, 1, 50_000)])
def test_shard_major_gather_equals_oracle_gather(dtype, D, n, R):
    """out[pos[j]] = table[sm_ids[j]] over the bucketize output: the oracle's gather in position order,
    bit for bit (FreeScale Algorithm 2 line 12: lookup on the shard-major IDs, ranged combine back)."""
    L, off, ids = _batch(D + n, 3000, 5.0, 1.2, 2048, R)
    perm, ro = _perm(L, n, "fbs")
    d = {k: torch.from_numpy(v).to(DEV) for k, v in dict(off=off, ids=ids, perm=perm, ro=ro).items()}
    g = B.fs_permute_bucketize(d["off"], d["ids"], d["perm"], d["ro"], R)
    B.check(g[-1])
    T = int(off[-1])
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    W = (torch.randn(R, D, generator=torch.Generator().manual_seed(R)) * 0.01).to(tdt)
    Wd = W.to(DEV)
    out, err = B.fs_emb_gather_shard_major(Wd, g[3], g[4], T=T)
    B.check(err)
    _, ids2 = oracle.permute_jagged(off, ids, perm)
    assert np.array_equal(to_np(out), oracle.emb_gather(to_np(W), ids2))
    ref, err = B.fs_emb_gather(Wd, g[1], T=T)
    B.check(err)
    assert torch.equal(out, ref)


def test_shard_major_gather_reports_bad_entries():
    R, D, T = 100, 64, 50
    W = torch.randn(R, D, device=DEV)
    sm = torch.arange(T, dtype=torch.int64, device=DEV)
    pos = torch.arange(T, dtype=torch.int32, device=DEV).flip(0).contiguous()
    sm[3] = R
    out = torch.full((T, D), 5.0, device=DEV)
    _, err = B.fs_emb_gather_shard_major(W, sm, pos, out=out)
    with pytest.raises(B.FsError) as e:
        B.check(err)
    assert e.value.code == 2
    o = to_np(out)
    assert (o[T - 1 - 3] == 5.0).all()                          # the bad entry's row is left untouched
    keep = [j for j in range(T) if j != 3]
    assert np.array_equal(o[[T - 1 - j for j in keep]], to_np(W)[keep])
    pos2 = pos.clone()
    pos2[0] = T
    _, err = B.fs_emb_gather_shard_major(W, torch.arange(T, dtype=torch.int64, device=DEV), pos2, out=out)
    with pytest.raises(B.FsError) as e:
        B.check(err)
    assert e.value.code == 3
