"""The update's sort per shard (fs_emb_sort_rows_sharded) against the sort of
the batch-major IDs (GPU).

The input is the bucketize output of the same batch (FreeScale §3.2,
Algorithm 2 line 8) and the collision flags in shard-major order; the gather
from the sorted entries and the update that follows must give the same bytes
as after fs_emb_sort_rows -- gathered rows, table and Adagrad state bit for
bit -- and the gathered rows must equal the oracle's gather.  Cases cover one
shard, many shards, empty shards, shards of one row, the maximum of 1024
shards, a hot shard spanning many tiles, ragged tails and tiny batches.
"""
import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from jagged_embedding_gb300 import synthetic
from tests.helpers import assert_table_close, to_np, update_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bitmap(rows, R):
    bm = np.zeros((R + 31) // 32, np.uint32)
    np.bitwise_or.at(bm, rows >> 5, (np.uint32(1) << (rows & 31).astype(np.uint32)))
    return torch.from_numpy(bm.view(np.int32))


def _case(seed, R, D, T, n, dtype, s=1.05):
    g = torch.Generator().manual_seed(seed)
    ids = synthetic.zipf_rows(R, s, T, g, "cpu")
    nxt = synthetic.zipf_rows(R, s, max(T // 2, 1), g, "cpu").numpy()
    is_co = np.isin(ids.numpy(), nxt).astype(np.uint8)
    _case.next_rows = nxt
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    W = (torch.randn(R, D, generator=g) * 0.01).to(tdt)
    G = torch.randn(T, D, generator=g).to(tdt)
    rio = torch.tensor([T * r // n for r in range(n + 1)], dtype=torch.int64)
    return ids, is_co, W, G, rio


def _bucketize(idd, riod, R):
    sm, pos, splits, so, err = B.fs_bucketize_rowwise(idd, riod, R)
    B.check(err)
    return sm, pos, so


@pytest.mark.parametrize("dtype,D,optim,T,R,n,two", [
    ("f32", 64, "adagrad", 400_000, 2_000_000, 256, True),      # large-table shape, scaled
    ("bf16", 128, "adagrad", 300_000, 1_000_000, 64, True),     # mid-size shape, scaled
    ("f32", 64, "adagrad", 100_000, 500_000, 1, True),          # one shard
    ("f32", 32, "sgd", 60_001, 30_000, 1024, True),             # 1024 shards of 30 rows
    ("bf16", 64, "adagrad", 50_000, 700, 512, True),            # shards of 2 rows, many empty
    ("f32", 64, "sgd", 20_000, 100, 256, False),                # more shards than rows, one phase
    ("bf16", 256, "adagrad", 80_000, 1 << 19, 1, False),        # a shard of 2^19 rows, one phase
    ("f32", 128, "adagrad", 5, 1000, 8, True),                  # tiny batch
    ("f32", 64, "sgd", 1, 1, 1, True),
])
def test_sharded_sort_equals_batch_major_sort(dtype, D, optim, T, R, n, two):
    ids, is_co, W, G, rio = _case(T + R + n, R, D, T, n, dtype)
    idd, Gd, riod = ids.to(DEV), G.to(DEV), rio.to(DEV)
    sm, pos, so = _bucketize(idd, riod, R)
    m_bm = torch.from_numpy(is_co).to(DEV)
    m_sm = m_bm[pos.long()].contiguous()
    co_rows = _bitmap(_case.next_rows, R).to(DEV)
    ph = B.PHASE_COLLISION_THEN_EXCLUSIVE if two else B.PHASE_ALL
    state = torch.rand(R, generator=torch.Generator().manual_seed(5)) if optim == "adagrad" else None
    res = []
    for sharded in ((False, True, "bitmap") if two else (False, True)):
        Wd = W.to(DEV)
        sd = state.to(DEV) if state is not None else None
        if sharded == "bitmap":          # the flags from the next batch's row bitmap
            ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, D, B.dtype_code(Wd), n), DEV)
            err = B.fs_emb_sort_rows_sharded(Wd, sm, pos, so, ws, phase=ph, co_rows=co_rows)
        elif sharded:
            ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, D, B.dtype_code(Wd), n), DEV)
            err = B.fs_emb_sort_rows_sharded(Wd, sm, pos, so, ws, phase=ph, is_co=m_sm if two else None)
        else:
            ws = B.workspace(B.backward_workspace_size(T, R, D, B.dtype_code(Wd)), DEV)
            err = B.fs_emb_sort_rows(Wd, idd, ws, phase=ph, is_co=m_bm if two else None)
        out, _ = B.fs_emb_gather_sorted(Wd, T, ws, phase=ph, err=err)
        B.fs_emb_update_sorted(Wd, sd, Gd, T, ws, optim, 0.01, 1e-8, phase=ph, err=err)
        B.check(err)
        res.append((to_np(out), to_np(Wd), to_np(sd) if sd is not None else None))
    for o2, w2, s2 in res[2:]:       # the bitmap form: the same bytes as the mask form
        assert np.array_equal(o2, res[1][0]) and np.array_equal(w2, res[1][1])
        if s2 is not None:
            assert np.array_equal(s2, res[1][2])
    (o0, w0, s0), (o1, w1, s1) = res[:2]
    assert np.array_equal(o1, o0)
    assert np.array_equal(o1, oracle.emb_gather(to_np(W), ids.numpy()))
    assert np.array_equal(w1, w0)
    if s0 is not None:
        assert np.array_equal(s1, s0)
    W_ref = to_np(W)
    s_ref = state.numpy().copy() if state is not None else None
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(G), optim, 0.01, 1e-8)
    assert_table_close(w1, W_ref, dtype, 0.01, scale=update_scale(ids.numpy(), to_np(G), R, optim, 0.01, 1e-8, s_ref))


def test_sharded_sort_hot_shard_and_repeated_calls():
    """One shard holds most entries (hundreds of tiles) and the others a few each; the call is repeated
    on the same workspace with another batch and gives the batch-major sort's result both times."""
    R, D, n = 1 << 20, 64, 128
    for call, T in enumerate((1_500_000, 700_003)):
        g = torch.Generator().manual_seed(40 + call)
        hot = torch.randint(0, R // n, (T * 9 // 10,), generator=g)                 # shard 0
        rest = torch.randint(0, R, (T - hot.numel(),), generator=g)
        ids = torch.cat([hot, rest])[torch.randperm(T, generator=g)]
        W = torch.randn(R, D, generator=g)
        idd = ids.to(DEV)
        rio = torch.tensor([T * r // n for r in range(n + 1)], dtype=torch.int64, device=DEV)
        sm, pos, so = _bucketize(idd, rio, R)
        Wd = W.to(DEV)
        ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, D, B.dtype_code(Wd), n), DEV)
        err = B.fs_emb_sort_rows_sharded(Wd, sm, pos, so, ws)
        out, _ = B.fs_emb_gather_sorted(Wd, T, ws, err=err)
        B.check(err)
        assert np.array_equal(to_np(out), to_np(W)[ids.numpy()]), call


def test_sharded_sort_argument_and_data_errors():
    R, D, T, n = 1000, 64, 4000, 8
    ids, is_co, W, G, rio = _case(3, R, D, T, n, "f32")
    idd, riod = ids.to(DEV), rio.to(DEV)
    sm, pos, so = _bucketize(idd, riod, R)
    Wd = W.to(DEV)
    ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, D, B.dtype_code(Wd), n), DEV)
    m = torch.from_numpy(is_co).to(DEV)[pos.long()].contiguous()
    two = B.PHASE_COLLISION_THEN_EXCLUSIVE
    with pytest.raises(B.FsError) as e:                                   # two phases need the flags
        B.fs_emb_sort_rows_sharded(Wd, sm, pos, so, ws, phase=two)
    assert e.value.code == 1
    with pytest.raises(B.FsError) as e:                                   # the workspace of the batch-major sort
        small = B.workspace(B.backward_workspace_size(T, R, D, B.dtype_code(Wd)), DEV)
        B.fs_emb_sort_rows_sharded(Wd, sm, pos, so, small, phase=two, is_co=m)
    assert e.value.code == 5
    with pytest.raises(B.FsError) as e:                                   # one shard of 2^20 rows + the phase bit
        B.fs_emb_sort_rows_sharded(torch.empty(1 << 20, 64, device=DEV), sm, pos,
                                   torch.tensor([0, T], dtype=torch.int64, device=DEV), ws, phase=two, is_co=m)
    assert e.value.code == 1
    # shard offsets that do not match the IDs: entries outside their shard are reported and left unsorted
    bad = so.clone()
    bad[1:n] = so[1:n] + 3
    out = torch.full((T, D), -3.0, device=DEV)
    err = B.fs_emb_sort_rows_sharded(Wd, sm, pos, bad, ws)
    B.fs_emb_gather_sorted(Wd, T, ws, out=out, err=err)
    with pytest.raises(B.FsError) as e:
        B.check(err)
    assert e.value.code == 3
    # offsets that are not non-decreasing are reported too (and the call stays inside its buffers)
    bad2 = so.clone()
    bad2[2] = T + 100
    err = B.fs_emb_sort_rows_sharded(Wd, sm, pos, bad2, ws)
    with pytest.raises(B.FsError) as e:
        B.check(err)
    assert e.value.code == 3
    # T = 0 does nothing
    B.check(B.fs_emb_sort_rows_sharded(Wd, sm[:0], pos[:0], torch.zeros(n + 1, dtype=torch.int64, device=DEV), ws,
                                       T=0))
