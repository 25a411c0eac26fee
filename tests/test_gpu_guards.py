"""Every C-ABI call writes only its outputs (GPU).

Each call runs at a ragged size with every output and every workspace sized
exactly (no slack) and placed between two guard bands of seeded bytes
(tests.helpers.Guarded); after the call the outputs must equal the oracle's
and no guard byte may have changed.  In-place arguments (the table, the
Adagrad state, the AutoTune corrections) are guarded the same way.
"""
import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from jagged_embedding_gb300 import synthetic
from tests.helpers import Guarded, assert_state_close, assert_table_close, to_np, update_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"
i32, i64, u8 = torch.int32, torch.int64, torch.uint8


def G(shape, dtype, init=None):
    return Guarded(shape, dtype, DEV, init)


def WS(nbytes):
    return Guarded(max(int(nbytes), 1), u8)


def _check_all(*gs):
    for k, g in enumerate(gs):
        g.check(f"output {k}")


def _lens(seed, S):
    return np.clip(np.round(np.random.default_rng(seed).lognormal(4.0, 1.3, S)), 1, 3000).astype(np.int32)


def test_partitions_write_only_their_outputs():
    S, n = 5003, 7
    L = _lens(1, S)
    Ld = torch.from_numpy(L).to(DEV)
    L_ = B.lib()
    perm, ro, ws = G(S, i32), G(n + 1, i64), WS(L_.fs_balance_fbs_workspace_size(S, n))
    B.fs_balance_fbs(Ld, n, perm=perm.t, rank_offsets=ro.t, err=(e := B.new_err(DEV)), ws=ws.t)
    B.check(e)
    p_ref, ro_ref = oracle.balance_fbs(L, n)
    assert np.array_equal(to_np(perm.t), p_ref) and np.array_equal(to_np(ro.t), ro_ref)
    _check_all(perm, ro, ws)
    for sort_by_len in (0, 1):
        perm, ro, sw = G(S, i32), G(n + 1, i64), G(n, i64)
        ws = WS(L_.fs_balance_vbs_workspace_size(S, n))
        B.fs_balance_vbs(Ld, n, 1.5, sort_by_len, perm=perm.t, rank_offsets=ro.t, seg_weight=sw.t, err=e, ws=ws.t)
        B.check(e)
        p_ref, ro_ref, sw_ref = oracle.balance_vbs(L, n, 1.5, sort_by_len)
        assert np.array_equal(to_np(perm.t), p_ref) and np.array_equal(to_np(ro.t), ro_ref)
        assert np.array_equal(to_np(sw.t).astype(np.uint64), sw_ref)
        _check_all(perm, ro, sw, ws)
    # AutoTune: the corrections are updated in place, then the tuned cut
    times = np.array([15, 10, 10, 11, 9, 10, 14], np.int64) * 1_000_000
    delta = G(n, i64, torch.zeros(n, dtype=i64))
    B.fs_vbs_autotune(torch.from_numpy(times).to(DEV), delta.t, err=e)
    d_ref = oracle.vbs_autotune(times, np.zeros(n, np.int64))
    perm, ro, sw = G(S, i32), G(n + 1, i64), G(n, i64)
    ws = WS(L_.fs_balance_vbs_workspace_size(S, n))
    B.fs_balance_vbs_tuned(Ld, n, 1.5, 1, delta.t, perm=perm.t, rank_offsets=ro.t, seg_weight=sw.t, err=e, ws=ws.t)
    B.check(e)
    p_ref, ro_ref, sw_ref = oracle.balance_vbs_tuned(L, n, 1.5, 1, d_ref)
    assert np.array_equal(to_np(delta.t), d_ref) and np.array_equal(to_np(ro.t), ro_ref)
    assert np.array_equal(to_np(perm.t), p_ref) and np.array_equal(to_np(sw.t).astype(np.uint64), sw_ref)
    _check_all(delta, perm, ro, sw, ws)


def _jagged(seed, S, R):
    L = _lens(seed, S).astype(np.int64)
    off = np.zeros(S + 1, np.int64)
    np.cumsum(L, out=off[1:])
    ids = synthetic.zipf_rows(R, 1.05, int(off[-1]), torch.Generator().manual_seed(seed), "cpu").numpy()
    return L.astype(np.int32), off, ids


def test_jagged_index_calls_write_only_their_outputs():
    S, n, R = 3001, 16, 200_003
    L, off, ids = _jagged(2, S, R)
    T = int(off[-1])
    perm, ro = oracle.balance_fbs(L, n)
    d = {k: torch.from_numpy(v).to(DEV) for k, v in dict(off=off, ids=ids, perm=perm, ro=ro).items()}
    Lb = B.lib()
    e = B.new_err(DEV)
    # permute
    o_off, o_val, rio = G(S + 1, i64), G(T, i64), G(n + 1, i64)
    ws = WS(Lb.fs_permute_jagged_workspace_size(S))
    B.fs_permute_jagged(d["off"], d["ids"], d["perm"], capacity=T, rank_offsets=d["ro"], out_offsets=o_off.t,
                        out_values=o_val.t, rank_id_offsets=rio.t, err=e, ws=ws.t)
    B.check(e)
    off2, ids2 = oracle.permute_jagged(off, ids, perm)
    assert np.array_equal(to_np(o_off.t), off2) and np.array_equal(to_np(o_val.t), ids2)
    _check_all(o_off, o_val, rio, ws)
    # bucketize
    sm, pos, spl, so = G(T, i64), G(T, i32), G((n, n), i64), G(n + 1, i64)
    ws = WS(Lb.fs_bucketize_rowwise_workspace_size(T, n))
    B.fs_bucketize_rowwise(o_val.t, rio.t, R, sm_ids=sm.t, pos=pos.t, splits=spl.t, shard_offsets=so.t, err=e,
                           ws=ws.t)
    B.check(e)
    r = oracle.bucketize_rowwise(ids2, off2[ro], n, R)
    for got, ref in zip((sm, pos, spl, so), r):
        assert np.array_equal(to_np(got.t), ref)
    _check_all(sm, pos, spl, so, ws)
    # fused permute + bucketize
    outs = [G(S + 1, i64), G(T, i64), G(n + 1, i64), G(T, i64), G(T, i32), G((n, n), i64), G(n + 1, i64)]
    ws = WS(Lb.fs_permute_bucketize_workspace_size(S, T, n))
    B.fs_permute_bucketize(d["off"], d["ids"], d["perm"], d["ro"], R, capacity=T, out_offsets=outs[0].t,
                           out_values=outs[1].t, rank_id_offsets=outs[2].t, sm_ids=outs[3].t, pos=outs[4].t,
                           splits=outs[5].t, shard_offsets=outs[6].t, err=e, ws=ws.t)
    B.check(e)
    for got, ref in zip(outs, (off2, ids2, off2[ro]) + tuple(r)):
        assert np.array_equal(to_np(got.t), ref)
    _check_all(*outs, ws)
    # keyed transpose (F features x B samples, per-feature row bases)
    F, Bs = 3, S // 3
    base = torch.tensor([0, 1000, 5000], dtype=i64, device=DEV)
    Tt = int(off[F * Bs])
    t_off, t_val = G(F * Bs + 1, i64), G(Tt, i64)
    ws = WS(Lb.fs_keyed_transpose_workspace_size(F, Bs))
    B.fs_keyed_transpose(d["off"][: F * Bs + 1], d["ids"][:Tt], F, Bs, row_base=base, capacity=Tt,
                         out_offsets=t_off.t, out_values=t_val.t, err=e, ws=ws.t)
    B.check(e)
    ko, kv = oracle.keyed_transpose(off[: F * Bs + 1], ids[:Tt], F, Bs, to_np(base))
    assert np.array_equal(to_np(t_off.t), ko) and np.array_equal(to_np(t_val.t), kv)
    _check_all(t_off, t_val, ws)


def test_collision_calls_write_only_their_outputs():
    R, n = 300_007, 8
    g = torch.Generator().manual_seed(3)
    a = synthetic.zipf_rows(R, 1.05, 100_003, g, "cpu")
    b = synthetic.zipf_rows(R, 1.05, 77_001, g, "cpu")
    ref = oracle.collision_split(a.numpy(), b.numpy(), R, n)
    cap = int(max(ref["co"].size, ref["ex_t"].size, ref["ex_next"].size))
    ad, bd = a.to(DEV), b.to(DEV)
    e = B.new_err(DEV)
    Lb = B.lib()
    for bitmaps in (False, True):
        gs = {"co": G(cap, i64), "ex_t": G(cap, i64), "ex_next": G(cap, i64), "counts": G(3, i64),
              "co_off": G(n + 1, i64), "ex_t_off": G(n + 1, i64), "ex_next_off": G(n + 1, i64),
              "is_co_t": G(a.numel(), u8), "is_co_next": G(b.numel(), u8)}
        out = {k: v.t for k, v in gs.items()}
        extra = []
        if bitmaps:
            words = int(Lb.fs_row_bitmap_words(R))
            bma, bmb = G(words, i32), G(words, i32)
            B.fs_row_bitmap(ad, R, bitmap=bma.t, err=e)
            B.fs_row_bitmap(bd, R, bitmap=bmb.t, err=e)
            ws = WS(Lb.fs_collision_split_bitmaps_workspace_size(R))
            B.fs_collision_split_bitmaps(ad, bma.t, bd, bmb.t, R, n, out, cap, err=e, ws=ws.t)
            extra = [bma, bmb]
        else:
            ws = WS(Lb.fs_collision_split_workspace_size(a.numel(), b.numel(), R, n))
            B.fs_collision_split(ad, bd, R, n, cap_rows=cap, out=out, err=e, ws=ws.t)
        B.check(e)
        c = to_np(out["counts"])
        assert np.array_equal(to_np(out["co"])[: c[0]], ref["co"])
        assert np.array_equal(to_np(out["ex_t"])[: c[1]], ref["ex_t"])
        assert np.array_equal(to_np(out["ex_next"])[: c[2]], ref["ex_next"])
        for k in ("co_off", "ex_t_off", "ex_next_off", "is_co_t", "is_co_next"):
            assert np.array_equal(to_np(out[k]), ref[k]), k
        _check_all(*gs.values(), ws, *extra)


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 128), ("f32", 24)])
def test_gathers_write_only_their_outputs(dtype, D):
    R, T = 50_001, 70_003
    g = torch.Generator().manual_seed(D)
    ids = synthetic.zipf_rows(R, 1.05, T, g, "cpu")
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    W = (torch.randn(R, D, generator=g) * 0.01).to(tdt)
    Wd, idd = W.to(DEV), ids.to(DEV)
    e = B.new_err(DEV)
    ref = oracle.emb_gather(to_np(W), ids.numpy())
    out = G((T, D), tdt)
    B.fs_emb_gather(Wd, idd, out=out.t, err=e)
    B.check(e)
    assert np.array_equal(to_np(out.t), ref)
    out.check("gather")
    mask = (torch.rand(T, generator=g) < 0.4).to(u8)
    init = torch.full((T, D), 3.0).to(tdt)
    out = G((T, D), tdt, init)
    B.fs_emb_gather(Wd, idd, out=out.t, mask=mask.to(DEV), sel=1, err=e)
    B.check(e)
    exp = to_np(init)
    oracle.emb_gather(to_np(W), ids.numpy(), mask=mask.numpy(), sel=1, out=exp)
    assert np.array_equal(to_np(out.t), exp)
    out.check("masked gather")
    # shard-major order: the entries of a bucketize of the same IDs into 8 shards
    rio = torch.tensor([T * r // 8 for r in range(9)], dtype=i64, device=DEV)
    sm, pos, _, _, e2 = B.fs_bucketize_rowwise(idd, rio, R)
    B.check(e2)
    out = G((T, D), tdt)
    B.fs_emb_gather_shard_major(Wd, sm, pos, out=out.t, err=e)
    B.check(e)
    assert np.array_equal(to_np(out.t), ref)
    out.check("shard-major gather")


@pytest.mark.parametrize("path", ["one-call", "sorted", "sharded"])
def test_updates_write_only_their_rows_and_outputs(path):
    R, D, T, n = 80_021, 64, 120_007, 16
    g = torch.Generator().manual_seed(11)
    ids = synthetic.zipf_rows(R, 1.05, T, g, "cpu")
    nxt = synthetic.zipf_rows(R, 1.05, T // 2, g, "cpu").numpy()
    is_co = torch.from_numpy(np.isin(ids.numpy(), nxt).astype(np.uint8))
    W = torch.randn(R, D, generator=g) * 0.01
    Gr = torch.randn(T, D, generator=g)
    st0 = torch.rand(R, generator=g)
    table, state = G((R, D), torch.float32, W), G(R, torch.float32, st0)
    idd, Gd, md = ids.to(DEV), Gr.to(DEV), is_co.to(DEV)
    e = B.new_err(DEV)
    CT = B.PHASE_COLLISION_THEN_EXCLUSIVE
    guards = [table, state]
    if path == "one-call":
        ws = WS(B.backward_workspace_size(T, R, D, B.F32))
        B.fs_emb_backward_adagrad(table.t, state.t, idd, Gd, "adagrad", 0.01, 1e-8, is_co=md, phase=CT, err=e,
                                  ws=ws.t)
    else:
        out = G((T, D), torch.float32)
        if path == "sorted":
            ws = WS(B.backward_workspace_size(T, R, D, B.F32))
            B.fs_emb_sort_rows(table.t, idd, ws.t, phase=CT, is_co=md, err=e)
        else:
            rio = torch.tensor([T * r // n for r in range(n + 1)], dtype=i64, device=DEV)
            sm, pos, _, so, e2 = B.fs_bucketize_rowwise(idd, rio, R)
            B.check(e2)
            ws = WS(B.sort_rows_sharded_workspace_size(T, R, D, B.F32, n))
            B.fs_emb_sort_rows_sharded(table.t, sm, pos, so, ws.t, phase=CT, is_co=md[pos.long()].contiguous(),
                                       err=e)
        B.fs_emb_gather_sorted(table.t, T, ws.t, out=out.t, phase=CT, err=e)
        B.fs_emb_update_sorted(table.t, state.t, Gd, T, ws.t, "adagrad", 0.01, 1e-8, phase=CT, err=e)
        B.check(e)
        assert np.array_equal(to_np(out.t), to_np(W)[ids.numpy()])
        guards.append(out)
    B.check(e)
    W_ref, s_ref = to_np(W), st0.numpy().copy()
    oracle.emb_backward(W_ref, s_ref, ids.numpy(), to_np(Gr), "adagrad", 0.01, 1e-8)
    assert_table_close(to_np(table.t), W_ref, "f32", 0.01,
                       scale=update_scale(ids.numpy(), to_np(Gr), R, "adagrad", 0.01, 1e-8, s_ref))
    assert_state_close(to_np(state.t), s_ref)
    _check_all(*guards, ws)
