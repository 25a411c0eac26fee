"""Whole-iteration parity on the workload recipes at reduced sizes (GPU).

Each case runs the GPU pipeline over consecutive iterations in the synchronous
order and compares with the oracle's synchronous run: every index output
bit-exact (partition, permuted IDs, shard-major IDs, positions, splits, shard
offsets, collision lists, shard offsets and masks), gathered rows bit-exact,
updated table and Adagrad state within tolerance.  Then the prioritized order
(FreeScale Algorithm 2) must give bit-identical gathered rows, table and state
to the synchronous order on the GPU, and two runs must be bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from jagged_embedding_gb300 import synthetic
from jagged_embedding_gb300.pipeline import Pipeline
from tests.helpers import assert_state_close, assert_table_close, batch_np, batch_to, to_np, update_scale

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

W = synthetic.WORKLOADS
CASES = {
    "tiny-fbs-sgd": W["tiny-fbs-sgd"],                                                  # full size
    "vbs-gather": W["vbs-gather"],                                                      # full size
    "mid-full-step": W["mid-full-step"].scaled(B=16, R=1_000_000),
    "long-seq-index": W["long-seq-index"].scaled(B=2, R=5_000_000),
    "large-table-full-step": W["large-table-full-step"].scaled(B=4, R=2_000_000),
    "composite-cand": W["composite-cand"],                                              # full size
    "long-seq-autotune": W["long-seq-autotune"].scaled(B=2, R=5_000_000),
}


def _times(w, device="cpu"):
    """The ranks' step times reported after each iteration (AutoTune recipes), else None."""
    return [synthetic.step_times(w, t, device) for t in range(w.iters)] if w.autotune else None


def _gpu_sync(w, batches_cpu, table0, grads_cpu, row_sorted=True):
    tab = table0.to(DEV)
    state = torch.zeros(w.R, dtype=torch.float32, device=DEV) if w.optim == "adagrad" else None
    bd = [batch_to(b, DEV) for b in batches_cpu]
    gd = [g.to(DEV) for g in grads_cpu] if grads_cpu else None
    pipe = Pipeline(w, DEV, max(b["T"] for b in batches_cpu), tab, state, row_sorted=row_sorted)
    K = len(bd)
    times = _times(w, DEV)
    rec = []
    pipe.prepare(bd[0], 0)
    cur = 0
    for t in range(K):
        s = pipe.slots[cur]
        T = s.T
        # the table as the gather of t reads it (the update of t-1 has landed)
        snap = {"table_before": to_np(tab), "state_before": to_np(state) if state is not None else None,
                "perm": to_np(s.perm[: w.S]), "rank_offsets": to_np(s.rank_offsets), "ids": to_np(s.ids[:T]),
                "offsets": to_np(s.offsets[: w.S + 1]), "rank_id_offsets": to_np(s.rank_id_offsets),
                "sm_ids": to_np(s.sm_ids[:T]), "pos": to_np(s.pos[:T]), "splits": to_np(s.splits),
                "shard_offsets": to_np(s.shard_offsets), "seg_weight": to_np(s.seg_weight)}
        if w.composite:
            nc = int(bd[t]["cand_offsets"][-1])
            snap["cand_offsets"] = to_np(s.cand_offsets[: w.S + 1])
            snap["cand_lens"] = to_np(s.cand_lens[:nc])
        has_next = t + 1 < K
        nxt = pipe.step_sync(cur, bd[t + 1] if has_next else None, gd[t] if gd else None, has_next=has_next,
                             want_masks=True, times=times[t] if times else None)
        B.check(pipe.err, f"iteration {t}")
        snap["out"] = to_np(pipe.out[0][:T])
        if has_next:
            c = {k: to_np(v) for k, v in pipe.coll.items()}
            counts = c["counts"]
            m = to_np(pipe.masks[cur][:T])
            if pipe.mask_layout[cur] == "shard":        # aligned with sm_ids: back to batch-major order
                bm = np.empty_like(m)
                bm[snap["pos"]] = m
                m = bm
            snap["coll"] = {"co": c["co"][: counts[0]], "ex_t": c["ex_t"][: counts[1]],
                            "ex_next": c["ex_next"][: counts[2]], "co_off": c["co_off"], "ex_t_off": c["ex_t_off"],
                            "ex_next_off": c["ex_next_off"], "is_co_t": m}
        rec.append(snap)
        cur = nxt
    return rec, to_np(tab), (to_np(state) if state is not None else None)


def _inputs(w):
    batches = [synthetic.batch(w, t) for t in range(w.iters)]
    table0 = synthetic.table(w)
    grads = [synthetic.grads(w, b["T"], t) for t, b in enumerate(batches)] if w.has_update else None
    return batches, table0, grads


@pytest.mark.parametrize("name", list(CASES))
def test_pipeline_matches_oracle(name):
    w = CASES[name]
    batches, table0, grads = _inputs(w)
    rec, tab_gpu, st_gpu = _gpu_sync(w, batches, table0, grads)
    nb = [batch_np(b) for b in batches]
    tab_ref = to_np(table0)
    st_ref = np.zeros(w.R, np.float32) if w.optim == "adagrad" else None
    g_np = [to_np(g) for g in grads] if grads else None
    times = _times(w)
    ref = oracle.run_sync(w, nb, tab_ref, st_ref, g_np, [to_np(x) for x in times] if times else None,
                          keep_tables=True)
    for t in range(w.iters):
        g, r = rec[t], ref[t]
        p = r["prep"]
        assert np.array_equal(g["perm"], p["perm"]), t
        assert np.array_equal(g["rank_offsets"], p["rank_offsets"]), t
        if w.autotune and t > 0:   # the corrections moved the cut away from the plain one
            assert not np.array_equal(p["rank_offsets"], oracle.balance_vbs(nb[t]["uih_len"], w.n, w.alpha,
                                                                            w.sort_by_len)[1]), t
        if p["seg_weight"] is not None:
            assert np.array_equal(g["seg_weight"].astype(np.uint64), p["seg_weight"]), t
        assert np.array_equal(g["offsets"], p["offsets"]), t
        assert np.array_equal(g["ids"], p["ids"]), t
        assert np.array_equal(g["rank_id_offsets"], p["rank_id_offsets"]), t
        assert np.array_equal(g["sm_ids"], p["sm_ids"]), t
        assert np.array_equal(g["pos"], p["pos"]), t
        assert np.array_equal(g["splits"], p["splits"]), t
        assert np.array_equal(g["shard_offsets"], p["shard_offsets"]), t
        if w.composite:
            assert np.array_equal(g["cand_offsets"], p["cand_offsets"]), t
            assert np.array_equal(g["cand_lens"], p["cand_lens"]), t
        if "coll" in r:
            # (the synchronous order does not ask for the mask of t+1)
            for k in ("co", "ex_t", "ex_next", "co_off", "ex_t_off", "ex_next_off", "is_co_t"):
                assert np.array_equal(g["coll"][k], r["coll"][k]), (t, k)
        # gathered rows: a byte copy, so bit-exact against the oracle's gather of the table the GPU
        # gather read (the table before step t); that table is the oracle's within the update tolerance
        assert np.array_equal(g["out"], oracle.emb_gather(g["table_before"], p["ids"])), t
        if t == 0 or not w.has_update:
            assert np.array_equal(g["out"], r["out"]), t
            assert np.array_equal(g["table_before"], r["table_before"]), t
        else:
            ids_prev = np.concatenate([ref[k]["prep"]["ids"] for k in range(t)])
            g_prev = np.concatenate(g_np[:t])
            sc = update_scale(ids_prev, g_prev, w.R, w.optim, w.lr, w.eps, r["state_before"])
            assert_table_close(g["table_before"], r["table_before"], w.dtype, w.lr, scale=sc, ulps=t)
            if st_ref is not None:
                assert_state_close(g["state_before"], r["state_before"])
        if w.has_update:
            # the update of t writes the rows of uniq(I^t) and no other row (FreeScale Algorithm 2,
            # lines 7 and 20: each row of the batch is updated once, by its phase)
            after = rec[t + 1]["table_before"] if t + 1 < w.iters else tab_gpu
            changed = np.flatnonzero((after != g["table_before"]).any(axis=1))
            uniq = np.unique(p["ids"])
            assert np.isin(changed, uniq).all(), t
            moved = np.flatnonzero((r["table_after"] != r["table_before"]).any(axis=1))
            assert np.isin(moved, changed).all(), t
    if w.has_update:
        ids_all = np.concatenate([r["prep"]["ids"] for r in ref])
        g_all = np.concatenate(g_np)
        scale = update_scale(ids_all, g_all, w.R, w.optim, w.lr, w.eps, st_ref)
        assert_table_close(tab_gpu, tab_ref, w.dtype, w.lr, scale=scale, ulps=w.iters)
        if st_ref is not None:
            assert_state_close(st_gpu, st_ref)
    else:
        assert np.array_equal(tab_gpu, tab_ref)


@pytest.mark.parametrize("streams", [False, True])
@pytest.mark.parametrize("name", ["tiny-fbs-sgd", "mid-full-step", "large-table-full-step", "long-seq-autotune"])
def test_prioritized_order_equals_sync_order_on_gpu(name, streams):
    """Algorithm 2's order gathers exactly what the synchronous order gathers (FreeScale §3.2), on one
    stream and with the exclusive-row work on a side stream."""
    w = CASES[name]
    batches, table0, grads = _inputs(w)
    rec, tab_sync, st_sync = _gpu_sync(w, batches, table0, grads)
    tab = table0.to(DEV)
    state = torch.zeros(w.R, dtype=torch.float32, device=DEV) if w.optim == "adagrad" else None
    pipe = Pipeline(w, DEV, max(b["T"] for b in batches), tab, state, two_outputs=True, streams=streams)
    outs = {}
    pipe.run_prioritized([batch_to(b, DEV) for b in batches], [g.to(DEV) for g in grads] if grads else None,
                         on_output=lambda t, o: outs.__setitem__(t, to_np(o)), times_list=_times(w, DEV))
    B.check(pipe.err, "prioritized")
    for t in range(w.iters):
        assert np.array_equal(outs[t], rec[t]["out"]), t
    assert np.array_equal(to_np(tab), tab_sync)
    if state is not None:
        assert np.array_equal(to_np(state), st_sync)


@pytest.mark.parametrize("name", ["tiny-fbs-sgd", "mid-full-step", "large-table-full-step", "composite-cand"])
def test_row_sorted_step_equals_unsorted_step(name):
    """Gathering from the update's sorted entries changes nothing: every iteration's output, the
    table and the state are bit-identical to the step that gathers in position order."""
    w = CASES[name]
    batches, table0, grads = _inputs(w)
    a = _gpu_sync(w, batches, table0, grads, row_sorted=True)
    b = _gpu_sync(w, batches, table0, grads, row_sorted=False)
    for t in range(w.iters):
        assert np.array_equal(a[0][t]["out"], b[0][t]["out"]), t
    assert np.array_equal(a[1], b[1])
    if a[2] is not None:
        assert np.array_equal(a[2], b[2])


def test_runs_are_bit_identical():
    w = CASES["large-table-full-step"]
    batches, table0, grads = _inputs(w)
    a = _gpu_sync(w, batches, table0, grads)
    b = _gpu_sync(w, batches, table0, grads)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    for t in range(w.iters):
        assert np.array_equal(a[0][t]["out"], b[0][t]["out"])
