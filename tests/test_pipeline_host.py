"""Host-side sequencing of pipeline.py (CPU only).

The C-ABI calls are replaced by recorders, so these tests check only which
calls one iteration issues, in which order and with which phase: the
synchronous step (the update's sort before the lookup, the fallbacks), the
VBS AutoTune hook, and Algorithm 2's order (FreeScale, Algorithm 2 lines 7-21).
Nothing here runs a kernel.
"""
import pytest
import torch

from jagged_embedding_gb300 import binding as B
from jagged_embedding_gb300 import pipeline as P
from jagged_embedding_gb300 import synthetic

CALLS = ["fs_emb_gather_shard_major", "fs_balance_fbs", "fs_balance_vbs", "fs_balance_vbs_tuned", "fs_vbs_autotune", "fs_permute_jagged",
         "fs_bucketize_rowwise", "fs_permute_bucketize", "fs_row_bitmap", "fs_collision_split_bitmaps", "fs_emb_gather",
         "fs_emb_gather_sorted", "fs_emb_sort_rows", "fs_emb_sort_rows_sharded", "fs_emb_update_sorted",
         "fs_emb_backward_adagrad"]


KWARGS = {}   # keyword arguments of the last call of each name


@pytest.fixture
def calls(monkeypatch):
    log = []
    KWARGS.clear()
    for name in CALLS:
        def rec(*a, _n=name, **kw):
            log.append((_n, kw.get("phase")))
            KWARGS[_n] = kw
        monkeypatch.setattr(P.B, name, rec)
    return log


def _pipe(w, **kw):
    table = torch.zeros(w.R, w.D, dtype=torch.float32 if w.dtype == "f32" else torch.bfloat16)
    state = torch.zeros(w.R) if w.optim == "adagrad" else None
    return P.Pipeline(w, "cpu", 1000, table, state, **kw)


def _batch(w):
    S = w.S
    return {"uih_len": torch.ones(S, dtype=torch.int32), "offsets": torch.arange(S + 1, dtype=torch.int64),
            "ids": torch.zeros(S, dtype=torch.int64), "T": S}


def _names(log, skip=("fs_balance_fbs", "fs_permute_bucketize", "fs_permute_jagged", "fs_row_bitmap")):
    return [(n, ph) for n, ph in log if n not in skip]


TINY = synthetic.WORKLOADS["tiny-fbs-sgd"].scaled(R=1000)


def test_sync_step_sorts_before_the_lookup(calls):
    pipe = _pipe(TINY)
    pipe.prepare(_batch(TINY), 0)
    calls.clear()
    nxt = pipe.step_sync(0, _batch(TINY), torch.zeros(1, TINY.D))
    CT = B.PHASE_COLLISION_THEN_EXCLUSIVE
    assert nxt == 1
    # the update sorts each shard's entries of the bucketize output (shards of 125 rows)
    assert _names(calls) == [("fs_collision_split_bitmaps", None), ("fs_emb_sort_rows_sharded", CT),
                             ("fs_emb_gather_sorted", CT), ("fs_emb_update_sorted", CT)]
    # its collision flags come from the next batch's row bitmap: no mask pass
    assert KWARGS["fs_emb_sort_rows_sharded"]["co_rows"] is pipe.slots[1].bitmap
    assert KWARGS["fs_collision_split_bitmaps"]["want_t_mask"] is False
    calls.clear()
    pipe.step_sync(1, _batch(TINY), torch.zeros(1, TINY.D), want_masks=True)   # masks asked for: shard-major
    assert pipe.mask_layout == ["shard", "shard"]
    assert KWARGS["fs_collision_split_bitmaps"]["want_t_mask"] is True
    # the batch is prepared (balanced, permuted and bucketized in one call, marked) before the split
    assert [n for n, _ in calls[:3]] == ["fs_balance_fbs", "fs_permute_bucketize", "fs_row_bitmap"]
    assert KWARGS["fs_row_bitmap"]["T"] == TINY.S


def test_sync_step_sorts_batch_major_ids_when_shards_are_too_large(calls):
    w = TINY.scaled(n=1, B=TINY.S, R=(1 << 19) + 1)  # one shard: 2^19 + 1 rows and the phase bit
    pipe = _pipe(w)
    pipe.step_sync(0, _batch(w), torch.zeros(1, w.D))
    CT = B.PHASE_COLLISION_THEN_EXCLUSIVE
    assert _names(calls)[-3:] == [("fs_emb_sort_rows", CT), ("fs_emb_gather_sorted", CT),
                                  ("fs_emb_update_sorted", CT)]
    assert pipe.mask_layout[0] == "batch"                  # the batch-major sort reads the mask of t
    assert KWARGS["fs_collision_split_bitmaps"]["want_t_mask"] is True
    calls.clear()
    pipe.step_sync(0, None, torch.zeros(1, w.D), has_next=False)   # one phase: 20 bits fit
    assert _names(calls)[0] == ("fs_emb_sort_rows_sharded", B.PHASE_ALL)


def test_last_iteration_sorts_every_row_in_one_phase(calls):
    pipe = _pipe(TINY)
    pipe.step_sync(0, None, torch.zeros(1, TINY.D), has_next=False)
    A = B.PHASE_ALL
    assert _names(calls) == [("fs_emb_sort_rows_sharded", A), ("fs_emb_gather_sorted", A),
                             ("fs_emb_update_sorted", A)]


def test_position_order_step_when_asked_or_when_the_phase_bit_does_not_fit(calls):
    CT = B.PHASE_COLLISION_THEN_EXCLUSIVE
    pipe = _pipe(TINY, row_sorted=False)
    pipe.step_sync(0, _batch(TINY), torch.zeros(1, TINY.D))
    assert _names(calls)[-2:] == [("fs_emb_gather", None), ("fs_emb_backward_adagrad", CT)]
    calls.clear()
    pipe = _pipe(TINY)
    pipe.w = TINY.scaled(R=(1 << 30) + 1)          # rows beyond 2^30: no room for the phase bit
    pipe.step_sync(0, _batch(TINY), torch.zeros(1, TINY.D))
    assert _names(calls)[-2:] == [("fs_emb_gather", None), ("fs_emb_backward_adagrad", CT)]


def test_gather_only_workload_gathers_in_shard_major_order(calls):
    w = synthetic.WORKLOADS["vbs-gather"].scaled(R=1000)
    pipe = _pipe(w)
    pipe.step_sync(0, _batch(w), None)
    names = [n for n, _ in calls]
    # the lookup reads the shard-major IDs (each shard's rows together) and scatters to batch-major positions
    assert "fs_balance_vbs" in names and names[-1] == "fs_emb_gather_shard_major"
    assert not {"fs_emb_sort_rows", "fs_emb_sort_rows_sharded", "fs_emb_update_sorted", "fs_vbs_autotune"} & set(names)
    assert KWARGS["fs_collision_split_bitmaps"]["want_t_mask"] is False       # nothing reads the masks


def test_autotune_folds_the_times_in_before_the_next_cut(calls):
    w = synthetic.WORKLOADS["long-seq-autotune"].scaled(B=2, R=1000)
    pipe = _pipe(w)
    assert pipe.batch_delta is not None and pipe.batch_delta.shape == (w.n,)
    pipe.step_sync(0, _batch(w), None, times=torch.zeros(w.n, dtype=torch.int64))
    names = [n for n, _ in calls]
    assert names.index("fs_vbs_autotune") < names.index("fs_balance_vbs_tuned")
    assert "fs_balance_vbs" not in names
    calls.clear()
    pipe.step_sync(0, _batch(w), None)              # no times reported: the corrections stay as they are
    assert "fs_vbs_autotune" not in [n for n, _ in calls]


def test_prioritized_order_follows_algorithm_2(calls):
    pipe = _pipe(TINY, two_outputs=True)
    K = 3
    pipe.run_prioritized([_batch(TINY) for _ in range(K)], [torch.zeros(1, TINY.D)] * K)
    C, X, A = B.PHASE_COLLISION, B.PHASE_EXCLUSIVE, B.PHASE_ALL
    seq = [(n, ph) for n, ph in _names(calls) if n != "fs_collision_split_bitmaps"]
    expect = [("fs_emb_gather", None)]                                    # forward of the first batch
    for t in range(K):
        if t > 0:
            expect.append(("fs_emb_backward_adagrad", X))                 # line 7: exclusive rows of t-1
        if t + 1 < K:
            expect.append(("fs_emb_gather", None))                        # line 12: prefetch exclusive rows of t+1
            expect.append(("fs_emb_backward_adagrad", C))                 # line 20: collision rows of t
            expect.append(("fs_emb_gather", None))                        # line 21: collision rows of t+1
        else:
            expect.append(("fs_emb_backward_adagrad", A))
    assert seq == expect
    assert pipe.mask_layout == ["batch"] * 3        # the masked lookups and updates read batch-major masks
    assert len(pipe.slots) == 3                     # batches t-1 (deferred update), t and t+1
