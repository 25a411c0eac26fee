"""Every row of the batch is updated exactly once, and no other row (GPU).

FreeScale Algorithm 2 (lines 7 and 20) splits uniq(I^t) into collision and
exclusive rows and updates each part once, collision rows first; the update
reduces the gradients of a row's positions and applies one optimizer step to
the row.  These tests count the updates in closed form instead of against a
second implementation: the table starts at zero, every gradient element is 1
and SGD's rate is 1, so a row that appears c times in the batch must end at
exactly -c (integers of at most 2^24 are exact in fp32; in bf16 the one
rounding of -c is what the expected value takes too).  A row updated twice ends
at -2c, a row skipped stays 0, a row updated for another ends non-zero where it
should be 0, and a carry lost between two reduce tiles gives a partial count.
Row-wise Adagrad from a zero state must leave state c^2 and weight -lr.

The multiplicities mix many rows seen 1..40 times with a few rows seen
thousands and hundreds of thousands of times (their runs cross many reduce
tiles and the block sums of the carry chains), in random positions.  Each
update entry point is covered: the one-call update, its two single-phase
calls, the batch-major sort + sorted update, and the per-shard sort from the
bucketize output + sorted update.
"""
import numpy as np
import pytest
import torch

from jagged_embedding_gb300 import binding as B
from tests.helpers import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _batch(seed, R, n_rows, hot_counts):
    """IDs in which row r appears count[r] times, in a random order; per-row collision flag."""
    rng = np.random.default_rng(seed)
    rows = rng.choice(R, size=n_rows + len(hot_counts), replace=False).astype(np.int64)
    counts = np.concatenate([rng.integers(1, 41, size=n_rows), np.asarray(hot_counts, np.int64)])
    ids = rng.permutation(np.repeat(rows, counts))
    co_row = rng.random(R) < 0.5
    count = np.zeros(R, np.int64)
    count[rows] = counts
    return ids, count, co_row


def _expected_sgd(count, dtype, phase_rows=None):
    c = count if phase_rows is None else np.where(phase_rows, count, 0)
    w = torch.from_numpy((-c).astype(np.float32))            # integer negation: untouched rows stay +0
    if dtype == torch.bfloat16:
        w = w.to(torch.bfloat16)                           # one rounding of the exact -c
    return to_np(w)


def _check_sgd(W, count, dtype, phase_rows=None):
    got = to_np(W)
    exp = _expected_sgd(count, dtype, phase_rows)
    assert np.array_equal(got, np.repeat(exp[:, None], got.shape[1], axis=1)), (
        "rows updated other than once: %d" % int((got != exp[:, None]).any(axis=1).sum()))


CASES = [
    # R, D, dtype, rows seen 1..40 times, rows seen many times
    (400_000, 64, torch.float32, 150_000, [3_000, 150_000]),
    (100_000, 128, torch.bfloat16, 40_000, [5_000, 70_000]),
    (64, 32, torch.float32, 60, [100_000]),                 # few rows, one of them in most positions
]


@pytest.mark.parametrize("R,D,dtype,n_rows,hot", CASES)
def test_one_call_update_touches_each_row_once(R, D, dtype, n_rows, hot):
    n_rows = min(n_rows, R - len(hot))
    ids, count, co_row = _batch(R + D, R, n_rows, hot)
    T = ids.size
    idd = torch.from_numpy(ids).to(DEV)
    G = torch.ones(T, D, dtype=dtype, device=DEV)
    is_co = torch.from_numpy(co_row[ids].astype(np.uint8)).to(DEV)

    W = torch.zeros(R, D, dtype=dtype, device=DEV)
    B.check(B.fs_emb_backward_adagrad(W, None, idd, G, "sgd", 1.0))
    _check_sgd(W, count, dtype)

    # the two phases of Algorithm 2, one call each: collision rows only, then the rest
    W = torch.zeros(R, D, dtype=dtype, device=DEV)
    B.check(B.fs_emb_backward_adagrad(W, None, idd, G, "sgd", 1.0, is_co=is_co, phase=B.PHASE_COLLISION))
    _check_sgd(W, count, dtype, phase_rows=co_row)
    B.check(B.fs_emb_backward_adagrad(W, None, idd, G, "sgd", 1.0, is_co=is_co, phase=B.PHASE_EXCLUSIVE))
    _check_sgd(W, count, dtype)


@pytest.mark.parametrize("R,D,dtype,n_rows,hot", CASES)
@pytest.mark.parametrize("sharded", [False, True])
def test_sorted_update_touches_each_row_once(R, D, dtype, n_rows, hot, sharded):
    n_rows = min(n_rows, R - len(hot))
    ids, count, co_row = _batch(R + 2 * D, R, n_rows, hot)
    T = ids.size
    n = 16 if R >= 16 else 1
    idd = torch.from_numpy(ids).to(DEV)
    G = torch.ones(T, D, dtype=dtype, device=DEV)
    is_co = torch.from_numpy(co_row[ids].astype(np.uint8)).to(DEV)
    two = B.PHASE_COLLISION_THEN_EXCLUSIVE
    for phase in (B.PHASE_ALL, two):
        W = torch.zeros(R, D, dtype=dtype, device=DEV)
        if sharded:
            rio = torch.tensor([T * r // n for r in range(n + 1)], dtype=torch.int64, device=DEV)
            sm, pos, _, so, err = B.fs_bucketize_rowwise(idd, rio, R)
            B.check(err)
            ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, D, B.dtype_code(W), n), DEV)
            err = B.fs_emb_sort_rows_sharded(W, sm, pos, so, ws, phase=phase,
                                             is_co=is_co[pos.long()].contiguous() if phase == two else None)
        else:
            ws = B.workspace(B.backward_workspace_size(T, R, D, B.dtype_code(W)), DEV)
            err = B.fs_emb_sort_rows(W, idd, ws, phase=phase, is_co=is_co if phase == two else None)
        B.fs_emb_update_sorted(W, None, G, T, ws, "sgd", 1.0, phase=phase, err=err)
        B.check(err)
        _check_sgd(W, count, dtype)


@pytest.mark.parametrize("sharded", [False, True])
def test_adagrad_state_counts_each_row_once(sharded):
    R, D = 200_000, 64
    ids, count, co_row = _batch(7, R, 80_000, [500, 20_000])
    T = ids.size
    idd = torch.from_numpy(ids).to(DEV)
    G = torch.ones(T, D, dtype=torch.float32, device=DEV)
    is_co = torch.from_numpy(co_row[ids].astype(np.uint8)).to(DEV)
    W = torch.zeros(R, D, device=DEV)
    s = torch.zeros(R, device=DEV)
    two = B.PHASE_COLLISION_THEN_EXCLUSIVE
    if sharded:
        n = 64
        rio = torch.tensor([T * r // n for r in range(n + 1)], dtype=torch.int64, device=DEV)
        sm, pos, _, so, err = B.fs_bucketize_rowwise(idd, rio, R)
        B.check(err)
        ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, D, B.dtype_code(W), n), DEV)
        err = B.fs_emb_sort_rows_sharded(W, sm, pos, so, ws, phase=two, is_co=is_co[pos.long()].contiguous())
    else:
        ws = B.workspace(B.backward_workspace_size(T, R, D, B.dtype_code(W)), DEV)
        err = B.fs_emb_sort_rows(W, idd, ws, phase=two, is_co=is_co)
    lr = 0.25
    B.fs_emb_update_sorted(W, s, G, T, ws, "adagrad", lr, 0.0, phase=two, err=err)
    B.check(err)
    s_got, w_got = to_np(s), to_np(W)
    seen = count > 0
    # s = c^2 (exact in fp32 up to c = 4096; relative 1e-6 above), weight -lr (one division)
    assert np.allclose(s_got[seen], count[seen].astype(np.float64) ** 2, rtol=1e-6, atol=0)
    assert np.allclose(w_got[seen], -lr, rtol=1e-6, atol=0)
    assert not s_got[~seen].any() and not w_got[~seen].any()
