"""The oracle's multi-threaded variants (used only to time the oracle on every
host core) give exactly the single-threaded oracle's results: index outputs,
collision lists and masks, gathered rows, and updated tables and states bit for
bit, at several thread counts, on seeded workload-shaped inputs (CPU)."""
import numpy as np
import pytest

import oracle
from jagged_embedding_gb300 import synthetic
from tests.helpers import batch_np, to_np


@pytest.fixture(autouse=True)
def _single_threaded_after():
    yield
    oracle.set_threads(1)


def _run(w, threads, table, grads):
    oracle.set_threads(threads)
    b = [batch_np(synthetic.batch(w, t)) for t in range(2)]
    p = [oracle.prepare(w, x) for x in b]
    coll = oracle.collision_split(p[0]["ids"], p[1]["ids"], w.R, w.n)
    out = oracle.emb_gather(table, p[0]["ids"])
    masked = np.full_like(out, 7)
    oracle.emb_gather(table, p[0]["ids"], mask=coll["is_co_t"], sel=0, out=masked)
    tab = table.copy()
    st = np.zeros(w.R, np.float32) if w.optim == "adagrad" else None
    if w.has_update:
        for ph in (1, 2):
            oracle.emb_backward(tab, st, p[0]["ids"], grads, w.optim, w.lr, w.eps, is_co=coll["is_co_t"], phase=ph)
        oracle.emb_backward(tab, st, p[0]["ids"], grads, w.optim, w.lr, w.eps)
    return p, coll, out, masked, tab, st


@pytest.mark.parametrize("name,kw", [("tiny-fbs-sgd", {}), ("mid-full-step", dict(B=4, R=200_000)),
                                     ("large-table-full-step", dict(B=2, R=300_000, lmax=4096)),
                                     ("long-seq-index", dict(B=1, R=400_000, lmax=4096)),
                                     ("composite-cand", {})])
def test_threads_give_the_single_threaded_results(name, kw):
    w = synthetic.WORKLOADS[name].scaled(**kw)
    table = to_np(synthetic.table(w))
    T0 = synthetic.batch(w, 0)["T"]
    grads = to_np(synthetic.grads(w, T0, 0)) if w.has_update else None
    ref = _run(w, 1, table, grads)
    for k in (2, 3, 8):
        got = _run(w, k, table, grads)
        for t in range(2):
            for key, v in ref[0][t].items():
                if v is not None:
                    assert np.array_equal(got[0][t][key], v), (k, t, key)
        for key, v in ref[1].items():
            assert np.array_equal(got[1][key], v), (k, key)
        for a, b in zip(got[2:], ref[2:]):
            assert (a is None and b is None) or np.array_equal(a, b), k


def test_threads_on_degenerate_sizes():
    for k in (1, 4, 64):
        oracle.set_threads(k)
        off, val = oracle.permute_jagged(np.zeros(1, np.int64), np.zeros(0, np.int64), np.zeros(0, np.int32))
        assert off.tolist() == [0] and val.size == 0
        sm, pos, splits, so = oracle.bucketize_rowwise(np.array([5, 0, 9], np.int64), np.array([0, 3], np.int64), 1,
                                                       10)
        assert sm.tolist() == [5, 0, 9] and pos.tolist() == [0, 1, 2] and so.tolist() == [0, 3]
        c = oracle.collision_split(np.array([3, 3, 1], np.int64), np.array([1, 2], np.int64), 4, 2)
        assert c["co"].tolist() == [1] and c["ex_t"].tolist() == [3] and c["ex_next"].tolist() == [2]
        assert c["is_co_t"].tolist() == [0, 0, 1] and c["is_co_next"].tolist() == [1, 0]
        assert c["co_off"].tolist() == [0, 1, 1]
        with pytest.raises(oracle.OracleError):
            oracle.bucketize_rowwise(np.array([10], np.int64), np.array([0, 1], np.int64), 1, 10)
