"""The prioritized schedule reaches the synchronous result (CPU only).

FreeScale (arXiv 2604.24073) §3.2: enforcing write-read order on the collision
rows keeps numerical parity with the synchronized baseline; §5.4 reports the
same NE curves.  The oracle's Algorithm-2 ordering (exclusive rows prefetched,
collision rows updated first, exclusive updates deferred one iteration) must
give bit-identical gathered embeddings, tables and states.
"""
import numpy as np
import pytest

import oracle
from jagged_embedding_gb300 import synthetic


def _np(b):
    return {k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in b.items()}


def _table_np(w):
    t = synthetic.table(w)
    if w.dtype == "bf16":
        import torch
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def _grads_np(w, T, it):
    g = synthetic.grads(w, T, it)
    if w.dtype == "bf16":
        import torch
        return g.view(torch.int16).numpy().view(np.uint16).copy()
    return g.numpy().copy()


CASES = [
    synthetic.WORKLOADS["tiny-fbs-sgd"].scaled(iters=3),
    synthetic.WORKLOADS["mid-full-step"].scaled(n=4, B=8, R=5000, lmax=512, mu=4.0, iters=3),
    synthetic.WORKLOADS["large-table-full-step"].scaled(n=8, B=8, R=20000, lmax=1024, mu=4.5, iters=4),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_prioritized_equals_synchronous(w):
    batches = [_np(synthetic.batch(w, t)) for t in range(w.iters)]
    grads = [_grads_np(w, b["T"], t) for t, b in enumerate(batches)]
    t0 = _table_np(w)
    ta, tb = t0.copy(), t0.copy()
    sa, sb = np.zeros(w.R, np.float32), np.zeros(w.R, np.float32)
    ra = oracle.run_sync(w, batches, ta, sa, grads)
    rb = oracle.run_prioritized(w, batches, tb, sb, grads)
    for t in range(w.iters):
        assert np.array_equal(ra[t]["out"], rb[t]["out"]), t
    assert np.array_equal(ta, tb) and np.array_equal(sa, sb)
    assert not np.array_equal(ta, t0)                      # the updates did something


def test_stale_prefetch_differs():
    """Prefetching every row of t+1 before the update of t (no prioritization) reads stale rows."""
    w = CASES[0]
    batches = [_np(synthetic.batch(w, t)) for t in range(2)]
    grads = [_grads_np(w, b["T"], t) for t, b in enumerate(batches)]
    t0 = _table_np(w)
    ta = t0.copy()
    ra = oracle.run_sync(w, batches, ta, None, grads)
    p1 = oracle.prepare(w, batches[1])
    stale = oracle.emb_gather(t0, p1["ids"])               # gathered before the update of t = 0
    c = ra[0]["coll"]
    co_next = c["is_co_next"].astype(bool)
    assert co_next.any()
    assert not np.array_equal(stale[co_next], ra[1]["out"][co_next])   # collision rows are stale
    assert np.array_equal(stale[~co_next], ra[1]["out"][~co_next])     # exclusive rows are not
