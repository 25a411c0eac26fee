"""Parity at the full sizes of the gated workloads (GPU, slow).

The mid-size full step (64 x 256 samples, 10M x 128 bf16, Adagrad), the
long-sequence index workload (512 x 64 samples up to 16K IDs, 50M rows,
three iterations) and the large-table full step (256 x 512 samples, 100M x 64
f32 + Adagrad state, about 303M IDs per batch) run through the synchronous
pipeline at their own sizes, in the launch configuration the benchmark times
(inputs generated on the device, one gradient pool whose first T rows are
batch t's), and are checked against the CPU oracle:

* every index output bit for bit: partition, permuted offsets and IDs, rank ID
  ranges, shard-major IDs, positions, send splits, shard offsets, the
  collision / exclusive lists with their shard offsets and the collision mask
  of t (FreeScale Algorithm 1; Algorithm 2 lines 8 and 10);
* gathered rows at 100k seeded positions per iteration, bit for bit against
  the oracle's gather of the table rows the GPU read (Algorithm 2 line 12);
* the update (Algorithm 2 lines 18-20): for 10k seeded rows of uniq(I^t) and
  its two hottest rows (millions of positions) the oracle recomputes the new weights and Adagrad state from those rows' own
  positions and gradients (the update is per row, so the subset result is
  exact), within the update tolerance; 10k seeded rows outside uniq(I^t) must
  not change at all.

The oracle runs beside the GPU in a thread of its own (its calls release the
interpreter lock) on every host core: its multi-threaded variants, which the
CPU tests (tests/test_oracle_threads.py) prove identical to the
single-threaded functions, because the single-threaded oracle needs minutes
per 300M-ID batch.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from jagged_embedding_gb300 import synthetic
from jagged_embedding_gb300.pipeline import Pipeline
from tests.helpers import assert_state_close, assert_table_close, batch_np, to_np, update_scale

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda")

# iterations checked per workload (the long-sequence workload's three, so both collision pairs)
ITERS = {"mid-full-step": 2, "long-seq-index": 3, "large-table-full-step": 2}
GATHER_SAMPLE = 100_000
ROW_SAMPLE = 10_000


@pytest.fixture(autouse=True)
def _free_cached_memory():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    yield
    oracle.set_threads(1)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _index_outputs(w, s, T):
    snap = {"perm": to_np(s.perm[: w.S]), "rank_offsets": to_np(s.rank_offsets), "offsets": to_np(s.offsets[: w.S + 1]),
            "ids": to_np(s.ids[:T]), "rank_id_offsets": to_np(s.rank_id_offsets), "sm_ids": to_np(s.sm_ids[:T]),
            "pos": to_np(s.pos[:T]), "splits": to_np(s.splits), "shard_offsets": to_np(s.shard_offsets)}
    if w.balance == "vbs":
        snap["seg_weight"] = to_np(s.seg_weight)
    return snap


def _assert_prep_equal(g, p, t):
    for k in ("perm", "rank_offsets", "offsets", "ids", "rank_id_offsets", "sm_ids", "pos", "splits",
              "shard_offsets"):
        assert np.array_equal(g[k], p[k]), (t, k)
    if "seg_weight" in g:
        assert np.array_equal(g["seg_weight"].astype(np.uint64), p["seg_weight"]), t


@pytest.mark.parametrize("name", list(ITERS))
def test_full_size_matches_oracle(name):
    w = synthetic.WORKLOADS[name]
    K = ITERS[name]
    batches = [synthetic.batch(w, t, DEV) for t in range(K)]
    synthetic._cdf_cache.clear()
    Ts = [b["T"] for b in batches]
    table = synthetic.table(w, DEV)
    state = torch.zeros(w.R, dtype=torch.float32, device=DEV) if w.optim == "adagrad" else None
    grads = synthetic.grads(w, max(Ts), 0, DEV) if w.has_update else None
    nb = [batch_np(b) for b in batches]

    oracle.set_threads(os.cpu_count() or 1)
    pool = cf.ThreadPoolExecutor(max_workers=1)    # one oracle step at a time, each on every core
    preps = [pool.submit(oracle.prepare, w, nb[t]) for t in range(K)]

    def coll_of(t):
        return oracle.collision_split(preps[t].result()["ids"], preps[t + 1].result()["ids"], w.R, w.n)

    colls = [pool.submit(coll_of, t) for t in range(K - 1)]

    pipe = Pipeline(w, DEV, max(Ts), table, state)
    rng = np.random.default_rng(7000 + w.seed_base)
    pipe.prepare(batches[0], 0)
    cur = 0
    for t in range(K):
        s = pipe.slots[cur]
        T = s.T
        assert T == Ts[t]
        has_next = t + 1 < K
        torch.cuda.synchronize()
        got = _index_outputs(w, s, T)
        ids_d = s.ids[:T]

        # rows the checks read from the table as the gather of t sees it
        gpos = np.sort(rng.choice(T, size=min(T, GATHER_SAMPLE), replace=False))
        grows = got["ids"][gpos]
        p = preps[t].result()
        _assert_prep_equal(got, p, t)
        coll = colls[t].result() if has_next else None
        if coll is not None:
            uniq = np.concatenate([coll["co"], coll["ex_t"]])
            uniq.sort()
        else:
            uniq = np.unique(p["ids"])
        # seeded rows of the batch plus its two hottest (Zipf ranks 0 and 1: millions of positions,
        # carries across thousands of reduce tiles)
        hot = np.array([(k * synthetic.scramble_multiplier(w.R)) % w.R for k in (0, 1)], np.int64)
        urows = np.union1d(rng.choice(uniq, size=min(uniq.size, ROW_SAMPLE), replace=False),
                           hot[np.isin(hot, uniq)])
        others = np.setdiff1d(rng.integers(0, w.R, size=4 * ROW_SAMPLE), uniq)[:ROW_SAMPLE]
        need = np.union1d(np.union1d(grows, urows), others)
        need_d = torch.from_numpy(need).to(DEV)
        tab_before = to_np(table[need_d])
        st_before = to_np(state[need_d]) if state is not None else None

        # (want_masks: the masks are written for the check below; the step's calls are the benchmark's)
        nxt = pipe.step_sync(cur, batches[t + 1] if has_next else None, grads[:T] if grads is not None else None,
                             has_next=has_next, want_masks=True)
        B.check(pipe.err, f"{name} iteration {t}")

        # gathered rows: bit for bit
        out_s = to_np(pipe.out[0][torch.from_numpy(gpos).to(DEV)])
        ref_s = oracle.emb_gather(tab_before, np.searchsorted(need, grows))
        assert np.array_equal(out_s, ref_s), t

        if coll is not None:
            c = {k: to_np(v) for k, v in pipe.coll.items()}
            counts = c["counts"]
            assert np.array_equal(c["co"][: counts[0]], coll["co"]), t
            assert np.array_equal(c["ex_t"][: counts[1]], coll["ex_t"]), t
            assert np.array_equal(c["ex_next"][: counts[2]], coll["ex_next"]), t
            for k in ("co_off", "ex_t_off", "ex_next_off"):
                assert np.array_equal(c[k], coll[k]), (t, k)
            m = to_np(pipe.masks[cur][:T])
            if pipe.mask_layout[cur] == "shard":        # aligned with the shard-major IDs
                assert np.array_equal(m, coll["is_co_t"][got["pos"]]), t
            else:
                assert np.array_equal(m, coll["is_co_t"]), t

        if w.has_update:
            # the oracle's update of the sampled rows, from their own positions (ascending)
            ur_d = torch.from_numpy(urows).to(DEV)
            idx_d = torch.nonzero(torch.isin(ids_d, ur_d)).flatten()
            idx = to_np(idx_d)
            sub_ids = np.searchsorted(urows, got["ids"][idx])
            G = to_np(grads[idx_d])
            at = np.searchsorted(need, urows)
            sub_tab = np.ascontiguousarray(tab_before[at])
            sub_st = np.ascontiguousarray(st_before[at]) if st_before is not None else None
            st0 = None if sub_st is None else sub_st.copy()
            if coll is not None:
                m = np.ascontiguousarray(coll["is_co_t"][idx])
                oracle.emb_backward(sub_tab, sub_st, sub_ids, G, w.optim, w.lr, w.eps, is_co=m, phase=1)
                oracle.emb_backward(sub_tab, sub_st, sub_ids, G, w.optim, w.lr, w.eps, is_co=m, phase=2)
            else:
                oracle.emb_backward(sub_tab, sub_st, sub_ids, G, w.optim, w.lr, w.eps)
            scale = update_scale(sub_ids, G, urows.size, w.optim, w.lr, w.eps, sub_st)
            assert_table_close(to_np(table[ur_d]), sub_tab, w.dtype, w.lr, scale=scale, ulps=1)
            if state is not None:
                assert_state_close(to_np(state[ur_d]), sub_st)
                assert (sub_st > st0).all()
            # rows outside the batch keep their bits
            oat = np.searchsorted(need, others)
            assert np.array_equal(to_np(table[torch.from_numpy(others).to(DEV)]), tab_before[oat]), t
        else:
            assert np.array_equal(to_np(table[need_d]), tab_before), t
        cur = nxt
    pool.shutdown()
    oracle.set_threads(1)
