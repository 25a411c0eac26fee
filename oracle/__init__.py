"""CPU oracle of the FreeScale jagged index + embedding hot path.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and
by the CPU-baseline / reference arm of bench.py, never by the CUDA library or
its binding.  It shares no code with the CUDA path.  The arithmetic lives in
oracle.cpp (plain C++17, fp64 accumulation); this module only marshals numpy
arrays through ctypes and sequences the steps of one training iteration
(FreeScale, arXiv 2604.24073, Algorithm 2) in the synchronous and in the
prioritized order.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

ERRORS = {1: "invalid argument", 2: "ID outside [0, R)", 3: "malformed offsets or permutation"}


class OracleError(RuntimeError):
    pass


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i64, i32, f64, u8 = C.c_int64, C.c_int32, C.c_double, C.c_uint8
        sig = {
            "oracle_balance_fbs": [P, i64, i32, P, P],
            "oracle_balance_vbs": [P, i64, i32, f64, i32, P, P, P],
            "oracle_vbs_autotune": [P, i32, i64, i32, P],
            "oracle_balance_vbs_tuned": [P, i64, i32, f64, i32, P, P, P, P],
            "oracle_permute_jagged": [P, P, i64, P, P, P],
            "oracle_keyed_transpose": [P, P, i64, i64, P, P, P],
            "oracle_bucketize_rowwise": [P, i64, P, i32, i64, P, P, P, P],
            "oracle_collision_split": [P, i64, P, i64, i64, i32, P, P, P, i64, P, P, P, P, P, P],
            "oracle_emb_gather": [P, i64, i64, P, i64, P, u8, P],
            "oracle_emb_backward": [P, P, i64, i32, i32, i32, P, P, i64, P, i32, f64, f64, P, P, P],
            "oracle_permute_jagged_mt": [P, P, i64, P, P, P, i32],
            "oracle_bucketize_rowwise_mt": [P, i64, P, i32, i64, P, P, P, P, i32],
            "oracle_collision_split_mt": [P, i64, P, i64, i64, i32, P, P, P, i64, P, P, P, P, P, P, i32],
            "oracle_emb_gather_mt": [P, i64, i64, P, i64, P, u8, P, i32],
            "oracle_emb_backward_mt": [P, P, i64, i32, i32, i32, P, P, i64, P, i32, f64, f64, i32],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = C.c_int
        L.oracle_vbs_weight.argtypes = [i32, f64]
        L.oracle_vbs_weight.restype = C.c_uint64
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_bf16_to_double.restype = f64
        L.oracle_double_to_bf16.argtypes = [f64]
        L.oracle_double_to_bf16.restype = C.c_uint16
        _lib = L
    return _lib


_threads = 1


def set_threads(k):
    """Host threads the oracle's steps use from now on (1 = the single-threaded functions).  With k > 1 the
    permute, bucketize, collision split, gather and update run their *_mt variants, which give the same
    results; the balance stays single-threaded (a sort of the S sample lengths)."""
    global _threads
    _threads = max(1, int(k))


def threads():
    return _threads


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc):
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"error {rc}"))


# --------------------------------------------------------------- partition

def balance_fbs(uih_len, n):
    L = _c(uih_len, np.int32)
    S = L.shape[0]
    perm = np.empty(S, np.int32)
    ro = np.empty(n + 1, np.int64)
    _check(lib().oracle_balance_fbs(_p(L), S, n, _p(perm), _p(ro)))
    return perm, ro


def vbs_weight(L, alpha):
    return int(lib().oracle_vbs_weight(int(L), float(alpha)))


def balance_vbs(uih_len, n, alpha, sort_by_len):
    L = _c(uih_len, np.int32)
    S = L.shape[0]
    perm = np.empty(S, np.int32)
    ro = np.empty(n + 1, np.int64)
    sw = np.empty(n, np.uint64)
    _check(lib().oracle_balance_vbs(_p(L), S, n, float(alpha), int(bool(sort_by_len)), _p(perm), _p(ro), _p(sw)))
    return perm, ro, sw


def vbs_autotune(times, delta, step=1, tol_ppm=0):
    """One AutoTune update: returns the new per-rank batch corrections."""
    t = _c(times, np.int64)
    d = _c(delta, np.int64).copy()
    if d.shape != t.shape:
        raise OracleError("times and delta differ in length")
    _check(lib().oracle_vbs_autotune(_p(t), t.shape[0], int(step), int(tol_ppm), _p(d)))
    return d


def balance_vbs_tuned(uih_len, n, alpha, sort_by_len, delta):
    L = _c(uih_len, np.int32)
    d = _c(delta, np.int64)
    if d.shape != (n,):
        raise OracleError("delta must hold n values")
    S = L.shape[0]
    perm = np.empty(S, np.int32)
    ro = np.empty(n + 1, np.int64)
    sw = np.empty(n, np.uint64)
    _check(lib().oracle_balance_vbs_tuned(_p(L), S, n, float(alpha), int(bool(sort_by_len)), _p(d), _p(perm),
                                          _p(ro), _p(sw)))
    return perm, ro, sw


# --------------------------------------------------------------- jagged ids

def permute_jagged(offsets, values, perm):
    off = _c(offsets, np.int64)
    val = _c(values, np.int64)
    pm = _c(perm, np.int32)
    S = off.shape[0] - 1
    out_off = np.empty(S + 1, np.int64)
    out_val = np.empty(val.shape[0], np.int64)
    if _threads > 1:
        _check(lib().oracle_permute_jagged_mt(_p(off), _p(val), S, _p(pm), _p(out_off), _p(out_val), _threads))
    else:
        _check(lib().oracle_permute_jagged(_p(off), _p(val), S, _p(pm), _p(out_off), _p(out_val)))
    return out_off, out_val


def keyed_transpose(offsets, values, F, B, row_base=None):
    off = _c(offsets, np.int64)
    val = _c(values, np.int64)
    rb = None if row_base is None else _c(row_base, np.int64)
    out_off = np.empty(F * B + 1, np.int64)
    out_val = np.empty(val.shape[0], np.int64)
    _check(lib().oracle_keyed_transpose(_p(off), _p(val), int(F), int(B), None if rb is None else _p(rb),
                                        _p(out_off), _p(out_val)))
    return out_off, out_val


def bucketize_rowwise(ids, rank_id_offsets, n, R):
    x = _c(ids, np.int64)
    rio = _c(rank_id_offsets, np.int64)
    T = x.shape[0]
    sm = np.empty(T, np.int64)
    pos = np.empty(T, np.int32)
    splits = np.empty(n * n, np.int64)
    so = np.empty(n + 1, np.int64)
    if _threads > 1:
        _check(lib().oracle_bucketize_rowwise_mt(_p(x), T, _p(rio), n, R, _p(sm), _p(pos), _p(splits), _p(so),
                                                 _threads))
    else:
        _check(lib().oracle_bucketize_rowwise(_p(x), T, _p(rio), n, R, _p(sm), _p(pos), _p(splits), _p(so)))
    return sm, pos, splits.reshape(n, n), so


def collision_split(ids_t, ids_next, R, n):
    a = _c(ids_t, np.int64)
    b = _c(ids_next, np.int64)
    cap = a.shape[0] + b.shape[0]
    co = np.empty(cap, np.int64)
    ext = np.empty(cap, np.int64)
    exn = np.empty(cap, np.int64)
    counts = np.empty(3, np.int64)
    offs = [np.empty(n + 1, np.int64) for _ in range(3)]
    m_t = np.empty(a.shape[0], np.uint8)
    m_n = np.empty(b.shape[0], np.uint8)
    args = (_p(a), a.shape[0], _p(b), b.shape[0], R, n, _p(co), _p(ext), _p(exn), cap, _p(counts), _p(offs[0]),
            _p(offs[1]), _p(offs[2]), _p(m_t), _p(m_n))
    if _threads > 1:
        _check(lib().oracle_collision_split_mt(*args, _threads))
    else:
        _check(lib().oracle_collision_split(*args))
    c0, c1, c2 = (int(v) for v in counts)
    return {"co": co[:c0].copy(), "ex_t": ext[:c1].copy(), "ex_next": exn[:c2].copy(),
            "co_off": offs[0], "ex_t_off": offs[1], "ex_next_off": offs[2],
            "is_co_t": m_t, "is_co_next": m_n}


# --------------------------------------------------------------- embeddings

def _dtype_code(arr):
    if arr.dtype == np.float32:
        return 0
    if arr.dtype == np.uint16:  # bf16 bit patterns
        return 1
    raise TypeError("table must be float32 or uint16 (bf16 bits)")


def emb_gather(table, ids, mask=None, sel=1, out=None):
    """table: [R, D] float32 or uint16 (bf16 bits); returns / fills out [T, D]."""
    tb = np.ascontiguousarray(table)
    x = _c(ids, np.int64)
    T = x.shape[0]
    if out is None:
        out = np.zeros((T,) + tb.shape[1:], tb.dtype)
    m = None if mask is None else _c(mask, np.uint8)
    rb = tb.dtype.itemsize * (tb.shape[1] if tb.ndim > 1 else 1)
    if _threads > 1:
        _check(lib().oracle_emb_gather_mt(_p(tb), tb.shape[0], rb, _p(x), T, _p(m), int(sel), _p(out), _threads))
    else:
        _check(lib().oracle_emb_gather(_p(tb), tb.shape[0], rb, _p(x), T, _p(m), int(sel), _p(out)))
    return out


def emb_backward(table, state, ids, grads, optim, lr, eps=0.0, is_co=None, phase=0, want_sums=False):
    """In-place update of table (and state).  optim: 'sgd' | 'adagrad'.

    phase: 0 all positions, 1 collision rows (is_co == 1), 2 exclusive rows.
    Returns (rows, fp64 sums) when want_sums, else None.
    """
    assert table.flags.c_contiguous and grads.flags.c_contiguous
    dt = _dtype_code(table)
    assert grads.dtype == table.dtype
    R, D = table.shape
    x = _c(ids, np.int64)
    T = x.shape[0]
    m = None if is_co is None else _c(is_co, np.uint8)
    oc = {"sgd": 0, "adagrad": 1}[optim]
    if oc == 1:
        assert state is not None and state.dtype == np.float32 and state.flags.c_contiguous
    g_out = rows = None
    nrows = np.zeros(1, np.int64)
    if want_sums:
        g_out = np.empty((T, D), np.float64)
        rows = np.empty(T, np.int64)
    if _threads > 1 and not want_sums:
        _check(lib().oracle_emb_backward_mt(_p(table), _p(state) if oc == 1 else None, R, D, dt, oc, _p(x),
                                            _p(grads), T, _p(m), int(phase), float(lr), float(eps), _threads))
        return None
    _check(lib().oracle_emb_backward(_p(table), _p(state) if oc == 1 else None, R, D, dt, oc, _p(x), _p(grads), T,
                                     _p(m), int(phase), float(lr), float(eps), _p(g_out), _p(rows), _p(nrows)))
    if want_sums:
        k = int(nrows[0])
        return rows[:k].copy(), g_out[:k].copy()
    return None


def bf16_to_double(h):
    return lib().oracle_bf16_to_double(int(h))


def double_to_bf16(x):
    return int(lib().oracle_double_to_bf16(float(x)))


# --------------------------------------------------------------- one iteration

def prepare(w, b, delta=None):
    """Balance, permute and bucketize one batch (FreeScale Algorithm 1, Algorithm 2 line 8).

    w: a synthetic.Workload; b: a batch dict of numpy arrays (uih_len, offsets, ids; with composite
    candidates also cand_offsets, cand_lens); delta: the VBS AutoTune corrections, when w.autotune.
    """
    if w.balance == "fbs":
        perm, ro = balance_fbs(b["uih_len"], w.n)
        sw = None
    elif w.autotune:
        perm, ro, sw = balance_vbs_tuned(b["uih_len"], w.n, w.alpha, w.sort_by_len,
                                         np.zeros(w.n, np.int64) if delta is None else delta)
    else:
        perm, ro, sw = balance_vbs(b["uih_len"], w.n, w.alpha, w.sort_by_len)
    off2, ids2 = permute_jagged(b["offsets"], b["ids"], perm)
    rio = off2[ro]
    sm, pos, splits, so = bucketize_rowwise(ids2, rio, w.n, w.R)
    res = {"perm": perm, "rank_offsets": ro, "seg_weight": sw, "offsets": off2, "ids": ids2,
           "rank_id_offsets": rio, "sm_ids": sm, "pos": pos, "splits": splits, "shard_offsets": so}
    if "cand_lens" in b:
        # composite candidates (Algorithm 1 Stage II): their lengths move with the samples
        res["cand_offsets"], res["cand_lens"] = permute_jagged(b["cand_offsets"], b["cand_lens"], perm)
    return res


def _prepare_all(w, batches, times_list):
    """Prepare every batch; with AutoTune on, the times reported in iteration t
    update the corrections before batch t+1 is cut (FreeScale §4.1)."""
    delta = np.zeros(w.n, np.int64)
    preps = []
    for t, b in enumerate(batches):
        if t > 0 and w.autotune and times_list is not None:
            delta = vbs_autotune(times_list[t - 1], delta, w.tune_step, w.tune_tol_ppm)
        preps.append(prepare(w, b, delta))
    return preps


def run_sync(w, batches, table, state, grads_list, times_list=None, keep_tables=False):
    """Synchronous schedule: for each iteration t, out_t = gather(W, I_t), then W <- update(W, G_t, I_t).

    Collision rows of t (rows shared with t+1) are updated before exclusive rows
    (same result: the two row sets are disjoint).  Returns per-iteration dicts
    and updates table/state in place.  keep_tables also records copies of the
    table (and state) before the gather of t and of the table after its update.
    """
    preps = _prepare_all(w, batches, times_list)
    res = []
    for t, pr in enumerate(preps):
        r = {"prep": pr}
        if keep_tables:
            r["table_before"] = table.copy()
            r["state_before"] = None if state is None else state.copy()
        out = emb_gather(table, pr["ids"])
        r["out"] = out
        if t + 1 < len(preps):
            r["coll"] = collision_split(pr["ids"], preps[t + 1]["ids"], w.R, w.n)
        if w.has_update:
            G = grads_list[t]
            if "coll" in r:
                m = r["coll"]["is_co_t"]
                emb_backward(table, state, pr["ids"], G, w.optim, w.lr, w.eps, is_co=m, phase=1)
                emb_backward(table, state, pr["ids"], G, w.optim, w.lr, w.eps, is_co=m, phase=2)
            else:
                emb_backward(table, state, pr["ids"], G, w.optim, w.lr, w.eps)
        if keep_tables:
            r["table_after"] = table.copy()
        res.append(r)
    return res


def run_prioritized(w, batches, table, state, grads_list, times_list=None):
    """Prioritized schedule of FreeScale Algorithm 2.

    Forward of iteration t: finish the exclusive update of t-1, prepare t+1,
    split collision / exclusive rows of (t, t+1), prefetch the exclusive rows
    of t+1.  Backward of t: update the collision rows of t first, then gather
    the collision rows of t+1.  The exclusive rows of the last iteration are
    updated at the end.
    """
    preps = _prepare_all(w, batches, times_list)
    K = len(preps)
    outs = [None] * K
    colls = [None] * K
    outs[0] = emb_gather(table, preps[0]["ids"])
    pending_ex = None
    for t in range(K):
        if pending_ex is not None:                       # Algorithm 2 line 7
            ids_prev, G_prev, m_prev = pending_ex
            emb_backward(table, state, ids_prev, G_prev, w.optim, w.lr, w.eps, is_co=m_prev, phase=2)
            pending_ex = None
        if t + 1 < K:                                    # lines 8-12
            colls[t] = collision_split(preps[t]["ids"], preps[t + 1]["ids"], w.R, w.n)
            nxt = np.zeros((preps[t + 1]["ids"].shape[0],) + table.shape[1:], table.dtype)
            emb_gather(table, preps[t + 1]["ids"], mask=colls[t]["is_co_next"], sel=0, out=nxt)
            outs[t + 1] = nxt
        if w.has_update:                                 # lines 18-21
            G = grads_list[t]
            if colls[t] is not None:
                m = colls[t]["is_co_t"]
                emb_backward(table, state, preps[t]["ids"], G, w.optim, w.lr, w.eps, is_co=m, phase=1)
                pending_ex = (preps[t]["ids"], G, m)
            else:
                emb_backward(table, state, preps[t]["ids"], G, w.optim, w.lr, w.eps)
        if t + 1 < K:
            emb_gather(table, preps[t + 1]["ids"], mask=colls[t]["is_co_next"], sel=1, out=outs[t + 1])
    if pending_ex is not None:
        ids_prev, G_prev, m_prev = pending_ex
        emb_backward(table, state, ids_prev, G_prev, w.optim, w.lr, w.eps, is_co=m_prev, phase=2)
    return [{"prep": preps[t], "out": outs[t], "coll": colls[t]} for t in range(K)]
