"""Pins of the oracle's embedding gather and backward (CPU only).

FreeScale (arXiv 2604.24073) Algorithm 2: Lookup (line 12), merge (line 15),
split of the gradients (line 18) and update_embedding (lines 7 and 20).  The
optimizer is not named on the pages; the checks pin the standard SGD and
row-wise Adagrad (Duchi, Hazan & Singer 2011) through library reductions
(torch.index_add_ in fp64), closed forms and exact rational rounding.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ------------------------------------------------------------------ gather

@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_gather_is_row_indexing(dtype):
    rng = np.random.default_rng(1)
    R, D, T = 300, 64 if dtype == np.float32 else 128, 2000
    table = rng.integers(0, 2**16 if dtype == np.uint16 else 2**31, (R, D)).astype(dtype)
    ids = rng.integers(0, R, T)
    out = oracle.emb_gather(table, ids)
    assert np.array_equal(out, table[ids])                      # numpy fancy indexing
    ref = torch.nn.functional.embedding(torch.from_numpy(ids), torch.from_numpy(table.astype(np.int64)))
    assert np.array_equal(out.astype(np.int64), ref.numpy())


def test_gather_masked_leaves_other_rows():
    rng = np.random.default_rng(2)
    table = rng.standard_normal((50, 64)).astype(np.float32)
    ids = rng.integers(0, 50, 500)
    mask = rng.integers(0, 2, 500).astype(np.uint8)
    canary = np.full((500, 64), np.float32(-7.25))
    out = oracle.emb_gather(table, ids, mask=mask, sel=0, out=canary.copy())
    assert np.array_equal(out[mask == 0], table[ids[mask == 0]])
    assert (out[mask == 1] == np.float32(-7.25)).all()
    # merge: the two masked halves together are the full gather (Algorithm 2 line 15)
    oracle.emb_gather(table, ids, mask=mask, sel=1, out=out)
    assert np.array_equal(out, table[ids])


def test_gather_rejects_bad_id():
    with pytest.raises(oracle.OracleError):
        oracle.emb_gather(np.zeros((4, 4), np.float32), np.array([0, 4]))


# ------------------------------------------------------------------ bf16 rounding

def _nearest_bf16_exact(x: float) -> int:
    """Nearest bf16 (ties to even) by exact rational comparison against neighbours."""
    f = Fraction(x)
    lo_bits = int(_bf16_bits(np.array([x], np.float32))[0])            # a nearby bf16, then walk
    best = None
    for cand in range(lo_bits - 3, lo_bits + 4):
        c = cand & 0xFFFF
        v = Fraction(float(_bf16_to_f64(np.array([c], np.uint16))[0]))
        key = (abs(v - f), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_double_to_bf16_single_rounding():
    rng = np.random.default_rng(3)
    xs = list(rng.standard_normal(300) * 0.01) + list(rng.standard_normal(100) * 100)
    # values on and next to bf16 ties: 1 + 2^-8 is a tie between 1 and 1+2^-7
    xs += [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -40, -(1.0 + 2 ** -8), 0.0078125 * (1 + 2 ** -8)]
    for x in xs:
        assert oracle.double_to_bf16(float(x)) == _nearest_bf16_exact(float(x)), x
    assert oracle.double_to_bf16(1.0 + 2 ** -8) == 0x3F80                    # tie -> even (1.0)
    assert oracle.double_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82                # tie -> even (1+2^-6)
    assert oracle.double_to_bf16(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81         # just above the tie


# ------------------------------------------------------------------ backward

def _case(rng, R, D, T, dtype, zipf=False):
    if zipf:
        ids = np.minimum(rng.zipf(1.3, T) - 1, R - 1).astype(np.int64)
    else:
        ids = rng.integers(0, R, T).astype(np.int64)
    W = (rng.standard_normal((R, D)) * 0.01).astype(np.float32)
    G = rng.standard_normal((T, D)).astype(np.float32)
    if dtype == "bf16":
        W, G = _bf16_bits(W), _bf16_bits(G)
    return ids, W, G


def _as_f64(a):
    return a.astype(np.float64) if a.dtype == np.float32 else _bf16_to_f64(a)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segment_sums_equal_index_add(dtype):
    rng = np.random.default_rng(4)
    R, D, T = 500, 64 if dtype == "f32" else 128, 4000
    ids, W, G = _case(rng, R, D, T, dtype, zipf=True)
    rows, sums = oracle.emb_backward(W.copy(), np.zeros(R, np.float32), ids, G, "adagrad", 0.01, 1e-8,
                                     want_sums=True)
    ref = torch.zeros(R, D, dtype=torch.float64)
    ref.index_add_(0, torch.from_numpy(ids), torch.from_numpy(_as_f64(G)))   # library segment sum, fp64
    uniq = np.unique(ids)
    assert np.array_equal(rows, uniq)
    np.testing.assert_allclose(sums, ref.numpy()[uniq], rtol=1e-12, atol=1e-12)
    # sum over rows of g_r = sum over positions of G_p
    np.testing.assert_allclose(sums.sum(0), _as_f64(G).sum(0), rtol=1e-10, atol=1e-9)


def test_sgd_update_closed_form():
    rng = np.random.default_rng(5)
    R, D, T = 200, 64, 3000
    ids, W, G = _case(rng, R, D, T, "f32")
    W1 = W.copy()
    oracle.emb_backward(W1, None, ids, G, "sgd", 0.01)
    g = torch.zeros(R, D, dtype=torch.float64).index_add_(0, torch.from_numpy(ids), torch.from_numpy(G.astype(np.float64)))
    expect = (W.astype(np.float64) - 0.01 * g.numpy()).astype(np.float32)
    assert np.array_equal(W1, expect)
    W2 = W.copy()
    oracle.emb_backward(W2, None, ids, G, "sgd", 0.0)                    # lr = 0: unchanged
    assert np.array_equal(W2, W)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_adagrad_single_occurrence_closed_form(dtype):
    """One occurrence with g = c * ones(D): s = c^2, W' = W - lr * c / (|c| + eps)."""
    R, D, lr, eps = 8, 64, 0.01, 1e-8
    W = np.full((R, D), 0.25, np.float32)
    c = np.float32(-1.5)
    G = np.full((1, D), c, np.float32)
    if dtype == "bf16":
        W, G = _bf16_bits(W), _bf16_bits(G)
    s = np.zeros(R, np.float32)
    oracle.emb_backward(W, s, np.array([3]), G, "adagrad", lr, eps)
    assert s[3] == np.float32(2.25) and (np.delete(s, 3) == 0).all()
    expect = 0.25 - lr * float(c) / (1.5 + eps)
    got = _as_f64(W)
    if dtype == "f32":
        assert (got[3] == np.float32(expect)).all()
    else:
        assert (W[3] == oracle.double_to_bf16(expect)).all()
    assert (np.delete(got, 3, axis=0) == 0.25).all()                     # untouched rows


def test_adagrad_two_steps_closed_form():
    R, D, lr, eps = 4, 64, 0.05, 1e-8
    W = np.zeros((R, D), np.float32)
    s = np.zeros(R, np.float32)
    G = np.full((1, D), 2.0, np.float32)
    oracle.emb_backward(W, s, np.array([1]), G, "adagrad", lr, eps)
    oracle.emb_backward(W, s, np.array([1]), G, "adagrad", lr, eps)
    assert s[1] == 8.0
    e1 = np.float32(0.0 - lr * 2.0 / (2.0 + eps))
    e2 = np.float32(float(e1) - lr * 2.0 / (np.sqrt(8.0) + eps))
    assert (W[1] == e2).all()


def test_adagrad_lr_zero_keeps_weights_accumulates_state():
    rng = np.random.default_rng(6)
    ids, W, G = _case(rng, 100, 64, 500, "f32")
    W1, s = W.copy(), np.zeros(100, np.float32)
    oracle.emb_backward(W1, s, ids, G, "adagrad", 0.0, 1e-8)
    assert np.array_equal(W1, W)
    g = torch.zeros(100, 64, dtype=torch.float64).index_add_(0, torch.from_numpy(ids), torch.from_numpy(G.astype(np.float64)))
    expect = (g.numpy() ** 2).mean(axis=1).astype(np.float32)
    np.testing.assert_allclose(s, expect, rtol=1e-6)


def test_phases_partition_rows_and_compose():
    """Collision phase then exclusive phase == one update of every row once (Algorithm 2 lines 7, 20)."""
    rng = np.random.default_rng(7)
    R, D, T = 300, 64, 3000
    ids, W, G = _case(rng, R, D, T, "f32", zipf=True)
    nxt = rng.integers(0, R, 2000)
    is_co = np.isin(ids, nxt).astype(np.uint8)
    Wa, sa = W.copy(), np.zeros(R, np.float32)
    rows1, _ = oracle.emb_backward(Wa, sa, ids, G, "adagrad", 0.01, 1e-8, is_co=is_co, phase=1, want_sums=True)
    rows2, _ = oracle.emb_backward(Wa, sa, ids, G, "adagrad", 0.01, 1e-8, is_co=is_co, phase=2, want_sums=True)
    assert set(rows1.tolist()).isdisjoint(rows2.tolist())
    assert sorted(rows1.tolist() + rows2.tolist()) == np.unique(ids).tolist()     # each row exactly once
    assert set(rows1.tolist()) == set(ids.tolist()) & set(nxt.tolist())
    Wb, sb = W.copy(), np.zeros(R, np.float32)
    oracle.emb_backward(Wb, sb, ids, G, "adagrad", 0.01, 1e-8)
    assert np.array_equal(Wa, Wb) and np.array_equal(sa, sb)
