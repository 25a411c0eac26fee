"""Shared test helpers: moving synthetic data between devices and tolerance checks."""
import numpy as np
import torch


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    return t.detach().cpu().numpy().copy()


def batch_np(b):
    return {k: (to_np(v) if torch.is_tensor(v) else v) for k, v in b.items()}


def batch_to(b, device):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in b.items()}


def bf16_bits_to_f64(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def as_f64(a):
    return a.astype(np.float64) if a.dtype != np.uint16 else bf16_bits_to_f64(a)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.float64(2.0 ** -126))
    return np.exp2(np.floor(np.log2(ax)) - 7)


def update_scale(ids, grads, R, optim, lr, eps=0.0, state=None):
    """Per-element size of the update's rounding-sensitive part.

    The GPU sums gradients in fp32, the oracle in fp64; the error of a sum is
    bounded by a multiple of sqrt(sum_p G_{p,d}^2), not of |sum_p G_{p,d}|
    (cancellation).  SGD moves W by lr * g, so its scale is lr * sqrt(sum G^2);
    row-wise Adagrad moves it by lr * g / (sqrt(s) + eps), so its scale is
    lr * sqrt(sum G^2) / (sqrt(s) + eps), floored at lr.
    """
    import torch as _t
    G = _t.from_numpy(as_f64(np.ascontiguousarray(grads)))
    sq = _t.zeros(R, G.shape[1], dtype=_t.float64).index_add_(0, _t.from_numpy(np.asarray(ids, np.int64)), G * G)
    root = np.sqrt(sq.numpy())
    if optim == "sgd":
        return lr * root
    s = np.sqrt(np.asarray(state, np.float64))[:, None] + eps
    return np.maximum(lr * root / np.maximum(s, 1e-30), lr)


def assert_table_close(got, ref, dtype, lr, rtol=None, scale=None, ulps=1):
    """Updated weights: |gpu - oracle| <= rtol * max(|oracle|, scale); bf16 also accepts `ulps` ulps.

    scale defaults to lr (the size of one normalised Adagrad step); pass
    update_scale(...) for the exact per-element bound.  A bf16 table is rounded
    once per iteration on each side (fp32 -> bf16 on the GPU, fp64 -> bf16 in
    the oracle), so after k iterations the two may sit k ulps apart.
    """
    g, r = as_f64(got), as_f64(ref)
    sc = lr if scale is None else scale
    if dtype == "f32":
        rtol = 1e-5 if rtol is None else rtol
        tol = rtol * np.maximum(np.abs(r), sc)
    else:
        rtol = 1e-2 if rtol is None else rtol
        tol = np.maximum(rtol * np.maximum(np.abs(r), sc), bf16_ulp(r) * (ulps + 0.0001))
    bad = np.abs(g - r) > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance; first {idx.tolist()}: "
                             f"gpu={g[tuple(idx[0])]} ref={r[tuple(idx[0])]} tol={tol[tuple(idx[0])]}")


def assert_state_close(got, ref, rtol=1e-5):
    g, r = got.astype(np.float64), ref.astype(np.float64)
    tol = rtol * np.maximum(np.abs(r), 1e-30)
    bad = np.abs(g - r) > tol
    if bad.any():
        i = int(np.argwhere(bad)[0][0])
        raise AssertionError(f"{int(bad.sum())} state entries out of tolerance; first row {i}: {g[i]} vs {r[i]}")


class Guarded:
    """A device tensor between two guard bands of seeded bytes (4 KB each).

    `t` is the tensor a call may write (exactly `shape`, no slack); `check()`
    asserts that neither band changed, i.e. that the call wrote nothing before
    or after its output.  `init` fills `t` first (for in-place arguments).
    """

    BAND = 4096

    def __init__(self, shape, dtype, device="cuda", init=None, seed=0):
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (int(shape),)
        numel = int(np.prod(shape)) if shape else 1
        esz = torch.empty(0, dtype=dtype).element_size()
        self.band = self.BAND // esz
        self.nbytes = self.band * esz
        self.buf = torch.empty(numel + 2 * self.band, dtype=dtype, device=device)
        g = torch.Generator().manual_seed(numel * 31 + seed)
        raw = self.buf.view(torch.uint8)
        self.pattern = torch.randint(0, 256, (raw.numel(),), dtype=torch.uint8, generator=g)
        raw.copy_(self.pattern.to(device))
        self.t = self.buf[self.band: self.band + numel].view(shape)
        if init is not None:
            self.t.copy_(init)

    def check(self, what=""):
        raw = self.buf.view(torch.uint8).cpu()
        nb = self.nbytes
        assert torch.equal(raw[:nb], self.pattern[:nb]), f"{what}: guard band before the output was written"
        assert torch.equal(raw[-nb:], self.pattern[-nb:]), f"{what}: guard band after the output was written"
