"""Seeded synthetic inputs shaped like the FreeScale workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no balancing, sorting, bucketing, collision or update).
Both the CUDA path and the CPU oracle consume exactly the arrays it returns.

Recipe (FreeScale, arXiv 2604.24073: §2.2 for the skewed UIH-length
distribution and its 16K plateau, §3.1 / Algorithm 1 for a sample = UIH IDs
plus candidates, §5.2 for synthetic embedding workloads):

* sample g (global index, rank-major g = r*B + b) has UIH length
  L_g = clip(round_half_even(lognormal(mu, sigma)), 1, L_max) and
  C_g ~ U{c_min..c_max} candidates, each candidate one ID -- or, in a recipe
  with composite candidates (Algorithm 1 Stage II), each candidate c carries
  K_c ~ U{k_min..k_max} IDs, and the batch also holds the candidate lengths
  as a jagged tensor (cand_offsets by C_g, cand_lens = K_c);
* the jagged row of a sample is [UIH IDs | candidate IDs];
* every ID is drawn i.i.d. from a bounded Zipf law P(k) ~ (k+1)^-s over
  k in [0, R) by inverse CDF, then scrambled row = (k * A) mod R with
  A = 0x9E3779B97F4A7C15 mod R (bumped until gcd(A, R) = 1) so that hot rows
  spread over the row-range shards instead of piling into shard 0;
* table rows ~ N(0, 0.01^2) (std 0.01), stored fp32 or bf16 (RNE cast);
* gradients ~ N(0, 1) in the table dtype;
* with VBS AutoTune on, the ranks' step times are simulated clock readings
  (step_times, rank_times below): seeded integers, never computed from the
  method's own arithmetic.

Seeds: a batch of workload w at iteration i uses seed w.seed_base + i; the
table uses w.seed_base + 500; gradients w.seed_base + 600 + i.  torch
generators are used on whichever device is asked for, so CPU- and
CUDA-generated data have the same law but different values.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch

SCRAMBLE_A = 0x9E3779B97F4A7C15


@dataclass(frozen=True)
class Workload:
    name: str
    n: int            # logical ranks
    B: int            # samples per rank
    mu: float         # lognormal mu of the UIH length
    sigma: float      # lognormal sigma
    lmax: int         # UIH length clip
    cmin: int         # candidates per sample, uniform in [cmin, cmax]
    cmax: int
    R: int            # table rows
    D: int            # embedding dim
    dtype: str        # "f32" | "bf16"
    zipf_s: float
    balance: str      # "fbs" | "vbs"
    alpha: float      # VBS exponent
    sort_by_len: bool # VBS: cut the length-sorted order (True) or the original order
    iters: int        # consecutive iterations in one run of the workload
    optim: str        # "none" (gather only) | "sgd" | "adagrad"
    lr: float
    eps: float
    seed_base: int
    kmin: int = 1     # IDs per candidate, uniform in [kmin, kmax] (composite when kmax > 1)
    kmax: int = 1
    autotune: bool = False  # VBS AutoTune: per-rank batch corrections from the ranks' step times
    tune_step: int = 1      # samples one AutoTune adjustment moves
    tune_tol_ppm: int = 0   # AutoTune dead band, parts per million of the average time

    @property
    def S(self) -> int:
        return self.n * self.B

    @property
    def row_bytes(self) -> int:
        return self.D * (4 if self.dtype == "f32" else 2)

    @property
    def has_update(self) -> bool:
        return self.optim != "none"

    @property
    def composite(self) -> bool:
        return self.kmax > 1

    def scaled(self, **kw) -> "Workload":
        """Same recipe with some sizes replaced (used for reduced parity cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 8 ranks x 64 samples, FBS, 100K x 64 fp32, SGD over 2 iterations.
    "tiny-fbs-sgd": Workload("tiny-fbs-sgd", 8, 64, 5.0, 1.2, 2048, 1, 8, 100_000, 64, "f32",
                             1.1, "fbs", 1.5, False, 2, "sgd", 0.01, 0.0, 0),
    # 16 ranks x 128 samples, VBS alpha=1.5 in original order, 1M x 64 fp32, gather only.
    "vbs-gather": Workload("vbs-gather", 16, 128, 6.0, 1.4, 4096, 0, 0, 1_000_000, 64, "f32",
                           1.1, "vbs", 1.5, False, 2, "none", 0.0, 0.0, 1000),
    # 64 ranks x 256 samples, FBS, 10M x 128 bf16, row-wise Adagrad.
    "mid-full-step": Workload("mid-full-step", 64, 256, 6.5, 1.5, 8192, 1, 32, 10_000_000, 128, "bf16",
                              1.05, "fbs", 1.5, False, 2, "adagrad", 0.01, 1e-8, 2000),
    # 512 ranks x 64 samples, VBS alpha=1.5 on the length-sorted order, 50M x 128 bf16, gather only.
    "long-seq-index": Workload("long-seq-index", 512, 64, 7.0, 1.6, 16384, 0, 0, 50_000_000, 128, "bf16",
                               1.05, "vbs", 1.5, True, 3, "none", 0.0, 0.0, 3000),
    # 256 ranks x 512 samples, FBS, 100M x 64 fp32 + row-wise Adagrad state, 4 iterations.
    "large-table-full-step": Workload("large-table-full-step", 256, 512, 6.8, 1.5, 16384, 1, 64, 100_000_000, 64,
                                      "f32", 1.0, "fbs", 1.5, False, 4, "adagrad", 0.01, 1e-8, 4000),
    # 16 ranks x 64 samples whose candidates carry 1..16 IDs each, FBS, 1M x 64 fp32, SGD over 2 iterations.
    "composite-cand": Workload("composite-cand", 16, 64, 5.0, 1.2, 2048, 1, 8, 1_000_000, 64, "f32",
                               1.1, "fbs", 1.5, False, 2, "sgd", 0.01, 0.0, 5000, 1, 16),
    # the long-sequence index workload with VBS AutoTune on: every step reports per-rank times
    # (every fourth rank 1.5x slower) and the next batch's cut takes the corrected batch sizes.
    "long-seq-autotune": Workload("long-seq-autotune", 512, 64, 7.0, 1.6, 16384, 0, 0, 50_000_000, 128, "bf16",
                                  1.05, "vbs", 1.5, True, 3, "none", 0.0, 0.0, 6000, autotune=True),
}


def scramble_multiplier(R: int) -> int:
    a = SCRAMBLE_A % R if R > 1 else 0
    if R <= 1:
        return 0
    if a == 0:
        a = 1
    while math.gcd(a, R) != 1:
        a = (a + 1) % R
        if a == 0:
            a = 1
    return a


_cdf_cache: dict = {}


def _zipf_cdf(R: int, s: float, device) -> torch.Tensor:
    key = (R, s, str(device))
    c = _cdf_cache.get(key)
    if c is None:
        # summed on the host, in order: a device scan may associate the fp64 sum
        # differently from run to run, which would move IDs at CDF boundaries
        k = torch.arange(1, R + 1, dtype=torch.float64)
        c = torch.cumsum(k.pow_(-s), 0)
        c /= c[-1].clone()
        _cdf_cache.clear()  # keep at most one table resident
        _cdf_cache[key] = c.to(device)
        c = _cdf_cache[key]
    return c


def zipf_rows(R: int, s: float, count: int, gen: torch.Generator, device, chunk: int = 1 << 25) -> torch.Tensor:
    """count i.i.d. bounded-Zipf ranks k in [0, R), scrambled to rows (k*A) mod R (int64)."""
    out = torch.empty(count, dtype=torch.int64, device=device)
    if count == 0:
        return out
    cdf = _zipf_cdf(R, s, device)
    a = scramble_multiplier(R)
    for lo in range(0, count, chunk):
        hi = min(count, lo + chunk)
        u = torch.rand(hi - lo, dtype=torch.float64, device=device, generator=gen)
        k = torch.searchsorted(cdf, u, right=True)
        k.clamp_(max=R - 1)
        out[lo:hi] = (k * a) % R
    return out


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def batch(w: Workload, it: int, device="cpu") -> dict:
    """One global batch (all n logical ranks, rank-major) of iteration `it`.

    Returns uih_len int32[S], num_cand int32[S], offsets int64[S+1] (jagged row
    offsets, row g = [UIH | candidates]), ids int64[T] and the host int T; with
    composite candidates also cand_offsets int64[S+1] (candidates per sample)
    and cand_lens int64[sum C] (IDs per candidate).
    """
    device = torch.device(device)
    g = _gen(w.seed_base + it, device)
    S = w.S
    L = torch.empty(S, dtype=torch.float64, device=device).log_normal_(w.mu, w.sigma, generator=g)
    L = torch.round(L).clamp_(1, w.lmax).to(torch.int32)
    if w.cmax > 0:
        C = torch.randint(w.cmin, w.cmax + 1, (S,), dtype=torch.int32, device=device, generator=g)
    else:
        C = torch.zeros(S, dtype=torch.int32, device=device)
    extra = {}
    if w.composite:
        cand_offsets = torch.zeros(S + 1, dtype=torch.int64, device=device)
        torch.cumsum(C.to(torch.int64), 0, out=cand_offsets[1:])
        K = torch.randint(w.kmin, w.kmax + 1, (int(cand_offsets[-1].item()),), dtype=torch.int64, device=device,
                          generator=g)
        ck = torch.zeros(K.numel() + 1, dtype=torch.int64, device=device)
        torch.cumsum(K, 0, out=ck[1:])
        cand_ids = ck[cand_offsets[1:]] - ck[cand_offsets[:-1]]   # IDs of each sample's candidates
        lens = L.to(torch.int64) + cand_ids
        extra = {"cand_offsets": cand_offsets, "cand_lens": K}
    else:
        lens = (L + C).to(torch.int64)
    offsets = torch.zeros(S + 1, dtype=torch.int64, device=device)
    torch.cumsum(lens, 0, out=offsets[1:])
    T = int(offsets[-1].item())
    ids = zipf_rows(w.R, w.zipf_s, T, g, device)
    return {"uih_len": L, "num_cand": C, "offsets": offsets, "ids": ids, "T": T, **extra}


def table(w: Workload, device="cpu") -> torch.Tensor:
    """Embedding table [R, D], N(0, 0.01^2), in the workload dtype."""
    device = torch.device(device)
    g = _gen(w.seed_base + 500, device)
    if w.dtype == "f32":
        t = torch.empty(w.R, w.D, dtype=torch.float32, device=device)
        t.normal_(0.0, 0.01, generator=g)
        return t
    t = torch.empty(w.R, w.D, dtype=torch.bfloat16, device=device)
    rows = max(1, (1 << 26) // w.D)
    for lo in range(0, w.R, rows):
        hi = min(w.R, lo + rows)
        t[lo:hi] = torch.empty(hi - lo, w.D, dtype=torch.float32, device=device).normal_(0.0, 0.01, generator=g)
    return t


def grads(w: Workload, T: int, it: int = 0, device="cpu") -> torch.Tensor:
    """Gradient rows [T, D] ~ N(0, 1) in the workload dtype (one per batch-major position)."""
    device = torch.device(device)
    g = _gen(w.seed_base + 600 + it, device)
    if w.dtype == "f32":
        return torch.empty(T, w.D, dtype=torch.float32, device=device).normal_(0.0, 1.0, generator=g)
    out = torch.empty(T, w.D, dtype=torch.bfloat16, device=device)
    rows = max(1, (1 << 26) // w.D)
    for lo in range(0, T, rows):
        hi = min(T, lo + rows)
        out[lo:hi] = torch.empty(hi - lo, w.D, dtype=torch.float32, device=device).normal_(0.0, 1.0, generator=g)
    return out


def rank_speed(n: int):
    """Per-rank slowdown of the simulated clocks: every fourth rank runs 1.5x slower."""
    return [1.5 if r % 4 == 0 else 1.0 for r in range(n)]


def step_times(w: Workload, it: int, device="cpu") -> torch.Tensor:
    """Seeded per-rank step times [n] (int64 ns) reported after iteration `it`:
    rank_speed(r) * 10 ms * (1 + 0.02 * N(0, 1)).  They do not depend on the
    cut, so every benchmarked step does the same work; the feedback loop itself
    (times that follow the cut) is what rank_times below drives."""
    g = _gen(w.seed_base + 700 + it, "cpu")
    jitter = torch.randn(w.n, generator=g, dtype=torch.float64)
    t = torch.tensor(rank_speed(w.n), dtype=torch.float64) * 1.0e7 * (1.0 + 0.02 * jitter)
    return torch.round(t).clamp_(min=0).to(torch.int64).to(device)


def rank_times(uih_len, perm, rank_offsets, speed, beta: float, ns_per_unit: float = 1.0):
    """Simulated local execution times of the ranks, integer nanoseconds, for
    driving the VBS AutoTune loop without a trainer: rank r takes
    speed[r] * sum over its samples of L^beta (times ns_per_unit), rounded.
    The per-rank speed factors stand for what the L^alpha weights cannot see
    (slower hosts, stragglers).  A stand-in for the trainer's clock, not part of
    the method: only its output, the times, is handed to the AutoTune update."""
    L = torch.as_tensor(uih_len).to("cpu", torch.float64)
    p = torch.as_tensor(perm).to("cpu", torch.int64)
    ro = torch.as_tensor(rank_offsets).to("cpu", torch.int64)
    cost = torch.zeros(p.numel() + 1, dtype=torch.float64)
    torch.cumsum(L[p] ** beta, 0, out=cost[1:])
    per_rank = cost[ro[1:]] - cost[ro[:-1]]
    t = torch.as_tensor(speed, dtype=torch.float64) * per_rank * ns_per_unit
    return torch.round(t).to(torch.int64).numpy()
