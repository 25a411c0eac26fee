"""Benchmark: jagged IDs/s of the FreeScale jagged index + embedding path on GB300.

One step = one training iteration of the hot path over one global batch of
n logical ranks: balance (FBS/VBS) + jagged permute + row-wise bucketize of the
next batch, collision split of (t, t+1), embedding gather of t and, for
workloads with an optimizer, the gradient segment-reduce + row update of t
(collision rows first, then exclusive rows).  value = IDs of the gathered
batches / device time; the roofline fraction uses the algorithmic bytes of
the step (see algorithmic_bytes()).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gpu|reference]
                [--schedule sync|prioritized]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (weak scaling, no data-path collective); the timing is the
maximum over ranks and value sums the IDs of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "jagged IDs/s (balance+bucketize+collision+gather+update); % of HBM roofline"
DEFAULT_WORKLOAD = "large-table-full-step"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # the vendor's HBM3e figure for GB300 (context beside the measured peak)


# --------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def step_roofline(by_stage, K, secs, hbm_gbs):
    """Whole-step roofline keys of the result line: bytes per step by stage (summed over the K timed
    steps in `by_stage`), and the fraction of the measured and of the nominal HBM bandwidth."""
    total = sum(by_stage.values())
    return {"hbm_roofline_frac_step": total / secs / (hbm_gbs * 1e9),
            "hbm_nominal_frac_step": total / secs / (NOMINAL_HBM_GBS * 1e9),
            "algorithmic_bytes_per_step": total / K,
            "algorithmic_bytes_per_step_by_stage": {k: v / K for k, v in by_stage.items()}}


def algorithmic_bytes(w, S, T, U, R, n_cand=0, masks=False):
    """Bytes the method must move for one step (one batch), by stage.

    prep (balance + permute + bucketize)      16 S + 16 T + 20 T
      (+ 16 S + 16 C with composite candidates: their lengths move with the samples, C candidates)
    collision split, per pair                  8 T + 3 R / 8 + 16 U
      (+ 2 T when the per-position collision masks are written: the prioritized order's masked
       lookups and updates read them; the synchronous step's update reads t+1's row bitmap instead)
    gather                                     (8 + RB) T + RB U
      (+ 4 T when it gathers in shard-major order: the batch-major position of each entry; the
       gather-only workloads do)
    backward (segment-reduce + update)         (8 + RB) T + (2 RB + 8) U
    VBS AutoTune (when on)                     48 n: times in, corrections read and written,
                                               corrections read again and segment ends moved by the cut
    RB = row bytes; U = unique rows of the batch; n = logical ranks.
    """
    RB = w.row_bytes
    b = {
        "prep": 16 * S + 36 * T + ((16 * S + 16 * n_cand) if w.composite else 0),
        "collision": (10 if masks else 8) * T + 3 * R / 8 + 16 * U,
        "gather": gather_bytes(w, T, U),
    }
    if w.autotune:
        b["autotune"] = 48 * w.n
    if w.has_update:
        b["backward"] = (8 + RB) * T + (2 * RB + (8 if w.optim == "adagrad" else 0)) * U
    return b


def gather_bytes(w, T, U):
    """The lookup: IDs in, rows out, each distinct row read once; the gather-only workloads read the
    shard-major IDs and their batch-major positions (4 more bytes per ID)."""
    return (8 + (0 if w.has_update else 4) + w.row_bytes) * T + w.row_bytes * U


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    pw.append(float(parts[3]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s, p in zip(sm, pw) if p > 0.3 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist
    rank, local = int(os.environ["RANK"]), int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(ids_local, seconds_local, ws, device=None):
    """Whole-job (sum of IDs over ranks, max of elapsed seconds over ranks)."""
    if ws <= 1:
        return float(ids_local), float(seconds_local)
    import torch
    import torch.distributed as dist
    dev = device if device is not None else "cpu"
    t = torch.tensor([float(ids_local)], dtype=torch.float64, device=dev)
    s = torch.tensor([float(seconds_local)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(t.item()), float(s.item())


# --------------------------------------------------------------------------- oracle arm

def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_sample(w, steps, max_seconds=20.0, samples_per_rank=None, table_np=None, device=None, warmup=0,
                  threads=1):
    """Time the CPU oracle, as it stands, on a bounded sample of workload w.

    The sample keeps the workload's recipe (ranks, rows, dim, dtype, Zipf law,
    optimizer) with fewer samples per rank.  One timed unit mirrors one GPU
    step: prepare(t+1) + collision(t, t+1) + gather(t) + backward(t).  With
    threads > 1 the oracle's multi-threaded variants run (same results, the
    work of each step split over that many host threads).
    Returns (IDs/s, description, IDs timed, seconds).
    """
    import oracle

    oracle.set_threads(threads)
    try:
        return _oracle_sample(w, steps, max_seconds, samples_per_rank, table_np, device, warmup, threads)
    finally:
        oracle.set_threads(1)


def _oracle_sample(w, steps, max_seconds, samples_per_rank, table_np, device, warmup, threads):
    import numpy as np
    import torch

    import oracle
    from jagged_embedding_gb300 import synthetic

    spr = samples_per_rank or max(1, min(w.B, 8))
    ws_ = w.scaled(B=spr)
    gen_dev = device if device is not None else "cpu"
    nb = steps + 1
    batches = []
    for t in range(nb):
        b = synthetic.batch(ws_, t, gen_dev)
        batches.append({k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in b.items()})
    if table_np is None:
        tab = synthetic.table(ws_, gen_dev).cpu()
        table_np = tab.view(torch.int16).numpy().view(np.uint16) if w.dtype == "bf16" else tab.numpy()
    state = np.zeros(w.R, np.float32) if w.optim == "adagrad" else None
    maxT = max(b["T"] for b in batches)
    g = synthetic.grads(ws_, maxT, 0, gen_dev).cpu()
    G = g.view(torch.int16).numpy().view(np.uint16) if w.dtype == "bf16" else g.numpy()
    ids_done, secs, n_timed = 0, 0.0, 0
    delta = np.zeros(w.n, np.int64)
    times = [synthetic.step_times(ws_, t).numpy() for t in range(steps)] if w.autotune else None
    prep_t = oracle.prepare(ws_, batches[0], delta)
    for t in range(steps):
        timed = t >= warmup
        t0 = time.perf_counter()
        if w.autotune:
            delta = oracle.vbs_autotune(times[t], delta, w.tune_step, w.tune_tol_ppm)
        prep_n = oracle.prepare(ws_, batches[t + 1], delta)
        coll = oracle.collision_split(prep_t["ids"], prep_n["ids"], w.R, w.n)
        oracle.emb_gather(table_np, prep_t["ids"])
        if w.has_update:
            T = prep_t["ids"].shape[0]
            oracle.emb_backward(table_np, state, prep_t["ids"], G[:T], w.optim, w.lr, w.eps,
                                is_co=coll["is_co_t"], phase=1)
            oracle.emb_backward(table_np, state, prep_t["ids"], G[:T], w.optim, w.lr, w.eps,
                                is_co=coll["is_co_t"], phase=2)
        if timed:
            secs += time.perf_counter() - t0
            ids_done += int(prep_t["ids"].shape[0])
            n_timed += 1
        prep_t = prep_n
        if secs > max_seconds:
            break
    who = "single-threaded C++ oracle" if threads == 1 else f"C++ oracle on {threads} host threads"
    desc = (f"{w.name} recipe with {spr} samples/rank (S={ws_.S}), {ids_done} IDs over "
            f"{n_timed} timed steps after {warmup} untimed, R={w.R}, {who}")
    return ids_done / secs, desc, ids_done, secs


def workload_config(w, n_gpus):
    """The workload keys both arms report (the GPU arm adds its measured IDs per step and the L2 note)."""
    cfg = {"workload": w.name, "n_logical_ranks": w.n, "samples_per_rank": w.B, "rows": w.R, "dim": w.D,
           "table_dtype": w.dtype, "optimizer": w.optim, "balance": w.balance, "iterations_cycled": w.iters,
           "schedule": "sync order, collision rows updated before exclusive rows",
           "parallelism": f"replicas x{n_gpus}"}
    if w.autotune:
        cfg["vbs_autotune"] = {"step": w.tune_step, "tol_ppm": w.tune_tol_ppm,
                               "times": "seeded per-rank step times, every fourth rank 1.5x slower"}
    return cfg


def run_reference(args):
    """`--impl reference`: the CPU oracle timed on the host cores (rank 0 only)."""
    rank, ws, _ = dist_setup()
    from jagged_embedding_gb300 import synthetic
    w = synthetic.WORKLOADS[args.workload]
    if rank != 0:
        return 0
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    # warm-up steps are run (untimed) inside the same sample; the oracle runs on every host core
    cores = host_cores()
    rate, desc, ids, secs = oracle_sample(w, args.steps + args.warmup, max_seconds=150.0,
                                          samples_per_rank=args.ref_samples_per_rank, device=dev,
                                          warmup=args.warmup, threads=cores)
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "IDs/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * secs / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": f"int64/{w.dtype}",
            "data": "synthetic", "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": rate, "unit": "IDs/s", "cores": cores, "kind": "oracle", "sample": desc,
                             "host_cores": cores},
            "e2e": {"value": rate, "unit": "IDs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch

    from jagged_embedding_gb300 import binding as B
    from jagged_embedding_gb300 import build as cuda_build
    from jagged_embedding_gb300 import synthetic
    from jagged_embedding_gb300.pipeline import Pipeline

    rank, ws, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cuda_build.build()
    B.lib()
    w0 = synthetic.WORKLOADS[args.workload]
    w = w0.scaled(seed_base=w0.seed_base + 100 * rank)
    K, W = args.steps, args.warmup
    prio = args.schedule == "prioritized"

    # ---- resident inputs (all iterations' batches, table, state, gradients)
    batches = [synthetic.batch(w, t, dev) for t in range(w.iters)]
    synthetic._cdf_cache.clear()
    Ts = [b["T"] for b in batches]
    max_T = max(Ts)
    table = synthetic.table(w, dev)
    state = torch.zeros(w.R, dtype=torch.float32, device=dev) if w.optim == "adagrad" else None
    # gradient rows of the dense model's backward: one N(0,1) pool, batch t uses its first T_t rows
    grads = synthetic.grads(w, max_T, 0, dev) if w.has_update else None
    if prio:
        # Algorithm 2 needs the output of t+1 beside that of t and a third batch slot
        need = max_T * (w.row_bytes + 8 * 3 + 5) + w.R // 4
        free, _ = torch.cuda.mem_get_info(dev)
        if need > 0.9 * free:
            raise SystemExit(f"the prioritized order of {w.name} needs about {need / 1e9:.0f} GB more device "
                             f"memory than the {free / 1e9:.0f} GB free")
    pipe = Pipeline(w, dev, max_T, table, state, two_outputs=prio, streams=prio)
    # VBS AutoTune: the per-rank step times each iteration reports (seeded clock readings)
    times = [synthetic.step_times(w, t, dev) for t in range(w.iters)] if w.autotune else None
    torch.cuda.synchronize()

    def step(i, cur):
        nb = batches[(i + 1) % w.iters]
        tm = times[i % w.iters] if times else None
        if prio:   # one iteration of Algorithm 2: batch i % iters is slot i % 3
            T = Ts[i % w.iters]
            pipe.prio_step(nb, grads[:T] if grads is not None else None, times=tm)
            return (i + 1) % 3
        return pipe.step_sync(cur, nb, grads[: pipe.slots[cur].T] if grads is not None else None, times=tm)

    cur = 0
    if prio:
        pipe.prio_begin(batches[0])
    else:
        pipe.prepare(batches[0], 0)
    for i in range(W):
        cur = step(i, cur)
    torch.cuda.synchronize()
    B.check(pipe.err, "warm-up")

    stream = torch.cuda.current_stream(dev)
    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    u0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    u1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ids_timed = 0
    step_batches = []
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = B.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    t_start.record(stream)
    orig_gather, orig_update, orig_backward = pipe.gather, pipe.update_sorted, pipe.backward
    for k in range(K):
        i = W + k
        step_batches.append(i % w.iters)
        ids_timed += Ts[i % w.iters]
        if not prio:
            # the gather and the update of the synchronous step, timed with events on the stream
            # they run on (the prioritized order splits both into masked parts on two streams)
            def timed_gather(*a, _k=k, **kw):
                g0[_k].record(stream)
                orig_gather(*a, **kw)
                g1[_k].record(stream)

            def timed_update(*a, _k=k, _f=orig_update, **kw):
                u0[_k].record(stream)
                _f(*a, **kw)
                u1[_k].record(stream)

            def timed_backward(*a, _k=k, _f=orig_backward, **kw):
                u0[_k].record(stream)
                _f(*a, **kw)
                u1[_k].record(stream)

            pipe.gather, pipe.update_sorted, pipe.backward = timed_gather, timed_update, timed_backward
        cur = step(i, cur)
    pipe.gather, pipe.update_sorted, pipe.backward = orig_gather, orig_update, orig_backward
    t_end.record(stream)          # (the prioritized step leaves the side stream joined to this one)
    torch.cuda.synchronize()
    barrier(ws)
    launches = B.launch_count() - launches0
    clk = clocks.stop()
    B.check(pipe.err, "timed steps")
    secs = t_start.elapsed_time(t_end) / 1000.0
    gather_ms = update_ms = None
    if not prio:
        gather_ms = sum(a.elapsed_time(b) for a, b in zip(g0, g1)) / K
        update_ms = sum(a.elapsed_time(b) for a, b in zip(u0, u1)) / K if w.has_update else None
    if prio:
        pipe.prio_finish()
        torch.cuda.synchronize()

    # unique rows per batch (|co| + |ex_t| of its pair with the next batch), for the byte model
    U = {}
    for t in range(w.iters):
        out, err = B.fs_collision_split(batches[t]["ids"], batches[(t + 1) % w.iters]["ids"], w.R, w.n)
        B.check(err, "unique rows")
        c = out["counts"].cpu().tolist()
        U[t] = c[0] + c[1]
        del out
    torch.cuda.synchronize()
    hbm_gbs, peak_kind = measured_peaks()
    by_stage = {}
    gbytes = 0.0
    ubytes = 0.0
    for t in step_batches:
        n_cand = int(batches[t]["cand_offsets"][-1]) if w.composite else 0
        bb = algorithmic_bytes(w, w.S, Ts[t], U[t], w.R, n_cand, masks=prio)
        for k, v in bb.items():
            by_stage[k] = by_stage.get(k, 0.0) + v
        gbytes += gather_bytes(w, Ts[t], U[t])
        ubytes += bb.get("backward", 0.0)
    gbytes /= K
    ubytes /= K

    ids_all, secs_max = aggregate(ids_timed, secs, ws, dev)
    value = ids_all / secs_max

    # ---- end to end through the public API with host inputs (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e and not prio:
        e2e = run_e2e(w, pipe, batches, grads, K, W, dev, ws, times)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tab_host = table.cpu()
        tab_np = tab_host.view(torch.int16).numpy().view("uint16") if w.dtype == "bf16" else tab_host.numpy()
        cores = host_cores()
        # the oracle on every host core, then single-threaded, each on a bounded sample of the workload
        rate, desc, _, _ = oracle_sample(w, 4, max_seconds=15.0, samples_per_rank=args.ref_samples_per_rank,
                                         table_np=tab_np, device=dev, warmup=1, threads=cores)
        rate1, desc1, _, _ = oracle_sample(w, 4, max_seconds=15.0, samples_per_rank=args.ref_samples_per_rank,
                                           table_np=tab_np, device=dev, warmup=1, threads=1)
        cpu = {"value": rate, "unit": "IDs/s", "cores": cores, "kind": "oracle", "sample": desc,
               "host_cores": cores, "single_thread": {"value": rate1, "unit": "IDs/s", "cores": 1, "sample": desc1}}

    cfg = dict(workload_config(w0, ws), ids_per_step=ids_timed / K,
               l2="no flush: inputs larger than L2 (table %.1f GB, %.1f GB of IDs per batch)"
                  % (table.numel() * table.element_size() / 1e9, max_T * 8 / 1e9))
    if prio:
        cfg["schedule"] = ("FreeScale Algorithm 2: exclusive rows of t+1 prefetched and exclusive updates of t "
                           "deferred on a side stream; collision rows of t updated, then gathered for t+1")
    line = {
        "metric": METRIC, "value": value, "unit": "IDs/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": 1000.0 * secs_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"int64/{w.dtype}", "data": "synthetic", "config": cfg,
        **step_roofline(by_stage, K, secs, hbm_gbs),
        "roofline": None, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
    }
    if not prio:
        sorted_gather = w.has_update and pipe.row_sorted
        ga = gbytes / (gather_ms / 1000.0) / 1e9
        gk = SORTED_GATHER_KERNEL if sorted_gather else (GATHER_KERNEL if w.has_update else SHARD_GATHER_KERNEL)
        calls = {"gather": {"kernel": gk, "bound": "hbm",
                            "achieved": ga, "peak": hbm_gbs, "peak_kind": peak_kind, "unit": "GB/s",
                            "frac": ga / hbm_gbs, "traffic": recorded_traffic("gather", w0.name, sorted_gather),
                            "algorithmic_bytes_per_launch": gbytes, "avg_launch_ms": gather_ms}}
        if update_ms:
            # the update's segment-reduce + row update (both phases), timed like the gather
            ua = ubytes / (update_ms / 1000.0) / 1e9
            calls["update"] = {
                "kernel": "fs_emb_update_sorted (reduce_ring_kernel x2, block sums, fixup)" if sorted_gather
                else "fs_emb_backward_adagrad (sort, reduce_ring_kernel, block sums, fixup)",
                "bound": "hbm", "achieved": ua, "peak": hbm_gbs, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": ua / hbm_gbs, "traffic": recorded_traffic("update", w0.name, sorted_gather),
                "algorithmic_bytes_per_launch": ubytes, "avg_launch_ms": update_ms}
        # the dominant call of the step: the one that takes longer
        dom = max(calls, key=lambda c: calls[c]["avg_launch_ms"])
        line["roofline"] = dict(calls[dom], call=dom)
        for c, v in calls.items():
            line[f"roofline_{c}"] = v
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def recorded_traffic(call, workload, sorted_gather):
    """DRAM bytes per launch of `call` on `workload` from profiles/traffic.json (scaled from a small-case ncu
    capture), or None when there is no record or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{call}/{workload}")
    if not rec or rec.get("kernel_hash") != kernel_hash(call, sorted_gather):
        return None
    return rec.get("bytes_per_launch")


# the synchronous step's gather: from the update's sorted entries when the workload has an update, in
# shard-major order from the bucketize output otherwise (the position-order gather when neither applies)
GATHER_KERNEL = "fs_emb_gather (gather_bulk_kernel<4, 2>)"
SORTED_GATHER_KERNEL = "fs_emb_gather_sorted (gather_sorted_kernel)"
SHARD_GATHER_KERNEL = "fs_emb_gather_shard_major (gather_scatter_kernel)"


def kernel_hash(call="gather", sorted_gather=False):
    """Hash of the sources of a call's kernels (a recorded DRAM traffic is valid for these only)."""
    import hashlib
    names = {("gather", False): ("gather.cu",), ("gather", True): ("backward.cu", "radix.cuh"),
             ("update", False): ("backward.cu", "radix.cuh", "bulk.cuh"),
             ("update", True): ("backward.cu", "radix.cuh", "bulk.cuh")}[(call, sorted_gather)]
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "jagged_embedding_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gpu_numa_cpus(dev):
    """(node, CPUs) of the host NUMA node the GPU is attached to, or None when the host does not say."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            node = int(f.read())
        if node < 0:
            return None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            cl = f.read().strip()
        cpus = set()
        for part in cl.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return (node, cpus) if cpus else None
    except Exception:
        return None


def run_e2e(w, pipe, batches, grads, K, W, dev, ws, times=None):
    """Same steps, inputs copied from pinned host memory inside the timed region.

    A copy stream brings batch i+2 while batch i is processed (a ring of three
    device staging buffers); each step reads back the collision counts and the
    error word.  Gradient rows stand for the dense model's output and stay on
    the device.  With AutoTune on, each step's rank times (8 n bytes) are
    copied in on the compute stream just before the step uses them.
    """
    import torch

    from jagged_embedding_gb300 import binding as B

    # pinned host copies of the batches, their pages placed (first touch) on the NUMA node the GPU is
    # attached to when the host has more than one
    numa = gpu_numa_cpus(dev)
    old_aff = os.sched_getaffinity(0)
    if numa:
        os.sched_setaffinity(0, numa[1])
    try:
        host = []
        for b in batches:
            host.append({k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in b.items()})
    finally:
        if numa:
            os.sched_setaffinity(0, old_aff)
    max_S1 = max(h["offsets"].numel() for h in host)
    max_T = pipe.max_T
    ring = [{"uih_len": torch.empty(max_S1 - 1, dtype=torch.int32, device=dev),
             "offsets": torch.empty(max_S1, dtype=torch.int64, device=dev),
             "ids": torch.empty(max_T, dtype=torch.int64, device=dev)} for _ in range(3)]
    if w.composite:  # candidate lengths travel with the batch
        max_C = max(h["cand_lens"].numel() for h in host)
        for r in ring:
            r["cand_offsets"] = torch.empty(max_S1, dtype=torch.int64, device=dev)
            r["cand_lens"] = torch.empty(max(max_C, 1), dtype=torch.int64, device=dev)
    copy_stream = torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    done = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    used = [torch.cuda.Event() for _ in range(3)]
    readback = torch.empty(4, dtype=torch.int64).pin_memory()
    host_times = [x.cpu().pin_memory() for x in times] if times else None
    times_dev = torch.empty(w.n, dtype=torch.int64, device=dev) if times else None

    def stage(i):
        h = host[i % w.iters]
        slot = ring[i % 3]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(used[i % 3])
            c0 = None
            if copy_ev is not None:
                c0 = torch.cuda.Event(enable_timing=True)
                c0.record(copy_stream)
            S1 = h["offsets"].numel()
            slot["uih_len"][: S1 - 1].copy_(h["uih_len"], non_blocking=True)
            slot["offsets"][:S1].copy_(h["offsets"], non_blocking=True)
            slot["ids"][: h["T"]].copy_(h["ids"], non_blocking=True)
            if w.composite:
                nc = h["cand_lens"].numel()
                slot["cand_offsets"][:S1].copy_(h["cand_offsets"], non_blocking=True)
                slot["cand_lens"][:nc].copy_(h["cand_lens"], non_blocking=True)
            done[i % 3].record(copy_stream)
            if copy_ev is not None:
                copy_ev.append((c0, done[i % 3]))
        nbytes = h["uih_len"].numel() * 4 + h["offsets"].numel() * 8 + h["T"] * 8
        b = {"uih_len": slot["uih_len"][: S1 - 1], "offsets": slot["offsets"][:S1],
             "ids": slot["ids"][: h["T"]], "T": h["T"]}
        if w.composite:
            nc = h["cand_lens"].numel()
            nbytes += S1 * 8 + nc * 8
            b["cand_offsets"], b["cand_lens"] = slot["cand_offsets"][:S1], slot["cand_lens"][:nc]
        return b, nbytes

    copy_ev = None  # (start, end) events of the timed steps' host-to-device copies

    def run(steps, measure):
        staged = {}
        b0, n0 = stage(0)
        staged[0] = b0
        staged[1], n1 = stage(1)
        main.wait_event(done[0])
        pipe.prepare(staged[0], 0)
        used[0].record(main)
        cur = 0
        total_ids, h2d_bytes = 0, n0 + n1
        for i in range(steps):
            staged[i + 2], nb = stage(i + 2)
            h2d_bytes += nb
            main.wait_event(done[(i + 1) % 3])
            total_ids += pipe.slots[cur].T
            gsl = grads[: pipe.slots[cur].T] if grads is not None else None
            if host_times is not None:
                times_dev.copy_(host_times[i % w.iters], non_blocking=True)
                h2d_bytes += 8 * w.n
            cur = pipe.step_sync(cur, staged[i + 1], gsl, times=times_dev)
            used[(i + 1) % 3].record(main)
            readback[:3].copy_(pipe.coll["counts"], non_blocking=True)
            readback[3:4].copy_(pipe.err.to(torch.int64), non_blocking=True)
            staged.pop(i, None)
        return total_ids, h2d_bytes

    run(W, False)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    copy_ev = []
    t0.record(main)
    ids, h2d_bytes = run(K, True)
    t1.record(main)
    torch.cuda.synchronize()
    barrier(ws)
    B.check(pipe.err, "e2e")
    secs = t0.elapsed_time(t1) / 1000.0
    # each copy's duration is read before its `done` event is recorded again (three-slot ring,
    # synchronised above): the last three are exact, earlier ones were re-recorded, so keep those
    copy_ms = [a.elapsed_time(b) for a, b in copy_ev[-3:]]
    ids_all, secs_max = aggregate(ids, secs, ws, dev)
    return {"value": ids_all / secs_max, "unit": "IDs/s", "h2d_bytes_per_step": h2d_bytes / K,
            "d2h_bytes_per_step": 32, "h2d_copy_ms_last": [round(x, 3) for x in copy_ms],
            "host_numa_node": numa[0] if numa else None,
            "note": "batch IDs + lengths + offsets from pinned host memory, "
                    "copy of batch i+2 overlapped with step i; gradients device-resident; "
                    "h2d_copy_ms_last: durations of the last timed copies (a step waits for its batch's copy)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--schedule", default="sync", choices=["sync", "prioritized"],
                    help="sync: the synchronous order (default); prioritized: FreeScale Algorithm 2 on two streams")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-samples-per-rank", type=int, default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
