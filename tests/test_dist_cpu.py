"""Multi-process host logic of the benchmark on CPU (gloo, world size 2).

Each GPU runs an independent replica (weak scaling, no data-path collective);
the only cross-rank steps are the barrier around the timed region and the
whole-job aggregation: IDs summed over ranks, elapsed time = max over ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    ids, secs = bench.aggregate(1000 * (rank + 1), 0.5 + rank, world)
    q.put((rank, ids, secs))
    bench.barrier(world)
    dist.destroy_process_group()


def test_aggregate_sums_ids_and_takes_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ids, secs in got:
        assert ids == 3000.0 and secs == 1.5


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(123, 0.25, 1) == (123.0, 0.25)


def test_algorithmic_bytes_model():
    import bench
    from jagged_embedding_gb300 import synthetic
    w = synthetic.WORKLOADS["large-table-full-step"]
    b = bench.algorithmic_bytes(w, w.S, 3.0e8, 3.7e7, w.R)
    per_id = sum(b.values()) / 3.0e8
    assert 640 < per_id < 700          # about 670 bytes per ID for a full step with 256-byte rows
    g = synthetic.WORKLOADS["vbs-gather"]
    b = bench.algorithmic_bytes(g, g.S, 2.0e6, 2.0e5, g.R)
    assert "backward" not in b
    # the collision masks (a byte written and read per position) count only where they are written
    bm = bench.algorithmic_bytes(w, w.S, 3.0e8, 3.7e7, w.R, masks=True)
    assert bm["collision"] - bench.algorithmic_bytes(w, w.S, 3.0e8, 3.7e7, w.R)["collision"] == 2 * 3.0e8


def test_algorithmic_bytes_autotune_and_config():
    import bench
    from jagged_embedding_gb300 import synthetic
    w = synthetic.WORKLOADS["long-seq-autotune"]
    plain = synthetic.WORKLOADS["long-seq-index"]
    b = bench.algorithmic_bytes(w, w.S, 9.3e7, 1.06e7, w.R)
    b0 = bench.algorithmic_bytes(plain, plain.S, 9.3e7, 1.06e7, plain.R)
    assert b["autotune"] == 48 * w.n and "autotune" not in b0
    assert sum(b.values()) - sum(b0.values()) == 48 * w.n      # nothing else changes
    cfg = bench.workload_config(w, 1)
    assert cfg["vbs_autotune"]["step"] == 1 and "vbs_autotune" not in bench.workload_config(plain, 1)
    # the update's bytes: (8 + RB) per ID, 2 RB + 8 per unique row with Adagrad state
    big = synthetic.WORKLOADS["large-table-full-step"]
    assert bench.algorithmic_bytes(big, big.S, 10, 3, big.R)["backward"] == 264 * 10 + 520 * 3


def test_step_times_are_seeded_and_slow_every_fourth_rank():
    import torch

    from jagged_embedding_gb300 import synthetic
    w = synthetic.WORKLOADS["long-seq-autotune"]
    a, b = synthetic.step_times(w, 2), synthetic.step_times(w, 2)
    assert a.dtype == torch.int64 and a.shape == (w.n,) and torch.equal(a, b)
    assert not torch.equal(a, synthetic.step_times(w, 3))
    slow, fast = a[::4].double().mean(), torch.cat([a[1::4], a[2::4], a[3::4]]).double().mean()
    assert 1.4 < float(slow / fast) < 1.6
