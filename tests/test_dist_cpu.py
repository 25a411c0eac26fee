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


def test_step_roofline_keys():
    import bench
    from jagged_embedding_gb300 import synthetic
    w = synthetic.WORKLOADS["large-table-full-step"]
    by_stage = {}
    for T, U in ((3.0e8, 3.7e7), (3.1e8, 3.8e7)):      # two timed steps
        for k, v in bench.algorithmic_bytes(w, w.S, T, U, w.R).items():
            by_stage[k] = by_stage.get(k, 0.0) + v
    total = sum(by_stage.values())
    secs = 0.08
    r = bench.step_roofline(by_stage, 2, secs, 6666.6)
    assert r["algorithmic_bytes_per_step"] == total / 2
    assert abs(sum(r["algorithmic_bytes_per_step_by_stage"].values()) - total / 2) <= 1e-6 * total
    assert set(r["algorithmic_bytes_per_step_by_stage"]) == {"prep", "collision", "gather", "backward"}
    assert r["hbm_roofline_frac_step"] == total / secs / 6666.6e9
    assert abs(r["hbm_nominal_frac_step"] / r["hbm_roofline_frac_step"] - 6666.6 / 7900.0) < 1e-12


def test_step_times_are_seeded_and_slow_every_fourth_rank():
    import torch

    from jagged_embedding_gb300 import synthetic
    w = synthetic.WORKLOADS["long-seq-autotune"]
    a, b = synthetic.step_times(w, 2), synthetic.step_times(w, 2)
    assert a.dtype == torch.int64 and a.shape == (w.n,) and torch.equal(a, b)
    assert not torch.equal(a, synthetic.step_times(w, 3))
    slow, fast = a[::4].double().mean(), torch.cat([a[1::4], a[2::4], a[3::4]]).double().mean()
    assert 1.4 < float(slow / fast) < 1.6


def test_recorded_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    """A DRAM traffic record is printed only while the call's kernel sources hash to the recorded value."""
    import json
    import bench
    src = tmp_path / "jagged_embedding_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in ("backward.cu", "radix.cuh", "bulk.cuh", "gather.cu"):
        (src / name).write_text(f"// {name}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"gather/large-table-full-step": {"kernel_hash": bench.kernel_hash("gather", True), "bytes_per_launch": 7},
           "update/large-table-full-step": {"kernel_hash": bench.kernel_hash("update", True), "bytes_per_launch": 9}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("gather", "large-table-full-step", True) == 7
    assert bench.recorded_traffic("update", "large-table-full-step", True) == 9
    assert bench.recorded_traffic("gather", "mid-full-step", True) is None         # no record for that workload
    (src / "backward.cu").write_text("// changed\n")                             # the gather and update kernels' file
    assert bench.recorded_traffic("gather", "large-table-full-step", True) is None
    assert bench.recorded_traffic("update", "large-table-full-step", True) is None
    (src / "backward.cu").write_text("// backward.cu\n")
    (src / "bulk.cuh").write_text("// changed\n")                                # the update's only
    assert bench.recorded_traffic("gather", "large-table-full-step", True) == 7
    assert bench.recorded_traffic("update", "large-table-full-step", True) is None


def test_gpu_numa_node_without_a_device_is_none():
    import bench
    assert bench.gpu_numa_cpus(0) is None or isinstance(bench.gpu_numa_cpus(0)[1], set)
