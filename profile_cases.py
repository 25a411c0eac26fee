"""One hot-path call on seeded synthetic input, for profiling a single kernel.

    python profile_cases.py <op> <T> <R> [reps]

These are the small cases that the ncu summaries under profiles/ were taken
on (a few GB on the device, one kernel at a time).

op is one of
  gather    -- fs_emb_gather, unmasked, f32 rows of 64, T bounded-Zipf(1.0) IDs over R rows
  backward  -- fs_emb_backward_adagrad (sort + reduce + fixup), same IDs, f32, row-wise Adagrad,
               collision rows (half of the rows, by a hash of the row) updated before exclusive rows
  backward-bf16 -- the same with bf16 rows of 128 (the mid-size full step's table)
  bucketize -- fs_bucketize_rowwise of the same IDs into 256 row-range shards
  prep      -- fs_permute_bucketize: T IDs in samples of lognormal(6.8, 1.5) lengths up to 16384 dealt to
               256 ranks by FBS, permuted and bucketized into 256 row-range shards over R rows
  sorted-step -- the large-table step's update path on the same IDs (256 ranks and shards, f32 rows of 64,
               row-wise Adagrad, half the rows collision rows): fs_bucketize_rowwise, the mask in
               shard-major order, fs_emb_sort_rows_sharded, fs_emb_gather_sorted, fs_emb_update_sorted;
               prints each call's median time and the bandwidth of its algorithmic bytes
  transpose -- fs_keyed_transpose of about T IDs in R features x 65536 samples (lengths uniform, per-feature
               row bases); prints the time per call and the bandwidth of its algorithmic bytes
  gather-sorted -- the same IDs and table as gather: fs_emb_sort_rows once, then fs_emb_gather_sorted and
               fs_emb_gather each timed alone (median of reps calls, CUDA events), with the bandwidth of
               the algorithmic bytes (8 + 256 per ID, 256 per distinct row)
  bitmap    -- fs_row_bitmap of T bounded-Zipf(1.0) IDs over R rows, in the shard-major order the pipeline
               marks them in (fs_bucketize_rowwise into 256 row-range shards first); prints the median
               time and the bandwidth of the IDs read
  collision -- fs_collision_split_bitmaps of two batches of T bounded-Zipf(1.0) IDs over R rows (their row
               bitmaps built first, no masks): the compact of the collision / exclusive lists with
               256 shard offsets; prints the median time and the list lengths
  autotune  -- VBS AutoTune with T samples over R logical ranks (lognormal(7, 1.6) lengths up to 16384,
               alpha 1.5, length-sorted cut): fs_vbs_autotune, fs_balance_vbs_tuned and the plain
               fs_balance_vbs, each timed alone (median of reps calls, CUDA events)
Inputs come from jagged_embedding_gb300.synthetic; every call goes through the C ABI.
Exits non-zero if a call reports an error.
"""
from __future__ import annotations

import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from jagged_embedding_gb300 import binding as B  # noqa: E402
from jagged_embedding_gb300 import build as cuda_build  # noqa: E402
from jagged_embedding_gb300 import synthetic  # noqa: E402

DIM = 64
SHARDS = 256


def main(argv) -> int:
    if len(argv) < 3 or argv[0] not in ("gather", "backward", "backward-bf16", "bucketize", "transpose",
                                        "autotune", "gather-sorted", "prep", "sorted-step", "bitmap", "collision"):
        print(__doc__)
        return 2
    op, T, R = argv[0], int(argv[1]), int(argv[2])
    reps = int(argv[3]) if len(argv) > 3 else 2
    cuda_build.build()
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if op == "transpose":
        return _transpose(T, R, reps, dev, g, err)
    if op == "autotune":
        return _autotune(T, R, reps, dev, g, err)
    if op == "prep":
        return _prep(T, R, reps, dev, g, err)
    ids = synthetic.zipf_rows(R, 1.0, T, g, dev)
    if op == "sorted-step":
        return _sorted_step(ids, T, R, reps, dev, g, err)
    if op == "bitmap":
        return _bitmap(ids, T, R, reps, dev, err)
    if op == "collision":
        return _collision(ids, synthetic.zipf_rows(R, 1.0, T, g, dev), T, R, reps, dev, err)
    if op == "gather-sorted":
        return _gather_sorted(ids, T, R, reps, dev, g, err)
    if op == "gather":
        table = torch.empty(R, DIM, device=dev).normal_(0, 0.01, generator=g)
        out = torch.empty(T, DIM, device=dev)
        for _ in range(reps):
            B.fs_emb_gather(table, ids, out=out, err=err)
    elif op in ("backward", "backward-bf16"):
        dim, dt = (DIM, torch.float32) if op == "backward" else (128, torch.bfloat16)
        table = torch.empty(R, dim, device=dev).normal_(0, 0.01, generator=g).to(dt)
        state = torch.zeros(R, device=dev)
        grads = torch.empty(T, dim, device=dev).normal_(generator=g).to(dt)
        ws = B.workspace(B.backward_workspace_size(T, R, dim, B.dtype_code(table)), dev)
        is_co = (((ids * 0x9E3779B1) >> 7) & 1).to(torch.uint8)
        for _ in range(reps):
            B.fs_emb_backward_adagrad(table, state, ids, grads, "adagrad", 0.01, 1e-8, is_co=is_co,
                                      phase=B.PHASE_COLLISION_THEN_EXCLUSIVE, err=err, ws=ws)
    else:
        rio = torch.linspace(0, T, SHARDS + 1, device=dev).round().to(torch.int64)
        for _ in range(reps):
            B.fs_bucketize_rowwise(ids, rio, R, err=err)
    torch.cuda.synchronize()
    B.check(err, op)
    print(f"{op} T={T} R={R} reps={reps}: ok")
    return 0


def _transpose(T, F, reps, dev, g, err):
    Bs = 65536
    mean = max(1, T // (F * Bs))
    lens = torch.randint(0, 2 * mean + 1, (F * Bs,), device=dev, generator=g)
    off = torch.zeros(F * Bs + 1, dtype=torch.int64, device=dev)
    off[1:] = torch.cumsum(lens, 0)
    n = int(off[-1])
    val = torch.randint(0, 1 << 30, (n,), dtype=torch.int64, device=dev, generator=g)
    base = torch.arange(F, dtype=torch.int64, device=dev) * (1 << 30)
    out_off = torch.empty_like(off)
    out_val = torch.empty_like(val)
    ws = B.workspace(B.lib().fs_keyed_transpose_workspace_size(F, Bs), dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    best = None
    for _ in range(max(reps, 2)):
        ev[0].record()
        B.fs_keyed_transpose(off, val, F, Bs, row_base=base, out_offsets=out_off, out_values=out_val, err=err, ws=ws)
        ev[1].record()
        torch.cuda.synchronize()
        ms = ev[0].elapsed_time(ev[1])
        best = ms if best is None else min(best, ms)
    B.check(err, "transpose")
    byts = 16 * n + 16 * (F * Bs + 1) + 8 * F
    print(f"transpose F={F} B={Bs} IDs={n}: {best:.3f} ms, {byts / best / 1e6:.0f} GB/s of algorithmic bytes")
    return 0


def _median_ms(fn, reps):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    fn()
    for a, b in ev:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    return ms[len(ms) // 2]


def _gather_sorted(ids, T, R, reps, dev, g, err):
    reps = max(reps, 5)
    table = torch.empty(R, DIM, device=dev).normal_(0, 0.01, generator=g)
    out = torch.empty(T, DIM, device=dev)
    ws = B.workspace(B.backward_workspace_size(T, R, DIM, B.dtype_code(table)), dev)
    B.fs_emb_sort_rows(table, ids, ws, err=err)
    t_sorted = _median_ms(lambda: B.fs_emb_gather_sorted(table, T, ws, out=out, err=err), reps)
    t_plain = _median_ms(lambda: B.fs_emb_gather(table, ids, out=out, err=err), reps)
    torch.cuda.synchronize()
    B.check(err, "gather-sorted")
    U = int(torch.unique(ids).numel())
    byts = (8 + 4 * DIM) * T + 4 * DIM * U
    print(f"gather-sorted T={T} R={R} U={U}: sorted {t_sorted:.3f} ms ({byts / t_sorted / 1e6:.0f} GB/s), "
          f"position order {t_plain:.3f} ms ({byts / t_plain / 1e6:.0f} GB/s) (median of {reps})")
    return 0


def _prep(T, R, reps, dev, g, err):
    reps = max(reps, 3)
    n = SHARDS
    L = torch.empty(T // 2000 + 1, dtype=torch.float64, device=dev).log_normal_(6.8, 1.5, generator=g)
    L = L.round().clamp_(1, 16384).to(torch.int64)
    S = (L.numel() // n) * n
    L = L[:S]
    off = torch.zeros(S + 1, dtype=torch.int64, device=dev)
    off[1:] = torch.cumsum(L, 0)
    Tn = int(off[-1])
    ids = synthetic.zipf_rows(R, 1.0, Tn, g, dev)
    perm, ro, e0 = B.fs_balance_fbs(L.to(torch.int32), n)
    B.check(e0, "prep balance")
    outs = [torch.empty(S + 1, dtype=torch.int64, device=dev), torch.empty(Tn, dtype=torch.int64, device=dev),
            torch.empty(n + 1, dtype=torch.int64, device=dev), torch.empty(Tn, dtype=torch.int64, device=dev),
            torch.empty(Tn, dtype=torch.int32, device=dev), torch.empty(n, n, dtype=torch.int64, device=dev),
            torch.empty(n + 1, dtype=torch.int64, device=dev)]
    ws = B.workspace(B.lib().fs_permute_bucketize_workspace_size(S, Tn, n), dev)

    def call():
        B.fs_permute_bucketize(off, ids, perm, ro, R, capacity=Tn, out_offsets=outs[0], out_values=outs[1],
                               rank_id_offsets=outs[2], sm_ids=outs[3], pos=outs[4], splits=outs[5],
                               shard_offsets=outs[6], err=err, ws=ws)
    t = _median_ms(call, reps)
    B.check(err, "prep")
    byts = 16 * S + 36 * Tn
    print(f"prep S={S} T={Tn} R={R}: {t:.3f} ms, {byts / t / 1e6:.0f} GB/s of algorithmic bytes (median of {reps})")
    return 0


def _sorted_step(ids, T, R, reps, dev, g, err):
    reps = max(reps, 3)
    n = SHARDS
    table = torch.empty(R, DIM, device=dev).normal_(0, 0.01, generator=g)
    state = torch.zeros(R, device=dev)
    grads = torch.empty(T, DIM, device=dev).normal_(generator=g)
    rio = torch.linspace(0, T, n + 1, device=dev).round().to(torch.int64)
    sm, pos, _, so, e0 = B.fs_bucketize_rowwise(ids, rio, R)
    B.check(e0, "sorted-step bucketize")
    is_co = (((sm * 0x9E3779B1) >> 7) & 1).to(torch.uint8)             # half the rows, shard-major
    out = torch.empty(T, DIM, device=dev)
    ws = B.workspace(B.sort_rows_sharded_workspace_size(T, R, DIM, B.dtype_code(table), n), dev)
    ph = B.PHASE_COLLISION_THEN_EXCLUSIVE
    t_sort = _median_ms(lambda: B.fs_emb_sort_rows_sharded(table, sm, pos, so, ws, phase=ph, is_co=is_co, err=err),
                        reps)
    t_gather = _median_ms(lambda: B.fs_emb_gather_sorted(table, T, ws, out=out, phase=ph, err=err), reps)
    t_update = _median_ms(lambda: B.fs_emb_update_sorted(table, state, grads, T, ws, "adagrad", 0.01, 1e-8,
                                                         phase=ph, err=err), reps)
    torch.cuda.synchronize()
    B.check(err, "sorted-step")
    U = int(torch.unique(ids).numel())
    rb = 4 * DIM
    gb, ub = (8 + rb) * T + rb * U, (8 + rb) * T + (2 * rb + 8) * U
    print(f"sorted-step T={T} R={R} U={U}: sort {t_sort:.3f} ms, gather {t_gather:.3f} ms "
          f"({gb / t_gather / 1e6:.0f} GB/s), update {t_update:.3f} ms ({ub / t_update / 1e6:.0f} GB/s) "
          f"(median of {reps}); algorithmic bytes gather {gb}, update {ub}")
    return 0


def _bitmap(ids, T, R, reps, dev, err):
    reps = max(reps, 5)
    rio = torch.linspace(0, T, SHARDS + 1, device=dev).round().to(torch.int64)
    sm, _, _, _, e0 = B.fs_bucketize_rowwise(ids, rio, R)
    B.check(e0, "bitmap bucketize")
    bm = torch.empty(int(B.lib().fs_row_bitmap_words(R)), dtype=torch.int32, device=dev)
    t = _median_ms(lambda: B.fs_row_bitmap(sm, R, bitmap=bm, err=err), reps)
    B.check(err, "bitmap")
    print(f"bitmap T={T} R={R}: {t:.3f} ms, {8 * T / t / 1e6:.0f} GB/s of IDs read (median of {reps})")
    return 0


def _collision(a, b, T, R, reps, dev, err):
    reps = max(reps, 5)
    n = SHARDS
    bma, _ = B.fs_row_bitmap(a, R, err=err)
    bmb, _ = B.fs_row_bitmap(b, R, err=err)
    cap = min(2 * T, R)
    out = {k: torch.empty(cap, dtype=torch.int64, device=dev) for k in ("co", "ex_t", "ex_next")}
    out.update({"counts": torch.zeros(3, dtype=torch.int64, device=dev)})
    out.update({k: torch.empty(n + 1, dtype=torch.int64, device=dev) for k in ("co_off", "ex_t_off", "ex_next_off")})
    ws = B.workspace(B.lib().fs_collision_split_bitmaps_workspace_size(R), dev)
    t = _median_ms(lambda: B.fs_collision_split_bitmaps(a, bma, b, bmb, R, n, out, cap, err=err, ws=ws,
                                                        want_t_mask=False, want_next_mask=False), reps)
    B.check(err, "collision")
    print(f"collision T={T} R={R}: {t:.3f} ms, lists {out['counts'].tolist()} (median of {reps})")
    return 0


def _autotune(S, n, reps, dev, g, err):
    reps = max(reps, 5)
    L = torch.empty(S, dtype=torch.float64, device=dev).log_normal_(7.0, 1.6, generator=g)
    L = L.round().clamp_(1, 16384).to(torch.int32)
    times = (torch.rand(n, dtype=torch.float64, device=dev, generator=g) * 1e7 + 1e7).to(torch.int64)
    delta = torch.zeros(n, dtype=torch.int64, device=dev)
    perm = torch.empty(S, dtype=torch.int32, device=dev)
    ro = torch.empty(n + 1, dtype=torch.int64, device=dev)
    sw = torch.empty(n, dtype=torch.int64, device=dev)
    ws = B.workspace(B.lib().fs_balance_vbs_workspace_size(S, n), dev)
    # a few updates first, so that the timed cut moves real corrections (step 0 keeps them fixed while timing)
    for _ in range(8):
        B.fs_vbs_autotune(times, delta, 1, 0, err=err)
    t_upd = _median_ms(lambda: B.fs_vbs_autotune(times, delta, 0, 0, err=err), reps)
    t_tuned = _median_ms(lambda: B.fs_balance_vbs_tuned(L, n, 1.5, 1, delta, perm=perm, rank_offsets=ro,
                                                         seg_weight=sw, err=err, ws=ws), reps)
    t_plain = _median_ms(lambda: B.fs_balance_vbs(L, n, 1.5, 1, perm=perm, rank_offsets=ro, seg_weight=sw,
                                                  err=err, ws=ws), reps)
    torch.cuda.synchronize()
    B.check(err, "autotune")
    print(f"autotune S={S} n={n}: update {1000 * t_upd:.1f} us, tuned VBS cut {1000 * t_tuned:.1f} us, "
          f"plain VBS cut {1000 * t_plain:.1f} us (median of {reps})")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
