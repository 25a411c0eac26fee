"""One FreeScale training iteration's jagged index + embedding path on one GPU.

Sequences the C-ABI calls of binding.py over preallocated device buffers
(FreeScale, arXiv 2604.24073: Algorithm 1 for the balance + shuffle,
Algorithm 2 for the collision split, lookups and updates).  n logical ranks
live in one GPU's memory, so the AllGathers of Algorithm 1 are the identity
and every AllToAll is a device-memory permutation done by the kernels.

Two orders are provided:
  * step_sync   -- gather of iteration t, then the update of t (collision rows
                   first, then exclusive rows); the IDs of t+1 are prepared
                   and split against t before the update, as Algorithm 2 does.
                   With an update, the update's sort runs first and the
                   gather reads its sorted entries (each distinct row once).
  * run_prioritized -- Algorithm 2's order: exclusive rows of t+1 prefetched
                   before the update of t, collision rows of t updated first,
                   then gathered for t+1; exclusive updates of t deferred to
                   the next forward.  It needs a second output buffer and a
                   third batch slot.  With streams=True the exclusive-row work
                   (the deferred updates and the prefetch, Algorithm 2's
                   "C.stream") runs on a side stream, ordered against the main
                   stream by events only where the two touch the same data.
"""
from __future__ import annotations

import torch

from . import binding as B


class Slot:
    """Device buffers of one prepared batch (balance, permute, bucketize)."""

    def __init__(self, w, max_S, max_T, device):
        n = w.n
        self.perm = torch.empty(max_S, dtype=torch.int32, device=device)
        self.rank_offsets = torch.empty(n + 1, dtype=torch.int64, device=device)
        self.seg_weight = torch.empty(n, dtype=torch.int64, device=device)
        self.offsets = torch.empty(max_S + 1, dtype=torch.int64, device=device)
        self.ids = torch.empty(max_T, dtype=torch.int64, device=device)
        self.rank_id_offsets = torch.empty(n + 1, dtype=torch.int64, device=device)
        self.sm_ids = torch.empty(max_T, dtype=torch.int64, device=device)
        self.pos = torch.empty(max_T, dtype=torch.int32, device=device)
        self.splits = torch.empty(n, n, dtype=torch.int64, device=device)
        self.shard_offsets = torch.empty(n + 1, dtype=torch.int64, device=device)
        # presence bitmap of the batch's rows: built once, used by both collision
        # pairs the batch belongs to
        self.bitmap = torch.empty((w.R + 31) // 32, dtype=torch.int32, device=device)
        if w.composite:  # candidate lengths, permuted with the samples (Algorithm 1 Stage II)
            self.cand_offsets = torch.empty(max_S + 1, dtype=torch.int64, device=device)
            self.cand_lens = torch.empty(max_S * max(w.cmax, 1), dtype=torch.int64, device=device)
        self.T = 0


class Pipeline:
    def __init__(self, w, device, max_T, table, state=None, max_S=None, two_outputs=False, row_sorted=True,
                 streams=False):
        self.w = w
        # synchronous order with an update: sort once, gather and update from the sorted entries
        self.row_sorted = row_sorted
        self.dev = torch.device(device)
        self.max_T = int(max_T)
        self.max_S = int(max_S or w.S)
        self.table = table
        self.state = state
        dev = self.dev
        # the prioritized order keeps three batches: t-1 (its exclusive update is deferred), t and t+1
        self.slots = [Slot(w, self.max_S, self.max_T, dev) for _ in range(3 if two_outputs else 2)]
        cap = min(2 * self.max_T, w.R)
        self.cap_rows = cap
        self.coll = {
            "co": torch.empty(cap, dtype=torch.int64, device=dev),
            "ex_t": torch.empty(cap, dtype=torch.int64, device=dev),
            "ex_next": torch.empty(cap, dtype=torch.int64, device=dev),
            "counts": torch.zeros(3, dtype=torch.int64, device=dev),
            "co_off": torch.empty(w.n + 1, dtype=torch.int64, device=dev),
            "ex_t_off": torch.empty(w.n + 1, dtype=torch.int64, device=dev),
            "ex_next_off": torch.empty(w.n + 1, dtype=torch.int64, device=dev),
        }
        self.masks = [torch.zeros(self.max_T, dtype=torch.uint8, device=dev) for _ in self.slots]
        # order of each slot's mask: "batch" (aligned with ids) or "shard" (aligned with sm_ids)
        self.mask_layout = ["batch"] * len(self.slots)
        self.out = [torch.empty(self.max_T, w.D, dtype=table.dtype, device=dev)]
        if two_outputs:
            self.out.append(torch.empty(self.max_T, w.D, dtype=table.dtype, device=dev))
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # VBS AutoTune: per-rank batch-size corrections, carried across iterations
        self.batch_delta = torch.zeros(w.n, dtype=torch.int64, device=dev) if w.autotune else None
        L = B.lib()
        ws_bytes = max(
            L.fs_balance_vbs_workspace_size(self.max_S, w.n),
            L.fs_balance_fbs_workspace_size(self.max_S, w.n),
            L.fs_permute_jagged_workspace_size(self.max_S),
            L.fs_bucketize_rowwise_workspace_size(self.max_T, w.n),
            L.fs_permute_bucketize_workspace_size(self.max_S, self.max_T, w.n),
            L.fs_collision_split_bitmaps_workspace_size(w.R),
            B.backward_workspace_size(self.max_T, w.R, w.D, B.dtype_code(table)) if w.has_update else 0,
            B.sort_rows_sharded_workspace_size(self.max_T, w.R, w.D, B.dtype_code(table), w.n)
            if w.has_update and w.n <= 1024 else 0,
        )
        # one workspace, reused by every call (calls on one stream run in order)
        self.ws = B.workspace(ws_bytes, dev)
        # Algorithm 2's side stream: the deferred exclusive updates sort in a workspace of their own
        self.side = None
        if streams:
            self.side = torch.cuda.Stream(dev)
            self.ws_side = B.workspace(B.backward_workspace_size(self.max_T, w.R, w.D, B.dtype_code(table))
                                       if w.has_update else 256, dev)

    # -------------------------------------------------------------- stages
    def prepare(self, batch, slot):
        """Balance + permute + bucketize one batch into slot, and its rows' presence bitmap
        (Algorithm 1; Algorithm 2 line 8)."""
        w, s = self.w, self.slots[slot]
        if w.balance == "fbs":
            B.fs_balance_fbs(batch["uih_len"], w.n, perm=s.perm, rank_offsets=s.rank_offsets, err=self.err, ws=self.ws)
        elif w.autotune:
            B.fs_balance_vbs_tuned(batch["uih_len"], w.n, w.alpha, w.sort_by_len, self.batch_delta, perm=s.perm,
                                   rank_offsets=s.rank_offsets, seg_weight=s.seg_weight, err=self.err, ws=self.ws)
        else:
            B.fs_balance_vbs(batch["uih_len"], w.n, w.alpha, w.sort_by_len, perm=s.perm, rank_offsets=s.rank_offsets,
                             seg_weight=s.seg_weight, err=self.err, ws=self.ws)
        T = int(batch["T"])
        # the shuffle and the ranged dispatch in one call: the source IDs are read once (§4.2)
        B.fs_permute_bucketize(batch["offsets"], batch["ids"], s.perm[: batch["uih_len"].numel()], s.rank_offsets,
                               w.R, capacity=self.max_T, out_offsets=s.offsets[: batch["offsets"].numel()],
                               out_values=s.ids, rank_id_offsets=s.rank_id_offsets, sm_ids=s.sm_ids, pos=s.pos,
                               splits=s.splits, shard_offsets=s.shard_offsets, err=self.err, ws=self.ws)
        if w.composite:
            B.fs_permute_jagged(batch["cand_offsets"], batch["cand_lens"], s.perm[: batch["uih_len"].numel()],
                                capacity=s.cand_lens.numel(), out_offsets=s.cand_offsets[: batch["offsets"].numel()],
                                out_values=s.cand_lens, err=self.err, ws=self.ws)
        # the row set does not depend on the order; in shard-major order the IDs a warp marks
        # fall in one shard's stretch of the bitmap
        B.fs_row_bitmap(s.sm_ids, w.R, bitmap=s.bitmap, err=self.err, T=T)
        s.T = T

    def autotune(self, times):
        """VBS AutoTune (FreeScale §4.1): fold the ranks' latest step times [n] (int64 ns, device)
        into the batch-size corrections that the next prepared batch's cut takes."""
        w = self.w
        B.fs_vbs_autotune(times, self.batch_delta, step=w.tune_step, tol_ppm=w.tune_tol_ppm, err=self.err)

    def collision(self, slot_t, slot_next, want_t_mask=True, want_next_mask=True, shard_major=False):
        """Collision / exclusive split of (t, t+1) (Algorithm 2 line 10).

        The mask of t gives the update its phases; the mask of t+1 only serves
        the prioritized order's masked gathers of t+1.  The masks are aligned
        with the batch-major IDs, or with the shard-major IDs when shard_major
        (Algorithm 2 computes the split on the shard-major form; the sets are
        the same either way).
        """
        a, b = self.slots[slot_t], self.slots[slot_next]
        out = dict(self.coll)
        out["is_co_t"] = self.masks[slot_t]
        out["is_co_next"] = self.masks[slot_next]
        ids_t, ids_n = (a.sm_ids, b.sm_ids) if shard_major else (a.ids, b.ids)
        B.fs_collision_split_bitmaps(ids_t, a.bitmap, ids_n, b.bitmap, self.w.R, self.w.n, out, self.cap_rows,
                                     err=self.err, ws=self.ws, T_t=a.T, T_next=b.T, want_t_mask=want_t_mask,
                                     want_next_mask=want_next_mask)
        layout = "shard" if shard_major else "batch"
        if want_t_mask:
            self.mask_layout[slot_t] = layout
        if want_next_mask:
            self.mask_layout[slot_next] = layout

    def gather(self, slot, out_idx=0, mask=None, sel=1, sorted_phase=None, shard_major=False):
        """Lookup of the batch in `slot` (Algorithm 2 lines 12, 15); with sorted_phase, from the entries
        sort_rows left in the workspace (each distinct row read once); with shard_major, from the
        bucketize output (each shard's rows looked up together, then put at their batch-major positions)."""
        s = self.slots[slot]
        if sorted_phase is not None:
            B.fs_emb_gather_sorted(self.table, s.T, self.ws, out=self.out[out_idx], phase=sorted_phase, err=self.err)
        elif shard_major:
            assert mask is None
            B.fs_emb_gather_shard_major(self.table, s.sm_ids, s.pos, out=self.out[out_idx], err=self.err, T=s.T)
        else:
            B.fs_emb_gather(self.table, s.ids, out=self.out[out_idx], mask=mask, sel=sel, err=self.err, T=s.T)

    def sort_rows(self, slot, phase, co_rows=None):
        """The update's sort of the batch in `slot`, ahead of its gather: per shard from the shard-major
        IDs when the shards allow it (collision flags from co_rows, the next batch's row bitmap, when
        given, else from the batch's shard-major mask), else over the batch-major IDs (flags from the
        batch-major mask)."""
        s = self.slots[slot]
        two = phase != B.PHASE_ALL
        if self._sharded_ok(phase):
            if two and co_rows is None:
                assert self.mask_layout[slot] == "shard"
            B.fs_emb_sort_rows_sharded(self.table, s.sm_ids, s.pos, s.shard_offsets, self.ws, phase=phase,
                                       is_co=self.masks[slot] if two and co_rows is None else None,
                                       co_rows=co_rows if two else None, err=self.err, T=s.T)
        else:
            assert not two or self.mask_layout[slot] == "batch"
            B.fs_emb_sort_rows(self.table, s.ids, self.ws, phase=phase, is_co=self.masks[slot] if two else None,
                               err=self.err, T=s.T)

    def update_sorted(self, slot, grads, phase):
        w, s = self.w, self.slots[slot]
        B.fs_emb_update_sorted(self.table, self.state, grads, s.T, self.ws, w.optim, w.lr, w.eps, phase=phase,
                               err=self.err)

    def _sharded_ok(self, phase):
        # the per-shard sort: at most 1024 shards; a shard's row offsets (and the phase bit) in 20 bits
        block = -(-self.w.R // self.w.n)
        limit = 1 << (19 if phase != B.PHASE_ALL else 20)
        return self.row_sorted and self.w.n <= 1024 and block <= limit

    def _sorted_ok(self, phase):
        # the phase bit must fit beside the row bits; 16-byte aligned rows for the gather
        return (self.row_sorted and (phase == B.PHASE_ALL or self.w.R <= (1 << 30))
                and self.table.data_ptr() % 16 == 0 and self.out[0].data_ptr() % 16 == 0)

    def backward(self, slot, grads, phase=B.PHASE_ALL, co_rows=None, ws=None):
        """Update of the batch in `slot`; the phase's collision flags come from the batch's mask, or
        from co_rows (the row bitmap of the next batch) when given."""
        w, s = self.w, self.slots[slot]
        use_mask = phase != B.PHASE_ALL and co_rows is None
        B.fs_emb_backward_adagrad(self.table, self.state, s.ids, grads, w.optim, w.lr, w.eps,
                                  is_co=self.masks[slot] if use_mask else None, phase=phase,
                                  err=self.err, ws=self.ws if ws is None else ws, T=s.T, co_rows=co_rows)

    # -------------------------------------------------------------- orders
    def step_sync(self, cur, nxt_batch, grads, has_next=True, want_masks=False, times=None):
        """One iteration in the synchronous order; slot `cur` holds iteration t already prepared.

        The update's collision flags: the per-shard sort looks each entry's row up
        in t+1's row bitmap (its entries come shard-major, so the lookups of a
        tile stay in one shard's stretch of the bitmap); the batch-major sort and
        the one-call update read the mask of t instead (in batch-major order a
        bitmap lookup per entry was measured slower than the mask pass).
        want_masks also writes the masks of t and t+1 (shard-major unless the
        update reads them batch-major: self.mask_layout says which).  With AutoTune on,
        `times` (the ranks' latest step times) is folded into the corrections
        before t+1 is prepared.
        Returns the slot that now holds t+1.
        """
        nxt = 1 - cur
        # one sort, collision rows updated first, then exclusive rows
        phase = B.PHASE_COLLISION_THEN_EXCLUSIVE if has_next else B.PHASE_ALL
        sharded = self.w.has_update and self._sorted_ok(phase) and self._sharded_ok(phase)
        # the per-shard sort reads the collision rows from t+1's row bitmap; only the other updates read
        # the mask of t (batch-major).  Masks asked for (want_masks) are shard-major unless those read them.
        batch_major_update = self.w.has_update and not sharded
        if has_next:
            if times is not None and self.w.autotune:
                self.autotune(times)
            self.prepare(nxt_batch, nxt)
            self.collision(cur, nxt, want_t_mask=want_masks or batch_major_update, want_next_mask=want_masks,
                           shard_major=not batch_major_update)
        if not self.w.has_update:
            self.gather(cur, shard_major=True)
            return nxt
        if self._sorted_ok(phase):
            self.sort_rows(cur, phase, co_rows=self.slots[nxt].bitmap if (sharded and has_next) else None)
            self.gather(cur, sorted_phase=phase)
            self.update_sorted(cur, grads, phase)
        else:
            self.gather(cur)
            self.backward(cur, grads, phase)
        return nxt

    # ------------------------------------------------ Algorithm 2, one iteration at a time
    def prio_begin(self, batch0):
        """Prioritized order: prepare the first batch and gather it whole (slot 0, output 0)."""
        assert len(self.out) == 2 and len(self.slots) == 3
        self.prepare(batch0, 0)
        self.gather(0, out_idx=0)
        self._t = 0
        self._pending_ex = None                # (slot, grads, event after its split) of the deferred update
        self._slot_free = [None] * 3           # side-stream event after which a slot may be rewritten

    def _exclusive_update(self, slot, grads, ev_split):
        """Algorithm 2 line 7: the deferred update of the batch in `slot`'s exclusive rows (side stream)."""
        if self.side is None:
            self.backward(slot, grads, B.PHASE_EXCLUSIVE)
            return
        self.side.wait_event(ev_split)
        with torch.cuda.stream(self.side):
            self.backward(slot, grads, B.PHASE_EXCLUSIVE, ws=self.ws_side)
        ev = torch.cuda.Event()
        ev.record(self.side)
        self._slot_free[slot] = ev

    def prio_step(self, next_batch, grads, times=None, on_output=None):
        """Iteration t of Algorithm 2 (t counts calls since prio_begin); next_batch is None for the last.

        Batch t lives in slot t % 3 and its output in out[t % 2]; on_output(t, rows) sees it whole.
        Main stream: prepare t+1, the split of (t, t+1), the collision rows of t (line 20), then
        their lookup for t+1 (line 21).  Side stream (or the main one): the deferred exclusive update
        of t-1 (line 7), then the prefetch of t+1's exclusive rows (line 12), which may read rows
        that update wrote.  The two streams touch disjoint rows: the exclusive rows of t-1 are not
        rows of t, and those of t+1 are not rows of t either.
        """
        t = self._t
        cur, nxt = t % 3, (t + 1) % 3
        side = self.side
        main = torch.cuda.current_stream(self.dev) if side is not None else None
        if self._pending_ex is not None:                                 # line 7
            self._exclusive_update(*self._pending_ex)
            self._pending_ex = None
        ev_split = ev_pref = None
        if next_batch is not None:                                       # lines 8-12
            if self._slot_free[nxt] is not None:                         # batch t-2's deferred update read it
                main.wait_event(self._slot_free[nxt])
                self._slot_free[nxt] = None
            if times is not None and self.w.autotune:
                self.autotune(times)
            self.prepare(next_batch, nxt)
            self.collision(cur, nxt)
            if side is not None:
                ev_split = torch.cuda.Event()
                ev_split.record(main)
                side.wait_event(ev_split)
                with torch.cuda.stream(side):
                    self.gather(nxt, out_idx=(t + 1) % 2, mask=self.masks[nxt], sel=0)
                ev_pref = torch.cuda.Event()
                ev_pref.record(side)
            else:
                self.gather(nxt, out_idx=(t + 1) % 2, mask=self.masks[nxt], sel=0)
        if on_output is not None:
            on_output(t, self.out[t % 2][: self.slots[cur].T])
        if self.w.has_update:                                            # lines 18-20
            if next_batch is not None:
                self.backward(cur, grads, B.PHASE_COLLISION)
                self._pending_ex = (cur, grads, ev_split)
            else:
                self.backward(cur, grads, B.PHASE_ALL)
        if next_batch is not None:                                       # line 21
            self.gather(nxt, out_idx=(t + 1) % 2, mask=self.masks[nxt], sel=1)
            if ev_pref is not None:
                main.wait_event(ev_pref)                                 # the output of t+1 is whole
        self._t = t + 1

    def prio_finish(self):
        """The exclusive update still deferred after the last iteration; the side stream joins the main one."""
        if self._pending_ex is not None:
            self._exclusive_update(*self._pending_ex)
            self._pending_ex = None
        if self.side is not None:
            ev = torch.cuda.Event()
            ev.record(self.side)
            torch.cuda.current_stream(self.dev).wait_event(ev)
        self._slot_free = [None] * 3

    def run_prioritized(self, batches, grads_list, on_output=None, times_list=None):
        """Algorithm 2 order over len(batches) iterations.  on_output(t, out_tensor) sees each batch's output;
        with AutoTune on, times_list[t] is folded in before t+1 is prepared (as in step_sync)."""
        K = len(batches)
        self.prio_begin(batches[0])
        for t in range(K):
            self.prio_step(batches[t + 1] if t + 1 < K else None, grads_list[t] if grads_list else None,
                           times=times_list[t] if times_list is not None else None, on_output=on_output)
        self.prio_finish()
