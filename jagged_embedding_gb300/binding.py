"""Thin Python binding of the C ABI in include/fs_jagged.h (ctypes).

Argument marshalling only: every step runs in the CUDA library
(libfsjagged.so, built in-tree by build.py).  torch supplies device memory and
the current stream.  There is no fallback: if the library is missing or the
device is not a CUDA device, the calls raise.

Each function has the name of the C entry point it wraps.  Outputs and
workspace may be passed in (the benchmark does, to keep allocations out of the
timed region); otherwise they are allocated with torch.  Data errors found on
the device land in the int32 `err` tensor (first error wins); `check(err)`
waits for the stream and raises on a non-zero code.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfsjagged.so")

F32, BF16 = 0, 1
SGD, ROWWISE_ADAGRAD = 0, 1
PHASE_ALL, PHASE_COLLISION, PHASE_EXCLUSIVE, PHASE_COLLISION_THEN_EXCLUSIVE = 0, 1, 2, 3

STATUS = {0: "ok", 1: "invalid argument", 2: "ID outside [0, num_rows)", 3: "malformed offsets or permutation",
          4: "output capacity exceeded", 5: "workspace too small", 6: "bounded inter-block wait gave up",
          7: "CUDA runtime error", 8: "misaligned pointer"}

EXPORTS = [
    "fs_balance_fbs_workspace_size", "fs_balance_fbs", "fs_balance_fbs_noalloc", "fs_balance_vbs_workspace_size",
    "fs_balance_vbs", "fs_balance_vbs_tuned", "fs_vbs_autotune",
    "fs_permute_jagged_workspace_size", "fs_permute_jagged", "fs_keyed_transpose_workspace_size",
    "fs_keyed_transpose", "fs_bucketize_rowwise_workspace_size",
    "fs_bucketize_rowwise", "fs_permute_bucketize_workspace_size", "fs_permute_bucketize",
    "fs_collision_split_workspace_size", "fs_collision_split", "fs_row_bitmap_words",
    "fs_row_bitmap", "fs_collision_split_bitmaps_workspace_size", "fs_collision_split_bitmaps", "fs_emb_gather", "fs_emb_gather_shard_major",
    "fs_emb_backward_adagrad_workspace_size", "fs_emb_backward_adagrad", "fs_emb_sort_rows",
    "fs_emb_gather_sorted", "fs_emb_update_sorted", "fs_emb_sort_rows_sharded_workspace_size",
    "fs_emb_sort_rows_sharded", "fs_check", "fs_status_string",
    "fs_set_spin_limit", "fs_get_spin_limit", "fs_debug_skip_publish", "fs_launch_count", "fs_version",
]


class FsError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, 'status %d' % self.code)} (code {self.code})")


_lib = None


def lib():
    """Load libfsjagged.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FsError(7, f"CUDA library not built ({LIB_PATH}); run jagged_embedding_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    P, i64, i32, f64, f32, sz, u8 = C.c_void_p, C.c_int64, C.c_int32, C.c_double, C.c_float, C.c_size_t, C.c_uint8
    sig = {
        "fs_balance_fbs_workspace_size": ([i64, i32], sz),
        "fs_balance_fbs": ([P, i64, i32, P, P, P, P, sz, P], C.c_int),
        "fs_balance_fbs_noalloc": ([P, i64, i32, P, P, P, P], C.c_int),
        "fs_balance_vbs_workspace_size": ([i64, i32], sz),
        "fs_balance_vbs": ([P, i64, i32, f64, i32, P, P, P, P, P, sz, P], C.c_int),
        "fs_balance_vbs_tuned": ([P, i64, i32, f64, i32, P, P, P, P, P, P, sz, P], C.c_int),
        "fs_vbs_autotune": ([P, i32, i64, i32, P, P, P], C.c_int),
        "fs_permute_jagged_workspace_size": ([i64], sz),
        "fs_permute_jagged": ([P, P, i64, P, P, P, i64, P, i32, P, P, P, sz, P], C.c_int),
        "fs_keyed_transpose_workspace_size": ([i64, i64], sz),
        "fs_keyed_transpose": ([P, P, i64, i64, P, P, P, i64, P, P, sz, P], C.c_int),
        "fs_bucketize_rowwise_workspace_size": ([i64, i32], sz),
        "fs_bucketize_rowwise": ([P, i64, P, i32, i64, P, P, P, P, P, P, sz, P], C.c_int),
        "fs_permute_bucketize_workspace_size": ([i64, i64, i32], sz),
        "fs_permute_bucketize": ([P, P, i64, P, P, i32, i64, P, P, i64, P, P, P, P, P, P, P, sz, P], C.c_int),
        "fs_collision_split_workspace_size": ([i64, i64, i64, i32], sz),
        "fs_collision_split": ([P, i64, P, i64, i64, i32, P, P, P, i64, P, P, P, P, P, P, P, P, sz, P], C.c_int),
        "fs_row_bitmap_words": ([i64], sz),
        "fs_row_bitmap": ([P, i64, i64, P, P, P], C.c_int),
        "fs_collision_split_bitmaps_workspace_size": ([i64], sz),
        "fs_collision_split_bitmaps": ([P, i64, P, P, i64, P, i64, i32, P, P, P, i64, P, P, P, P, P, P, P, P, sz, P],
                                       C.c_int),
        "fs_emb_gather": ([P, i64, i32, C.c_int, P, i64, P, u8, P, P, P], C.c_int),
        "fs_emb_gather_shard_major": ([P, i64, i32, C.c_int, P, P, i64, P, P, P], C.c_int),
        "fs_emb_backward_adagrad_workspace_size": ([i64, i64, i32, C.c_int], sz),
        "fs_emb_sort_rows": ([i64, i32, C.c_int, P, i64, P, P, C.c_int, P, P, sz, P], C.c_int),
        "fs_emb_gather_sorted": ([P, i64, i32, C.c_int, i64, C.c_int, P, P, P, sz, P], C.c_int),
        "fs_emb_sort_rows_sharded_workspace_size": ([i64, i64, i32, C.c_int, i32], sz),
        "fs_emb_sort_rows_sharded": ([i64, i32, C.c_int, P, P, i64, P, i32, P, P, C.c_int, P, P, sz, P], C.c_int),
        "fs_emb_update_sorted": ([P, P, i64, i32, C.c_int, C.c_int, P, i64, C.c_int, f32, f32, P, P, sz, P],
                                 C.c_int),
        "fs_emb_backward_adagrad": ([P, P, i64, i32, C.c_int, C.c_int, P, P, i64, P, P, C.c_int, f32, f32, P, P, sz,
                                     P], C.c_int),
        "fs_check": ([P, P], C.c_int),
        "fs_status_string": ([C.c_int], C.c_char_p),
        "fs_set_spin_limit": ([i64], None),
        "fs_get_spin_limit": ([], i64),
        "fs_debug_skip_publish": ([i64], None),
        "fs_launch_count": ([], i64),
        "fs_version": ([], C.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    env = os.environ.get("FS_SPIN_LIMIT")
    if env:  # bounded waits: polls before giving up with FS_ERR_TIMEOUT
        try:
            polls = int(env)
        except ValueError:
            raise FsError(1, f"FS_SPIN_LIMIT={env!r} is not an integer") from None
        if polls < 1:
            raise FsError(1, f"FS_SPIN_LIMIT={env!r} must be positive")
        L.fs_set_spin_limit(polls)
    _lib = L
    return L


# ------------------------------------------------------------------ helpers

def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(device):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, dtype, name, numel=None):
    if t.device.type != "cuda":
        raise FsError(1, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise FsError(1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise FsError(1, f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise FsError(1, f"{name} too small: {t.numel()} < {numel}")


def _ok(rc, where):
    if rc != 0:
        raise FsError(rc, where)


def new_err(device):
    return torch.zeros(1, dtype=torch.int32, device=device)


def workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def check(err, where="fs"):
    """Wait for the current stream and raise if the device error word is set."""
    rc = lib().fs_check(_ptr(err), _stream(err.device))
    _ok(rc, where)


def dtype_code(t):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise FsError(1, f"table dtype {t.dtype} not supported")


def launch_count():
    return int(lib().fs_launch_count())


def set_spin_limit(polls):
    lib().fs_set_spin_limit(int(polls))


def spin_limit():
    return int(lib().fs_get_spin_limit())


def debug_skip_publish(tile):
    lib().fs_debug_skip_publish(int(tile))


def version():
    return lib().fs_version().decode()


# ------------------------------------------------------------------ partition

def fs_balance_fbs(uih_len, n, perm=None, rank_offsets=None, err=None, ws=None):
    dev = uih_len.device
    _need(uih_len, torch.int32, "uih_len")
    S = uih_len.numel()
    perm = torch.empty(S, dtype=torch.int32, device=dev) if perm is None else perm
    rank_offsets = torch.empty(n + 1, dtype=torch.int64, device=dev) if rank_offsets is None else rank_offsets
    err = new_err(dev) if err is None else err
    need = lib().fs_balance_fbs_workspace_size(S, n)
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_balance_fbs(_ptr(uih_len), S, n, _ptr(perm), _ptr(rank_offsets), _ptr(err), _ptr(ws), ws.numel(),
                             _stream(dev)), "fs_balance_fbs")
    return perm, rank_offsets, err


def fs_balance_fbs_noalloc(uih_len, n, perm, rank_offsets, err):
    """FBS partition that allocates nothing: the caller passes every output, the
    scratch is a fixed array inside the library (S <= 262144; calls must not overlap)."""
    dev = uih_len.device
    _need(uih_len, torch.int32, "uih_len")
    _need(perm, torch.int32, "perm", uih_len.numel())
    _need(rank_offsets, torch.int64, "rank_offsets", n + 1)
    _need(err, torch.int32, "err", 1)
    _ok(lib().fs_balance_fbs_noalloc(_ptr(uih_len), uih_len.numel(), n, _ptr(perm), _ptr(rank_offsets), _ptr(err),
                                     _stream(dev)), "fs_balance_fbs_noalloc")
    return perm, rank_offsets, err


def fs_balance_vbs(uih_len, n, alpha, sort_by_len, perm=None, rank_offsets=None, seg_weight=None, err=None, ws=None):
    dev = uih_len.device
    _need(uih_len, torch.int32, "uih_len")
    S = uih_len.numel()
    perm = torch.empty(S, dtype=torch.int32, device=dev) if perm is None else perm
    rank_offsets = torch.empty(n + 1, dtype=torch.int64, device=dev) if rank_offsets is None else rank_offsets
    seg_weight = torch.empty(n, dtype=torch.int64, device=dev) if seg_weight is None else seg_weight
    err = new_err(dev) if err is None else err
    need = lib().fs_balance_vbs_workspace_size(S, n)
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_balance_vbs(_ptr(uih_len), S, n, float(alpha), int(bool(sort_by_len)), _ptr(perm),
                             _ptr(rank_offsets), _ptr(seg_weight), _ptr(err), _ptr(ws), ws.numel(), _stream(dev)),
        "fs_balance_vbs")
    return perm, rank_offsets, seg_weight, err


def fs_balance_vbs_tuned(uih_len, n, alpha, sort_by_len, batch_delta, perm=None, rank_offsets=None, seg_weight=None,
                         err=None, ws=None):
    """VBS cut with the AutoTune correction batch_delta [n] (int64, device) applied to its segment ends."""
    dev = uih_len.device
    _need(uih_len, torch.int32, "uih_len")
    _need(batch_delta, torch.int64, "batch_delta", n)
    S = uih_len.numel()
    perm = torch.empty(S, dtype=torch.int32, device=dev) if perm is None else perm
    rank_offsets = torch.empty(n + 1, dtype=torch.int64, device=dev) if rank_offsets is None else rank_offsets
    seg_weight = torch.empty(n, dtype=torch.int64, device=dev) if seg_weight is None else seg_weight
    err = new_err(dev) if err is None else err
    need = lib().fs_balance_vbs_workspace_size(S, n)
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_balance_vbs_tuned(_ptr(uih_len), S, n, float(alpha), int(bool(sort_by_len)), _ptr(batch_delta),
                                   _ptr(perm), _ptr(rank_offsets), _ptr(seg_weight), _ptr(err), _ptr(ws), ws.numel(),
                                   _stream(dev)), "fs_balance_vbs_tuned")
    return perm, rank_offsets, seg_weight, err


def fs_vbs_autotune(times, batch_delta, step=1, tol_ppm=0, err=None):
    """One AutoTune update of batch_delta [n] (int64, device, in place) from the ranks' times [n] (int64, device)."""
    dev = times.device
    n = times.numel()
    _need(times, torch.int64, "times")
    _need(batch_delta, torch.int64, "batch_delta", n)
    err = new_err(dev) if err is None else err
    _ok(lib().fs_vbs_autotune(_ptr(times), n, int(step), int(tol_ppm), _ptr(batch_delta), _ptr(err), _stream(dev)),
        "fs_vbs_autotune")
    return batch_delta, err


# ------------------------------------------------------------------ jagged ids

def fs_permute_jagged(offsets, values, perm, capacity=None, rank_offsets=None, out_offsets=None, out_values=None,
                      rank_id_offsets=None, err=None, ws=None):
    dev = offsets.device
    _need(offsets, torch.int64, "offsets")
    _need(values, torch.int64, "values")
    _need(perm, torch.int32, "perm")
    S = offsets.numel() - 1
    cap = values.numel() if capacity is None else int(capacity)
    out_offsets = torch.empty(S + 1, dtype=torch.int64, device=dev) if out_offsets is None else out_offsets
    out_values = torch.empty(cap, dtype=torch.int64, device=dev) if out_values is None else out_values
    n = 0
    if rank_offsets is not None:
        _need(rank_offsets, torch.int64, "rank_offsets")
        n = rank_offsets.numel() - 1
        rank_id_offsets = torch.empty(n + 1, dtype=torch.int64, device=dev) if rank_id_offsets is None else rank_id_offsets
    err = new_err(dev) if err is None else err
    need = lib().fs_permute_jagged_workspace_size(S)
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_permute_jagged(_ptr(offsets), _ptr(values), S, _ptr(perm), _ptr(out_offsets), _ptr(out_values), cap,
                                _ptr(rank_offsets), n, _ptr(rank_id_offsets), _ptr(err), _ptr(ws), ws.numel(),
                                _stream(dev)), "fs_permute_jagged")
    return out_offsets, out_values, rank_id_offsets, err


def fs_keyed_transpose(offsets, values, F, B, row_base=None, capacity=None, out_offsets=None, out_values=None,
                       err=None, ws=None):
    """Feature-major [F x B] jagged IDs to batch-major [B x F]; row_base (int64 [F]) shifts feature f's IDs."""
    dev = offsets.device
    _need(offsets, torch.int64, "offsets", F * B + 1)
    _need(values, torch.int64, "values")
    if row_base is not None:
        _need(row_base, torch.int64, "row_base", F)
    cap = values.numel() if capacity is None else int(capacity)
    out_offsets = torch.empty(F * B + 1, dtype=torch.int64, device=dev) if out_offsets is None else out_offsets
    out_values = torch.empty(cap, dtype=torch.int64, device=dev) if out_values is None else out_values
    err = new_err(dev) if err is None else err
    need = lib().fs_keyed_transpose_workspace_size(int(F), int(B))
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_keyed_transpose(_ptr(offsets), _ptr(values), int(F), int(B), _ptr(row_base), _ptr(out_offsets),
                                 _ptr(out_values), cap, _ptr(err), _ptr(ws), ws.numel(), _stream(dev)),
        "fs_keyed_transpose")
    return out_offsets, out_values, err


def fs_bucketize_rowwise(ids, rank_id_offsets, num_rows, sm_ids=None, pos=None, splits=None, shard_offsets=None,
                         err=None, ws=None, T=None):
    dev = ids.device
    _need(ids, torch.int64, "ids")
    _need(rank_id_offsets, torch.int64, "rank_id_offsets")
    n = rank_id_offsets.numel() - 1
    T = ids.numel() if T is None else int(T)
    sm_ids = torch.empty(T, dtype=torch.int64, device=dev) if sm_ids is None else sm_ids
    pos = torch.empty(T, dtype=torch.int32, device=dev) if pos is None else pos
    splits = torch.empty(n, n, dtype=torch.int64, device=dev) if splits is None else splits
    shard_offsets = torch.empty(n + 1, dtype=torch.int64, device=dev) if shard_offsets is None else shard_offsets
    err = new_err(dev) if err is None else err
    need = lib().fs_bucketize_rowwise_workspace_size(T, n)
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_bucketize_rowwise(_ptr(ids), T, _ptr(rank_id_offsets), n, int(num_rows), _ptr(sm_ids), _ptr(pos),
                                   _ptr(splits), _ptr(shard_offsets), _ptr(err), _ptr(ws), ws.numel(), _stream(dev)),
        "fs_bucketize_rowwise")
    return sm_ids, pos, splits, shard_offsets, err


def fs_permute_bucketize(offsets, values, perm, rank_offsets, num_rows, capacity=None, out_offsets=None,
                         out_values=None, rank_id_offsets=None, sm_ids=None, pos=None, splits=None,
                         shard_offsets=None, err=None, ws=None):
    """fs_permute_jagged (with rank_offsets) then fs_bucketize_rowwise, in one call that reads the source IDs
    once.  Returns (out_offsets, out_values, rank_id_offsets, sm_ids, pos, splits, shard_offsets, err)."""
    dev = offsets.device
    _need(offsets, torch.int64, "offsets")
    _need(values, torch.int64, "values")
    _need(perm, torch.int32, "perm")
    _need(rank_offsets, torch.int64, "rank_offsets")
    S = offsets.numel() - 1
    n = rank_offsets.numel() - 1
    cap = values.numel() if capacity is None else int(capacity)
    new = lambda t, k, dt: torch.empty(k, dtype=dt, device=dev) if t is None else t  # noqa: E731
    out_offsets = new(out_offsets, S + 1, torch.int64)
    out_values = new(out_values, cap, torch.int64)
    rank_id_offsets = new(rank_id_offsets, n + 1, torch.int64)
    sm_ids = new(sm_ids, cap, torch.int64)
    pos = new(pos, cap, torch.int32)
    splits = torch.empty(n, n, dtype=torch.int64, device=dev) if splits is None else splits
    shard_offsets = new(shard_offsets, n + 1, torch.int64)
    for t, nm, dt, k in ((out_values, "out_values", torch.int64, cap), (sm_ids, "sm_ids", torch.int64, cap),
                         (pos, "pos", torch.int32, cap), (out_offsets, "out_offsets", torch.int64, S + 1)):
        _need(t, dt, nm, k)
    err = new_err(dev) if err is None else err
    need = lib().fs_permute_bucketize_workspace_size(S, cap, n)
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_permute_bucketize(_ptr(offsets), _ptr(values), S, _ptr(perm), _ptr(rank_offsets), n, int(num_rows),
                                   _ptr(out_offsets), _ptr(out_values), cap, _ptr(rank_id_offsets), _ptr(sm_ids),
                                   _ptr(pos), _ptr(splits), _ptr(shard_offsets), _ptr(err), _ptr(ws), ws.numel(),
                                   _stream(dev)), "fs_permute_bucketize")
    return out_offsets, out_values, rank_id_offsets, sm_ids, pos, splits, shard_offsets, err


def fs_collision_split(ids_t, ids_next, num_rows, n, cap_rows=None, out=None, err=None, ws=None, T_t=None,
                       T_next=None, want_next_mask=True):
    """Returns dict with co/ex_t/ex_next (capacity-sized; counts on device), shard offsets and masks."""
    dev = ids_t.device
    _need(ids_t, torch.int64, "ids_t")
    _need(ids_next, torch.int64, "ids_next")
    Tt = ids_t.numel() if T_t is None else int(T_t)
    Tn = ids_next.numel() if T_next is None else int(T_next)
    cap = min(Tt + Tn, int(num_rows)) if cap_rows is None else int(cap_rows)
    if out is None:
        out = {
            "co": torch.empty(cap, dtype=torch.int64, device=dev),
            "ex_t": torch.empty(cap, dtype=torch.int64, device=dev),
            "ex_next": torch.empty(cap, dtype=torch.int64, device=dev),
            "counts": torch.empty(3, dtype=torch.int64, device=dev),
            "co_off": torch.empty(n + 1, dtype=torch.int64, device=dev),
            "ex_t_off": torch.empty(n + 1, dtype=torch.int64, device=dev),
            "ex_next_off": torch.empty(n + 1, dtype=torch.int64, device=dev),
            "is_co_t": torch.empty(Tt, dtype=torch.uint8, device=dev),
            "is_co_next": torch.empty(Tn, dtype=torch.uint8, device=dev),
        }
    err = new_err(dev) if err is None else err
    need = lib().fs_collision_split_workspace_size(Tt, Tn, int(num_rows), n)
    ws = workspace(need, dev) if ws is None else ws
    o = out
    _ok(lib().fs_collision_split(_ptr(ids_t), Tt, _ptr(ids_next), Tn, int(num_rows), n, _ptr(o["co"]),
                                 _ptr(o["ex_t"]), _ptr(o["ex_next"]), cap, _ptr(o["counts"]), _ptr(o["co_off"]),
                                 _ptr(o["ex_t_off"]), _ptr(o["ex_next_off"]), _ptr(o.get("is_co_t")),
                                 _ptr(o.get("is_co_next") if want_next_mask else None), _ptr(err), _ptr(ws),
                                 ws.numel(), _stream(dev)),
        "fs_collision_split")
    return out, err


def fs_row_bitmap(ids, num_rows, bitmap=None, err=None, T=None):
    dev = ids.device
    _need(ids, torch.int64, "ids")
    T = ids.numel() if T is None else int(T)
    words = int(lib().fs_row_bitmap_words(int(num_rows)))
    bitmap = torch.empty(words, dtype=torch.int32, device=dev) if bitmap is None else bitmap
    err = new_err(dev) if err is None else err
    _ok(lib().fs_row_bitmap(_ptr(ids), T, int(num_rows), _ptr(bitmap), _ptr(err), _stream(dev)), "fs_row_bitmap")
    return bitmap, err


def fs_collision_split_bitmaps(ids_t, bm_t, ids_next, bm_next, num_rows, n, out, cap_rows, err=None, ws=None,
                               T_t=None, T_next=None, want_t_mask=True, want_next_mask=True):
    """Same outputs as fs_collision_split (into the caller's `out` dict), from two row bitmaps."""
    dev = bm_t.device
    Tt = ids_t.numel() if T_t is None else int(T_t)
    Tn = ids_next.numel() if T_next is None else int(T_next)
    err = new_err(dev) if err is None else err
    need = lib().fs_collision_split_bitmaps_workspace_size(int(num_rows))
    ws = workspace(need, dev) if ws is None else ws
    o = out
    _ok(lib().fs_collision_split_bitmaps(
        _ptr(ids_t), Tt, _ptr(bm_t), _ptr(ids_next), Tn, _ptr(bm_next), int(num_rows), n, _ptr(o["co"]),
        _ptr(o["ex_t"]), _ptr(o["ex_next"]), int(cap_rows), _ptr(o["counts"]), _ptr(o["co_off"]), _ptr(o["ex_t_off"]),
        _ptr(o["ex_next_off"]), _ptr(o.get("is_co_t") if want_t_mask else None),
        _ptr(o.get("is_co_next") if want_next_mask else None), _ptr(err), _ptr(ws), ws.numel(), _stream(dev)),
        "fs_collision_split_bitmaps")
    return out, err


# ------------------------------------------------------------------ embeddings

def fs_emb_gather(table, ids, out=None, mask=None, sel=1, err=None, T=None):
    dev = table.device
    _need(ids, torch.int64, "ids")
    if table.dim() != 2 or not table.is_contiguous():
        raise FsError(1, "table must be a contiguous [R, D] tensor")
    R, D = table.shape
    T = ids.numel() if T is None else int(T)
    out = torch.empty(T, D, dtype=table.dtype, device=dev) if out is None else out
    if mask is not None:
        _need(mask, torch.uint8, "mask")
    err = new_err(dev) if err is None else err
    _ok(lib().fs_emb_gather(_ptr(table), R, D, dtype_code(table), _ptr(ids), T, _ptr(mask), int(sel), _ptr(out),
                            _ptr(err), _stream(dev)), "fs_emb_gather")
    return out, err


def fs_emb_gather_shard_major(table, sm_ids, pos, out=None, err=None, T=None):
    """out[pos[j]] = table[sm_ids[j]]: the gather from the bucketize output (the same bytes as fs_emb_gather)."""
    dev = table.device
    _need(sm_ids, torch.int64, "sm_ids")
    _need(pos, torch.int32, "pos")
    R, D = _table_shape(table)
    T = sm_ids.numel() if T is None else int(T)
    out = torch.empty(T, D, dtype=table.dtype, device=dev) if out is None else out
    if out.dtype != table.dtype or not out.is_contiguous() or out.numel() < T * D:
        raise FsError(1, "out must be contiguous [>= T, D] with the table dtype")
    err = new_err(dev) if err is None else err
    _ok(lib().fs_emb_gather_shard_major(_ptr(table), R, D, dtype_code(table), _ptr(sm_ids), _ptr(pos), T, _ptr(out),
                                        _ptr(err), _stream(dev)), "fs_emb_gather_shard_major")
    return out, err


def backward_workspace_size(T, num_rows, dim, dtype):
    return int(lib().fs_emb_backward_adagrad_workspace_size(int(T), int(num_rows), int(dim), int(dtype)))


def fs_emb_backward_adagrad(table, state, ids, grads, optim, lr, eps=0.0, is_co=None, phase=PHASE_ALL, err=None,
                            ws=None, T=None, co_rows=None):
    """is_co: uint8 collision flag per position; co_rows: int32 bitmap of the collision rows (one of the two
    unless phase is PHASE_ALL)."""
    dev = table.device
    _need(ids, torch.int64, "ids")
    if table.dim() != 2 or not table.is_contiguous():
        raise FsError(1, "table must be a contiguous [R, D] tensor")
    R, D = table.shape
    T = ids.numel() if T is None else int(T)
    if grads.dtype != table.dtype or not grads.is_contiguous():
        raise FsError(1, "grads must be contiguous with the table dtype")
    oc = {"sgd": SGD, "adagrad": ROWWISE_ADAGRAD}[optim] if isinstance(optim, str) else int(optim)
    if oc == ROWWISE_ADAGRAD:
        _need(state, torch.float32, "state", R)
    if is_co is not None:
        _need(is_co, torch.uint8, "is_co")
    if co_rows is not None:
        _need(co_rows, torch.int32, "co_rows", (R + 31) // 32)
    err = new_err(dev) if err is None else err
    need = backward_workspace_size(T, R, D, dtype_code(table))
    ws = workspace(need, dev) if ws is None else ws
    _ok(lib().fs_emb_backward_adagrad(_ptr(table), _ptr(state) if oc == ROWWISE_ADAGRAD else None, R, D,
                                      dtype_code(table), oc, _ptr(ids), _ptr(grads), T, _ptr(is_co), _ptr(co_rows),
                                      int(phase), float(lr), float(eps), _ptr(err), _ptr(ws), ws.numel(),
                                      _stream(dev)),
        "fs_emb_backward_adagrad")
    return err


# ------------------------------------------------------------------ row-sorted path

def _table_shape(table):
    if table.dim() != 2 or not table.is_contiguous():
        raise FsError(1, "table must be a contiguous [R, D] tensor")
    return table.shape


def fs_emb_sort_rows(table, ids, ws, phase=PHASE_ALL, is_co=None, co_rows=None, err=None, T=None):
    """Sort the batch's entries by (phase bit, row) into ws, for fs_emb_gather_sorted / fs_emb_update_sorted.
    `table` only gives num_rows, dim and dtype (it is not read)."""
    dev = ids.device
    _need(ids, torch.int64, "ids")
    R, D = _table_shape(table)
    T = ids.numel() if T is None else int(T)
    if is_co is not None:
        _need(is_co, torch.uint8, "is_co")
    if co_rows is not None:
        _need(co_rows, torch.int32, "co_rows", (R + 31) // 32)
    err = new_err(dev) if err is None else err
    _ok(lib().fs_emb_sort_rows(R, D, dtype_code(table), _ptr(ids), T, _ptr(is_co), _ptr(co_rows), int(phase),
                               _ptr(err), _ptr(ws), ws.numel(), _stream(dev)), "fs_emb_sort_rows")
    return err


def sort_rows_sharded_workspace_size(T, num_rows, dim, dtype, n):
    return int(lib().fs_emb_sort_rows_sharded_workspace_size(int(T), int(num_rows), int(dim), int(dtype), int(n)))


def fs_emb_sort_rows_sharded(table, sm_ids, pos, shard_offsets, ws, phase=PHASE_ALL, is_co=None, co_rows=None,
                             err=None, T=None):
    """The update's sort from the bucketize output (entries grouped by shard): the same sorted entries as
    fs_emb_sort_rows, in ws.  is_co: the collision flag of each shard-major entry; co_rows: the collision
    rows as an int32 bitmap (one of the two for two phases).  `table` only gives num_rows, dim and dtype."""
    dev = sm_ids.device
    _need(sm_ids, torch.int64, "sm_ids")
    _need(pos, torch.int32, "pos")
    _need(shard_offsets, torch.int64, "shard_offsets")
    R, D = _table_shape(table)
    T = sm_ids.numel() if T is None else int(T)
    n = shard_offsets.numel() - 1
    if is_co is not None:
        _need(is_co, torch.uint8, "is_co")
    if co_rows is not None:
        _need(co_rows, torch.int32, "co_rows", (R + 31) // 32)
    err = new_err(dev) if err is None else err
    _ok(lib().fs_emb_sort_rows_sharded(R, D, dtype_code(table), _ptr(sm_ids), _ptr(pos), T, _ptr(shard_offsets), n,
                                       _ptr(is_co), _ptr(co_rows), int(phase), _ptr(err), _ptr(ws), ws.numel(),
                                       _stream(dev)),
        "fs_emb_sort_rows_sharded")
    return err


def fs_emb_gather_sorted(table, T, ws, out=None, phase=PHASE_ALL, err=None):
    """out[p] = table[ids[p]] from the entries fs_emb_sort_rows left in ws."""
    dev = table.device
    R, D = _table_shape(table)
    out = torch.empty(int(T), D, dtype=table.dtype, device=dev) if out is None else out
    if out.dtype != table.dtype or not out.is_contiguous() or out.numel() < int(T) * D:
        raise FsError(1, "out must be contiguous [>= T, D] with the table dtype")
    err = new_err(dev) if err is None else err
    _ok(lib().fs_emb_gather_sorted(_ptr(table), R, D, dtype_code(table), int(T), int(phase), _ptr(out), _ptr(err),
                                   _ptr(ws), ws.numel(), _stream(dev)), "fs_emb_gather_sorted")
    return out, err


def fs_emb_update_sorted(table, state, grads, T, ws, optim, lr, eps=0.0, phase=PHASE_ALL, err=None):
    """Segment-reduce + row update of the entries fs_emb_sort_rows left in ws."""
    dev = table.device
    R, D = _table_shape(table)
    if grads.dtype != table.dtype or not grads.is_contiguous():
        raise FsError(1, "grads must be contiguous with the table dtype")
    oc = {"sgd": SGD, "adagrad": ROWWISE_ADAGRAD}[optim] if isinstance(optim, str) else int(optim)
    if oc == ROWWISE_ADAGRAD:
        _need(state, torch.float32, "state", R)
    err = new_err(dev) if err is None else err
    _ok(lib().fs_emb_update_sorted(_ptr(table), _ptr(state) if oc == ROWWISE_ADAGRAD else None, R, D,
                                   dtype_code(table), oc, _ptr(grads), int(T), int(phase), float(lr), float(eps),
                                   _ptr(err), _ptr(ws), ws.numel(), _stream(dev)), "fs_emb_update_sorted")
    return err
