"""The C-ABI library loads, exports every symbol the header declares, and rejects
bad arguments on the host (no GPU needed: nothing is launched for these)."""
import ctypes as C
import os
import re

import pytest

from jagged_embedding_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fs_jagged.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fs_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ["fs_balance_fbs", "fs_balance_vbs", "fs_permute_jagged", "fs_keyed_transpose", "fs_bucketize_rowwise",
              "fs_collision_split",
              "fs_emb_gather", "fs_emb_backward_adagrad"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = B.lib()
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert missing == []
    assert sorted(_declared()) == sorted(B.EXPORTS)


def test_status_strings_and_version():
    L = B.lib()
    for code, text in B.STATUS.items():
        assert L.fs_status_string(code).decode() == text
    assert "sm_103a" in B.version()


def test_workspace_queries():
    L = B.lib()
    assert L.fs_balance_fbs_workspace_size(131072, 256) > 4 * 131072 * 4
    assert L.fs_balance_vbs_workspace_size(32768, 512) > L.fs_balance_fbs_workspace_size(32768, 512)
    assert L.fs_permute_jagged_workspace_size(131072) >= 131072 * 8
    assert L.fs_bucketize_rowwise_workspace_size(10 ** 6, 256) > 0
    # two presence bitmaps of R bits
    assert L.fs_collision_split_workspace_size(0, 0, 10 ** 8, 256) >= 2 * 10 ** 8 // 8
    # key/value ping-pong of the backward sort: 16 bytes per ID at least
    assert L.fs_emb_backward_adagrad_workspace_size(10 ** 6, 10 ** 7, 64, 0) >= 16 * 10 ** 6
    assert L.fs_balance_fbs_workspace_size(-1, 4) == 0


NULL = None


def test_host_argument_errors_return_without_launching():
    L = B.lib()
    err = C.c_void_p(0x1000)  # never dereferenced: every call below fails host checks first
    ws = C.c_void_p(0x2000)
    assert L.fs_balance_fbs(NULL, 10, 0, NULL, NULL, err, ws, 1 << 30, NULL) == 1            # n < 1
    assert L.fs_balance_fbs(NULL, 10, 4, NULL, C.c_void_p(0x3000), err, ws, 1 << 30, NULL) == 1  # NULL input
    assert L.fs_balance_fbs(C.c_void_p(0x10), 10, 4, C.c_void_p(0x20), C.c_void_p(0x3000), err, ws, 16, NULL) == 5
    assert L.fs_balance_vbs(C.c_void_p(0x10), 10, 4, -1.0, 0, C.c_void_p(0x20), C.c_void_p(0x3000),
                            C.c_void_p(0x4000), err, ws, 1 << 30, NULL) == 1                   # alpha < 0
    # VBS AutoTune: a correction is required (8-byte aligned); 1 <= n <= 65536, step >= 0, tol in [0, 10^6]
    vbs_out = (C.c_void_p(0x20), C.c_void_p(0x3000), C.c_void_p(0x4000), err, ws, 1 << 30, NULL)
    assert L.fs_balance_vbs_tuned(C.c_void_p(0x10), 10, 4, 1.5, 0, NULL, *vbs_out) == 1
    assert L.fs_balance_vbs_tuned(C.c_void_p(0x10), 10, 4, 1.5, 0, C.c_void_p(0x5004), *vbs_out) == 8
    assert L.fs_balance_vbs_tuned(C.c_void_p(0x10), 10, 0, 1.5, 0, C.c_void_p(0x5000), *vbs_out) == 1
    tune = dict(times=C.c_void_p(0x100), delta=C.c_void_p(0x200))
    assert L.fs_vbs_autotune(tune["times"], 0, 1, 0, tune["delta"], err, NULL) == 1
    assert L.fs_vbs_autotune(tune["times"], 65537, 1, 0, tune["delta"], err, NULL) == 1
    assert L.fs_vbs_autotune(tune["times"], 4, -1, 0, tune["delta"], err, NULL) == 1
    assert L.fs_vbs_autotune(tune["times"], 4, 1, 1000001, tune["delta"], err, NULL) == 1
    assert L.fs_vbs_autotune(tune["times"], 4, 1, 0, NULL, err, NULL) == 1
    assert L.fs_vbs_autotune(C.c_void_p(0x104), 4, 1, 0, tune["delta"], err, NULL) == 8
    assert L.fs_bucketize_rowwise(C.c_void_p(0x10), 10, C.c_void_p(0x100), 1025, 100, C.c_void_p(0x20),
                                  C.c_void_p(0x30), C.c_void_p(0x40), C.c_void_p(0x50), err, ws, 1 << 30, NULL) == 1
    assert L.fs_bucketize_rowwise(C.c_void_p(0x13), 10, C.c_void_p(0x100), 4, 100, C.c_void_p(0x20),
                                  C.c_void_p(0x30), C.c_void_p(0x40), C.c_void_p(0x50), err, ws, 1 << 30, NULL) == 8
    # keyed transpose: F >= 1, F*B < 2^31, 8-byte aligned row bases
    assert L.fs_keyed_transpose(C.c_void_p(0x10), C.c_void_p(0x20), 0, 4, NULL, C.c_void_p(0x30), C.c_void_p(0x40),
                                10, err, ws, 1 << 30, NULL) == 1
    assert L.fs_keyed_transpose(C.c_void_p(0x10), C.c_void_p(0x20), 1 << 16, 1 << 16, NULL, C.c_void_p(0x30),
                                C.c_void_p(0x40), 10, err, ws, 1 << 30, NULL) == 1
    assert L.fs_keyed_transpose(C.c_void_p(0x10), C.c_void_p(0x20), 2, 4, C.c_void_p(0x54), C.c_void_p(0x30),
                                C.c_void_p(0x40), 10, err, ws, 1 << 30, NULL) == 8
    assert L.fs_keyed_transpose_workspace_size(4, 1000) >= L.fs_permute_jagged_workspace_size(4000)
    assert L.fs_emb_gather(C.c_void_p(0x100), 10, 0, 0, C.c_void_p(0x200), 5, NULL, 1, C.c_void_p(0x300), err,
                           NULL) == 1                                                           # dim < 1
    assert L.fs_emb_gather(C.c_void_p(0x100), 10, 64, 7, C.c_void_p(0x200), 5, NULL, 1, C.c_void_p(0x300), err,
                           NULL) == 1                                                           # bad dtype
    # backward: dim 48 unsupported, Adagrad without state, phase without mask
    args = dict(table=C.c_void_p(0x100), R=10, ids=C.c_void_p(0x200), grads=C.c_void_p(0x300), T=4)
    assert L.fs_emb_backward_adagrad(args["table"], C.c_void_p(0x400), 10, 48, 0, 1, args["ids"], args["grads"], 4,
                                     NULL, NULL, 0, C.c_float(0.01), C.c_float(1e-8), err, ws, 1 << 30, NULL) == 1
    assert L.fs_emb_backward_adagrad(args["table"], NULL, 10, 64, 0, 1, args["ids"], args["grads"], 4,
                                     NULL, NULL, 0, C.c_float(0.01), C.c_float(1e-8), err, ws, 1 << 30, NULL) == 1
    assert L.fs_emb_backward_adagrad(args["table"], C.c_void_p(0x400), 10, 64, 0, 1, args["ids"], args["grads"], 4,
                                     NULL, NULL, 1, C.c_float(0.01), C.c_float(1e-8), err, ws, 1 << 30, NULL) == 1
    # a phase needs exactly one of is_co / co_rows; co_rows 4-byte aligned
    assert L.fs_emb_backward_adagrad(args["table"], C.c_void_p(0x400), 10, 64, 0, 1, args["ids"], args["grads"], 4,
                                     C.c_void_p(0x500), C.c_void_p(0x600), 1, C.c_float(0.01), C.c_float(1e-8), err,
                                     ws, 1 << 30, NULL) == 1
    assert L.fs_emb_backward_adagrad(args["table"], C.c_void_p(0x400), 10, 64, 0, 1, args["ids"], args["grads"], 4,
                                     NULL, C.c_void_p(0x602), 3, C.c_float(0.01), C.c_float(1e-8), err, ws, 1 << 30,
                                     NULL) == 8
    # row-sorted path: only the phases that keep every entry; the phase bit must fit (rows <= 2^30);
    # the workspace of the one-call update; 16-byte aligned table and output for the gather
    big = L.fs_emb_backward_adagrad_workspace_size(100, 1000, 64, 0)
    assert L.fs_emb_sort_rows(1000, 64, 0, C.c_void_p(0x200), 100, C.c_void_p(0x500), NULL, 1, err, ws, big,
                              NULL) == 1                                                    # COLLISION alone
    assert L.fs_emb_sort_rows((1 << 31) + 5, 64, 0, C.c_void_p(0x200), 100, C.c_void_p(0x500), NULL, 3, err, ws,
                              1 << 40, NULL) == 1                                           # phase bit does not fit
    assert L.fs_emb_sort_rows(1000, 64, 0, C.c_void_p(0x200), 100, NULL, NULL, 0, err, ws, 16, NULL) == 5
    assert L.fs_emb_sort_rows(1000, 48, 0, C.c_void_p(0x200), 100, NULL, NULL, 0, err, ws, big, NULL) == 1
    assert L.fs_emb_sort_rows(1000, 64, 0, C.c_void_p(0x204), 100, NULL, NULL, 0, err, ws, big, NULL) == 8
    assert L.fs_emb_gather_sorted(C.c_void_p(0x100), 1000, 64, 0, 100, 0, C.c_void_p(0x308), err, ws, big,
                                  NULL) == 8                                                # out 8-byte aligned
    assert L.fs_emb_gather_sorted(C.c_void_p(0x100), 1000, 64, 0, 100, 2, C.c_void_p(0x300), err, ws, big,
                                  NULL) == 1                                                # EXCLUSIVE alone
    assert L.fs_emb_update_sorted(C.c_void_p(0x100), NULL, 1000, 64, 0, 1, C.c_void_p(0x300), 100, 0,
                                  C.c_float(0.01), C.c_float(1e-8), err, ws, big, NULL) == 1  # Adagrad, no state
    assert L.fs_emb_update_sorted(C.c_void_p(0x100), NULL, 1000, 64, 0, 0, C.c_void_p(0x300), 0, 0,
                                  C.c_float(0.01), C.c_float(0.0), err, NULL, 0, NULL) == 0  # T = 0: nothing to do
    # fused permute + bucketize: rank offsets required, n <= 1024, 8-byte aligned outputs, workspace
    pb = [C.c_void_p(0x10), C.c_void_p(0x20), 10, C.c_void_p(0x30), C.c_void_p(0x40), 4, 100, C.c_void_p(0x50),
          C.c_void_p(0x60), 64, C.c_void_p(0x70), C.c_void_p(0x80), C.c_void_p(0x90), C.c_void_p(0xa0),
          C.c_void_p(0xb0), err, ws, 1 << 30, NULL]
    assert L.fs_permute_bucketize(*(pb[:4] + [NULL] + pb[5:])) == 1
    assert L.fs_permute_bucketize(*(pb[:5] + [1025] + pb[6:])) == 1
    assert L.fs_permute_bucketize(*(pb[:11] + [C.c_void_p(0x84)] + pb[12:])) == 8
    assert L.fs_permute_bucketize(*(pb[:17] + [16] + pb[18:])) == 5
    assert L.fs_permute_bucketize_workspace_size(10, 64, 4) > 0 and L.fs_permute_bucketize_workspace_size(10, 64, 0) == 0
    # per-shard update sort: n <= 1024, the phase bit beside shards of at most 2^19 rows, the flags for two phases
    big_s = L.fs_emb_sort_rows_sharded_workspace_size(100, 1000, 64, 0, 8)
    assert big_s > L.fs_emb_backward_adagrad_workspace_size(100, 1000, 64, 0)
    sh = [1000, 64, 0, C.c_void_p(0x200), C.c_void_p(0x300), 100, C.c_void_p(0x400), 8, C.c_void_p(0x500), NULL, 3,
          err, ws, big_s, NULL]
    assert L.fs_emb_sort_rows_sharded(*(sh[:7] + [1025] + sh[8:])) == 1
    assert L.fs_emb_sort_rows_sharded(*([(1 << 19) + 1] + sh[1:7] + [1] + sh[8:13] + [1 << 40] + sh[14:])) == 1
    assert L.fs_emb_sort_rows_sharded(*(sh[:8] + [NULL] + sh[9:])) == 1                 # no flags
    assert L.fs_emb_sort_rows_sharded(*(sh[:9] + [C.c_void_p(0x600)] + sh[10:])) == 1   # both flag forms
    assert L.fs_emb_sort_rows_sharded(*(sh[:8] + [NULL, C.c_void_p(0x602)] + sh[10:])) == 8
    assert L.fs_emb_sort_rows_sharded(*(sh[:4] + [C.c_void_p(0x302)] + sh[5:])) == 8
    assert L.fs_emb_sort_rows_sharded(*(sh[:13] + [big_s - 256] + sh[14:])) == 5
    # shard-major gather: positions 4-byte aligned, IDs 8-byte aligned, a known dtype
    gs = [C.c_void_p(0x100), 10, 64, 0, C.c_void_p(0x200), C.c_void_p(0x300), 5, C.c_void_p(0x400), err, NULL]
    assert L.fs_emb_gather_shard_major(*(gs[:4] + [C.c_void_p(0x204)] + gs[5:])) == 8
    assert L.fs_emb_gather_shard_major(*(gs[:5] + [C.c_void_p(0x302)] + gs[6:])) == 8
    assert L.fs_emb_gather_shard_major(*(gs[:3] + [9] + gs[4:])) == 1
    assert L.fs_emb_gather_shard_major(*(gs[:5] + [NULL] + gs[6:])) == 1
    assert L.fs_collision_split(C.c_void_p(0x10), 5, C.c_void_p(0x20), 5, (1 << 32) + 1, 4, NULL, NULL, NULL, 0,
                                C.c_void_p(0x30), C.c_void_p(0x40), C.c_void_p(0x50), C.c_void_p(0x60),
                                C.c_void_p(0x70), C.c_void_p(0x80), err, ws, 1 << 30, NULL) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(B.FsError):
        B.fs_balance_fbs(torch.zeros(4, dtype=torch.int32), 2)


def test_profiling_cases_print_usage_without_arguments():
    import profile_cases
    assert profile_cases.main([]) == 2
    assert profile_cases.main(["nosuchop", "1", "1"]) == 2


def _spin_limit_in_child(env_value):
    import subprocess
    import sys
    env = dict(os.environ)
    env.pop("FS_SPIN_LIMIT", None)
    if env_value is not None:
        env["FS_SPIN_LIMIT"] = env_value
    code = ("from jagged_embedding_gb300 import binding as B\n"
            "try:\n    print(B.spin_limit())\nexcept B.FsError as e:\n    print('error', e.code)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    return r.stdout.split()


def test_spin_limit_from_the_environment():
    """FS_SPIN_LIMIT sets the bounded waits' poll limit when the binding loads the library."""
    assert _spin_limit_in_child(None) == [str(1 << 22)]
    assert _spin_limit_in_child("12345") == ["12345"]
    assert _spin_limit_in_child("0") == ["error", "1"]
    assert _spin_limit_in_child("many") == ["error", "1"]
    L = B.lib()
    before = L.fs_get_spin_limit()
    try:
        L.fs_set_spin_limit(-5)                     # clamped to one poll
        assert L.fs_get_spin_limit() == 1
    finally:
        L.fs_set_spin_limit(before)
