"""The FBS entry point that allocates nothing (GPU).

Callers that cannot allocate device memory at the time they partition a batch
(a frozen or tearing-down memory pool, a plugin running inside a process whose
allocator it does not own, a fixed memory plan) use fs_balance_fbs_noalloc: it
keeps the sort's scratch in a fixed array inside the library.  These checks
call it through the C ABI, twice in a row with different batches, and compare
with the CPU oracle's FBS partition and with fs_balance_fbs, which takes a
caller workspace.  This file is collected last on purpose and must pass both
alone and after every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from jagged_embedding_gb300 import binding as B
from tests.helpers import Guarded, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _lens(seed, S):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.clip(np.round(rng.lognormal(6.8, 1.5, S)), 1, 16384).astype(np.int32)).to(DEV)


def _noalloc(L, n):
    S = L.numel()
    # outputs between guard bands: the call writes nothing before or after them
    perm = Guarded(S, torch.int32, DEV, torch.full((S,), -1, dtype=torch.int32))
    ro = Guarded(n + 1, torch.int64, DEV, torch.full((n + 1,), -1, dtype=torch.int64))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.fs_balance_fbs_noalloc(L, n, perm.t, ro.t, err)
    B.check(err, "fs_balance_fbs_noalloc")
    perm.check("perm")
    ro.check("rank_offsets")
    return perm.t, ro.t


@pytest.mark.parametrize("n,S", [(256, 131072), (64, 16384), (3, 7)])
def test_noalloc_matches_workspace_entry_point_twice(n, S):
    for call in range(2):                          # two calls in a row share the fixed scratch array
        L = _lens(1000 * call + S, S)
        perm, ro = _noalloc(L, n)
        p_ora, ro_ora = oracle.balance_fbs(to_np(L), n)
        assert np.array_equal(to_np(perm), p_ora), call
        assert np.array_equal(to_np(ro), ro_ora), call
        p_ref, ro_ref, err = B.fs_balance_fbs(L, n)
        B.check(err, "fs_balance_fbs")
        assert torch.equal(perm, p_ref), call
        assert torch.equal(ro, ro_ref), call


def test_noalloc_at_the_size_limit_and_beyond():
    S = 1 << 18
    L = _lens(7, S)
    perm, ro = _noalloc(L, 512)
    p_ora, ro_ora = oracle.balance_fbs(to_np(L), 512)
    assert np.array_equal(to_np(perm), p_ora) and np.array_equal(to_np(ro), ro_ora)
    p_ref, ro_ref, err = B.fs_balance_fbs(L, 512)
    B.check(err)
    assert torch.equal(perm, p_ref) and torch.equal(ro, ro_ref)
    too_big = torch.ones(S + 1, dtype=torch.int32, device=DEV)
    with pytest.raises(B.FsError) as e:
        B.fs_balance_fbs_noalloc(too_big, 4, torch.empty(S + 1, dtype=torch.int32, device=DEV),
                                 torch.empty(5, dtype=torch.int64, device=DEV),
                                 torch.zeros(1, dtype=torch.int32, device=DEV))
    assert e.value.code == 1


def test_noalloc_call_leaves_free_device_memory_unchanged():
    L = _lens(3, 50_000)
    perm = torch.empty(50_000, dtype=torch.int32, device=DEV)
    ro = torch.empty(65, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.fs_balance_fbs_noalloc(L, 64, perm, ro, err)   # first call on the device: module and array are loaded
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        B.fs_balance_fbs_noalloc(L, 64, perm, ro, err)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    B.check(err)
    assert free1 == free0
