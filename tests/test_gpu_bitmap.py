"""Row presence bitmaps (fs_row_bitmap) against the set of rows (GPU).

The bitmap of a batch is the set uniq(I) that the collision split of FreeScale
Algorithm 2 (line 10) intersects; bit r % 32 of word r / 32 is set exactly
when row r occurs.  The marking goes through a shared-memory window of the
bitmap when a block's IDs are grouped by row range (shard-major order) and
straight to global memory otherwise, so the cases cover both: shard-major
IDs, sorted IDs, IDs in random order over a large table, runs that jump
across the table, row counts that are not a multiple of 32, and tiny inputs.
"""
import numpy as np
import pytest
import torch

from jagged_embedding_gb300 import binding as B
from tests.helpers import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(bm, R):
    words = to_np(bm).view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")
    assert not bits[R:].any()                       # nothing beyond the last row
    return np.flatnonzero(bits[:R])


def _zipf_like(rng, R, T, s=1.05):
    # heavy-headed ranks, scrambled over the table (stand-in for the workloads' ID law)
    k = np.minimum(rng.zipf(1.0 + s, T) - 1, R - 1).astype(np.int64)
    return (k * 2654435761) % R


def _shard_major(ids, R, n):
    block = -(-R // n)
    return ids[np.argsort(ids // block, kind="stable")]


@pytest.mark.parametrize("R,n,T", [(100_000_000, 256, 3_000_000), (10_000_000, 64, 2_600_000),
                                   (50_000_000, 512, 1_000_003), (1_000_003, 7, 300_000)])
def test_bitmap_of_shard_major_ids(R, n, T):
    rng = np.random.default_rng(R % 1000 + T)
    ids = _shard_major(_zipf_like(rng, R, T), R, n)
    bm, err = B.fs_row_bitmap(torch.from_numpy(ids).to(DEV), R)
    B.check(err)
    assert np.array_equal(_rows(bm, R), np.unique(ids))


@pytest.mark.parametrize("order", ["sorted", "random", "runs"])
def test_bitmap_orders(order):
    R, T = 40_000_037, 2_000_000
    rng = np.random.default_rng(11)
    ids = rng.integers(0, R, T).astype(np.int64)
    if order == "sorted":
        ids.sort()
    elif order == "runs":   # sorted runs of 5000 IDs, each near a random place of the table
        base = rng.integers(0, R - 2_000_000, T // 5000)
        ids = (np.repeat(base, 5000) + rng.integers(0, 2_000_000, T)).astype(np.int64)
    bm, err = B.fs_row_bitmap(torch.from_numpy(ids).to(DEV), R)
    B.check(err)
    assert np.array_equal(_rows(bm, R), np.unique(ids))


@pytest.mark.parametrize("R,T", [(1, 5), (31, 100), (33, 1), (1000, 0), (5_000, 8191), (5_000, 8193), (70_001, 20_000)])
def test_bitmap_small(R, T):
    rng = np.random.default_rng(R * 3 + T)
    ids = rng.integers(0, R, T).astype(np.int64)
    bm = torch.full(((R + 31) // 32,), -1, dtype=torch.int32, device=DEV)   # stale bits are cleared
    _, err = B.fs_row_bitmap(torch.from_numpy(ids).to(DEV), R, bitmap=bm)
    B.check(err)
    assert np.array_equal(_rows(bm, R), np.unique(ids))


def test_bitmap_out_of_range_ids_set_the_error_and_mark_the_rest():
    R, T = 2_000_000, 100_000
    rng = np.random.default_rng(5)
    ids = np.sort(rng.integers(0, R, T)).astype(np.int64)
    bad = rng.choice(T, 7, replace=False)
    ids[bad[:4]] = R + rng.integers(0, 10, 4)
    ids[bad[4:]] = -1 - rng.integers(0, 10, 3)
    bm, err = B.fs_row_bitmap(torch.from_numpy(ids).to(DEV), R)
    with pytest.raises(B.FsError) as e:
        B.check(err)
    assert e.value.code == 2
    good = ids[(ids >= 0) & (ids < R)]
    assert np.array_equal(_rows(bm, R), np.unique(good))
