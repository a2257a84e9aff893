"""The row-gather probe (a timing aid beside the decode path) reads exactly the
rows it is given: the XOR of what each issue method read, against numpy on the
same pool, with skipped rows flagged. Sizes make every warp of the persistent
grid reuse its shared-memory slots several times."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def windows(pool, rows, pitch):
    win = 144 if pitch == 132 else 576
    r = rows.astype(np.int64)
    start = (r * pitch) & ~15
    ok = (r >= 0) & (start + win <= pool.size)
    return start[ok], win, (~ok).any()


@pytest.mark.parametrize("pitch,nrows,n", [(132, 5000, 400_003), (576, 2000, 120_001)])
@pytest.mark.parametrize("method", [0, 1, 2])
def test_probe_reads_the_listed_rows(cuda_lib, pitch, nrows, n, method):
    rng = np.random.default_rng(pitch + method)
    pool = rng.integers(0, 256, size=nrows * pitch, dtype=np.uint8)
    rows = rng.integers(0, nrows, size=n).astype(np.int32)
    rows[[5, 77, n - 1]] = [nrows - 1, 0, nrows - 1]  # the windows at both ends of the pool
    words = pool.view(np.uint32)
    start, win, _ = windows(pool, rows, pitch)
    if method == 0:
        idx = (start // 4)[:, None] + np.arange(win // 4)[None, :]
        want = np.bitwise_xor.reduce(words[idx].reshape(-1))
    else:
        want = np.bitwise_xor.reduce(words[start // 4])
    dpool = torch.from_numpy(pool).cuda()
    out = cuda_lib.pmqa_gather_probe(dpool, torch.from_numpy(rows).cuda(), pitch, method)
    got = out.cpu().numpy().view(np.uint32)
    assert got[0] == 0
    assert got[1] == want


@pytest.mark.parametrize("method", [0, 1, 2])
def test_rows_outside_the_pool_are_skipped_and_flagged(cuda_lib, method):
    pitch, nrows = 132, 3000
    rng = np.random.default_rng(9)
    pool = rng.integers(0, 256, size=nrows * pitch, dtype=np.uint8)
    rows = rng.integers(0, nrows, size=70_000).astype(np.int32)
    rows[[3, 40_000]] = [-1, nrows + 1]
    start, win, skipped = windows(pool, rows, pitch)
    assert skipped
    words = pool.view(np.uint32)
    if method == 0:
        want = np.bitwise_xor.reduce(words[(start // 4)[:, None] + np.arange(win // 4)].reshape(-1))
    else:
        want = np.bitwise_xor.reduce(words[start // 4])
    out = cuda_lib.pmqa_gather_probe(torch.from_numpy(pool).cuda(), torch.from_numpy(rows).cuda(),
                                     pitch, method)
    got = out.cpu().numpy().view(np.uint32)
    assert got[0] == cuda_lib.PMQA_DEV_BAD_CONTEXT
    assert got[1] == want
