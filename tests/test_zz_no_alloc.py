"""fs_prune_cells_static: the pool construction on the library's fixed scratch
array, compared with fs_prune_cells (caller workspace) on the same norms.

Pools are integer work, so the two entry points must agree exactly.  Two calls
in a row (different shapes) check that the shared array needs no clearing
between calls.  The file is named so that it is collected last; it also
passes on its own in a fresh process (the first call does the one-time
address lookup)."""
import numpy as np
import pytest
import torch

from long_context_lm_gb300 import fs

pytestmark = pytest.mark.gpu
PAGE = dict(w=512, s=32, K=4, P=64, W=8, Bq=128, rope_base=10000.0, rms_eps=1e-6, mode=0)


def _amax(B, H, N, seed, quant=0):
    rng = np.random.default_rng(seed)
    a = rng.lognormal(0, 0.5, size=(B, H, N // 32)).astype(np.float32)
    if quant:  # many exact ties between norms
        a = (np.round(a * quant) / quant).astype(np.float32)
    return torch.from_numpy(a).cuda()


@pytest.mark.parametrize("B,H,N,quant", [(1, 3, 8192 + 128, 0), (2, 16, 65536, 4)])
def test_static_scratch_matches_workspace_entry_point_twice(B, H, N, quant):
    params = dict(PAGE)
    amax = _amax(B, H, N, seed=N + H, quant=quant)
    ref_pool, ref_count = fs.fs_prune_cells(amax, N, params)
    nblk = N // 128
    pool = torch.empty((B, H, nblk, 72), device="cuda", dtype=torch.int32)
    count = torch.empty((B, H, nblk), device="cuda", dtype=torch.int32)
    for call in range(2):
        pool.fill_(-7)
        count.fill_(-7)
        fs.fs_prune_cells_static(amax, N, params, pool=pool, count=count)
        torch.cuda.synchronize()
        assert torch.equal(count, ref_count), call
        assert torch.equal(pool, ref_pool), call


def test_static_scratch_after_a_larger_shape():
    # a large call leaves lists in the array; a smaller one must not read them
    big = _amax(1, 16, 262144, seed=11)
    small = _amax(1, 2, 4096, seed=12)
    fs.fs_prune_cells_static(big, 262144, PAGE)
    pool, count = fs.fs_prune_cells_static(small, 4096, PAGE)
    ref_pool, ref_count = fs.fs_prune_cells(small, 4096, PAGE)
    torch.cuda.synchronize()
    assert torch.equal(pool, ref_pool) and torch.equal(count, ref_count)


def test_static_scratch_rejects_shapes_past_its_limit():
    assert fs.load().fs_prune_static_scratch_bytes() == 4 << 20
    # batch*H*ceil(N/2048) = 4097 lists per bank: one more than the array holds
    amax = torch.ones((1, 4097, 1), device="cuda", dtype=torch.float32)
    with pytest.raises(fs.FSError) as e:
        fs.fs_prune_cells_static(amax, 128, PAGE)
    assert e.value.status == fs.FS_ERR_SCRATCH_LIMIT
