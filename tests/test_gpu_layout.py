"""GPU checks of the token-layout kernels (through the C ABI), bit for bit
against the oracle: voxel reordering and its inverse on tiled and clipped
grids (d = 64 and 128), the 69K-token grid of the benchmarks, and the rolling
KV window over a sequence of chunks (fill, then roll with the sink kept)."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu


def bits(shape, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint64).astype(np.uint16)


@pytest.mark.parametrize("grid,voxel,d", [((4, 8, 8), (2, 4, 4), 128), ((5, 7, 9), (2, 3, 4), 64),
                                          ((18, 48, 80), (3, 8, 8), 128), ((18, 48, 80), (4, 6, 8), 64),
                                          ((1, 1, 1000), (1, 1, 128), 128), ((3, 1, 1), (2, 2, 2), 64)])
def test_voxel_permute_matches_oracle(grid, voxel, d):
    from video_dit_sparse_gb300 import binding as sa
    N = grid[0] * grid[1] * grid[2]
    x = bits((2, 3, N, d), seed=N + d)
    xd = P.to_dev(x)
    y = sa.sparse_attn_voxel_permute(xd, grid, voxel)
    z = sa.sparse_attn_voxel_permute(y, grid, voxel, inverse=True)
    torch.cuda.synchronize()
    want = oracle.voxel_permute(x, grid, voxel)
    assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), want)
    assert torch.equal(z.view(torch.int16), xd.view(torch.int16))


def test_voxel_permute_rejects_overlap_and_bad_args():
    from video_dit_sparse_gb300 import binding as sa
    x = P.to_dev(bits((1, 1, 256, 128), seed=1))
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_voxel_permute(x, (2, 8, 16), (2, 4, 4), out=x)
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_voxel_permute(x, (2, 8, 16), (0, 4, 4))


@pytest.mark.parametrize("S,L,d", [(4, 880, 128), (2, 64, 64), (3, 7, 128)])
def test_kv_window_append_matches_oracle(S, L, d):
    from video_dit_sparse_gb300 import binding as sa
    B, H = 1, 3
    ck = torch.zeros(B, H, S * L, d, dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    ref_k = np.zeros((B, H, S * L, d), dtype=np.uint16)
    ref_v = ref_k.copy()
    for n in range(S + 4):
        nk, nv = bits((B, H, L, d), seed=2 * n), bits((B, H, L, d), seed=2 * n + 1)
        valid = sa.sparse_attn_kv_window_append(ck, cv, P.to_dev(nk), P.to_dev(nv), n)
        ref_k, vref = oracle.kv_window_append(ref_k, nk, n)
        ref_v, _ = oracle.kv_window_append(ref_v, nv, n)
        torch.cuda.synchronize()
        assert valid == vref
        assert np.array_equal(ck.view(torch.int16).cpu().numpy().view(np.uint16)[:, :, :valid], ref_k[:, :, :valid])
        assert np.array_equal(cv.view(torch.int16).cpu().numpy().view(np.uint16)[:, :, :valid], ref_v[:, :, :valid])
