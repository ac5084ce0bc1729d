"""Pins for the oracle's token-layout steps (no GPU): the voxel reordering of
the Chipmunk review (Alg. 1) and the rolling KV window of the DiT page.

  * voxel order: a bijection; for grids the voxels tile, equal to the closed
    form reshape (T/vt, vt, H/vh, vh, W/vw, vw) -> transpose (0,2,4,1,3,5);
    every run of vt*vh*vw positions is one voxel (its t, h and w spans stay
    inside one voxel cell); the inverse undoes it; and it agrees with the
    separate permutation the input generator uses to lay out the workloads;
  * KV window: a chunk-by-chunk brute force with a Python list of chunks
    (append while there is room; then keep the first, drop the oldest of the
    rest); the sink never changes once written; the valid length.
"""
import numpy as np
import pytest

import oracle
from video_dit_sparse_gb300 import inputs as I


@pytest.mark.parametrize("grid,voxel", [((4, 8, 8), (2, 4, 4)), ((18, 48, 80), (3, 8, 8)),
                                        ((16, 32, 32), (2, 8, 8)), ((6, 6, 10), (3, 2, 5))])
def test_voxel_order_closed_form(grid, voxel):
    T, H, W = grid
    vt, vh, vw = voxel
    order = oracle.voxel_order(grid, voxel)
    ref = np.arange(T * H * W).reshape(T // vt, vt, H // vh, vh, W // vw, vw)
    ref = ref.transpose(0, 2, 4, 1, 3, 5).reshape(-1)
    np.testing.assert_array_equal(order, ref)
    np.testing.assert_array_equal(np.sort(order), np.arange(T * H * W))
    C = vt * vh * vw
    t, h, w = order // (H * W), (order // W) % H, order % W
    for c in range(0, order.size, C):
        assert len(set(t[c:c + C] // vt)) == 1 and len(set(h[c:c + C] // vh)) == 1
        assert len(set(w[c:c + C] // vw)) == 1


@pytest.mark.parametrize("grid,voxel", [((5, 7, 9), (2, 3, 4)), ((18, 48, 80), (4, 6, 8)),
                                        ((1, 1, 1000), (1, 1, 128))])
def test_voxel_order_clipped_edges(grid, voxel):
    T, H, W = grid
    order = oracle.voxel_order(grid, voxel)
    np.testing.assert_array_equal(np.sort(order), np.arange(T * H * W))
    # positions of each voxel are contiguous and hold exactly its tokens
    vt, vh, vw = voxel
    t, h, w = order // (H * W), (order // W) % H, order % W
    cell = (t // vt) * 10**6 + (h // vh) * 10**3 + w // vw
    changes = np.flatnonzero(np.diff(cell)) + 1
    cells = cell[np.concatenate([[0], changes])]
    assert len(cells) == len(set(cells.tolist()))  # each voxel appears as one run
    assert np.all(np.diff(cells) > 0)              # voxels in raster order


def test_voxel_permute_inverse_and_generator_agree():
    grid, voxel = (6, 16, 24), (3, 8, 8)
    x = np.random.default_rng(0).standard_normal((2, 3, 6 * 16 * 24, 4))
    y = oracle.voxel_permute(x, grid, voxel)
    np.testing.assert_array_equal(oracle.voxel_permute(y, grid, voxel, inverse=True), x)
    # the input generator's own permutation (perm[new] = old raster index)
    np.testing.assert_array_equal(oracle.voxel_order(grid, voxel), I.voxel_perm(grid, voxel))


def brute_window(chunks_seq, S):
    kept = []
    for c in chunks_seq:
        if len(kept) < S:
            kept.append(c)
        else:
            kept = [kept[0]] + kept[2:] + [c]
    return kept


@pytest.mark.parametrize("S", [2, 3, 4])
def test_kv_window_append_bruteforce(S):
    L, d = 5, 3
    rng = np.random.default_rng(S)
    cache = np.zeros((2, S * L, d))
    seq = []
    for n in range(9):
        new = rng.standard_normal((2, L, d))
        seq.append(new)
        cache, valid = oracle.kv_window_append(cache, new, n)
        kept = brute_window(seq, S)
        assert valid == len(kept) * L
        np.testing.assert_array_equal(cache[:, :valid], np.concatenate(kept, axis=-2))
        np.testing.assert_array_equal(cache[:, :L], seq[0])  # the sink stays
    # LongLive's window: sink + 2 most recent + current
    if S == 4:
        np.testing.assert_array_equal(cache, np.concatenate([seq[0], seq[6], seq[7], seq[8]], axis=-2))
