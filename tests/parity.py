"""Parity helpers shared by the GPU tests: move seeded inputs to the device,
compare the CUDA path with the fp64 oracle under the stated tolerances.

Tolerances (the method's acceptance bar):
  * attention output: max |o - o_ref| <= 2e-2 and mean |o - o_ref| <= 2e-3;
  * log-sum-exp: |lse - lse_ref| <= 1e-3 * max(|lse_ref|, 1) per row;
  * index lists: identical except keys whose fp64 score lies within
    1e-3 * max(|cut|, 1) of the oracle's selection cut.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from video_dit_sparse_gb300 import inputs as I

O_MAX, O_MEAN, LSE_REL, CUT_REL = 2e-2, 2e-3, 1e-3, 1e-3


def to_dev(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def cached_inputs(name: str, seed: int = 0):
    """Inputs of a named preset, generated once per test session (the
    69k-token sweep points share one tensor set)."""
    w = I.preset(name)
    key = (w.B, w.H, w.d, w.grid_q, w.grid_k, w.q_frame_offset, w.voxel, w.smooth)
    return _generate(key, w, seed)


_gen_cache: dict = {}


def _generate(key, w, seed):
    k = (key, seed)
    if k not in _gen_cache:
        if len(_gen_cache) >= 2:
            _gen_cache.pop(next(iter(_gen_cache)))
        _gen_cache[k] = I.make_inputs(w, seed)
    return _gen_cache[k]


def unit_coords(u: int, H: int, G: int):
    return u // (H * G), (u // G) % H, u % G


def compare_units(q, k, v, M, row_ptr, col_idx, units, o_dev, lse_dev, scale=None):
    """Runs the oracle on `units` and asserts the tolerances; returns stats."""
    B, H, Nq, d = q.shape
    G = -(-Nq // M)
    scale = scale if scale is not None else 1.0 / math.sqrt(d)
    units = np.asarray(units, dtype=np.int64)
    o_ref, lse_ref = oracle.forward(q, k, v, M, scale, row_ptr, col_idx, units)
    o_all = o_dev.view(B * H, Nq, d)
    lse_all = lse_dev.view(B * H, Nq) if lse_dev is not None else None
    abs_err = []
    worst_lse = 0.0
    for i, u in enumerate(units):
        b, h, g = unit_coords(int(u), H, G)
        r0, r1 = g * M, min((g + 1) * M, Nq)
        og = o_all[b * H + h, r0:r1].double().cpu().numpy()
        ref = o_ref[i, : r1 - r0]
        abs_err.append(np.abs(og - ref).ravel())
        if lse_all is not None:
            lg = lse_all[b * H + h, r0:r1].double().cpu().numpy()
            lr = lse_ref[i, : r1 - r0]
            empty = np.isneginf(lr)
            assert np.array_equal(np.isneginf(lg), empty), f"unit {u}: empty-row LSE mismatch"
            if (~empty).any():
                rel = np.abs(lg[~empty] - lr[~empty]) / np.maximum(np.abs(lr[~empty]), 1.0)
                worst_lse = max(worst_lse, float(rel.max()))
    e = np.concatenate(abs_err) if abs_err else np.zeros(1)
    stats = {"o_max": float(e.max()), "o_mean": float(e.mean()), "lse_rel": worst_lse}
    assert stats["o_max"] <= O_MAX, stats
    assert stats["o_mean"] <= O_MEAN, stats
    assert stats["lse_rel"] <= LSE_REL, stats
    return stats


def compare_lists(row_ptr_dev, col_dev, rows, ref_lists, ref_cut, ref_scores, Nk):
    """GPU lists of `rows` vs the oracle's: equal except near-cut keys."""
    rp = row_ptr_dev.cpu().numpy()
    n_near = 0
    for i, r in enumerate(rows):
        got = col_dev[int(rp[r]):int(rp[r + 1])].cpu().numpy()
        assert got.size > 0, f"row {r}: empty list"
        assert np.all(np.diff(got) > 0), f"row {r}: not strictly ascending"
        assert got.min() >= 0 and got.max() < Nk, f"row {r}: index out of range"
        ref = ref_lists[i]
        diff = np.setxor1d(got, ref)
        if diff.size:
            cut = ref_cut[i]
            tol = CUT_REL * max(abs(cut), 1.0)
            far = diff[np.abs(ref_scores[i][diff] - cut) > tol]
            assert far.size == 0, (f"row {r}: keys {far[:8]} differ, scores "
                                   f"{ref_scores[i][far[:8]]}, cut {cut}")
            n_near += diff.size
    return n_near
