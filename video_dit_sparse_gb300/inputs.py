"""Seeded synthetic inputs for column-sparse video-DiT attention.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds no attention or selection arithmetic: it only draws tensors,
rounds them to bf16 and puts tokens in voxel order.

Workload recipe (one spec for every preset):

* A latent grid (T, Hh, W); normalised positions t/T, h/Hh, w/W in [0, 1).
* For tensor X in {Q, K, V}, head h and channel c::

      X[h, n, c] = sum_{j<8} a * sin(2*pi*(kt*t_n + kh*h_n + kw*w_n) + phi) + eps

  with wave numbers kt in {0,1,2}, kh, kw in {0..3}, phase phi ~ U[0, 2*pi),
  amplitude a = 1 and eps ~ N(0, 0.5^2).  A smooth 3D field plus noise:
  neighbouring latent tokens are alike, which is what makes a voxel's mean
  query representative (Chipmunk review, voxel reordering; FG-Attn review,
  the pooling-mask premise).
* Tensor X draws from ``numpy.random.SeedSequence(3*seed + x)`` (x = 0, 1, 2
  for Q, K, V), spawned once per batch entry; each entry's sequence spawns
  H + 1 children.  Child 0 draws kt, kh, kw as integer arrays of shape
  (H, d, 8), then phi (H, d, 8); child 1 + h draws head h's noise, (N, d)
  float32.  The field is evaluated in float32 from float64 wave phases.
* Values are rounded to bf16 (round to nearest even) and then permuted to
  voxel order: voxels in raster order, tokens inside a voxel in raster order.

The tiny preset instead draws i.i.d. N(0, 1) values and uniform key lists.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "PRESETS", "preset", "make_inputs", "f32_to_bf16_bits",
    "bf16_bits_to_f32", "voxel_perm", "topk_count", "uniform_lists",
]

# Wave-number ranges of the field (kt in [0,3), kh/kw in [0,4)).
_KT, _KH, _KW = 3, 4, 4
_NWAVE = 8
_AMP = 1.0
_NOISE_STD = 0.5


@dataclass(frozen=True)
class Workload:
    """Shape and selection of one synthetic attention layer.

    ``grid_q``/``grid_k`` are latent grids (T, Hh, W) whose token counts are
    Nq/Nk; ``q_frame_offset`` places the query grid inside the key grid's
    time axis (rolling-window KV: queries are the newest chunk).
    ``voxel`` is None for raster order.  ``mode`` is "topk", "threshold",
    "mass" or "given" (index lists supplied by :func:`uniform_lists`), or a
    dense-step rule: "cached" (column max of the dense probabilities against
    ``threshold``, FG-Attn's cached mask) or "colsum" (top ``keep_pct`` % by
    column sums, Chipmunk's selection, followed by the sparse delta).
    """
    name: str
    B: int
    H: int
    d: int
    group: int
    grid_q: tuple
    grid_k: tuple
    q_frame_offset: int = 0
    voxel: tuple | None = None
    mode: str = "topk"
    keep_pct: float = 20.0
    threshold: float = 0.0
    mass: float = 0.99
    smooth: bool = True
    given_keep: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def Nq(self) -> int:
        return int(np.prod(self.grid_q))

    @property
    def Nk(self) -> int:
        return int(np.prod(self.grid_k))

    @property
    def G(self) -> int:
        return -(-self.Nq // self.group)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def topk(self) -> int:
        if self.mode == "given":
            return self.given_keep
        return topk_count(self.keep_pct, self.Nk)


def topk_count(pct: float, nk: int) -> int:
    """k = ceil(pct/100 * Nk), computed in integers when pct is integral."""
    if float(pct).is_integer():
        return min(nk, -(-int(pct) * nk // 100))
    return min(nk, int(math.ceil(pct * nk / 100.0)))


PRESETS = {
    # B=1, H=1, N=1024, d=64, i.i.d. N(0,1); 8 groups of 128 each keep 256
    # uniformly drawn keys.
    "tiny": Workload("tiny", 1, 1, 64, 128, (1, 1, 1024), (1, 1, 1024),
                     smooth=False, mode="given", given_keep=256),
    # H=24, d=128, 16x32x32 grid in (2,8,8) voxels, mean-query top 20 %.
    "wan16k_top20": Workload("wan16k_top20", 1, 24, 128, 128, (16, 32, 32),
                             (16, 32, 32), voxel=(2, 8, 8), keep_pct=20.0),
    # H=12, d=128, queries = newest chunk (8 frames x 22x40), keys = 4 chunks
    # (32 frames); raster order; 99 % retained mean-query softmax mass.
    "rollingkv_mass99": Workload("rollingkv_mass99", 1, 12, 128, 128,
                                 (8, 22, 40), (32, 22, 40), q_frame_offset=24,
                                 mode="mass", mass=0.99),
    # H=24, d=128, 18x48x80 grid in (3,8,8) voxels = chunks of C=192, top 10 %.
    "chunk192_top10": Workload("chunk192_top10", 1, 24, 128, 192, (18, 48, 80),
                               (18, 48, 80), voxel=(3, 8, 8), keep_pct=10.0),
}
for _p in (5, 10, 20, 40, 100):
    # H=24, d=128, 18x48x80 grid in (2,8,8) voxels, M=128, top p %.
    PRESETS[f"sweep69k_top{_p}"] = Workload(
        f"sweep69k_top{_p}", 1, 24, 128, 128, (18, 48, 80), (18, 48, 80),
        voxel=(2, 8, 8), keep_pct=float(_p))


# Dense-step workloads on the 18x48x80 grid: the cached mask of the FG-Attn
# review (keep a slice when one of its dense probabilities reaches 0.5/N,
# M = 128) and Chipmunk's column-sum top 10 % over C = 192 chunks with the
# sparse delta.
PRESETS["cached69k"] = Workload("cached69k", 1, 24, 128, 128, (18, 48, 80), (18, 48, 80),
                                voxel=(2, 8, 8), mode="cached", threshold=0.5 / 69120)
PRESETS["colsum192_top10"] = Workload("colsum192_top10", 1, 24, 128, 192, (18, 48, 80),
                                      (18, 48, 80), voxel=(3, 8, 8), mode="colsum",
                                      keep_pct=10.0)


# Token-layout workloads: voxel reordering of Q, K, V and back of O on the
# 69K grid ((3,8,8) voxels, C = 192), and rolling-window appends of one
# LongLive chunk (8 frames x 22x40 = 7040 tokens) to 4-slot K/V caches.
PRESETS["voxel69k"] = Workload("voxel69k", 1, 24, 128, 192, (18, 48, 80), (18, 48, 80),
                               voxel=(3, 8, 8), mode="layout")
PRESETS["kvwindow_rollingkv"] = Workload("kvwindow_rollingkv", 1, 12, 128, 128, (8, 22, 40),
                                         (32, 22, 40), mode="kvwindow")


# Mask-format conversions on the 69K grid, M = 128 (12960 index rows): a
# bit-packed keep-mask with 20 % of the bits set, and a block mask of
# 128-key blocks with 20 % kept.
PRESETS["bitmask69k_top20"] = Workload("bitmask69k_top20", 1, 24, 128, 128, (18, 48, 80),
                                       (18, 48, 80), mode="bitmask", keep_pct=20.0)
PRESETS["blockmask69k_top20"] = Workload("blockmask69k_top20", 1, 24, 128, 128, (18, 48, 80),
                                         (18, 48, 80), mode="blockmask", keep_pct=20.0)


def preset(name: str) -> Workload:
    return PRESETS[name]


# ---------------------------------------------------------------- bf16 bits
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ voxels
def voxel_perm(grid: tuple, voxel: tuple | None) -> np.ndarray:
    """perm[new] = old raster index; voxels raster-ordered, tokens likewise."""
    T, Hh, W = grid
    n = T * Hh * W
    if voxel is None:
        return np.arange(n, dtype=np.int64)
    vt, vh, vw = voxel
    if T % vt or Hh % vh or W % vw:
        raise ValueError(f"voxel {voxel} does not tile grid {grid}")
    idx = np.arange(n, dtype=np.int64).reshape(T // vt, vt, Hh // vh, vh, W // vw, vw)
    return idx.transpose(0, 2, 4, 1, 3, 5).reshape(n)


def _positions(grid: tuple, frame_offset: int, t_total: int) -> np.ndarray:
    T, Hh, W = grid
    t = (np.arange(T, dtype=np.float64) + frame_offset) / t_total
    h = np.arange(Hh, dtype=np.float64) / Hh
    w = np.arange(W, dtype=np.float64) / W
    tt, hh, ww = np.meshgrid(t, h, w, indexing="ij")
    return np.stack([tt.ravel(), hh.ravel(), ww.ravel()], axis=1)


def _field_tensor(ss: np.random.SeedSequence, H: int, d: int, pos: np.ndarray,
                  perm: np.ndarray) -> np.ndarray:
    """One of Q/K/V for one batch entry: bf16 bits [H, N, d] in token order."""
    children = ss.spawn(H + 1)
    rng = np.random.default_rng(children[0])
    kt = rng.integers(0, _KT, size=(H, d, _NWAVE))
    kh = rng.integers(0, _KH, size=(H, d, _NWAVE))
    kw = rng.integers(0, _KW, size=(H, d, _NWAVE))
    phi = rng.uniform(0.0, 2.0 * math.pi, size=(H, d, _NWAVE))
    # The 48 distinct wave vectors; sin(theta + phi) = sin(theta)cos(phi) + cos(theta)sin(phi).
    waves = np.array([(a, b, c) for a in range(_KT) for b in range(_KH) for c in range(_KW)],
                     dtype=np.float64)
    theta = 2.0 * math.pi * (pos @ waves.T)             # [N, 48]
    basis = np.concatenate([np.sin(theta), np.cos(theta)], axis=1).astype(np.float32)
    nw = waves.shape[0]
    widx = (kt * _KH + kh) * _KW + kw                    # [H, d, 8]
    N = pos.shape[0]
    out = np.empty((H, N, d), dtype=np.uint16)
    cols = np.broadcast_to(np.arange(d)[:, None], (d, _NWAVE))

    def head(h: int) -> None:
        coef = np.zeros((2 * nw, d), dtype=np.float64)
        np.add.at(coef, (widx[h], cols), _AMP * np.cos(phi[h]))
        np.add.at(coef, (widx[h] + nw, cols), _AMP * np.sin(phi[h]))
        f = basis @ coef.astype(np.float32)
        noise = np.random.default_rng(children[1 + h]).standard_normal((N, d), dtype=np.float32)
        f += noise * np.float32(_NOISE_STD)
        out[h] = f32_to_bf16_bits(f)[perm]

    with ThreadPoolExecutor(max_workers=min(H, os.cpu_count() or 1)) as ex:
        list(ex.map(head, range(H)))
    return out


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Return {"q","k","v"}: uint16 bf16 bit arrays [B, H, N, d] (+ "lists")."""
    out = {}
    if not w.smooth:
        for x, name in enumerate("qkv"):
            rng = np.random.default_rng(3 * seed + x)
            n = w.Nq if name == "q" else w.Nk
            a = rng.standard_normal((w.B, w.H, n, w.d), dtype=np.float32)
            out[name] = f32_to_bf16_bits(a).reshape(w.B, w.H, n, w.d)
    else:
        t_total = w.grid_k[0]
        pos_q = _positions(w.grid_q, w.q_frame_offset, t_total)
        pos_k = _positions(w.grid_k, 0, t_total)
        perm_q = voxel_perm(w.grid_q, w.voxel)
        perm_k = voxel_perm(w.grid_k, w.voxel)
        for x, name in enumerate("qkv"):
            ss = np.random.SeedSequence(3 * seed + x)
            pos, perm = (pos_q, perm_q) if name == "q" else (pos_k, perm_k)
            bits = np.empty((w.B, w.H, pos.shape[0], w.d), dtype=np.uint16)
            for b, ssb in enumerate(ss.spawn(w.B)):
                bits[b] = _field_tensor(ssb, w.H, w.d, pos, perm)
            out[name] = bits
    if w.mode == "given":
        out["row_ptr"], out["col_idx"] = uniform_lists(w, seed)
    return out


def uniform_lists(w: Workload, seed: int = 0):
    """Per (b,h,g): ``given_keep`` distinct keys drawn uniformly, ascending."""
    rng = np.random.default_rng(1000 + seed)
    rows = w.B * w.H * w.G
    keep = min(w.given_keep, w.Nk)
    col = np.empty((rows, keep), dtype=np.int32)
    for r in range(rows):
        col[r] = np.sort(rng.choice(w.Nk, size=keep, replace=False))
    row_ptr = np.arange(rows + 1, dtype=np.int64) * keep
    return row_ptr, col.reshape(-1)


def custom(name: str, B: int, H: int, d: int, group: int, grid_q: tuple,
           grid_k: tuple | None = None, **kw) -> Workload:
    """A field workload of arbitrary (small) shape for parity tests."""
    return Workload(name, B, H, d, group, grid_q, grid_k or grid_q, **kw)
