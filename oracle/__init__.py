"""fp64 CPU oracle for mean-query column-sparse attention (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package's smoke
check and by the benchmark's CPU-baseline leg, never by the product path.
The arithmetic lives in ``oracle.c``; this file only marshals numpy arrays.
It shares no code with the CUDA path.

Modes follow the C side: 0 = TOPK, 1 = THRESHOLD, 2 = MASS, 3 = LEVEL (the
statistic itself reaches tau; used for dense-step lists).  Column
statistics: 0 = MAX, 1 = SUM over a group's queries of the dense-step
attention probabilities.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

TOPK, THRESHOLD, MASS, LEVEL = 0, 1, 2, 3
MODES = {"topk": TOPK, "threshold": THRESHOLD, "mass": MASS, "level": LEVEL}
STAT_MAX, STAT_SUM = 0, 1
STATS = {"max": STAT_MAX, "sum": STAT_SUM}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (IEEE fp64, no FMA
    contraction, so x86 and Arm hosts produce the same bits)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC",
                        "-shared", "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_mean_query.argtypes = [p, i64, i64, i64, i64, i64, p, i64, p]
    lib.oracle_group_scores.argtypes = [p, p, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_double, p, i64, p, ctypes.c_int]
    lib.oracle_select.argtypes = [p, i64, i64, ctypes.c_int, i64, ctypes.c_double,
                                  ctypes.c_double, p, p, p, ctypes.c_int]
    lib.oracle_forward.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64,
                                   ctypes.c_double, p, p, p, i64, p, p, ctypes.c_int]
    lib.oracle_column_stats.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_double, ctypes.c_int, p, i64, p, ctypes.c_int]
    lib.oracle_forward_delta.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_double,
                                         p, p, p, p, ctypes.c_double, p, i64, p, ctypes.c_int]
    for f in (lib.oracle_mean_query, lib.oracle_group_scores, lib.oracle_select,
              lib.oracle_forward, lib.oracle_column_stats, lib.oracle_forward_delta):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def _units(units, total):
    if units is None:
        units = np.arange(total, dtype=np.int64)
    return np.ascontiguousarray(units, dtype=np.int64)


def mean_query(q, M: int, units=None) -> np.ndarray:
    """q: uint16 [B,H,Nq,d] -> float64 [n_units, d]."""
    q = _bits(q)
    B, H, Nq, d = q.shape
    G = -(-Nq // M)
    units = _units(units, B * H * G)
    out = np.empty((units.size, d), dtype=np.float64)
    rc = _load().oracle_mean_query(_ptr(q), B, H, Nq, d, M, _ptr(units), units.size, _ptr(out))
    if rc:
        raise ValueError("oracle_mean_query rejected its arguments")
    return out


def group_scores(q, k, M: int, scale: float, units=None, threads: int | None = None):
    """Mean-query scores: float64 [n_units, Nk]."""
    q, k = _bits(q), _bits(k)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    units = _units(units, B * H * G)
    out = np.empty((units.size, Nk), dtype=np.float64)
    rc = _load().oracle_group_scores(_ptr(q), _ptr(k), B, H, Nq, Nk, d, M, float(scale),
                                     _ptr(units), units.size, _ptr(out),
                                     threads or default_threads())
    if rc:
        raise ValueError("oracle_group_scores rejected its arguments")
    return out


def select(scores, mode, topk: int = 0, tau: float = 0.0, rho: float = 0.99,
           threads: int | None = None):
    """Returns (lists, cut): ascending int32 index arrays per row, cut scores."""
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    n_rows, Nk = scores.shape
    mode = MODES.get(mode, mode)
    counts = np.empty(n_rows, dtype=np.int64)
    idx = np.empty((n_rows, max(Nk, 1)), dtype=np.int32)
    cut = np.empty(n_rows, dtype=np.float64)
    rc = _load().oracle_select(_ptr(scores), n_rows, Nk, int(mode), int(topk), float(tau),
                               float(rho), _ptr(counts), _ptr(idx), _ptr(cut),
                               threads or default_threads())
    if rc:
        raise ValueError("oracle_select rejected its arguments")
    return [idx[r, :counts[r]].copy() for r in range(n_rows)], cut


def build_index(q, k, M: int, scale: float, mode, topk: int = 0, tau: float = 0.0,
                rho: float = 0.99, units=None, threads: int | None = None):
    """Scores + selection for the listed units: (lists, cut, scores)."""
    sc = group_scores(q, k, M, scale, units, threads)
    lists, cut = select(sc, mode, topk, tau, rho, threads)
    return lists, cut, sc


def to_csr(lists):
    """Concatenate per-row lists into (row_ptr int64, col_idx int32)."""
    counts = np.array([len(x) for x in lists], dtype=np.int64)
    row_ptr = np.zeros(len(lists) + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    col = np.concatenate(lists).astype(np.int32) if lists else np.zeros(0, np.int32)
    return row_ptr, col


def forward(q, k, v, M: int, scale: float, row_ptr, col_idx, units=None,
            threads: int | None = None):
    """Restricted attention of the listed units.

    row_ptr has B*H*G+1 entries indexed by unit id.  Returns o float64
    [n_units, M, d] (rows past Nq are zero) and lse float64 [n_units, M].
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    units = _units(units, B * H * G)
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    if row_ptr.size != B * H * G + 1:
        raise ValueError("row_ptr must have B*H*G+1 entries")
    if col_idx.size == 0:
        col_idx = np.zeros(1, dtype=np.int32)
    o = np.empty((units.size, M, d), dtype=np.float64)
    lse = np.empty((units.size, M), dtype=np.float64)
    rc = _load().oracle_forward(_ptr(q), _ptr(k), _ptr(v), B, H, Nq, Nk, d, M, float(scale),
                                _ptr(row_ptr), _ptr(col_idx), _ptr(units), units.size,
                                _ptr(o), _ptr(lse), threads or default_threads())
    if rc:
        raise ValueError("oracle_forward rejected its arguments")
    return o, lse


def dense_lse(q, k, scale: float, M: int | None = None, units=None, threads: int | None = None):
    """Row log-sum-exp over all Nk keys (the dense step), computed by the
    restricted-attention oracle with every key kept.  Without `units`:
    float64 [B, H, Nq]; with `units` (query groups of M rows): [n_units, M]."""
    q, k = _bits(q), _bits(k)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if M is None:
        M = Nq  # one group per head
    G = -(-Nq // M)
    full = units is None
    units = _units(units, B * H * G)
    # CSR in which each listed unit keeps every key (the others stay empty)
    counts = np.zeros(B * H * G, dtype=np.int64)
    counts[units] = Nk
    row_ptr = np.zeros(B * H * G + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    col = np.tile(np.arange(Nk, dtype=np.int32), units.size)
    _, lse = forward(q, k, k, M, scale, row_ptr, col, units, threads)
    if full:
        return lse.reshape(B, H, G * M)[:, :, :Nq]
    return lse


def column_stats(q, k, lse, M: int, scale: float, stat, units=None, threads: int | None = None):
    """ln of the per-key column statistic of each listed unit: float64
    [n_units, Nk].  stat "max": max over the group's queries of
    exp(s q.k - lse); "sum": their sum.  lse: [B, H, Nq] (any float type)."""
    q, k = _bits(q), _bits(k)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    units = _units(units, B * H * G)
    lse = np.ascontiguousarray(lse, dtype=np.float64).reshape(B, H, Nq)
    out = np.empty((units.size, Nk), dtype=np.float64)
    rc = _load().oracle_column_stats(_ptr(q), _ptr(k), _ptr(lse), B, H, Nq, Nk, d, M,
                                     float(scale), int(STATS.get(stat, stat)), _ptr(units),
                                     units.size, _ptr(out), threads or default_threads())
    if rc:
        raise ValueError("oracle_column_stats rejected its arguments")
    return out


def dense_index(q, k, lse, M: int, scale: float, stat, mode, topk: int = 0, tau: float = 0.0,
                rho: float = 0.99, units=None, threads: int | None = None):
    """Dense-step lists: column statistics + selection.  mode "threshold"
    means LEVEL here (the statistic itself reaches tau).  Returns
    (lists, cut, ln-statistics)."""
    st = column_stats(q, k, lse, M, scale, stat, units, threads)
    m = MODES.get(mode, mode)
    if m == THRESHOLD:
        m = LEVEL
    lists, cut = select(st, m, topk, tau, rho, threads)
    return lists, cut, st


def forward_delta(q, k, v, M: int, scale: float, row_ptr, col_idx, lse, base=None,
                  sign: float = 1.0, units=None, threads: int | None = None):
    """Sparse-delta attention: o_i = base_i + sign * sum over kept j of
    exp(s q_i.k_j - lse_i) v_j.  Returns float64 [n_units, M, d]."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    units = _units(units, B * H * G)
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    if row_ptr.size != B * H * G + 1:
        raise ValueError("row_ptr must have B*H*G+1 entries")
    if col_idx.size == 0:
        col_idx = np.zeros(1, dtype=np.int32)
    lse = np.ascontiguousarray(lse, dtype=np.float64).reshape(B, H, Nq)
    if base is not None:
        base = np.ascontiguousarray(base, dtype=np.float64).reshape(B, H, Nq, d)
    o = np.empty((units.size, M, d), dtype=np.float64)
    rc = _load().oracle_forward_delta(_ptr(q), _ptr(k), _ptr(v), B, H, Nq, Nk, d, M, float(scale),
                                      _ptr(row_ptr), _ptr(col_idx), _ptr(lse),
                                      None if base is None else _ptr(base), float(sign),
                                      _ptr(units), units.size, _ptr(o), threads or default_threads())
    if rc:
        raise ValueError("oracle_forward_delta rejected its arguments")
    return o


# ------------------------------------------------------------ token layout
# Chipmunk review, "What carries the argument" / Alg. 1 (voxel reordering):
# tokens of a (T, Hh, W) latent grid are reordered so that contiguous chunks
# are spatio-temporal voxels.  Reading: voxels of (vt, vh, vw) tokens in
# raster order over the voxel grid, tokens raster-ordered inside each voxel;
# at the grid's far edges voxels are clipped to what remains.

def voxel_order(grid, voxel):
    """order[n] = raster index (t*Hh*W + h*W + w) of the token at position n
    of the voxel-ordered sequence; built by enumerating voxels one by one."""
    T, Hh, W = grid
    vt, vh, vw = voxel
    order = []
    for t0 in range(0, T, vt):
        for h0 in range(0, Hh, vh):
            for w0 in range(0, W, vw):
                for t in range(t0, min(t0 + vt, T)):
                    for h in range(h0, min(h0 + vh, Hh)):
                        for w in range(w0, min(w0 + vw, W)):
                            order.append((t * Hh + h) * W + w)
    return np.asarray(order, dtype=np.int64)


def voxel_permute(x, grid, voxel, inverse: bool = False):
    """x [..., N, d] (any dtype): raster -> voxel order (y[n] = x[order[n]]),
    or back (y[order[n]] = x[n]) when inverse."""
    order = voxel_order(grid, voxel)
    if inverse:
        y = np.empty_like(x)
        y[..., order, :] = x
        return y
    return x[..., order, :]


# DiT page, "The Architecture" (KV window of 4 chunks: the first chunk is a
# permanent attention sink, then the 2 most recent chunks and the current one)
# and its per-chunk loop ("roll the cache if the 4-chunk window is full (sink
# stays)").  Reading: the cache holds S chunk slots in chronological order.

def kv_window_append(cache, new, chunks_before: int):
    """cache [..., S*L, d], new [..., L, d]; returns (cache after appending the
    chunk, number of valid key tokens).  While slots are free the chunk fills
    the next one; once full, slot 0 (the sink) stays, every other chunk moves
    one slot towards the sink (the oldest non-sink chunk leaves) and the new
    chunk takes the last slot."""
    L = new.shape[-2]
    S = cache.shape[-2] // L
    chunks = [cache[..., s * L:(s + 1) * L, :].copy() for s in range(S)]
    if chunks_before < S:
        chunks[chunks_before] = new.copy()
    else:
        chunks = [chunks[0]] + chunks[2:] + [new.copy()]
    return np.concatenate(chunks, axis=-2), min(chunks_before + 1, S) * L


# ------------------------------------------------------------ index formats
# Chipmunk review, "Bitpacked Sparsity Masks": a boolean keep-mask stored one
# bit per entry (8x smaller than one byte per entry).  Reading: per index row
# (query group), ceil(Nk/32) little-endian uint32 words, key j is bit j % 32 of
# word j // 32; bits past Nk are ignored.
# FG-Attn review, "The pith" and Fig. 6: block-sparse masks (M x M tiles) can
# be fed to the slice kernel.  Reading: a byte per (query group, key block of
# block_k keys); a kept block keeps all of its keys (the last block ragged).

def lists_from_bitmask(words, Nk: int):
    """words uint32 [rows, ceil(Nk/32)] -> ascending key lists per row."""
    words = np.ascontiguousarray(words, dtype=np.uint32)
    out = []
    for r in range(words.shape[0]):
        keep = []
        for j in range(Nk):
            if (int(words[r, j // 32]) >> (j % 32)) & 1:
                keep.append(j)
        out.append(np.asarray(keep, dtype=np.int32))
    return out


def lists_from_block_mask(blocks, Nk: int, block_k: int):
    """blocks uint8 [rows, ceil(Nk/block_k)] (non-zero = kept) -> key lists."""
    out = []
    for r in range(blocks.shape[0]):
        keep = []
        for b in range(blocks.shape[1]):
            if blocks[r, b]:
                keep.extend(range(b * block_k, min((b + 1) * block_k, Nk)))
        out.append(np.asarray(keep, dtype=np.int32))
    return out
