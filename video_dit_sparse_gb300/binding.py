"""ctypes binding of ``libsparse_attn.so`` (declared in include/sparse_attn.h).

Argument marshalling only: torch CUDA tensors are passed as raw device
pointers together with ``torch.cuda.current_stream()``.  Every step of the
path runs in the library's kernels; there is no CPU or PyTorch fallback, and
a missing library raises at import.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsparse_attn.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CAPACITY = 0, 1, 2, 3
SA_ERR_BAD_INDEX, SA_ERR_TIMEOUT, SA_ERR_CUDA = 4, 5, 6
SA_DEVERR_ROW_PTR, SA_DEVERR_INDEX, SA_DEVERR_TIMEOUT, SA_DEVERR_CAPACITY = 1, 2, 4, 8
SA_SELECT_TOPK, SA_SELECT_THRESHOLD, SA_SELECT_MASS = 0, 1, 2
_MODES = {"topk": SA_SELECT_TOPK, "threshold": SA_SELECT_THRESHOLD, "mass": SA_SELECT_MASS}
SA_COLSTAT_MAX, SA_COLSTAT_SUM = 0, 1
_STATS = {"max": SA_COLSTAT_MAX, "sum": SA_COLSTAT_SUM}


class SparseAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {sparse_attn_status_string(status)} (status {status})")


class sa_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Nq", ctypes.c_int32),
                ("Nk", ctypes.c_int32), ("d", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int32)]


SA_OUT_BF16, SA_OUT_FP32 = 0, 1
_OUT = {torch.bfloat16: SA_OUT_BF16, torch.float32: SA_OUT_FP32}


class sa_select(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("topk", ctypes.c_int64),
                ("threshold", ctypes.c_double), ("mass", ctypes.c_double)]


class sa_voxel_grid(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("Hh", ctypes.c_int32), ("W", ctypes.c_int32),
                ("vt", ctypes.c_int32), ("vh", ctypes.c_int32), ("vw", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc, sm_103a). There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    P, i64, vp = ctypes.POINTER, ctypes.c_int64, ctypes.c_void_p
    lib.sparse_attn_build_index_workspace_size.argtypes = [P(sa_problem)]
    lib.sparse_attn_build_index_workspace_size.restype = ctypes.c_size_t
    lib.sparse_attn_build_index.argtypes = [P(sa_problem), P(sa_select), vp, vp, vp, vp, i64,
                                            P(ctypes.c_int64), vp, ctypes.c_size_t, vp]
    lib.sparse_attn_build_index.restype = ctypes.c_int
    lib.sparse_attn_build_index_dense.argtypes = [P(sa_problem), P(sa_select), ctypes.c_int32, vp,
                                                  vp, vp, vp, vp, i64, P(ctypes.c_int64), vp,
                                                  ctypes.c_size_t, vp]
    lib.sparse_attn_build_index_dense.restype = ctypes.c_int
    lib.sparse_attn_forward.argtypes = [P(sa_problem), vp, vp, vp, vp, vp, i64, vp, vp, vp, vp]
    lib.sparse_attn_forward.restype = ctypes.c_int
    lib.sparse_attn_forward_delta.argtypes = [P(sa_problem), vp, vp, vp, vp, vp, i64, vp, vp,
                                              ctypes.c_float, vp, vp, vp]
    lib.sparse_attn_forward_delta.restype = ctypes.c_int
    lib.sparse_attn_layer_from_host.argtypes = [P(sa_problem), P(sa_select), vp, vp, vp, vp, vp, vp,
                                                vp, vp, vp, vp, vp, vp, i64, vp, ctypes.c_size_t,
                                                ctypes.c_int32, vp, vp, vp]
    lib.sparse_attn_layer_from_host.restype = ctypes.c_int
    lib.sparse_attn_index_from_bitmask.argtypes = [P(sa_problem), vp, vp, vp, i64, P(ctypes.c_int64), vp]
    lib.sparse_attn_index_from_bitmask.restype = ctypes.c_int
    lib.sparse_attn_index_from_block_mask.argtypes = [P(sa_problem), ctypes.c_int32, vp, vp, vp, i64,
                                                      P(ctypes.c_int64), vp]
    lib.sparse_attn_index_from_block_mask.restype = ctypes.c_int
    lib.sparse_attn_voxel_permute.argtypes = [P(sa_voxel_grid), ctypes.c_int32, ctypes.c_int32, vp,
                                              vp, ctypes.c_int32, vp]
    lib.sparse_attn_voxel_permute.restype = ctypes.c_int
    lib.sparse_attn_kv_window_append.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, i64, vp, vp, vp, vp,
                                                 P(ctypes.c_int64), vp]
    lib.sparse_attn_kv_window_append.restype = ctypes.c_int
    lib.sparse_attn_validate_index.argtypes = [P(sa_problem), vp, vp, i64, vp, vp]
    lib.sparse_attn_validate_index.restype = ctypes.c_int
    lib.sparse_attn_status_string.argtypes = [ctypes.c_int]
    lib.sparse_attn_status_string.restype = ctypes.c_char_p
    lib.sparse_attn_version.argtypes = []
    lib.sparse_attn_version.restype = ctypes.c_int32
    return lib


lib = _load()


def sparse_attn_status_string(status: int) -> str:
    return lib.sparse_attn_status_string(int(status)).decode()


def sparse_attn_version() -> int:
    return int(lib.sparse_attn_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def problem(q: torch.Tensor, k: torch.Tensor, group_size: int, scale: float | None = None,
            out_dtype=torch.bfloat16):
    """sa_problem for bf16 [B,H,N,d] tensors."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("k must be [B, H, Nk, d] with q's B, H and d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype not in _OUT:
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    return sa_problem(B, H, Nq, k.shape[2], d, group_size, scale, _OUT[out_dtype])


def _check(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


def sparse_attn_build_index_workspace_size(p: sa_problem) -> int:
    return int(lib.sparse_attn_build_index_workspace_size(ctypes.byref(p)))


def _build(q, k, mode, topk, threshold, mass, group_size, scale, col_capacity, workspace,
           stream, sync_nnz, stat=None, lse=None):
    _check(q, torch.bfloat16, "q")
    _check(k, torch.bfloat16, "k")
    p = problem(q, k, group_size, scale)
    G = -(-p.Nq // group_size)
    rows = p.B * p.H * G
    m = _MODES.get(mode, mode)
    sel = sa_select(m, int(topk), float(threshold), float(mass))
    dev = q.device
    row_ptr = torch.empty(rows + 1, dtype=torch.int64, device=dev)
    if col_capacity is None:
        col_capacity = rows * (min(max(int(topk), 1), p.Nk) if m == SA_SELECT_TOPK else p.Nk)
    col_idx = torch.empty(max(col_capacity, 1), dtype=torch.int32, device=dev)
    ws_bytes = sparse_attn_build_index_workspace_size(p)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if sync_nnz is None:
        sync_nnz = True
    nnz = ctypes.c_int64(0)
    nnz_ref = ctypes.byref(nnz) if sync_nnz else None
    if stat is None:
        st = lib.sparse_attn_build_index(ctypes.byref(p), ctypes.byref(sel), _ptr(q), _ptr(k),
                                         _ptr(row_ptr), _ptr(col_idx), int(col_capacity), nnz_ref,
                                         _ptr(workspace), workspace.numel(), _stream(stream))
        where = "sparse_attn_build_index"
    else:
        _check(lse, torch.float32, "lse")
        st = lib.sparse_attn_build_index_dense(ctypes.byref(p), ctypes.byref(sel),
                                               _STATS.get(stat, stat), _ptr(q), _ptr(k), _ptr(lse),
                                               _ptr(row_ptr), _ptr(col_idx), int(col_capacity),
                                               nnz_ref, _ptr(workspace), workspace.numel(),
                                               _stream(stream))
        where = "sparse_attn_build_index_dense"
    if st != SA_OK:
        raise SparseAttnError(st, where)
    n = nnz.value if sync_nnz else rows * min(max(int(topk), 1), p.Nk)
    return row_ptr, col_idx[:n], n


def sparse_attn_build_index(q: torch.Tensor, k: torch.Tensor, mode="topk", *, topk: int = 0,
                            threshold: float = 0.0, mass: float = 0.99, group_size: int = 128,
                            scale: float | None = None, col_capacity: int | None = None,
                            workspace: torch.Tensor | None = None, stream=None,
                            sync_nnz: bool | None = None):
    """Builds CSR key lists from mean-query scores; returns (row_ptr int64,
    col_idx int32, nnz).

    By default the call synchronises and raises on any device-side error
    (capacity, timeout).  ``sync_nnz=False`` keeps a TOPK call fully
    asynchronous (nnz is then known up front).  For THRESHOLD/MASS col_idx is
    allocated for the worst case (every key) unless col_capacity is given;
    col_idx is returned trimmed to nnz (a view).
    """
    return _build(q, k, mode, topk, threshold, mass, group_size, scale, col_capacity, workspace,
                  stream, sync_nnz)


def sparse_attn_build_index_dense(q: torch.Tensor, k: torch.Tensor, lse: torch.Tensor,
                                  stat="max", mode="threshold", *, topk: int = 0,
                                  threshold: float = 0.0, mass: float = 0.99,
                                  group_size: int = 128, scale: float | None = None,
                                  col_capacity: int | None = None,
                                  workspace: torch.Tensor | None = None, stream=None,
                                  sync_nnz: bool | None = None):
    """Key lists from a dense step's attention probabilities (column max or
    column sum over each group of exp(scale q.k - lse)); `lse` fp32
    [B,H,Nq] as the dense forward writes it.  THRESHOLD compares the
    statistic itself with `threshold` (the cached mask: stat "max",
    threshold 0.5/Nk).  Returns (row_ptr, col_idx, nnz) like
    sparse_attn_build_index."""
    return _build(q, k, mode, topk, threshold, mass, group_size, scale, col_capacity, workspace,
                  stream, sync_nnz, stat=stat, lse=lse)


def _fwd_common(q, k, v, row_ptr, col_idx, group_size, scale, nnz, out, out_dtype):
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, torch.bfloat16, n)
    if (row_ptr is None) != (col_idx is None):
        raise ValueError("row_ptr and col_idx are both given or both None (dense)")
    if row_ptr is not None:
        _check(row_ptr, torch.int64, "row_ptr")
        _check(col_idx, torch.int32, "col_idx")
    if v.shape != k.shape:
        raise ValueError("v must have k's shape")
    if out is not None:
        _check(out, out.dtype, "out")
        out_dtype = out.dtype
    p = problem(q, k, group_size, scale, out_dtype)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if row_ptr is None:
        return p, out, None, None, 0
    if nnz is None:
        nnz = col_idx.numel()
    return p, out, _ptr(row_ptr), (_ptr(col_idx) if col_idx.numel() else None), int(nnz)


def sparse_attn_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        row_ptr: torch.Tensor | None, col_idx: torch.Tensor | None, *,
                        group_size: int = 128, scale: float | None = None,
                        nnz: int | None = None, out: torch.Tensor | None = None,
                        out_dtype=torch.bfloat16, lse: torch.Tensor | bool = True,
                        status: torch.Tensor | None = None, stream=None):
    """Column-sparse attention; returns (o [B,H,Nq,d] in out_dtype (bf16 or
    fp32; taken from `out` if given), lse fp32 [B,H,Nq] or None).
    row_ptr = col_idx = None: dense attention (every key kept)."""
    p, out, rp, ci, nnz = _fwd_common(q, k, v, row_ptr, col_idx, group_size, scale, nnz, out,
                                      out_dtype)
    if lse is True:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    st = lib.sparse_attn_forward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), rp, ci, nnz,
                                 _ptr(out), _ptr(lse), _ptr(status), _stream(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_forward")
    return out, lse


def sparse_attn_forward_delta(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                              row_ptr: torch.Tensor | None, col_idx: torch.Tensor | None,
                              lse_ref: torch.Tensor, *, base: torch.Tensor | None = None,
                              sign: float = 1.0, group_size: int = 128,
                              scale: float | None = None, nnz: int | None = None,
                              out: torch.Tensor | None = None, out_dtype=torch.float32,
                              status: torch.Tensor | None = None, stream=None):
    """Sparse delta: o = base + sign * sum over kept j of
    exp(scale q.k_j - lse_ref) v_j (fp32 base, fp32 output by default;
    out=base updates the cache in place)."""
    _check(lse_ref, torch.float32, "lse_ref")
    if base is not None:
        _check(base, torch.float32, "base")
    p, out, rp, ci, nnz = _fwd_common(q, k, v, row_ptr, col_idx, group_size, scale, nnz, out,
                                      out_dtype)
    st = lib.sparse_attn_forward_delta(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), rp, ci, nnz,
                                       _ptr(lse_ref), _ptr(base), float(sign), _ptr(out),
                                       _ptr(status), _stream(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_forward_delta")
    return out


def sparse_attn_validate_index(row_ptr: torch.Tensor, col_idx: torch.Tensor, *, B: int, H: int,
                               Nq: int, Nk: int, d: int = 128, group_size: int = 128,
                               status: torch.Tensor | None = None, stream=None) -> int:
    """Returns SA_OK or SA_ERR_BAD_INDEX (synchronises)."""
    _check(row_ptr, torch.int64, "row_ptr")
    _check(col_idx, torch.int32, "col_idx")
    p = sa_problem(B, H, Nq, Nk, d, group_size, 1.0 / math.sqrt(d), SA_OUT_BF16)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=row_ptr.device)
    st = lib.sparse_attn_validate_index(ctypes.byref(p), _ptr(row_ptr),
                                        _ptr(col_idx) if col_idx.numel() else None,
                                        col_idx.numel(), _ptr(status), _stream(stream))
    if st not in (SA_OK, SA_ERR_BAD_INDEX):
        raise SparseAttnError(st, "sparse_attn_validate_index")
    return st


def _from_mask(mask, B, H, Nq, Nk, d, group_size, block_k, col_capacity, stream):
    p = sa_problem(B, H, Nq, Nk, d, group_size, 1.0 / math.sqrt(d), SA_OUT_BF16)
    G = -(-Nq // group_size)
    rows = B * H * G
    dev = mask.device
    row_ptr = torch.empty(rows + 1, dtype=torch.int64, device=dev)
    cap = rows * Nk if col_capacity is None else int(col_capacity)
    col_idx = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    nnz = ctypes.c_int64(0)
    if block_k is None:
        st = lib.sparse_attn_index_from_bitmask(ctypes.byref(p), _ptr(mask), _ptr(row_ptr),
                                                _ptr(col_idx), cap, ctypes.byref(nnz), _stream(stream))
        where = "sparse_attn_index_from_bitmask"
    else:
        st = lib.sparse_attn_index_from_block_mask(ctypes.byref(p), int(block_k), _ptr(mask),
                                                   _ptr(row_ptr), _ptr(col_idx), cap,
                                                   ctypes.byref(nnz), _stream(stream))
        where = "sparse_attn_index_from_block_mask"
    if st != SA_OK:
        raise SparseAttnError(st, where)
    return row_ptr, col_idx[:nnz.value], nnz.value


def sparse_attn_index_from_bitmask(mask_words: torch.Tensor, *, B: int, H: int, Nq: int, Nk: int,
                                   d: int = 128, group_size: int = 128,
                                   col_capacity: int | None = None, stream=None):
    """uint32 words [B*H*G, ceil(Nk/32)] (torch.int32 storage), key j = bit j%32
    of word j//32 -> (row_ptr, col_idx, nnz).  Synchronises."""
    _check(mask_words, torch.int32, "mask_words")
    return _from_mask(mask_words, B, H, Nq, Nk, d, group_size, None, col_capacity, stream)


def sparse_attn_index_from_block_mask(block_mask: torch.Tensor, block_k: int, *, B: int, H: int,
                                      Nq: int, Nk: int, d: int = 128, group_size: int = 128,
                                      col_capacity: int | None = None, stream=None):
    """uint8 [B*H*G, ceil(Nk/block_k)] (non-zero = keep the key block) ->
    (row_ptr, col_idx, nnz).  Synchronises."""
    _check(block_mask, torch.uint8, "block_mask")
    return _from_mask(block_mask, B, H, Nq, Nk, d, group_size, block_k, col_capacity, stream)


def sparse_attn_voxel_permute(x: torch.Tensor, grid, voxel, *, inverse: bool = False,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """x bf16 [B, H, N, d] (N = T*Hh*W) -> the same tokens in voxel order
    (or back to raster order when inverse)."""
    _check(x, torch.bfloat16, "x")
    if x.dim() != 4:
        raise ValueError("x must be [B, H, N, d]")
    B, H, N, d = x.shape
    g = sa_voxel_grid(*grid, *voxel)
    if out is None:
        out = torch.empty_like(x)
    _check(out, torch.bfloat16, "out")
    st = lib.sparse_attn_voxel_permute(ctypes.byref(g), B * H, d, _ptr(x), _ptr(out),
                                       1 if inverse else 0, _stream(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_voxel_permute")
    return out


def sparse_attn_kv_window_append(cache_k: torch.Tensor, cache_v: torch.Tensor,
                                 new_k: torch.Tensor, new_v: torch.Tensor, chunks_before: int, *,
                                 stream=None) -> int:
    """Appends one chunk ([B, H, L, d]) to the rolling caches ([B, H, S*L, d],
    slot 0 = sink) in place; returns the number of valid key tokens."""
    for t, n in ((cache_k, "cache_k"), (cache_v, "cache_v"), (new_k, "new_k"), (new_v, "new_v")):
        _check(t, torch.bfloat16, n)
    B, H, SL, d = cache_k.shape
    L = new_k.shape[2]
    if cache_v.shape != cache_k.shape or new_v.shape != new_k.shape or SL % L:
        raise ValueError("caches must be [B, H, S*L, d] and chunks [B, H, L, d]")
    valid = ctypes.c_int64(0)
    st = lib.sparse_attn_kv_window_append(B * H, d, L, SL // L, int(chunks_before), _ptr(cache_k),
                                          _ptr(cache_v), _ptr(new_k), _ptr(new_v),
                                          ctypes.byref(valid), _stream(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_kv_window_append")
    return int(valid.value)


class HostLayer:
    """One attention layer from pinned host tensors (sparse_attn_layer_from_host):
    device staging, one chunk's scratch and two copy streams, allocated once
    for a shape.  Calling it enqueues the copies in, the build + forward per
    chunk of heads and the copies out; `synchronize()` waits for the layer."""

    def __init__(self, B, H, Nq, Nk, d, *, group_size=128, mode="topk", topk=0, threshold=0.0,
                 mass=0.99, heads_per_chunk=0, out_dtype=torch.bfloat16, with_lse=True,
                 device=None):
        dev = torch.device(device or "cuda")
        self.p = sa_problem(B, H, Nq, Nk, d, group_size, 1.0 / math.sqrt(d), _OUT[out_dtype])
        m = _MODES.get(mode, mode)
        self.sel = sa_select(m, int(topk), float(threshold), float(mass))
        BH = B * H
        mid = BH - 2 if BH > 2 else 0
        self.hc = heads_per_chunk if heads_per_chunk > 0 else (-(-mid // 3) if mid > 0 else BH)
        self.hc = min(self.hc, BH)
        G = -(-Nq // group_size)
        kmax = min(max(int(topk), 1), Nk) if m == SA_SELECT_TOPK else Nk
        cp = sa_problem(1, self.hc, Nq, Nk, d, group_size, self.p.scale, self.p.out_dtype)
        self.ws = torch.empty(sparse_attn_build_index_workspace_size(cp), dtype=torch.uint8, device=dev)
        self.row_ptr = torch.empty(self.hc * G + 1, dtype=torch.int64, device=dev)
        self.cap = self.hc * G * kmax
        self.col = torch.empty(self.cap, dtype=torch.int32, device=dev)
        self.q = torch.empty(B, H, Nq, d, dtype=torch.bfloat16, device=dev)
        self.k = torch.empty(B, H, Nk, d, dtype=torch.bfloat16, device=dev)
        self.v = torch.empty_like(self.k)
        self.o = torch.empty(B, H, Nq, d, dtype=out_dtype, device=dev)
        self.lse = torch.empty(B, H, Nq, dtype=torch.float32, device=dev) if with_lse else None
        self.copy_in = torch.cuda.Stream(device=dev)
        self.copy_out = torch.cuda.Stream(device=dev)

    def __call__(self, q_host, k_host, v_host, o_host, lse_host=None, stream=None):
        for t in (q_host, k_host, v_host, o_host):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("host tensors must be contiguous CPU tensors (pinned to overlap)")
        if (lse_host is None) != (self.lse is None):
            raise ValueError("lse_host must be given exactly when the layer keeps lse")
        st = lib.sparse_attn_layer_from_host(
            ctypes.byref(self.p), ctypes.byref(self.sel), _ptr(q_host), _ptr(k_host), _ptr(v_host),
            _ptr(o_host), _ptr(lse_host), _ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.o),
            _ptr(self.lse), _ptr(self.row_ptr), _ptr(self.col), self.cap, _ptr(self.ws),
            self.ws.numel(), int(self.hc), _stream(stream), _stream(self.copy_in),
            _stream(self.copy_out))
        if st != SA_OK:
            raise SparseAttnError(st, "sparse_attn_layer_from_host")

    def synchronize(self, stream=None):
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()


# Short aliases for Python callers.
build_index = sparse_attn_build_index
build_index_dense = sparse_attn_build_index_dense
forward = sparse_attn_forward
forward_delta = sparse_attn_forward_delta
validate_index = sparse_attn_validate_index
voxel_permute = sparse_attn_voxel_permute
index_from_bitmask = sparse_attn_index_from_bitmask
index_from_block_mask = sparse_attn_index_from_block_mask
kv_window_append = sparse_attn_kv_window_append
