"""sparse_attn_build_index_noalloc: the index builder for callers that
cannot allocate device memory (its scratch is a fixed 32 MiB array owned by
the library).  Called through the C ABI, it must give the same lists as
sparse_attn_build_index with a caller-provided workspace, on two calls in a
row whose problems differ (the second call starts from the first call's
leftover scratch), and must refuse a problem whose scratch does not fit.
This file is collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest
import torch

from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _lib():
    from video_dit_sparse_gb300 import binding as sa
    f = sa.lib.sparse_attn_build_index_noalloc
    P = ctypes.POINTER
    f.argtypes = [P(sa.sa_problem), P(sa.sa_select), ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, P(ctypes.c_int64),
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    return sa, f


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _inputs(H, d, grid_q, grid_k, seed):
    w = I.custom("noalloc", 1, H, d, 128, grid_q, grid_k)
    x = I.make_inputs(w, seed)
    return _dev(x["q"]), _dev(x["k"])


def _select(sa, mode, kw):
    return sa.sa_select(sa._MODES[mode], kw.get("topk", 0), kw.get("threshold", 0.0),
                        kw.get("mass", 0.99))


def _noalloc(sa, f, q, k, mode, M, cap=None, with_nnz=True, stream=None, **kw):
    p = sa.problem(q, k, M)
    sel = _select(sa, mode, kw)
    rows = p.B * p.H * (-(-p.Nq // M))
    cap = rows * p.Nk if cap is None else cap
    row_ptr = torch.full((rows + 1,), -1, dtype=torch.int64, device="cuda")
    col = torch.full((max(cap, 1),), -1, dtype=torch.int32, device="cuda")
    nnz = ctypes.c_int64(-1)
    st = f(ctypes.byref(p), ctypes.byref(sel), sa._ptr(q), sa._ptr(k), sa._ptr(row_ptr),
           sa._ptr(col), cap, ctypes.byref(nnz) if with_nnz else None, sa._stream(stream))
    torch.cuda.synchronize()
    return st, row_ptr, col[:max(nnz.value, 0)], nnz.value


CASES = [
    dict(H=2, d=128, grid_q=(4, 16, 16), grid_k=(8, 16, 16), mode="topk", M=128, kw={"topk": 300}),
    dict(H=3, d=64, grid_q=(5, 10, 20), grid_k=(7, 10, 10), mode="mass", M=192, kw={"mass": 0.95}),
    dict(H=2, d=128, grid_q=(3, 12, 20), grid_k=(5, 12, 20), mode="threshold", M=128,
         kw={"threshold": 0.5 / 1200}),
]


def test_noalloc_matches_workspace_builder_on_two_calls_in_a_row():
    sa, f = _lib()
    for i, c in enumerate(CASES):
        q, k = _inputs(c["H"], c["d"], c["grid_q"], c["grid_k"], seed=i)
        st, rp, col, _ = _noalloc(sa, f, q, k, c["mode"], c["M"], **c["kw"])
        assert st == sa.SA_OK, sa.sparse_attn_status_string(st)
        ref_rp, ref_col, ref_nnz = sa.sparse_attn_build_index(q, k, c["mode"], group_size=c["M"],
                                                              **c["kw"])
        torch.cuda.synchronize()
        assert torch.equal(rp, ref_rp)
        assert col.numel() == ref_nnz and torch.equal(col, ref_col)


def test_noalloc_on_a_side_stream():
    sa, f = _lib()
    c = CASES[0]
    q, k = _inputs(c["H"], c["d"], c["grid_q"], c["grid_k"], seed=5)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    st, rp, col, _ = _noalloc(sa, f, q, k, c["mode"], c["M"], stream=side, **c["kw"])
    assert st == sa.SA_OK, sa.sparse_attn_status_string(st)
    ref_rp, ref_col, ref_nnz = sa.sparse_attn_build_index(q, k, c["mode"], group_size=c["M"], **c["kw"])
    torch.cuda.synchronize()
    assert torch.equal(rp, ref_rp) and torch.equal(col, ref_col)


def test_noalloc_capacity_rules():
    sa, f = _lib()
    # TOPK: the need is known up front, reported without a launch
    c = CASES[0]
    q, k = _inputs(c["H"], c["d"], c["grid_q"], c["grid_k"], seed=6)
    rows = c["H"] * (q.shape[2] // c["M"])
    st, _, _, nnz = _noalloc(sa, f, q, k, "topk", c["M"], cap=rows * 300 - 1, topk=300)
    assert st == sa.SA_ERR_CAPACITY and nnz == rows * 300
    # MASS: data-dependent; a short capacity runs, then reports the need
    c = CASES[1]
    q, k = _inputs(c["H"], c["d"], c["grid_q"], c["grid_k"], seed=7)
    _, ref_col, ref_nnz = sa.sparse_attn_build_index(q, k, "mass", group_size=c["M"], mass=0.95)
    torch.cuda.synchronize()
    st, _, _, nnz = _noalloc(sa, f, q, k, "mass", c["M"], cap=ref_nnz // 2, mass=0.95)
    assert st == sa.SA_ERR_CAPACITY and nnz == ref_nnz
    # without nnz_out_host a data-dependent selection needs room for every key
    st, _, _, _ = _noalloc(sa, f, q, k, "mass", c["M"], cap=ref_nnz, with_nnz=False, mass=0.95)
    assert st == sa.SA_ERR_INVALID_ARG


def test_noalloc_rejects_problems_larger_than_its_scratch():
    sa, f = _lib()
    q = torch.zeros(1, 8, 16384, 128, dtype=torch.bfloat16, device="cuda")
    p = sa.problem(q, q, 128)
    assert sa.sparse_attn_build_index_workspace_size(p) > (32 << 20)
    rows = 8 * 128
    row_ptr = torch.empty(rows + 1, dtype=torch.int64, device="cuda")
    col = torch.empty(rows * 16, dtype=torch.int32, device="cuda")
    sel = sa.sa_select(sa.SA_SELECT_TOPK, 16, 0.0, 0.0)
    st = f(ctypes.byref(p), ctypes.byref(sel), sa._ptr(q), sa._ptr(q), sa._ptr(row_ptr),
           sa._ptr(col), col.numel(), None, sa._stream(None))
    assert st == sa.SA_ERR_UNSUPPORTED
