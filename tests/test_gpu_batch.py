"""Batch dimension B = 2 through every entry point (GPU, C ABI): the mean-query
builder (all three modes), the forward on its lists, the dense mode, the
dense-step builder and the sparse delta, each against the oracle; units are
ordered (b, h, g) with b slowest."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def batch_inputs(seed=0):
    w = I.custom("b2", 2, 3, 128, 128, (5, 10, 20), (7, 10, 10))  # Nq 1000, Nk 700
    x = I.make_inputs(w, seed)
    return w, x


@pytest.mark.parametrize("mode,kw", [("topk", {"topk": 140}), ("mass", {"mass": 0.9}),
                                     ("threshold", {"threshold": 0.002})])
def test_batch_builder_and_forward(mode, kw):
    from video_dit_sparse_gb300 import binding as sa
    w, x = batch_inputs(1)
    qd, kd, vd = P.to_dev(x["q"]), P.to_dev(x["k"]), P.to_dev(x["v"])
    rp, col, nnz = sa.sparse_attn_build_index(qd, kd, mode, group_size=128, **kw)
    o, lse = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = w.B * w.H * w.G
    okw = {"topk": kw.get("topk", 0), "tau": kw.get("threshold", 0.0), "rho": kw.get("mass", 0.99)}
    lists, cut, sc = oracle.build_index(x["q"], x["k"], 128, w.scale, mode, **okw)
    P.compare_lists(rp, col, range(rows), lists, cut, sc, w.Nk)
    P.compare_units(x["q"], x["k"], x["v"], 128, rp.cpu().numpy(), col.cpu().numpy(), np.arange(rows), o, lse)


def test_batch_dense_step_and_delta():
    from video_dit_sparse_gb300 import binding as sa
    w, x = batch_inputs(2)
    qd, kd, vd = P.to_dev(x["q"]), P.to_dev(x["k"]), P.to_dev(x["v"])
    rows = w.B * w.H * w.G
    o, lse = sa.sparse_attn_forward(qd, kd, vd, None, None, group_size=128, out_dtype=torch.float32)
    rp_full, col_full = oracle.to_csr([np.arange(w.Nk, dtype=np.int32)] * rows)
    P.compare_units(x["q"], x["k"], x["v"], 128, rp_full, col_full, np.arange(rows), o, lse)
    rp, col, nnz = sa.sparse_attn_build_index_dense(qd, kd, lse, "sum", "topk", topk=70, group_size=128)
    cache = sa.sparse_attn_forward_delta(qd, kd, vd, rp, col, lse, base=o, sign=-1.0, group_size=128)
    torch.cuda.synchronize()
    lse64 = lse.double().cpu().numpy()
    lists, cut, st = oracle.dense_index(x["q"], x["k"], lse64, 128, w.scale, "sum", "topk", topk=70)
    P.compare_lists(rp, col, range(rows), lists, cut, st, w.Nk)
    d_ref = oracle.forward_delta(x["q"], x["k"], x["v"], 128, w.scale, rp.cpu().numpy(), col.cpu().numpy(),
                                 lse64, o.double().cpu().numpy(), -1.0)
    got = cache.view(w.B * w.H, w.Nq, w.d).double().cpu().numpy()
    ref = d_ref.reshape(w.B * w.H, w.G * 128, w.d)[:, :w.Nq]
    err = np.abs(got - ref)
    assert err.max() <= P.O_MAX and err.mean() <= P.O_MEAN, (err.max(), err.mean())
