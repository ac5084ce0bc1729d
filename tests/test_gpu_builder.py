"""GPU parity of sparse_attn_build_index against the fp64 oracle (through the
C ABI): top-k, threshold and retained-mass selection on small field inputs
(several key tiles, ragged tails, ragged groups), bit-exact lists except for
keys within 1e-3 relative of the oracle's cut, then the GPU lists fed to the
GPU forward and compared end to end."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def field(B, H, d, grid_q, grid_k=None, seed=0, voxel=None):
    w = I.custom("t", B, H, d, 128, grid_q, grid_k, voxel=voxel)
    x = I.make_inputs(w, seed)
    return x["q"], x["k"], x["v"]


def gpu_build(q, k, M, mode, **kw):
    from video_dit_sparse_gb300 import binding as sa
    qd, kd = P.to_dev(q), P.to_dev(k)
    rp, col, nnz = sa.sparse_attn_build_index(qd, kd, mode, group_size=M, **kw)
    torch.cuda.synchronize()
    return rp, col, nnz


CASES = [
    # (d, M, grid_q, grid_k, mode, kwargs)
    (128, 128, (4, 16, 16), None, "topk", {"topk": 205}),
    (128, 128, (5, 10, 20), (7, 10, 10), "topk", {"topk": 1}),
    (128, 128, (5, 10, 20), (7, 10, 10), "topk", {"topk": 700}),
    (64, 128, (4, 16, 16), None, "topk", {"topk": 333}),
    (128, 192, (5, 10, 20), (9, 10, 10), "topk", {"topk": 90}),
    (128, 128, (4, 16, 16), None, "threshold", {"threshold": 5e-4}),
    (128, 128, (4, 16, 16), None, "threshold", {"threshold": 0.0}),
    (128, 128, (4, 16, 16), None, "threshold", {"threshold": 0.9}),
    (128, 128, (4, 16, 16), (8, 16, 16), "mass", {"mass": 0.99}),
    (128, 128, (4, 16, 16), None, "mass", {"mass": 0.5}),
    (64, 192, (5, 10, 20), (7, 10, 10), "mass", {"mass": 0.9}),
    (128, 128, (4, 16, 16), None, "mass", {"mass": 1.0}),
    # more keys than the selection's in-memory bracket: the sampled path
    (128, 128, (4, 16, 16), (10, 25, 40), "topk", {"topk": 2000}),
    (128, 128, (4, 16, 16), (10, 25, 40), "topk", {"topk": 9}),
    (128, 128, (4, 16, 16), (10, 25, 40), "topk", {"topk": 9990}),
    (128, 128, (4, 16, 16), (10, 25, 40), "mass", {"mass": 0.99}),
    (128, 128, (4, 16, 16), (10, 25, 40), "mass", {"mass": 0.3}),
]


@pytest.mark.parametrize("d,M,grid_q,grid_k,mode,kw", CASES)
def test_lists_match_oracle(d, M, grid_q, grid_k, mode, kw):
    q, k, v = field(1, 2, d, grid_q, grid_k, seed=M + d)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    rows = B * H * G
    scale = 1.0 / math.sqrt(d)
    rp, col, nnz = gpu_build(q, k, M, mode, **kw)
    ref_lists, ref_cut, ref_sc = oracle.build_index(q, k, M, scale, mode, topk=kw.get("topk", 0),
                                                    tau=kw.get("threshold", 0.0),
                                                    rho=kw.get("mass", 0.99))
    rpn = rp.cpu().numpy()
    assert rpn[0] == 0 and rpn[-1] == nnz and np.all(np.diff(rpn) >= 1)
    P.compare_lists(rp, col, range(rows), ref_lists, ref_cut, ref_sc, Nk)
    if mode == "topk":
        assert np.all(np.diff(rpn) == min(kw["topk"], Nk))
    # end to end: GPU lists -> GPU forward vs oracle forward on the same lists
    from video_dit_sparse_gb300 import binding as sa
    o, lse = sa.sparse_attn_forward(P.to_dev(q), P.to_dev(k), P.to_dev(v), rp, col, group_size=M,
                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    P.compare_units(q, k, v, M, rpn, col.cpu().numpy(), np.arange(rows), o, lse)


def test_capacity_report_for_mass():
    from video_dit_sparse_gb300 import binding as sa
    q, k, _ = field(1, 1, 128, (4, 16, 16))
    with pytest.raises(sa.SparseAttnError) as e:
        sa.sparse_attn_build_index(P.to_dev(q), P.to_dev(k), "mass", mass=0.99, col_capacity=10)
    assert e.value.status == sa.SA_ERR_CAPACITY


def test_builder_repeatable():
    q, k, _ = field(1, 2, 128, (4, 16, 16), (8, 16, 16))
    a = gpu_build(q, k, 128, "mass", mass=0.95)
    b = gpu_build(q, k, 128, "mass", mass=0.95)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
