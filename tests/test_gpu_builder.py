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


# ---------------------------------------------------------------- TOPK over >= 8192 keys
# These lists come from the path without a score matrix: sampled scores, a
# bracket around each row's cut, one classifying score pass, the exact cut
# among the bracketed candidates.  Rows it cannot bracket are selected from
# their full scores afterwards; `fallback_rows` reads how many there were
# (the int32 at the start of the workspace's last region: count, row list,
# unit flags), or -1 when the path was not taken (the workspace starts as
# 0xFF bytes and only that path clears the count).
def _workspace(qd, kd, M):
    from video_dit_sparse_gb300 import binding as sa
    ws = torch.full((sa.sparse_attn_build_index_workspace_size(sa.problem(qd, kd, M)),), 255,
                    dtype=torch.uint8, device="cuda")
    B, H, Nq, _ = qd.shape
    rows = B * H * (-(-Nq // M))
    return ws, ws.numel() - ((256 + 8 * rows + 255) // 256) * 256


def fallback_rows(ws, off):
    return int(ws[off:off + 4].view(torch.int32).item())


def build_topk(q, k, M, topk):
    from video_dit_sparse_gb300 import binding as sa
    qd, kd = P.to_dev(q), P.to_dev(k)
    ws, off = _workspace(qd, kd, M)
    rp, col, nnz = sa.sparse_attn_build_index(qd, kd, "topk", topk=topk, group_size=M, workspace=ws)
    torch.cuda.synchronize()
    return rp, col, nnz, fallback_rows(ws, off)


def check_topk(q, k, M, topk, rp, col):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    rows = B * H * (-(-Nq // M))
    ref_lists, ref_cut, ref_sc = oracle.build_index(q, k, M, 1.0 / math.sqrt(d), "topk", topk=topk)
    rpn = rp.cpu().numpy()
    assert np.all(np.diff(rpn) == min(topk, Nk)) and rpn[-1] == rows * min(topk, Nk)
    P.compare_lists(rp, col, range(rows), ref_lists, ref_cut, ref_sc, Nk)


DIRECT_CASES = [
    # (d, M, grid_q, grid_k, topk): ragged 128-row chunks of groups (G = 150),
    # d = 64, 192-row groups, a top key, nearly every key, every key
    (128, 128, (12, 40, 40), (10, 25, 40), 1500),
    (64, 128, (4, 16, 16), (16, 32, 32), 3277),
    (128, 192, (6, 16, 16), (10, 25, 40), 1000),
    (128, 128, (4, 16, 16), (8, 32, 32), 1),
    (128, 128, (4, 16, 16), (8, 32, 32), 8191),
    (128, 128, (4, 16, 16), (8, 32, 32), 8192),
]


@pytest.mark.parametrize("d,M,grid_q,grid_k,topk", DIRECT_CASES)
def test_topk_direct_matches_oracle(d, M, grid_q, grid_k, topk):
    q, k, _ = field(1, 2, d, grid_q, grid_k, seed=topk + d)
    rp, col, nnz, nf = build_topk(q, k, M, topk)
    check_topk(q, k, M, topk, rp, col)
    if topk < k.shape[2]:
        assert nf == 0  # field inputs: every row bracketed


def test_topk_direct_identical_keys_fall_back():
    # every score of a row ties: the bracket holds the whole row, more than
    # the finalize takes, so every row goes through the full-score selection
    # (lowest indices first among equal scores)
    q, k, _ = field(1, 2, 128, (4, 16, 16), (8, 32, 32), seed=5)
    k = np.ascontiguousarray(np.broadcast_to(k[:, :, :1], k.shape))
    rp, col, nnz, nf = build_topk(q, k, 128, 1000)
    rows = 2 * 8
    assert nf == rows
    check_topk(q, k, 128, 1000, rp, col)
    first = np.arange(1000, dtype=np.int32)
    c = col.cpu().numpy().reshape(rows, 1000)
    assert all(np.array_equal(c[r], first) for r in range(rows))


def _tall_keys(grid_k, seed, every):
    # every `every`-th key is all ones and the queries are offset by +3:
    # those keys tie far above every other key
    q, k, _ = field(1, 1, 128, (4, 16, 16), grid_k, seed=seed)
    one = np.uint16(np.float32(1.0).view(np.uint32) >> 16)
    qf = (q.astype(np.uint32) << 16).view(np.float32) + np.float32(3.0)
    q = (qf.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16: any bits are inputs
    k = k.copy()
    k[:, :, ::every, :] = one
    return q, k


def test_topk_direct_unrepresentative_sample_falls_back():
    # the sampled keys (every 8th) are the tied ones: the bracket sits among
    # them and holds fewer than k keys, so every row falls back
    q, k = _tall_keys((16, 32, 32), seed=6, every=8)
    rp, col, nnz, nf = build_topk(q, k, 128, 3277)
    assert nf == 8
    check_topk(q, k, 128, 3277, rp, col)


def test_topk_direct_ties_at_the_cut_by_index():
    # k below the 512 tied keys: the cut falls among equal scores and the
    # lowest indices are kept
    q, k = _tall_keys((8, 32, 32), seed=7, every=16)
    rp, col, nnz, nf = build_topk(q, k, 128, 500)
    assert nf == 0
    check_topk(q, k, 128, 500, rp, col)
    c = col.cpu().numpy().reshape(8, 500)
    assert all(np.array_equal(c[r], np.arange(0, 8000, 16)) for r in range(8))


def test_topk_direct_batch_of_two():
    # B = 2: rows of both batch entries' heads, 192-row groups, d = 64
    q, k, _ = field(2, 2, 64, (6, 16, 16), (8, 32, 32), seed=11)
    rp, col, nnz, nf = build_topk(q, k, 192, 777)
    assert nf == 0
    check_topk(q, k, 192, 777, rp, col)
