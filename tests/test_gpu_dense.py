"""GPU parity of the dense step and of the sparse delta (through the C ABI):

  * the forward's dense mode (no index lists) against the oracle with every
    key listed, and bit for bit against the same kernel given explicit
    all-key lists;
  * sparse_attn_build_index_dense (FG-Attn cached mask: column max of the
    dense probabilities against tau = 0.5/N; Chipmunk column sums with
    top-k; retained mass of the column sums) against the oracle's lists,
    with the oracle's lse given to both sides, and end to end from the GPU's
    own dense forward;
  * sparse_attn_forward_delta (masked full softmax with a stale normaliser)
    against the oracle, the cache round trip, in-place update and the
    all-keys case;
  * the 69K-token workload: dense forward, cached mask and sparse forward on
    the GPU's lists, sampled query groups checked by the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def field(B, H, d, grid_q, grid_k=None, seed=0):
    w = I.custom("t", B, H, d, 128, grid_q, grid_k)
    x = I.make_inputs(w, seed)
    return x["q"], x["k"], x["v"]


def full_csr(rows, Nk):
    return oracle.to_csr([np.arange(Nk, dtype=np.int32)] * rows)


@pytest.mark.parametrize("d,M", [(128, 128), (64, 128), (128, 192), (64, 64)])
def test_dense_forward_matches_oracle_and_full_lists(d, M):
    from video_dit_sparse_gb300 import binding as sa
    q, k, v = field(1, 2, d, (5, 10, 20), (7, 10, 10), seed=d + M)  # Nq 1000, Nk 700
    qd, kd, vd = P.to_dev(q), P.to_dev(k), P.to_dev(v)
    G = -(-1000 // M)
    o, lse = sa.sparse_attn_forward(qd, kd, vd, None, None, group_size=M, out_dtype=torch.float32)
    rp, col = full_csr(2 * G, 700)
    o2, lse2 = sa.sparse_attn_forward(qd, kd, vd, torch.from_numpy(rp).cuda(),
                                      torch.from_numpy(col).cuda(), group_size=M,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    P.compare_units(q, k, v, M, rp, col, np.arange(2 * G), o, lse)
    # and against dense attention by torch (fp32 reference of the same op)
    ref = torch.nn.functional.scaled_dot_product_attention(qd.float(), kd.float(), vd.float())
    assert (o - ref).abs().max().item() < 2e-2


def dense_case(d, M, seed):
    q, k, v = field(1, 2, d, (5, 10, 20), (7, 10, 10), seed=seed)
    scale = 1.0 / math.sqrt(d)
    lse = oracle.dense_lse(q, k, scale)
    lse32 = lse.astype(np.float32)
    return q, k, v, scale, lse32


@pytest.mark.parametrize("stat,mode,kw", [
    ("max", "threshold", {"threshold": 0.5 / 700}),
    ("max", "topk", {"topk": 140}),
    ("sum", "topk", {"topk": 70}),
    ("sum", "mass", {"mass": 0.9}),
    ("sum", "threshold", {"threshold": 0.2}),
    ("max", "mass", {"mass": 0.99}),
])
@pytest.mark.parametrize("d,M", [(128, 128), (64, 192), (128, 64)])
def test_dense_builder_matches_oracle(stat, mode, kw, d, M):
    from video_dit_sparse_gb300 import binding as sa
    q, k, _, scale, lse32 = dense_case(d, M, seed=3 * d + M)
    G = -(-1000 // M)
    rows = 2 * G
    rp, col, nnz = sa.sparse_attn_build_index_dense(
        P.to_dev(q), P.to_dev(k), torch.from_numpy(lse32).cuda(), stat, mode, group_size=M, **kw)
    torch.cuda.synchronize()
    okw = {"topk": kw.get("topk", 0), "tau": kw.get("threshold", 0.0), "rho": kw.get("mass", 0.99)}
    lists, cut, st = oracle.dense_index(q, k, lse32.astype(np.float64), M, scale, stat, mode, **okw)
    assert int(rp[-1].item()) == nnz
    P.compare_lists(rp, col, range(rows), lists, cut, st, 700)


def test_cached_mask_end_to_end_from_gpu_dense_step():
    from video_dit_sparse_gb300 import binding as sa
    q, k, v = field(1, 3, 128, (5, 10, 20), (7, 10, 10), seed=5)
    qd, kd, vd = P.to_dev(q), P.to_dev(k), P.to_dev(v)
    _, lse_gpu = sa.sparse_attn_forward(qd, kd, vd, None, None, group_size=128)
    rp, col, nnz = sa.sparse_attn_build_index_dense(qd, kd, lse_gpu, "max", "threshold",
                                                    threshold=0.5 / 700, group_size=128)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(128)
    lse = oracle.dense_lse(q, k, scale)
    lists, cut, st = oracle.dense_index(q, k, lse, 128, scale, "max", "threshold", tau=0.5 / 700)
    P.compare_lists(rp, col, range(3 * 8), lists, cut, st, 700)
    # the sparse steps then run on the cached lists
    o, l2 = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    P.compare_units(q, k, v, 128, rp.cpu().numpy(), col.cpu().numpy(), np.arange(24), o, l2)


def random_lists(rows, Nk, seed, sizes):
    rng = np.random.default_rng(seed)
    return [np.sort(rng.choice(Nk, size=min(int(sizes[r % len(sizes)]), Nk), replace=False)).astype(np.int32)
            for r in range(rows)]


def delta_compare(got, ref_units, B, H, Nq, M, d):
    G = -(-Nq // M)
    g = got.view(B * H, Nq, d).double().cpu().numpy()
    ref = ref_units.reshape(B * H, G * M, d)[:, :Nq]
    err = np.abs(g - ref)
    assert err.max() <= P.O_MAX and err.mean() <= P.O_MEAN, (err.max(), err.mean())
    return err


@pytest.mark.parametrize("d,M,sign", [(128, 128, 1.0), (64, 192, -1.0), (128, 64, 1.0)])
def test_delta_matches_oracle(d, M, sign):
    from video_dit_sparse_gb300 import binding as sa
    q0, k, v = field(1, 2, d, (5, 10, 20), (7, 10, 10), seed=d + M + 7)
    scale = 1.0 / math.sqrt(d)
    # stale normaliser: the lse of an earlier step's queries
    rng = np.random.default_rng(1)
    q1 = I.f32_to_bf16_bits((I.bf16_bits_to_f32(q0) + 0.2 * rng.standard_normal(q0.shape)).astype(np.float32))
    lse0 = oracle.dense_lse(q0, k, scale).astype(np.float32)
    G = -(-1000 // M)
    lists = random_lists(2 * G, 700, seed=M, sizes=[0, 1, 129, 700, 64, 300, 511])
    rp, col = oracle.to_csr(lists)
    base = rng.standard_normal((1, 2, 1000, d)).astype(np.float32)
    out = sa.sparse_attn_forward_delta(P.to_dev(q1), P.to_dev(k), P.to_dev(v),
                                       torch.from_numpy(rp).cuda(), torch.from_numpy(col).cuda(),
                                       torch.from_numpy(lse0).cuda(), base=torch.from_numpy(base).cuda(),
                                       sign=sign, group_size=M)
    torch.cuda.synchronize()
    ref = oracle.forward_delta(q1, k, v, M, scale, rp, col, lse0.astype(np.float64),
                               base.astype(np.float64), sign)
    delta_compare(out, ref, 1, 2, 1000, M, d)
    # empty lists leave the base untouched, bit for bit
    for u, lst in enumerate(lists):
        if len(lst) == 0:
            h, g = u // G, u % G
            r0, r1 = g * M, min((g + 1) * M, 1000)
            assert torch.equal(out[0, h, r0:r1].cpu(), torch.from_numpy(base[0, h, r0:r1]))


def test_delta_cache_roundtrip_in_place_and_dense():
    from video_dit_sparse_gb300 import binding as sa
    q, k, v = field(1, 2, 128, (5, 10, 20), (7, 10, 10), seed=21)
    qd, kd, vd = P.to_dev(q), P.to_dev(k), P.to_dev(v)
    o_dense, lse = sa.sparse_attn_forward(qd, kd, vd, None, None, out_dtype=torch.float32)
    lists = random_lists(16, 700, seed=2, sizes=[70, 140, 200, 1])
    rp, col = oracle.to_csr(lists)
    rpd, cold = torch.from_numpy(rp).cuda(), torch.from_numpy(col).cuda()
    cache = sa.sparse_attn_forward_delta(qd, kd, vd, rpd, cold, lse, base=o_dense, sign=-1.0)
    back = cache.clone()
    sa.sparse_attn_forward_delta(qd, kd, vd, rpd, cold, lse, base=back, sign=1.0, out=back)
    torch.cuda.synchronize()
    assert (back - o_dense).abs().max().item() < 1e-5
    # every key with the dense normaliser and no base is dense attention
    full = sa.sparse_attn_forward_delta(qd, kd, vd, None, None, lse)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(128)
    rpf, colf = full_csr(16, 700)
    ref = oracle.forward_delta(q, k, v, 128, scale, rpf, colf, lse.double().cpu().numpy())
    delta_compare(full, ref, 1, 2, 1000, 128, 128)


def test_delta_rejects_overlap_and_bad_args():
    from video_dit_sparse_gb300 import binding as sa
    q, k, v = field(1, 1, 128, (2, 8, 8), seed=3)
    qd, kd, vd = P.to_dev(q), P.to_dev(k), P.to_dev(v)
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    base = torch.zeros(1, 1, 128, 128, dtype=torch.float32, device="cuda")
    flat = base.view(torch.bfloat16).view(-1)
    with pytest.raises(sa.SparseAttnError):  # bf16 output in place over an fp32 base
        sa.sparse_attn_forward_delta(qd, kd, vd, None, None, lse, base=base,
                                     out=flat[:128 * 128].view(1, 1, 128, 128))
    with pytest.raises(sa.SparseAttnError):  # output overlapping the base, 16 bytes on
        sa.sparse_attn_forward_delta(qd, kd, vd, None, None, lse, base=base,
                                     out=flat[8:8 + 128 * 128].view(1, 1, 128, 128))
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_forward_delta(qd, kd, vd, None, None, lse, sign=float("nan"))


@pytest.mark.parametrize("stat", ["max", "sum"])
def test_dense_builder_rejects_bad_args(stat):
    from video_dit_sparse_gb300 import binding as sa
    q, k, _ = field(1, 1, 128, (2, 8, 8), seed=3)
    qd, kd = P.to_dev(q), P.to_dev(k)
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_build_index_dense(qd, kd, lse, 7, "topk", topk=4)
    with pytest.raises(sa.SparseAttnError):  # threshold beyond the statistic's range
        sa.sparse_attn_build_index_dense(qd, kd, lse, stat, "threshold", threshold=1e4)
    # a host pointer for lse is refused before any launch
    p = sa.problem(qd, kd, 128)
    sel = sa.sa_select(sa.SA_SELECT_TOPK, 4, 0.0, 0.99)
    ws = torch.empty(sa.sparse_attn_build_index_workspace_size(p), dtype=torch.uint8, device="cuda")
    rp = torch.empty(2, dtype=torch.int64, device="cuda")
    col = torch.empty(4, dtype=torch.int32, device="cuda")
    host_lse = torch.zeros(1, 1, 128, dtype=torch.float32)
    st = sa.lib.sparse_attn_build_index_dense(
        sa.ctypes.byref(p), sa.ctypes.byref(sel), sa._STATS[stat], sa._ptr(qd), sa._ptr(kd),
        sa._ptr(host_lse), sa._ptr(rp), sa._ptr(col), 4, None, sa._ptr(ws), ws.numel(), None)
    assert st == sa.SA_ERR_INVALID_ARG


def test_cached_mask_69k_sampled():
    """The 69K-token workload: dense forward (the refresh step), cached mask
    with tau = 0.5/N, then the sparse forward on those lists; sampled query
    groups are checked by the oracle one by one."""
    from video_dit_sparse_gb300 import binding as sa
    w = I.preset("sweep69k_top20")
    x = P.cached_inputs("sweep69k_top20")
    qd, kd, vd = P.to_dev(x["q"]), P.to_dev(x["k"]), P.to_dev(x["v"])
    Nk = w.Nk
    o_d, lse = sa.sparse_attn_forward(qd, kd, vd, None, None, group_size=128, out_dtype=torch.float32)
    rp, col, nnz = sa.sparse_attn_build_index_dense(qd, kd, lse, "max", "threshold",
                                                    threshold=0.5 / Nk, group_size=128)
    o_s, lse_s = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = w.B * w.H * w.G
    units = np.sort(np.random.default_rng(5).choice(rows, size=4, replace=False)).astype(np.int64)
    # the dense step on the sampled groups
    lse_ref = oracle.dense_lse(x["q"], x["k"], w.scale, M=128, units=units)
    lse_all = lse.view(-1).cpu().numpy()
    for i, u in enumerate(units):
        h, g = u // w.G, u % w.G
        got = lse_all[h * w.Nq + g * 128: h * w.Nq + (g + 1) * 128]
        assert np.all(np.abs(got - lse_ref[i]) <= 1e-3 * np.maximum(np.abs(lse_ref[i]), 1.0))
    # the oracle's statistic needs lse for every row of the group: place the sampled rows
    lse_full = np.zeros((w.B, w.H, w.Nq))
    for i, u in enumerate(units):
        h, g = u // w.G, u % w.G
        lse_full[0, h, g * 128:(g + 1) * 128] = lse_ref[i]
    lists, cut, st = oracle.dense_index(x["q"], x["k"], lse_full, 128, w.scale, "max", "threshold",
                                        tau=0.5 / Nk, units=units)
    P.compare_lists(rp, col, units, lists, cut, st, Nk)
    density = nnz / (rows * Nk)
    assert 0.0 < density < 1.0
    P.compare_units(x["q"], x["k"], x["v"], 128, rp.cpu().numpy(), col.cpu().numpy(), units, o_s, lse_s)


def test_colsum_delta_chunk192_sampled():
    """Chipmunk's dense step on the C = 192 chunk workload (69K tokens):
    dense forward, column-sum top 10 %, the cache (o minus the kept keys'
    terms) and the update that adds them back; sampled chunks checked by the
    oracle."""
    from video_dit_sparse_gb300 import binding as sa
    w = I.preset("colsum192_top10")
    x = P.cached_inputs("colsum192_top10")
    qd, kd, vd = P.to_dev(x["q"]), P.to_dev(x["k"]), P.to_dev(x["v"])
    o, lse = sa.sparse_attn_forward(qd, kd, vd, None, None, group_size=192, out_dtype=torch.float32)
    rp, col, nnz = sa.sparse_attn_build_index_dense(qd, kd, lse, "sum", "topk", topk=w.topk,
                                                    group_size=192)
    cache = sa.sparse_attn_forward_delta(qd, kd, vd, rp, col, lse, base=o, sign=-1.0, group_size=192)
    back = sa.sparse_attn_forward_delta(qd, kd, vd, rp, col, lse, base=cache, sign=1.0, group_size=192)
    torch.cuda.synchronize()
    rows = w.B * w.H * w.G
    assert nnz == rows * w.topk
    assert (back - o).abs().max().item() < 1e-4
    units = np.sort(np.random.default_rng(8).choice(rows, size=3, replace=False)).astype(np.int64)
    # the dense step of the sampled chunks: o and lse over every key
    uset = set(units.tolist())
    o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], 192, w.scale, *oracle.to_csr(
        [np.arange(w.Nk, dtype=np.int32) if u in uset else np.zeros(0, np.int32)
         for u in range(rows)]), units)
    lse_full = np.zeros((w.B, w.H, w.Nq))
    lse_all = lse.view(-1).cpu().numpy()
    for i, u in enumerate(units):
        h, g = u // w.G, u % w.G
        lse_full[0, h, g * 192:(g + 1) * 192] = lse_ref[i]
        got = lse_all[h * w.Nq + g * 192: h * w.Nq + (g + 1) * 192]
        assert np.all(np.abs(got - lse_ref[i]) <= 1e-3 * np.maximum(np.abs(lse_ref[i]), 1.0))
    lists, cut, st = oracle.dense_index(x["q"], x["k"], lse_full, 192, w.scale, "sum", "topk",
                                        topk=w.topk, units=units)
    P.compare_lists(rp, col, units, lists, cut, st, w.Nk)
    # the cache of the sampled chunks, on the GPU's lists and lse
    rpn, coln = rp.cpu().numpy(), col.cpu().numpy()
    lse_gpu = lse.double().cpu().numpy()
    d_ref = oracle.forward_delta(x["q"], x["k"], x["v"], 192, w.scale, rpn, coln, lse_gpu,
                                 None, -1.0, units)
    c_all = cache.view(w.B * w.H, w.Nq, w.d)
    for i, u in enumerate(units):
        h, g = u // w.G, u % w.G
        got = c_all[h, g * 192:(g + 1) * 192].double().cpu().numpy()
        err = np.abs(got - (o_ref[i] + d_ref[i]))
        assert err.max() <= P.O_MAX and err.mean() <= P.O_MEAN, (u, err.max(), err.mean())
