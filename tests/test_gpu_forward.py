"""GPU parity of sparse_attn_forward against the fp64 oracle (through the
C ABI), with index lists given by the test so that the forward is checked on
its own: random lists of every length (empty, single key, partial tiles,
several tiles, every key), ragged query groups, d in {64, 128} and group
sizes 64/128/160/192/224/256."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def random_lists(rows, Nk, seed, sizes=None):
    rng = np.random.default_rng(seed)
    out = []
    for r in range(rows):
        n = int(sizes[r % len(sizes)]) if sizes is not None else int(rng.integers(0, Nk + 1))
        n = min(n, Nk)
        out.append(np.sort(rng.choice(Nk, size=n, replace=False)).astype(np.int32))
    return out


def run_forward(q, k, v, M, row_ptr, col, **kw):
    from video_dit_sparse_gb300 import binding as sa
    qd, kd, vd = P.to_dev(q), P.to_dev(k), P.to_dev(v)
    rp = torch.from_numpy(row_ptr).cuda()
    cd = torch.from_numpy(col if col.size else np.zeros(1, np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw.setdefault("out_dtype", torch.float32)
    o, lse = sa.sparse_attn_forward(qd, kd, vd, rp, cd, group_size=M, nnz=col.size,
                                    status=status, **kw)
    torch.cuda.synchronize()
    return o, lse, int(status.item())


def field(B, H, d, grid_q, grid_k=None, seed=0):
    w = I.custom("t", B, H, d, 128, grid_q, grid_k)
    x = I.make_inputs(w, seed)
    return x["q"], x["k"], x["v"]


def test_tiny_preset_full_compare():
    w = I.preset("tiny")
    x = I.make_inputs(w, 0)
    o, lse, st = run_forward(x["q"], x["k"], x["v"], w.group, x["row_ptr"], x["col_idx"])
    assert st == 0
    stats = P.compare_units(x["q"], x["k"], x["v"], w.group, x["row_ptr"], x["col_idx"],
                            np.arange(w.G), o, lse)
    assert stats["o_max"] < 2e-2


@pytest.mark.parametrize("d,M", [(128, 128), (64, 128), (128, 192), (64, 192), (128, 64),
                                 (128, 256), (128, 160), (64, 224)])
def test_random_lists_every_length(d, M):
    # Nq = 1000 -> a ragged last group; Nk = 700 -> 6 key tiles, ragged tail
    q, k, v = field(1, 2, d, (5, 10, 20), (7, 10, 10), seed=d + M)
    G = -(-1000 // M)
    rows = 2 * G
    sizes = [0, 1, 2, 127, 128, 129, 300, 700, 64, 200, 511, 513]
    lists = random_lists(rows, 700, seed=M, sizes=sizes)
    row_ptr, col = oracle.to_csr(lists)
    o, lse, st = run_forward(q, k, v, M, row_ptr, col)
    assert st == 0
    P.compare_units(q, k, v, M, row_ptr, col, np.arange(rows), o, lse)


@pytest.mark.parametrize("d,M,scale", [(128, 128, -1.0 / math.sqrt(128)), (64, 192, -0.3),
                                       (128, 128, 0.05)])
def test_scale_of_either_sign(d, M, scale):
    """Any finite non-zero scale: a negative one negates every score (the
    softmax then favours the smallest q.k), and the oracle takes the same
    scale; lists of every length, ragged groups and tiles."""
    q, k, v = field(1, 2, d, (5, 10, 20), (7, 10, 10), seed=29)
    G = -(-1000 // M)
    rows = 2 * G
    lists = random_lists(rows, 700, seed=31, sizes=[1, 127, 128, 129, 300, 700, 513])
    row_ptr, col = oracle.to_csr(lists)
    o, lse, st = run_forward(q, k, v, M, row_ptr, col, scale=scale)
    assert st == 0
    P.compare_units(q, k, v, M, row_ptr, col, np.arange(rows), o, lse, scale=scale)
    # the bf16 launch is the same result rounded
    o16, _, _ = run_forward(q, k, v, M, row_ptr, col, scale=scale, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o.to(torch.bfloat16))


@pytest.mark.parametrize("d,M", [(128, 128), (64, 192)])
def test_bf16_output_is_rounded_fp32_output(d, M):
    q, k, v = field(1, 2, d, (5, 10, 20), (7, 10, 10), seed=11)
    G = -(-1000 // M)
    lists = random_lists(2 * G, 700, seed=4, sizes=[0, 5, 129, 700, 300])
    row_ptr, col = oracle.to_csr(lists)
    o32, l32, _ = run_forward(q, k, v, M, row_ptr, col)
    o16, l16, _ = run_forward(q, k, v, M, row_ptr, col, out_dtype=torch.bfloat16)
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)


def test_full_keep_equals_dense_attention():
    q, k, v = field(1, 2, 128, (4, 16, 16))  # 1024 tokens
    lists = [np.arange(1024, dtype=np.int32)] * 16
    row_ptr, col = oracle.to_csr(lists)
    o, lse, st = run_forward(q, k, v, 128, row_ptr, col)
    assert st == 0
    P.compare_units(q, k, v, 128, row_ptr, col, np.arange(16), o, lse)
    ref = torch.nn.functional.scaled_dot_product_attention(P.to_dev(q).float(), P.to_dev(k).float(),
                                                           P.to_dev(v).float())
    assert (o.float() - ref).abs().max().item() < 2e-2


def test_large_logits_rescale_path():
    """Scores that grow along the list force the running-max rescale."""
    rng = np.random.default_rng(3)
    Nk, d = 1024, 128
    base = rng.standard_normal((1, 1, 128, d)).astype(np.float32)
    q = I.f32_to_bf16_bits(base * 2.0)
    kk = rng.standard_normal((1, 1, Nk, d)).astype(np.float32)
    kk *= np.linspace(0.1, 4.0, Nk, dtype=np.float32)[None, None, :, None]
    k = I.f32_to_bf16_bits(kk)
    v = I.f32_to_bf16_bits(rng.standard_normal((1, 1, Nk, d)).astype(np.float32))
    row_ptr, col = oracle.to_csr([np.arange(Nk, dtype=np.int32)])
    o, lse, st = run_forward(q, k, v, 128, row_ptr, col)
    assert st == 0
    P.compare_units(q, k, v, 128, row_ptr, col, [0], o, lse)


@pytest.mark.parametrize("case", ["growing16", "late_outlier", "falling"])
def test_running_max_raised_by_a_later_tile(case):
    """A later tile whose scores sit far above the running max (set by the
    unit's first tile) makes its P against that max sum past the lazy-rescale
    bound: the kernel then takes the tile's max, rescales O and the sums and
    recomputes P.  Falling scores never raise it."""
    rng = np.random.default_rng(11)
    Nk, d = 1024, 128
    base = rng.standard_normal(d).astype(np.float32)
    q32 = (base[None, None, None, :] + 0.3 * rng.standard_normal((1, 1, 128, d))).astype(np.float32)
    k32 = rng.standard_normal((1, 1, Nk, d)).astype(np.float32)
    if case == "growing16":
        k32 *= np.linspace(0.05, 16.0, Nk, dtype=np.float32)[None, None, :, None]
    elif case == "late_outlier":
        k32[0, 0, 1000] = 3.0 * base  # score ~ 3 |base|^2 / sqrt(d) above every other key's
    else:
        k32 *= np.linspace(8.0, 0.05, Nk, dtype=np.float32)[None, None, :, None]
    q, k = I.f32_to_bf16_bits(q32), I.f32_to_bf16_bits(k32)
    v = I.f32_to_bf16_bits(rng.standard_normal((1, 1, Nk, d)).astype(np.float32))
    row_ptr, col = oracle.to_csr([np.arange(Nk, dtype=np.int32)])
    o, lse, st = run_forward(q, k, v, 128, row_ptr, col)
    assert st == 0
    P.compare_units(q, k, v, 128, row_ptr, col, [0], o, lse)


def test_permuted_and_duplicate_free_lists_match():
    q, k, v = field(1, 1, 128, (2, 8, 16), (4, 8, 16))
    rng = np.random.default_rng(5)
    lists = [np.sort(rng.choice(512, 300, replace=False)).astype(np.int32) for _ in range(2)]
    row_ptr, col = oracle.to_csr(lists)
    perm = [rng.permutation(x).astype(np.int32) for x in lists]
    _, col_p = oracle.to_csr(perm)
    o1, l1, _ = run_forward(q, k, v, 128, row_ptr, col)
    o2, l2, _ = run_forward(q, k, v, 128, row_ptr, col_p)
    assert (o1.float() - o2.float()).abs().max().item() < 1e-2
    assert (l1 - l2).abs().max().item() < 1e-4


def test_output_rows_sum_to_one_with_unit_values():
    q, k, _ = field(1, 1, 128, (2, 8, 16), (4, 8, 16))
    v = I.f32_to_bf16_bits(np.ones((1, 1, 512, 128), np.float32))
    lists = random_lists(2, 512, 9, sizes=[77, 400])
    row_ptr, col = oracle.to_csr(lists)
    o, _, _ = run_forward(q, k, v, 128, row_ptr, col)
    assert (o.float() - 1.0).abs().max().item() <= 2 ** -7


def test_empty_lists_give_zero_and_neg_inf():
    q, k, v = field(1, 1, 128, (2, 8, 16))
    row_ptr = np.zeros(3, dtype=np.int64)
    o, lse, st = run_forward(q, k, v, 128, row_ptr, np.zeros(0, np.int32))
    assert st == 0
    assert o.abs().max().item() == 0 and torch.isneginf(lse).all()


def test_bad_input_sets_status_without_fault():
    q, k, v = field(1, 1, 128, (2, 8, 16))
    from video_dit_sparse_gb300 import binding as sa
    # out-of-range index, negative index, row_ptr past nnz
    col = np.array([0, 5, 9999, -3, 7], dtype=np.int32)
    row_ptr = np.array([0, 3, 5], dtype=np.int64)
    _, _, st = run_forward(q, k, v, 128, row_ptr, col)
    assert st & sa.SA_DEVERR_INDEX
    row_ptr = np.array([0, 3, 9], dtype=np.int64)
    o, lse, st = run_forward(q, k, v, 128, row_ptr, col)
    assert st & sa.SA_DEVERR_ROW_PTR
    assert torch.isneginf(lse[0, 0, 128:]).all()  # the malformed unit is treated as empty


def test_validate_index():
    from video_dit_sparse_gb300 import binding as sa
    rp = torch.tensor([0, 3, 5], dtype=torch.int64, device="cuda")
    good = torch.tensor([1, 4, 9, 0, 2], dtype=torch.int32, device="cuda")
    kw = dict(B=1, H=1, Nq=256, Nk=16)
    assert sa.sparse_attn_validate_index(rp, good, **kw) == sa.SA_OK
    for bad in ([1, 4, 4, 0, 2], [1, 4, 16, 0, 2], [3, 1, 9, 0, 2], [1, 4, 9, -1, 2]):
        t = torch.tensor(bad, dtype=torch.int32, device="cuda")
        assert sa.sparse_attn_validate_index(rp, t, **kw) == sa.SA_ERR_BAD_INDEX
    rp_bad = torch.tensor([0, 6, 5], dtype=torch.int64, device="cuda")
    assert sa.sparse_attn_validate_index(rp_bad, good, **kw) == sa.SA_ERR_BAD_INDEX


def test_rejects_host_and_short_buffers():
    from video_dit_sparse_gb300 import binding as sa
    q = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    rp = torch.tensor([0, 1, 2], dtype=torch.int64, device="cuda")
    col = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(sa.SparseAttnError):  # nnz larger than col_idx's allocation
        sa.sparse_attn_forward(q, q, q, rp, col[:1], nnz=1 << 20)
    p = sa.problem(q, q, 128)
    host = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16)
    st = sa.lib.sparse_attn_forward(sa.ctypes.byref(p), sa._ptr(host), sa._ptr(q), sa._ptr(q),
                                    sa._ptr(rp), sa._ptr(col), 2, sa._ptr(q), None, None, None)
    assert st == sa.SA_ERR_INVALID_ARG
