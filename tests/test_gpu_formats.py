"""GPU checks of the mask-format conversions (through the C ABI): bit-packed
and block-sparse keep-masks give CSR lists identical to the oracle's (empty,
full and ragged rows, bits past Nk set), capacity reporting, and the forward
on block-sparse lists equals torch SDPA (fp32) with the dense block mask and
the oracle within the attention tolerances."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def check_csr(rp, col, nnz, lists):
    rpn, coln = rp.cpu().numpy(), col.cpu().numpy()
    ref_rp, ref_col = oracle.to_csr(lists)
    assert nnz == ref_rp[-1]
    np.testing.assert_array_equal(rpn, ref_rp)
    np.testing.assert_array_equal(coln[:nnz], ref_col)


@pytest.mark.parametrize("Nq,Nk,M,p", [(1000, 700, 128, 0.3), (256, 64, 64, 0.9), (384, 33, 192, 0.5),
                                       (128, 69120, 128, 0.2)])
def test_bitmask_to_csr(Nq, Nk, M, p):
    from video_dit_sparse_gb300 import binding as sa
    B, H = 1, 2
    rows = B * H * (-(-Nq // M))
    W = -(-Nk // 32)
    rng = np.random.default_rng(Nk)
    bitsarr = rng.random((rows, W * 32)) < p
    bitsarr[0, :] = False           # an empty row
    bitsarr[-1, :Nk] = True         # a full row (and garbage past Nk stays set)
    words = np.packbits(bitsarr, axis=1, bitorder="little").view("<u4").astype(np.uint32)
    rp, col, nnz = sa.sparse_attn_index_from_bitmask(torch.from_numpy(words.view(np.int32)).cuda(),
                                                     B=B, H=H, Nq=Nq, Nk=Nk, group_size=M)
    torch.cuda.synchronize()
    check_csr(rp, col, nnz, oracle.lists_from_bitmask(words, Nk))


@pytest.mark.parametrize("Nk,bk,M", [(700, 64, 128), (1000, 128, 192), (69120, 128, 128), (50, 7, 64)])
def test_block_mask_to_csr(Nk, bk, M):
    from video_dit_sparse_gb300 import binding as sa
    B, H, Nq = 1, 3, 640
    rows = B * H * (-(-Nq // M))
    nb = -(-Nk // bk)
    rng = np.random.default_rng(Nk + bk)
    blocks = ((rng.random((rows, nb)) < 0.35) * rng.integers(1, 256, (rows, nb))).astype(np.uint8)
    blocks[0] = 0
    blocks[-1] = 1
    rp, col, nnz = sa.sparse_attn_index_from_block_mask(torch.from_numpy(blocks).cuda(), bk, B=B, H=H,
                                                        Nq=Nq, Nk=Nk, group_size=M)
    torch.cuda.synchronize()
    check_csr(rp, col, nnz, oracle.lists_from_block_mask(blocks, Nk, bk))


def test_capacity_is_reported():
    from video_dit_sparse_gb300 import binding as sa
    blocks = np.ones((8, 10), dtype=np.uint8)
    with pytest.raises(sa.SparseAttnError) as e:
        sa.sparse_attn_index_from_block_mask(torch.from_numpy(blocks).cuda(), 64, B=1, H=1, Nq=1024,
                                             Nk=640, group_size=128, col_capacity=1000)
    assert e.value.status == sa.SA_ERR_CAPACITY


def test_block_sparse_forward_matches_sdpa_and_oracle():
    from video_dit_sparse_gb300 import binding as sa
    w = I.custom("t", 1, 2, 128, 128, (5, 10, 20), (7, 10, 10))  # Nq 1000, Nk 700
    x = I.make_inputs(w, 3)
    qd, kd, vd = P.to_dev(x["q"]), P.to_dev(x["k"]), P.to_dev(x["v"])
    G, bk = 8, 64
    nb = -(-700 // bk)
    rng = np.random.default_rng(9)
    blocks = (rng.random((2 * G, nb)) < 0.4).astype(np.uint8)
    blocks[:, 0] = 1
    rp, col, nnz = sa.sparse_attn_index_from_block_mask(torch.from_numpy(blocks).cuda(), bk, B=1, H=2,
                                                        Nq=1000, Nk=700, group_size=128)
    o, lse = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    P.compare_units(x["q"], x["k"], x["v"], 128, rp.cpu().numpy(), col.cpu().numpy(), np.arange(2 * G), o, lse)
    mask = np.repeat(np.repeat(blocks.reshape(1, 2, G, nb) != 0, 128, axis=2), bk, axis=3)[:, :, :1000, :700]
    ref = torch.nn.functional.scaled_dot_product_attention(qd.float(), kd.float(), vd.float(),
                                                           attn_mask=torch.from_numpy(mask).cuda())
    assert (o - ref).abs().max().item() < 2e-2
