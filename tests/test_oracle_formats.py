"""Pins for the oracle's index-format conversions (no GPU): the bit-packed
mask (Chipmunk review, "Bitpacked Sparsity Masks") against numpy's own
little-endian bit packing of a boolean mask, and the block-sparse mask
(FG-Attn review, Fig. 6) against a dense boolean mask built by numpy
repeat; then block-sparse attention through the slice oracle against torch
SDPA with the dense boolean block mask."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle import rand_qkv, vals


@pytest.mark.parametrize("rows,Nk,p", [(7, 100, 0.3), (3, 64, 0.0), (2, 33, 1.0), (5, 1000, 0.05)])
def test_bitmask_matches_numpy_packbits(rows, Nk, p):
    rng = np.random.default_rng(rows + Nk)
    dense = rng.random((rows, Nk)) < p
    W = -(-Nk // 32)
    padded = np.zeros((rows, W * 32), dtype=bool)
    padded[:, :Nk] = dense
    padded[:, Nk:] = rng.random((rows, W * 32 - Nk)) < 0.5  # bits past Nk must not count
    words = np.packbits(padded, axis=1, bitorder="little").view("<u4")
    lists = oracle.lists_from_bitmask(words, Nk)
    for r in range(rows):
        np.testing.assert_array_equal(lists[r], np.flatnonzero(dense[r]))


@pytest.mark.parametrize("rows,Nk,bk", [(4, 100, 16), (3, 128, 64), (6, 1000, 128)])
def test_block_mask_matches_numpy_repeat(rows, Nk, bk):
    rng = np.random.default_rng(Nk + bk)
    nb = -(-Nk // bk)
    blocks = (rng.random((rows, nb)) < 0.4).astype(np.uint8) * rng.integers(1, 255, (rows, nb)).astype(np.uint8)
    dense = np.repeat(blocks != 0, bk, axis=1)[:, :Nk]
    lists = oracle.lists_from_block_mask(blocks, Nk, bk)
    for r in range(rows):
        np.testing.assert_array_equal(lists[r], np.flatnonzero(dense[r]))


def test_block_sparse_attention_is_sdpa_with_block_mask():
    B, H, Nq, Nk, d, M, bk = 1, 2, 96, 80, 8, 32, 16
    q, k, v = rand_qkv(B, H, Nq, Nk, d, seed=3)
    G = Nq // M
    rng = np.random.default_rng(4)
    blocks = (rng.random((B * H * G, Nk // bk)) < 0.5).astype(np.uint8)
    blocks[:, 0] = 1  # no empty rows
    rp, col = oracle.to_csr(oracle.lists_from_block_mask(blocks, Nk, bk))
    o, lse = oracle.forward(q, k, v, M, 1 / math.sqrt(d), rp, col)
    mask = torch.from_numpy(np.repeat(np.repeat(blocks.reshape(B, H, G, -1) != 0, M, axis=2), bk, axis=3))
    tq, tk, tv = (torch.from_numpy(vals(x)) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).numpy()
    np.testing.assert_allclose(o.reshape(B, H, Nq, d), ref, rtol=1e-12, atol=1e-12)
