"""Pins for the oracle's dense-step lists and sparse-delta attention (no GPU).

Dense-step lists (FG-Attn review, cached mask: keep a slice when one of its
full-attention scores reaches tau_cached = 0.5/N; Chipmunk review, major
comment 2 / Alg. 4: top-k columns by column sums of the attention
probabilities) and sparse-delta attention (Chipmunk review, Eq. 1 with the
normalisation of an earlier step, Appendix B.2) are checked against:
  * a numpy/scipy brute force that materialises the dense probability matrix
    with scipy's softmax (no lse from the oracle involved);
  * closed forms: each probability row sums to 1, so the column sums of a
    group add up to its row count; single-query groups reduce both
    statistics to that query's own probabilities, so their top-k is the
    top-k of its logits; identical keys give p = 1/Nk everywhere;
    orthogonal one-hot keys make every query keep exactly its own key;
  * the delta's special cases: every key kept with the true normaliser is
    dense attention (torch SDPA); caching O minus the kept keys' terms and
    adding them back restores O; an empty list leaves the base.
"""
import math

import numpy as np
import pytest
import scipy.special as sp
import torch

from tests.test_oracle import bits, rand_qkv, random_lists, vals

SCALE = 0.25


def dense_probs(q, k, scale):
    Q, K = vals(q), vals(k)
    L = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    return sp.softmax(L, axis=-1), L


def brute_stats(q, k, M, scale, stat):
    P, _ = dense_probs(q, k, scale)
    B, H, Nq, Nk = P.shape
    G = -(-Nq // M)
    out = np.empty((B * H * G, Nk))
    for u in range(B * H * G):
        b, h, g = u // (H * G), (u // G) % H, u % G
        blk = P[b, h, g * M:min((g + 1) * M, Nq)]
        out[u] = blk.max(axis=0) if stat == "max" else blk.sum(axis=0)
    return out


@pytest.mark.parametrize("stat", ["max", "sum"])
@pytest.mark.parametrize("shape", [(1, 2, 100, 70, 16, 32), (2, 1, 64, 129, 8, 64)])
def test_column_stats_match_bruteforce(oracle_mod, stat, shape):
    B, H, Nq, Nk, d, M = shape
    q, k, _ = rand_qkv(B, H, Nq, Nk, d, seed=11)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    got = np.exp(oracle_mod.column_stats(q, k, lse, M, SCALE, stat))
    want = brute_stats(q, k, M, SCALE, stat)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=0)


def test_dense_lse_matches_scipy(oracle_mod):
    q, k, _ = rand_qkv(1, 3, 50, 90, 16, seed=2)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    _, L = dense_probs(q, k, SCALE)
    np.testing.assert_allclose(lse, sp.logsumexp(L, axis=-1), rtol=1e-13, atol=1e-13)


def test_column_sums_add_up_to_group_rows(oracle_mod):
    q, k, _ = rand_qkv(1, 2, 100, 77, 16, seed=3)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    tot = np.exp(oracle_mod.column_stats(q, k, lse, 32, SCALE, "sum")).sum(axis=1)
    np.testing.assert_allclose(tot, [32, 32, 32, 4] * 2, rtol=1e-12)


@pytest.mark.parametrize("stat", ["max", "sum"])
def test_single_query_groups_rank_by_logits(oracle_mod, stat):
    q, k, _ = rand_qkv(1, 1, 6, 40, 8, seed=4)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    lists, _, _ = oracle_mod.dense_index(q, k, lse, 1, SCALE, stat, "topk", topk=9)
    _, L = dense_probs(q, k, SCALE)
    for i in range(6):
        order = np.lexsort((np.arange(40), -L[0, 0, i]))
        np.testing.assert_array_equal(lists[i], np.sort(order[:9]))


def test_identical_keys_level(oracle_mod):
    Nk = 50
    rng = np.random.default_rng(5)
    q = bits(rng.standard_normal((1, 1, 64, 8)))
    k = bits(np.broadcast_to(rng.standard_normal(8), (1, 1, Nk, 8)))
    lse = oracle_mod.dense_lse(q, k, SCALE)
    st = np.exp(oracle_mod.column_stats(q, k, lse, 32, SCALE, "max"))
    np.testing.assert_allclose(st, 1.0 / Nk, rtol=1e-12)
    keep, _, _ = oracle_mod.dense_index(q, k, lse, 32, SCALE, "max", "threshold", tau=0.5 / Nk)
    assert all(len(x) == Nk for x in keep)
    none, cut, _ = oracle_mod.dense_index(q, k, lse, 32, SCALE, "max", "threshold", tau=2.0 / Nk)
    assert all(list(x) == [0] for x in none)  # nothing reaches tau: the top-ranked key
    assert np.allclose(cut, math.log(2.0 / Nk))


def test_one_hot_keys_keep_own_key(oracle_mod):
    # Nk = d orthogonal keys 16 e_j; query i points at key pi(i): its logit there is
    # 16 * 16 * 0.25 = 64, elsewhere 0, so p ~ 1 on its own key and ~e^-64 elsewhere.
    d = Nk = 16
    rng = np.random.default_rng(6)
    pi = rng.integers(0, Nk, size=48)
    q = bits((16.0 * np.eye(d)[pi])[None, None])
    k = bits((16.0 * np.eye(d))[None, None])
    lse = oracle_mod.dense_lse(q, k, SCALE)
    keep, _, _ = oracle_mod.dense_index(q, k, lse, 16, SCALE, "max", "threshold", tau=0.5 / Nk)
    for g in range(3):
        np.testing.assert_array_equal(keep[g], np.unique(pi[16 * g:16 * (g + 1)]))


def test_dense_mass_is_topk_of_its_size(oracle_mod):
    q, k, _ = rand_qkv(1, 2, 96, 80, 16, seed=7, std=1.5)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    mass, _, st = oracle_mod.dense_index(q, k, lse, 32, SCALE, "sum", "mass", rho=0.9)
    for r, lst in enumerate(mass):
        top, _ = oracle_mod.select(st[r:r + 1], "topk", topk=len(lst))
        np.testing.assert_array_equal(lst, top[0])
        s = np.exp(st[r])
        assert s[lst].sum() >= 0.9 * s.sum() - 1e-12
        if len(lst) > 1:
            smaller = np.sort(s)[::-1][:len(lst) - 1].sum()
            assert smaller < 0.9 * s.sum()


def test_rows_without_finite_lse_are_ignored(oracle_mod):
    q, k, _ = rand_qkv(1, 1, 32, 20, 8, seed=8)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    lse2 = lse.copy()
    lse2[0, 0, 5] = np.inf
    a = np.exp(oracle_mod.column_stats(q, k, lse2, 32, SCALE, "sum"))
    P, _ = dense_probs(q, k, SCALE)
    np.testing.assert_allclose(a[0], P[0, 0].sum(axis=0) - P[0, 0, 5], rtol=1e-11)


# ------------------------------------------------------------ sparse delta
def csr(lists):
    counts = np.array([len(x) for x in lists], dtype=np.int64)
    rp = np.zeros(len(lists) + 1, dtype=np.int64)
    np.cumsum(counts, out=rp[1:])
    return rp, (np.concatenate(lists).astype(np.int32) if lists else np.zeros(0, np.int32))


def to_bhnd(o_units, B, H, Nq, M):
    G = -(-Nq // M)
    d = o_units.shape[-1]
    return o_units.reshape(B, H, G * M, d)[:, :, :Nq]


def test_delta_all_keys_is_dense_attention(oracle_mod):
    B, H, Nq, Nk, d, M = 1, 2, 70, 50, 16, 32
    q, k, v = rand_qkv(B, H, Nq, Nk, d, seed=9)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    G = -(-Nq // M)
    rp, col = csr([np.arange(Nk, dtype=np.int32)] * (B * H * G))
    o = to_bhnd(oracle_mod.forward_delta(q, k, v, M, SCALE, rp, col, lse), B, H, Nq, M)
    tq, tk, tv = (torch.from_numpy(vals(x)) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=SCALE).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_delta_is_masked_full_softmax(oracle_mod):
    # stale normaliser: lse from the earlier step's queries, logits from the current ones
    B, H, Nq, Nk, d, M = 1, 2, 64, 40, 8, 32
    q0, k, v = rand_qkv(B, H, Nq, Nk, d, seed=10)
    q1 = bits(vals(q0) + 0.3 * np.random.default_rng(1).standard_normal(vals(q0).shape))
    lse0 = oracle_mod.dense_lse(q0, k, SCALE)
    G = Nq // M
    lists = random_lists(B * H * G, Nk, seed=12, lo=0, hi=25)
    rp, col = csr(lists)
    base = np.random.default_rng(2).standard_normal((B, H, Nq, d))
    o = to_bhnd(oracle_mod.forward_delta(q1, k, v, M, SCALE, rp, col, lse0, base, -1.0), B, H, Nq, M)
    L1 = SCALE * np.einsum("bhid,bhjd->bhij", vals(q1), vals(k))
    mask = np.zeros((B, H, Nq, Nk), dtype=bool)
    for u, lst in enumerate(lists):
        mask[u // (H * G), (u // G) % H, (u % G) * M:(u % G + 1) * M, lst] = True
    P = np.where(mask, np.exp(L1 - lse0[..., None]), 0.0)
    ref = base - np.einsum("bhij,bhjd->bhid", P, vals(v))
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_delta_cache_roundtrip_and_empty(oracle_mod):
    B, H, Nq, Nk, d, M = 1, 1, 96, 60, 16, 32
    q, k, v = rand_qkv(B, H, Nq, Nk, d, seed=13)
    lse = oracle_mod.dense_lse(q, k, SCALE)
    G = Nq // M
    rp_all, col_all = csr([np.arange(Nk, dtype=np.int32)] * G)
    dense = to_bhnd(oracle_mod.forward_delta(q, k, v, M, SCALE, rp_all, col_all, lse), B, H, Nq, M)
    lists = random_lists(G, Nk, seed=14, lo=1, hi=30)
    rp, col = csr(lists)
    cache = to_bhnd(oracle_mod.forward_delta(q, k, v, M, SCALE, rp, col, lse, dense, -1.0), B, H, Nq, M)
    back = to_bhnd(oracle_mod.forward_delta(q, k, v, M, SCALE, rp, col, lse, cache, 1.0), B, H, Nq, M)
    np.testing.assert_allclose(back, dense, rtol=0, atol=1e-13)
    rp0, col0 = csr([np.zeros(0, np.int32)] * G)
    same = to_bhnd(oracle_mod.forward_delta(q, k, v, M, SCALE, rp0, col0, lse, cache), B, H, Nq, M)
    np.testing.assert_array_equal(same, cache)
