"""Pins for the fp64 CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * torch's scaled_dot_product_attention in float64 with a boolean mask (a
    library routine whose masked softmax is exactly the restricted softmax
    over kept keys), and without a mask when every key is kept;
  * a numpy brute force that materialises the dense score matrix with an
    explicit -inf mask;
  * closed forms (V = 1 gives O = 1, a single key gives o = v_j exactly,
    identical keys give the mean of the kept values) and invariants
    (permuting a list changes nothing);
  * the restricted-vs-masked distinction of the Chipmunk review (major
    comment 1): the two must differ on a partial key set;
  * a brute-force full sort (numpy lexsort) for every selection mode, and
    hand-worked selections whose answer is known by inspection;
  * the shape arithmetic printed on the DiT page (tests/golden).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from video_dit_sparse_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    return I.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def vals(b):
    return I.bf16_bits_to_f32(b).astype(np.float64)


def rand_qkv(B, H, Nq, Nk, d, seed=0, std=1.0):
    rng = np.random.default_rng(seed)
    q = bits(rng.standard_normal((B, H, Nq, d)) * std)
    k = bits(rng.standard_normal((B, H, Nk, d)) * std)
    v = bits(rng.standard_normal((B, H, Nk, d)))
    return q, k, v


def random_lists(rows, Nk, seed, lo=1, hi=None):
    rng = np.random.default_rng(seed)
    hi = hi or Nk
    out = []
    for _ in range(rows):
        n = int(rng.integers(lo, hi + 1))
        out.append(np.sort(rng.choice(Nk, size=n, replace=False)).astype(np.int32))
    return out


def sdpa_reference(q, k, v, M, lists):
    """torch SDPA (float64, CPU) with a boolean keep-mask per query group."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    mask = torch.zeros(B, H, Nq, Nk, dtype=torch.bool)
    for u, lst in enumerate(lists):
        b, h, g = u // (H * G), (u // G) % H, u % G
        mask[b, h, g * M:min((g + 1) * M, Nq), torch.from_numpy(lst.astype(np.int64))] = True
    tq, tk, tv = (torch.from_numpy(vals(x)) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    logits = (tq @ tk.transpose(-1, -2)) / math.sqrt(d)
    lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)
    return o.numpy(), lse.numpy()


def brute_dense(q, k, v, M, lists):
    """Dense scores with an explicit -inf mask, softmax row by row (numpy)."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = -(-Nq // M)
    qf, kf, vf = vals(q), vals(k), vals(v)
    o = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    for u, lst in enumerate(lists):
        b, h, g = u // (H * G), (u // G) % H, u % G
        keep = np.full(Nk, -np.inf)
        keep[lst] = 0.0
        for i in range(g * M, min((g + 1) * M, Nq)):
            row = np.array([np.dot(qf[b, h, i], kf[b, h, j]) for j in range(Nk)]) / math.sqrt(d)
            row = row + keep
            mx = row.max()
            w = np.exp(row - mx)
            o[b, h, i] = (w[:, None] * vf[b, h]).sum(0) / w.sum()
            lse[b, h, i] = mx + math.log(w.sum())
    return o, lse


def oracle_dense(oracle_mod, q, k, v, M, lists):
    B, H, Nq, d = q.shape
    row_ptr, col = oracle_mod.to_csr(lists)
    o, lse = oracle_mod.forward(q, k, v, M, 1.0 / math.sqrt(d), row_ptr, col)
    G = -(-Nq // M)
    o = o.reshape(B, H, G * M, d)[:, :, :Nq]
    lse = lse.reshape(B, H, G * M)[:, :, :Nq]
    return o, lse


# ------------------------------------------------------------------ forward
@pytest.mark.parametrize("B,H,Nq,Nk,d,M", [(1, 2, 96, 80, 16, 32), (2, 1, 70, 50, 8, 16),
                                           (1, 1, 128, 200, 64, 128)])
def test_forward_matches_torch_sdpa_with_mask(oracle_mod, B, H, Nq, Nk, d, M):
    q, k, v = rand_qkv(B, H, Nq, Nk, d, seed=Nq + d)
    G = -(-Nq // M)
    lists = random_lists(B * H * G, Nk, seed=7)
    o, lse = oracle_dense(oracle_mod, q, k, v, M, lists)
    o_ref, lse_ref = sdpa_reference(q, k, v, M, lists)
    assert np.abs(o - o_ref).max() < 1e-12
    assert np.abs(lse - lse_ref).max() < 1e-12


def test_forward_matches_bruteforce_dense_mask(oracle_mod):
    q, k, v = rand_qkv(1, 2, 40, 24, 8, seed=3, std=2.0)
    lists = random_lists(2 * 3, 24, seed=11)  # M=16 -> G=3, ragged last group
    o, lse = oracle_dense(oracle_mod, q, k, v, 16, lists)
    o_b, lse_b = brute_dense(q, k, v, 16, lists)
    assert np.abs(o - o_b).max() < 1e-12
    assert np.abs(lse - lse_b).max() < 1e-12


def test_full_keep_equals_dense_sdpa(oracle_mod):
    q, k, v = rand_qkv(1, 2, 64, 48, 32, seed=5)
    lists = [np.arange(48, dtype=np.int32)] * 4
    o, lse = oracle_dense(oracle_mod, q, k, v, 32, lists)
    tq, tk, tv = (torch.from_numpy(vals(x)) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).numpy()
    assert np.abs(o - ref).max() < 1e-12
    ref_lse = torch.logsumexp((tq @ tk.transpose(-1, -2)) / math.sqrt(32), -1).numpy()
    assert np.abs(lse - ref_lse).max() < 1e-12


def test_rows_sum_to_one(oracle_mod):
    """V = 1 everywhere: o_i = sum_j p_ij, which must be exactly 1."""
    q, k, _ = rand_qkv(1, 1, 32, 40, 16, seed=9, std=3.0)
    v = bits(np.ones((1, 1, 40, 16)))
    lists = random_lists(2, 40, seed=2)
    o, _ = oracle_dense(oracle_mod, q, k, v, 16, lists)
    assert np.abs(o - 1.0).max() < 1e-14


def test_single_key_is_exact(oracle_mod):
    q, k, v = rand_qkv(1, 1, 16, 30, 8, seed=4)
    lists = [np.array([17], dtype=np.int32)]
    o, lse = oracle_dense(oracle_mod, q, k, v, 16, lists)
    vf, qf, kf = vals(v), vals(q), vals(k)
    assert np.array_equal(o[0, 0], np.broadcast_to(vf[0, 0, 17], (16, 8)))
    expect = (qf[0, 0] @ kf[0, 0, 17]) / math.sqrt(8)
    assert np.abs(lse[0, 0] - expect).max() < 1e-14


def test_identical_keys_average_values(oracle_mod):
    q, _, v = rand_qkv(1, 1, 16, 12, 8, seed=6)
    k = bits(np.tile(np.random.default_rng(1).standard_normal(8), (1, 1, 12, 1)))
    lst = np.array([0, 3, 4, 9, 11], dtype=np.int32)
    o, lse = oracle_dense(oracle_mod, q, k, v, 16, [lst])
    assert np.abs(o[0, 0] - vals(v)[0, 0, lst].mean(0)).max() < 1e-14
    # lse = l + ln(5) when all five logits are equal
    l0 = (vals(q)[0, 0] @ vals(k)[0, 0, 0]) / math.sqrt(8)
    assert np.abs(lse[0, 0] - (l0 + math.log(5))).max() < 1e-12


def test_permuted_list_same_output(oracle_mod):
    q, k, v = rand_qkv(1, 1, 32, 64, 16, seed=8)
    lst = np.sort(np.random.default_rng(3).choice(64, 20, replace=False)).astype(np.int32)
    perm = np.random.default_rng(4).permutation(lst).astype(np.int32)
    o1, l1 = oracle_dense(oracle_mod, q, k, v, 32, [lst])
    o2, l2 = oracle_dense(oracle_mod, q, k, v, 32, [perm])
    assert np.abs(o1 - o2).max() < 1e-13 and np.abs(l1 - l2).max() < 1e-13


def test_restricted_differs_from_masked_full_softmax(oracle_mod):
    """Restricted softmax (renormalised over kept keys) vs the masked full
    softmax of Chipmunk's Eq. 1: on a partial set they must differ, and the
    oracle must equal the restricted form."""
    q, k, v = rand_qkv(1, 1, 16, 32, 8, seed=10)
    lst = np.arange(0, 32, 3, dtype=np.int32)
    o, _ = oracle_dense(oracle_mod, q, k, v, 16, [lst])
    qf, kf, vf = vals(q)[0, 0], vals(k)[0, 0], vals(v)[0, 0]
    s = qf @ kf.T / math.sqrt(8)
    p_full = np.exp(s - s.max(1, keepdims=True))
    p_full /= p_full.sum(1, keepdims=True)
    masked = p_full[:, lst] @ vf[lst]
    restricted = (p_full[:, lst] / p_full[:, lst].sum(1, keepdims=True)) @ vf[lst]
    assert np.abs(o[0, 0] - restricted).max() < 1e-12
    assert np.abs(o[0, 0] - masked).max() > 1e-3


def test_empty_list_and_ragged_group(oracle_mod):
    q, k, v = rand_qkv(1, 1, 20, 10, 8, seed=12)
    lists = [np.zeros(0, dtype=np.int32), np.array([1, 2], dtype=np.int32)]
    row_ptr, col = oracle_mod.to_csr(lists)
    o, lse = oracle_mod.forward(q, k, v, 16, 1 / math.sqrt(8), row_ptr, col)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(o[1, 4:] == 0)  # rows 20..31 of group 1 do not exist
    ref, ref_lse = sdpa_reference(q, k, v, 16, [np.arange(10, dtype=np.int32), lists[1]])
    assert np.abs(o[1, :4] - ref[0, 0, 16:20]).max() < 1e-12


# ------------------------------------------------------------- mean / score
def test_mean_query_and_scores(oracle_mod):
    q, k, _ = rand_qkv(2, 2, 50, 30, 16, seed=13)
    M = 16
    qbar = oracle_mod.mean_query(q, M)
    qf = vals(q)
    G = 4
    ref = np.stack([qf[b, h, g * M:min((g + 1) * M, 50)].mean(0)
                    for b in range(2) for h in range(2) for g in range(G)])
    assert np.abs(qbar - ref).max() < 1e-15
    sc = oracle_mod.group_scores(q, k, M, 0.25)
    kf = vals(k)
    ref_sc = np.stack([0.25 * kf[u // (2 * G), (u // G) % 2] @ ref[u] for u in range(16)])
    assert np.abs(sc - ref_sc).max() < 1e-13
    # constant rows: the mean is that row exactly
    qc = bits(np.tile(np.arange(16, dtype=np.float32) / 4, (1, 1, 32, 1)))
    assert np.array_equal(oracle_mod.mean_query(qc, 16)[0], np.arange(16) / 4)


# ------------------------------------------------------------------ select
def brute_select(scores, mode, topk=0, tau=0.0, rho=0.99):
    out, cuts = [], []
    for row in scores:
        order = np.lexsort((np.arange(row.size), -row))  # score desc, index asc
        if mode == "topk":
            n = max(1, min(topk, row.size))
            cut = row[order[n - 1]]
        else:
            m = row.max()
            lse = m + math.log(np.exp(row - m).sum())
            p = np.exp(row[order] - lse)
            if mode == "threshold":
                n = max(1, int((p >= tau).sum()))
                cut = math.log(tau) if tau > 0 else -math.inf
                cut = cut + lse
            else:
                c = np.cumsum(p)
                hit = np.nonzero(c >= rho)[0]
                n = int(hit[0]) + 1 if hit.size else row.size
                cut = row[order[n - 1]]
        out.append(np.sort(order[:n]).astype(np.int32))
        cuts.append(cut)
    return out, np.array(cuts)


@pytest.mark.parametrize("mode,kw", [("topk", {"topk": 7}), ("topk", {"topk": 1}),
                                      ("threshold", {"tau": 0.02}), ("mass", {"rho": 0.9}),
                                      ("mass", {"rho": 0.5})])
def test_select_matches_bruteforce_sort(oracle_mod, mode, kw):
    rng = np.random.default_rng(21)
    scores = rng.standard_normal((40, 37)) * 2
    scores[::3, 5:9] = 1.25  # exact ties
    lists, cut = oracle_mod.select(scores, mode, **kw)
    ref, ref_cut = brute_select(scores, mode, **kw)
    for a, b in zip(lists, ref):
        assert np.array_equal(a, b)
    assert np.allclose(cut, ref_cut, rtol=0, atol=1e-12)


def test_select_worked_examples(oracle_mod):
    s = np.array([[1.0, 3.0, 2.0, 3.0]])
    assert oracle_mod.select(s, "topk", topk=2)[0][0].tolist() == [1, 3]
    assert oracle_mod.select(s, "topk", topk=1)[0][0].tolist() == [1]  # tie -> lower index
    assert oracle_mod.select(s, "topk", topk=3)[0][0].tolist() == [1, 2, 3]
    # probabilities 0.5, 0.3, 0.2 in that order of keys 2, 0, 1
    pm = np.log(np.array([[0.3, 0.2, 0.5]]))
    assert oracle_mod.select(pm, "mass", rho=0.75)[0][0].tolist() == [0, 2]
    assert oracle_mod.select(pm, "mass", rho=0.45)[0][0].tolist() == [2]
    assert oracle_mod.select(pm, "mass", rho=0.99)[0][0].tolist() == [0, 1, 2]
    assert oracle_mod.select(pm, "threshold", tau=0.25)[0][0].tolist() == [0, 2]
    assert oracle_mod.select(pm, "threshold", tau=0.9)[0][0].tolist() == [2]  # keeps >= 1


def test_select_closed_forms(oracle_mod):
    rng = np.random.default_rng(5)
    sc = rng.standard_normal((6, 50))
    allk = [np.arange(50)] * 6
    for lists in (oracle_mod.select(sc, "topk", topk=50)[0],
                  oracle_mod.select(sc, "threshold", tau=0.0)[0],
                  oracle_mod.select(sc, "mass", rho=1.0)[0]):
        assert all(np.array_equal(a, b) for a, b in zip(lists, allk))
    # TOPK(k) is contained in TOPK(k+1); MASS set equals TOPK of its size
    prev = None
    for kk in range(1, 12):
        cur = oracle_mod.select(sc, "topk", topk=kk)[0]
        if prev is not None:
            assert all(set(a) <= set(b) and len(b) == len(a) + 1 for a, b in zip(prev, cur))
        prev = cur
    mass = oracle_mod.select(sc, "mass", rho=0.8)[0]
    for r, lst in enumerate(mass):
        t = oracle_mod.select(sc[r:r + 1], "topk", topk=len(lst))[0][0]
        assert np.array_equal(t, lst)


def test_threshold_cut_is_log_tau_plus_lse(oracle_mod):
    sc = np.random.default_rng(8).standard_normal((3, 20))
    _, cut = oracle_mod.select(sc, "threshold", tau=0.03)
    lse = np.log(np.exp(sc).sum(1))
    assert np.abs(cut - (math.log(0.03) + lse)).max() < 1e-12


# ------------------------------------------------------------------ shapes
def test_rolling_window_shapes_match_dit_page():
    g = json.load(open(os.path.join(GOLDEN, "dit_page_shapes.json")))
    w = I.preset("rollingkv_mass99")
    assert g["tokens_per_latent_frame"] * g["latent_frames_per_chunk"] == g["tokens_per_chunk"]
    assert w.Nq == g["tokens_per_chunk"]
    assert w.Nk == g["kv_window_tokens"] == g["kv_window_chunks"] * g["tokens_per_chunk"]
    assert w.G == g["query_tiles_per_head"]
    assert w.Nk // g["tile_keys"] == g["key_pages_per_head"]
    assert w.G * (w.Nk // 128) == g["tiles_per_head"]
    assert g["tiles_per_head"] * g["heads"] == g["tiles_per_call_24_heads"]
    assert round(w.Nq * w.Nk * 2 / 1e6) == g["p_matrix_fp16_mb_approx"]
    # the page counts 1 MB = 1000 KB here: 148 x 256 KB = 37,888 KB
    assert round(g["tmem_sms"] * g["tmem_kb_per_sm"] / 1000, 1) == g["tmem_total_mb_approx"]


def test_presets_tile_their_grids():
    assert I.preset("wan16k_top20").G == 128 and I.preset("wan16k_top20").topk == 3277
    assert I.preset("chunk192_top10").G == 360 and I.preset("chunk192_top10").topk == 6912
    assert I.preset("sweep69k_top20").G == 540 and I.preset("sweep69k_top20").topk == 13824
    for name in ("wan16k_top20", "chunk192_top10", "sweep69k_top5"):
        w = I.preset(name)
        p = I.voxel_perm(w.grid_q, w.voxel)
        assert np.array_equal(np.sort(p), np.arange(w.Nq))
        # every group of M consecutive tokens is one whole voxel set
        vt, vh, vw = w.voxel
        T, Hh, W = w.grid_q
        t, h, x = np.unravel_index(p, (T, Hh, W))
        vox = (t // vt) * (Hh // vh) * (W // vw) + (h // vh) * (W // vw) + x // vw
        per_group = vox.reshape(-1, w.group)
        if w.group == vt * vh * vw:
            assert np.all(per_group == per_group[:, :1])


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.140625], dtype=np.float32)
    b = I.f32_to_bf16_bits(x)
    assert I.bf16_bits_to_f32(b).tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 3.140625]
    t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, t)
