"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (a dropped
term, a wrong sign or index, an off-by-one), compiles it on the CPU, swaps
it in for the real library and checks that at least one pin in
``test_oracle.py`` fails.  Nothing here touches a GPU.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins
from tests import test_oracle_dense as dpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "forward drops the scale": ("logits[j] = c->scale * dot;", "logits[j] = dot;"),
    "forward exp sign flipped": ("double p = exp(logits[j] - m);", "double p = exp(m - logits[j]);"),
    "lse drops the max": ("lse_unit[r] = m + log(sum);", "lse_unit[r] = log(sum);"),
    "key row ignores the list": ("c->k + (bh * s->Nk + list[j]) * d;\n      double dot = 0.0;\n"
                                 "      for (int64_t e = 0; e < d; ++e) dot += qrow[e] * bf16_value(krow[e]);\n"
                                 "      logits[j]",
                                 "c->k + (bh * s->Nk + j) * d;\n      double dot = 0.0;\n"
                                 "      for (int64_t e = 0; e < d; ++e) dot += qrow[e] * bf16_value(krow[e]);\n"
                                 "      logits[j]"),
    "delta key row ignores the list": ("c->k + (bh * s->Nk + list[j]) * d;\n      double dot = 0.0;\n"
                                       "      for (int64_t e = 0; e < d; ++e) dot += qrow[e] * bf16_value(krow[e]);\n"
                                       "      double p = exp(c->scale * dot - lse);",
                                       "c->k + (bh * s->Nk + j) * d;\n      double dot = 0.0;\n"
                                       "      for (int64_t e = 0; e < d; ++e) dot += qrow[e] * bf16_value(krow[e]);\n"
                                       "      double p = exp(c->scale * dot - lse);"),
    "value row ignores the list": ("c->v + (bh * s->Nk + list[j]) * d;\n      for (int64_t e = 0; e < d; ++e) orow[e] += p",
                                   "c->v + (bh * s->Nk + j) * d;\n      for (int64_t e = 0; e < d; ++e) orow[e] += p"),
    "delta value row ignores the list": ("c->v + (bh * s->Nk + list[j]) * d;\n      for (int64_t e = 0; e < d; ++e) orow[e] += c->sign",
                                         "c->v + (bh * s->Nk + j) * d;\n      for (int64_t e = 0; e < d; ++e) orow[e] += c->sign"),
    "output not normalised": ("for (int64_t e = 0; e < d; ++e) orow[e] /= sum;", ""),
    "mean divides by M": ("double n = (double)(r1 - r0);", "double n = (double)s->M;"),
    "score drops the scale": ("dst[j] = c->scale * dot;", "dst[j] = dot;"),
    "ties favour higher index": ("return (x->index > y->index) - (x->index < y->index);",
                                 "return (x->index < y->index) - (x->index > y->index);"),
    "ranking ascending": ("if (x->score > y->score) return -1;\n  if (x->score < y->score) return 1;",
                          "if (x->score < y->score) return -1;\n  if (x->score > y->score) return 1;"),
    "topk off by one": ("n = c->topk < Nk ? c->topk : Nk;", "n = c->topk < Nk ? c->topk - 1 : Nk;"),
    "mass stops one late": ("++n;\n        if (acc >= c->rho) break;",
                            "if (acc >= c->rho) break;\n        ++n;"),
    "select lse drops the max": ("double lse = m + log(z);", "double lse = log(z);"),
    "query row offset wrong": ("c->q + (bh * s->Nq + qi) * d;\n    for (int64_t e = 0; e < d; ++e) qrow[e] = bf16_value(qsrc[e]);\n    double m",
                               "c->q + (bh * s->Nq + r) * d;\n    for (int64_t e = 0; e < d; ++e) qrow[e] = bf16_value(qsrc[e]);\n    double m"),
    "delta query row offset wrong": ("c->q + (bh * s->Nq + qi) * d;\n    for (int64_t e = 0; e < d; ++e) qrow[e] = bf16_value(qsrc[e]);\n    for",
                                     "c->q + (bh * s->Nq + r) * d;\n    for (int64_t e = 0; e < d; ++e) qrow[e] = bf16_value(qsrc[e]);\n    for"),
    "column stat drops the lse": ("double p = exp(c->scale * dot - lse);\n      if (c->stat",
                                  "double p = exp(c->scale * dot);\n      if (c->stat"),
    "column max keeps the minimum": ("if (p > stat) stat = p;", "if (p < stat || stat == 0.0) stat = p;"),
    "column stat reads the wrong key": ("c->k + (bh * s->Nk + j) * d;", "c->k + (bh * s->Nk + (j + 1) % s->Nk) * d;"),
    "column stat lse row offset": ("double lse = c->lse[bh * s->Nq + r];",
                                   "double lse = c->lse[bh * s->Nq + r - r0];"),
    "level compares the log": ("exp(order[n].score) >= c->tau", "order[n].score >= c->tau"),
    "delta ignores the sign": ("orow[e] += c->sign * p * bf16_value(vrow[e]);",
                               "orow[e] += p * bf16_value(vrow[e]);"),
    "delta drops the base": ("orow[e] = c->base[(bh * s->Nq + qi) * d + e];", "orow[e] = 0.0;"),
    "delta drops the lse": ("double p = exp(c->scale * dot - lse);\n      const uint16_t* vrow",
                            "double p = exp(c->scale * dot);\n      const uint16_t* vrow"),
}

PINS = [
    lambda m: pins.test_forward_matches_torch_sdpa_with_mask(m, 2, 1, 70, 50, 8, 16),
    lambda m: pins.test_forward_matches_bruteforce_dense_mask(m),
    lambda m: pins.test_single_key_is_exact(m),
    lambda m: pins.test_mean_query_and_scores(m),
    lambda m: pins.test_select_worked_examples(m),
    lambda m: pins.test_select_matches_bruteforce_sort(m, "mass", {"rho": 0.9}),
    lambda m: pins.test_select_matches_bruteforce_sort(m, "threshold", {"tau": 0.02}),
    lambda m: pins.test_select_matches_bruteforce_sort(m, "topk", {"topk": 7}),
    lambda m: dpins.test_column_stats_match_bruteforce(m, "max", (1, 2, 100, 70, 16, 32)),
    lambda m: dpins.test_column_stats_match_bruteforce(m, "sum", (1, 2, 100, 70, 16, 32)),
    lambda m: dpins.test_identical_keys_level(m),
    lambda m: dpins.test_one_hot_keys_keep_own_key(m),
    lambda m: dpins.test_delta_is_masked_full_softmax(m),
    lambda m: dpins.test_delta_cache_roundtrip_and_empty(m),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", "-o", str(lib), str(mutant), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle._configure(ctypes.CDLL(str(lib))))
    caught = 0
    for pin in PINS:
        try:
            pin(oracle)
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin detects: {name}"


# Planted mistakes in the oracle's Python layout functions: each is applied to
# the function's source, the mutant replaces the real one, and a pin of
# test_oracle_layout.py must fail.
from tests import test_oracle_formats as fpins  # noqa: E402
from tests import test_oracle_layout as lpins  # noqa: E402

PY_MUTATIONS = {
    "voxel loops h and w swapped": ("voxel_order", "for h in range(h0, min(h0 + vh, Hh)):\n                        for w in range(w0, min(w0 + vw, W)):",
                                    "for w in range(w0, min(w0 + vw, W)):\n                        for h in range(h0, min(h0 + vh, Hh)):"),
    "voxel edge not clipped": ("voxel_order", "min(t0 + vt, T)", "t0 + vt"),
    "voxel raster index wrong": ("voxel_order", "(t * Hh + h) * W + w", "(t * W + h) * Hh + w"),
    "inverse applies forward": ("voxel_permute", "y[..., order, :] = x", "y = x[..., order, :]"),
    "window drops the sink": ("kv_window_append", "chunks = [chunks[0]] + chunks[2:] + [new.copy()]",
                              "chunks = chunks[1:] + [new.copy()]"),
    "window fills one slot late": ("kv_window_append", "if chunks_before < S:", "if chunks_before < S - 1:"),
    "bitmask bit order reversed": ("lists_from_bitmask", ">> (j % 32)", ">> (31 - j % 32)"),
    "bitmask word index wrong": ("lists_from_bitmask", "words[r, j // 32]", "words[r, min(j // 8, words.shape[1] - 1)]"),
    "block range not clipped": ("lists_from_block_mask", "min((b + 1) * block_k, Nk)", "(b + 1) * block_k"),
    "block keeps from the wrong start": ("lists_from_block_mask", "range(b * block_k,", "range(b * block_k + 1,"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_layout_pins_catch_mutation(name, monkeypatch):
    import inspect
    import textwrap
    fn, old, new = PY_MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn)))
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    if fn == "voxel_order":
        monkeypatch.setattr(oracle, "voxel_permute", ns["voxel_permute"])
    pins_ = [lambda: lpins.test_voxel_order_closed_form((4, 8, 8), (2, 4, 4)),
             lambda: lpins.test_voxel_order_clipped_edges((5, 7, 9), (2, 3, 4)),
             lambda: lpins.test_voxel_permute_inverse_and_generator_agree(),
             lambda: lpins.test_kv_window_append_bruteforce(4),
             lambda: fpins.test_bitmask_matches_numpy_packbits(7, 100, 0.3),
             lambda: fpins.test_block_mask_matches_numpy_repeat(4, 100, 16),
             lambda: fpins.test_block_sparse_attention_is_sdpa_with_block_mask()]
    caught = 0
    for pin in pins_:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught += 1
    assert caught > 0, f"no pin detects: {name}"
