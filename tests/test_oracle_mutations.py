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

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "forward drops the scale": ("logits[j] = c->scale * dot;", "logits[j] = dot;"),
    "forward exp sign flipped": ("double p = exp(logits[j] - m);", "double p = exp(m - logits[j]);"),
    "lse drops the max": ("lse_unit[r] = m + log(sum);", "lse_unit[r] = log(sum);"),
    "key row ignores the list": ("c->k + (bh * s->Nk + list[j]) * d", "c->k + (bh * s->Nk + j) * d"),
    "value row ignores the list": ("c->v + (bh * s->Nk + list[j]) * d", "c->v + (bh * s->Nk + j) * d"),
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
    "query row offset wrong": ("c->q + (bh * s->Nq + qi) * d", "c->q + (bh * s->Nq + r) * d"),
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
