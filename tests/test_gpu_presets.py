"""Full-size workloads (the five synthetic configurations) on the GPU, in the
launch configuration the benchmark times.  The oracle checks, one group at a
time, every list and every query group of one whole head (two heads of the
rolling-KV workload), the units of the forward's last round over the SMs
(the tail of the unit order), and seeded samples from the other heads; the
keep-everything sweep point is also checked against dense attention."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu

PRESETS = ["wan16k_top20", "rollingkv_mass99", "chunk192_top10", "sweep69k_top5",
           "sweep69k_top10", "sweep69k_top20", "sweep69k_top40", "sweep69k_top100"]


def sample(n_total, n, seed):
    rng = np.random.default_rng(seed)
    picks = rng.choice(n_total, size=min(n, n_total), replace=False)
    return np.unique(np.concatenate([picks, [0, n_total - 1]])).astype(np.int64)


def checked_units(w, name):
    """Every group of whole heads (seeded choice), the units of the last
    round over the SMs, and a seeded sample of the rest."""
    rows = w.B * w.H * w.G
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    n_heads = 2 if w.mode == "mass" else 1
    heads = rng.choice(w.B * w.H, size=n_heads, replace=False)
    full = np.concatenate([np.arange(h * w.G, (h + 1) * w.G) for h in heads])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tail = np.arange(rows - (rows % sms or sms), rows)
    return np.unique(np.concatenate([full, tail, sample(rows, 12, seed=1)])).astype(np.int64)


@pytest.mark.parametrize("name", PRESETS)
def test_preset_builder_and_forward(name):
    from video_dit_sparse_gb300 import binding as sa
    w = I.preset(name)
    x = P.cached_inputs(name)
    q, k, v = x["q"], x["k"], x["v"]
    qd, kd, vd = P.to_dev(q), P.to_dev(k), P.to_dev(v)
    rp, col, nnz = sa.sparse_attn_build_index(qd, kd, w.mode, topk=w.topk, mass=w.mass,
                                              threshold=w.threshold, group_size=w.group)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=w.group,
                                    out_dtype=torch.float32, status=status)
    # the benchmark's launch writes bf16: exactly the fp32 result, rounded
    o16, lse16 = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=w.group)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(o16, o.to(torch.bfloat16)) and torch.equal(lse16, lse)
    del o16, lse16
    rows = w.B * w.H * w.G
    rpn = rp.cpu().numpy()
    assert rpn[0] == 0 and rpn[-1] == nnz
    if w.mode == "topk":
        assert nnz == rows * w.topk
    # builder: whole heads, the tail and a sample, against the oracle's full
    # scoring + selection of each row
    units = checked_units(w, name)
    ref_lists, ref_cut, ref_sc = oracle.build_index(q, k, w.group, w.scale, w.mode, topk=w.topk,
                                                    tau=w.threshold, rho=w.mass, units=units)
    P.compare_lists(rp, col, units, ref_lists, ref_cut, ref_sc, w.Nk)
    del ref_lists, ref_sc
    # forward: the same units, same (GPU-built) lists on both sides
    coln = col.cpu().numpy()
    P.compare_units(q, k, v, w.group, rpn, coln, units, o, lse)
    if w.keep_pct == 100.0 and w.mode == "topk":
        for h in (0, w.H - 1):
            ref = torch.nn.functional.scaled_dot_product_attention(
                qd[:, h:h + 1], kd[:, h:h + 1], vd[:, h:h + 1])
            assert (o[:, h:h + 1].float() - ref.float()).abs().max().item() < 2e-2
