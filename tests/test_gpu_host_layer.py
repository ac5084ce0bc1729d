"""The host-memory layer runner (sparse_attn_layer_from_host, through the C
ABI): its output, copied back to pinned host memory chunk by chunk while the
next chunk computes, equals bit for bit the device-resident build + forward
of the whole layer (each (batch, head) is computed by the same kernels on
the same data), for TOPK and MASS, several chunk sizes including a ragged
last chunk, and on two calls in a row."""
import numpy as np
import pytest
import torch

from tests import parity as P
from video_dit_sparse_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,kw,hpc", [("topk", {"topk": 140}, 2), ("topk", {"topk": 140}, 0),
                                         ("mass", {"mass": 0.95}, 3), ("topk", {"topk": 70}, 5)])
def test_host_layer_matches_device_path(mode, kw, hpc):
    from video_dit_sparse_gb300 import binding as sa
    w = I.custom("host", 2, 3, 128, 128, (5, 10, 20), (7, 10, 10))  # B 2, H 3, Nq 1000, Nk 700
    x = I.make_inputs(w, 4)

    def host(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = host(x["q"]), host(x["k"]), host(x["v"])
    qd, kd, vd = hq.cuda(), hk.cuda(), hv.cuda()
    rp, col, nnz = sa.sparse_attn_build_index(qd, kd, mode, group_size=128, **kw)
    o_ref, lse_ref = sa.sparse_attn_forward(qd, kd, vd, rp, col, group_size=128)
    layer = sa.HostLayer(2, 3, 1000, 700, 128, group_size=128, mode=mode, heads_per_chunk=hpc, **kw)
    for _ in range(2):
        o_h = torch.empty(o_ref.shape, dtype=o_ref.dtype).pin_memory()
        l_h = torch.empty(lse_ref.shape, dtype=torch.float32).pin_memory()
        layer(hq, hk, hv, o_h, l_h)
        layer.synchronize()
        assert torch.equal(o_h.view(torch.int16), o_ref.cpu().view(torch.int16))
        assert torch.equal(l_h, lse_ref.cpu())


def test_host_layer_rejects_short_capacity():
    from video_dit_sparse_gb300 import binding as sa
    layer = sa.HostLayer(1, 2, 256, 256, 128, group_size=128, mode="topk", topk=16, heads_per_chunk=1)
    layer.cap = 8  # less than one chunk's lists
    z = torch.zeros(1, 2, 256, 128, dtype=torch.bfloat16).pin_memory()
    l = torch.zeros(1, 2, 256, dtype=torch.float32).pin_memory()
    with pytest.raises(sa.SparseAttnError) as e:
        layer(z, z, z, z.clone(), l)
    assert e.value.status == sa.SA_ERR_CAPACITY


def test_host_layer_checks_staging_buffers_before_any_copy():
    """An undersized device staging buffer is refused before the first copy
    is enqueued: nothing is written to it or to the host output."""
    from video_dit_sparse_gb300 import binding as sa
    B, H, N, d = 1, 24, 16384, 128  # 96 MiB per tensor
    layer = sa.HostLayer(B, H, N, N, d, group_size=128, mode="topk", topk=64, heads_per_chunk=4)
    torch.cuda.synchronize()
    # 2 MiB in a fresh allocation segment (no cached block to carve it from),
    # far smaller than the 96 MiB q needs
    torch.cuda.empty_cache()
    small = torch.full((1, 1, 8192, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    layer.q = small
    z = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    o_h = torch.full((B, H, N, d), 3.0, dtype=torch.bfloat16)
    l_h = torch.full((B, H, N), 5.0, dtype=torch.float32)
    with pytest.raises(sa.SparseAttnError) as e:
        layer(z, z, z, o_h, l_h)
    assert e.value.status == sa.SA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((layer.q == 7.0).all())
    assert bool((o_h == 3.0).all()) and bool((l_h == 5.0).all())
