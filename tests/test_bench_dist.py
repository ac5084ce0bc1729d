"""The benchmark's multi-rank path on CPU: world size 2 over gloo.  In the
real benchmark each rank runs its own layer (--split batch) or a share of one
layer's heads (--split heads) on its own GPU; heads are independent, so there
is no data exchange.  The only collective is the max-over-ranks step time and
the sum of the work, checked here without a GPU, together with the head
partition."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_info() == (world, rank, rank)
    ms, units = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), world)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, units in got:
        assert ms == 2.0  # slowest rank
        assert units == 300.0  # work of both ranks


def test_kept_pairs_counts_ragged_groups():
    import numpy as np
    import bench
    # 2 heads, Nq = 300, M = 128 -> groups of 128, 128, 44 rows
    counts = np.array([5, 6, 7, 1, 2, 3])
    row_ptr = np.concatenate([[0], np.cumsum(counts)])
    assert bench.kept_pairs(row_ptr, 1, 2, 300, 128) == 128 * (5 + 6 + 1 + 2) + 44 * (7 + 3)


def test_builder_and_gather_bytes():
    import bench
    # 24 heads x 16384 tokens, d = 128, groups of 128, 3277 keys per group
    rows = 24 * 128
    nnz = rows * 3277
    b, g = bench.builder_and_gather(1, 24, 16384, 16384, 128, 128, nnz, 0.2, 0.6, 6781.8, "measured")
    qk = 2 * 128 * (16384 + 16384) * 24  # Q and K read once: 201.3 MB
    assert b["bytes_per_step"] == qk + 4 * nnz + 8 * (rows + 1)
    assert abs(b["bytes_per_step"] - 241.6e6) < 0.1e6
    assert abs(b["achieved"] - b["bytes_per_step"] / 0.2e-3 / 1e9) < 1e-6
    assert abs(b["frac"] - b["achieved"] / 6781.8) < 1e-12 and b["unit"] == "GB/s"
    assert g["bytes_per_step"] == 4 * 128 * nnz  # 5.15 GB: one K and one V row per kept key
    assert abs(g["achieved"] - 4 * 128 * nnz / 0.6e-3 / 1e9) < 1e-6
    # a ragged last group still counts as one row of lists
    b2, _ = bench.builder_and_gather(2, 3, 300, 1000, 64, 128, 10, 1.0, 1.0, 1.0, "fallback")
    assert b2["bytes_per_step"] == 2 * 64 * 1300 * 6 + 40 + 8 * (2 * 3 * 3 + 1)


def _heads_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from video_dit_sparse_gb300 import inputs as I
    w = I.preset("sweep69k_top20")
    lw, seed, heads = bench.local_workload(w, "heads", world, rank)
    # each rank's share of the layer's work, summed by the benchmark's reduction
    _, pairs_total = bench.aggregate(float(rank), float(bench.topk_pairs(lw)), world)
    shares = [None] * world
    dist.all_gather_object(shares, heads)
    q.put((rank, lw.H, seed, heads, shares, pairs_total, bench.topk_pairs(w)))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_head_split_covers_every_head_once(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_heads_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    heads = [h for _, _, _, h, _, _, _ in got]
    covered = sorted(i for h0, h1 in heads for i in range(h0, h1))
    assert covered == list(range(24))  # every head exactly once
    for rank, H, seed, (h0, h1), shares, pairs_total, pairs_layer in got:
        assert H == h1 - h0 and seed == 0 and abs(H - 24 / world) < 1
        assert shares == heads  # every rank agrees on the partition
        assert pairs_total == pairs_layer  # the units add up to the whole layer


def test_partition_heads_rules():
    import bench
    assert [bench.partition_heads(24, 5, r) for r in range(5)] == [(0, 4), (4, 9), (9, 14), (14, 19), (19, 24)]
    assert bench.partition_heads(12, 1, 0) == (0, 12)
    with pytest.raises(ValueError):
        bench.partition_heads(2, 3, 0)  # more ranks than heads
    from video_dit_sparse_gb300 import inputs as I
    w = I.preset("wan16k_top20")
    assert bench.local_workload(w, "batch", 4, 3) == (w, 3, None)  # own layer, own seed
    assert bench.topk_pairs(w) == 24 * 16384 * 3277
    assert bench.topk_pairs(I.preset("rollingkv_mass99")) is None
