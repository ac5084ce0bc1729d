"""Benchmark: one step = the whole hot path (sparse_attn_build_index +
sparse_attn_forward) over one synthetic attention layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is effective TFLOP/s on kept scores
(4*d flops per kept query-key pair) for build + forward, inputs resident in
HBM; `e2e` is the same metric with host buffers (H2D of q, k, v and D2H of
o, lse inside the timed region); `roofline` is the forward kernel against
the measured bf16 tensor peak.  `--impl reference` times the fp64 CPU
oracle on a bounded sample of the same workload.

The default workload is the 69K-token density sweep at 20 % (24 heads,
18x48x80 latent grid in (2,8,8) voxels, M = 128, top 13824 keys per group).

Under torchrun (N > 1) the (batch, head) units are independent, so no
collective touches the data path:
  --split batch (default): rank r runs its own layer (batch element r, seeded
                 r): weak scaling, per-GPU work fixed;
  --split heads: rank r runs heads [r*H/N, (r+1)*H/N) of one layer: strong
                 scaling, total work fixed.
Rank 0 reports the slowest rank's step time and the work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective TFLOP/s on kept scores (4·d/pair) & ms/layer; % of GB300 dense BF16 TC peak"
DEFAULT_WORKLOAD = "sweep69k_top20"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def kernels_per_step(mode: str, topk: int = 0, Nk: int = 0) -> int:
    """Our kernels per step.  TOPK by mean query over at least 8192 keys (a
    multiple of 8): mean query, sample scores, bracket, classifying scores,
    finalize, the score and select kernels on the rows it left (usually
    none), forward; keeping every key: finalize, forward.  Other
    selections: mean query, scores, select, scan, [emit,] forward (TOPK lists
    are written by the select kernel; the other modes add the emit kernel
    once the row offsets are known).  Dense-step workloads: dense forward,
    column statistics, select, scan, [emit,] and the sparse forward (cached
    mask) or the two sparse deltas (column sums, TOPK)."""
    if mode == "cached":
        return 6
    if mode == "colsum":
        return 6
    if mode == "topk":
        if topk >= Nk:
            return 2
        return 8 if Nk >= 8192 and Nk % 8 == 0 else 5
    return 6


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "video_dit_sparse_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel, {}).get(workload)
    if not rec or rec.get("source_hash") != source_hash(*rec.get("sources", [])):
        return None
    return rec.get("dram_bytes_per_launch")


def kept_pairs(row_ptr: np.ndarray, B, H, Nq, M) -> int:
    """sum over units of |group rows| * |kept keys|."""
    G = -(-Nq // M)
    counts = np.diff(row_ptr).reshape(B * H, G)
    rows = np.full(G, M, dtype=np.int64)
    rows[-1] = Nq - (G - 1) * M
    return int((counts * rows[None, :]).sum())


def builder_and_gather(B, H, Nq, Nk, d, M, nnz, ms_build, ms_fwd, hbm_gbs, peak_kind):
    """The index builder against the HBM roofline, and the rate of the
    forward's gather.  The builder's algorithmic bytes are one read of Q and
    K (2·d bytes per token row) and the lists it writes (4 bytes per kept
    index, 8 per row offset); the gather moves 4·d bytes (one K and one V row)
    per (group, kept key) from L2 into shared memory inside the forward
    kernel, so it has no DRAM roofline of its own."""
    rows = B * H * (-(-Nq // M))
    build_bytes = 2 * d * (Nq + Nk) * B * H + 4 * nnz + 8 * (rows + 1)
    gbs = build_bytes / (ms_build * 1e-3) / 1e9
    builder = {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s",
               "frac": gbs / hbm_gbs, "bytes_per_step": int(build_bytes), "ms": ms_build,
               "peak_source": f"{peak_kind} hbm_gbs"}
    gather_bytes = 4 * d * nnz
    gather = {"source": "L2", "achieved": gather_bytes / (ms_fwd * 1e-3) / 1e9, "unit": "GB/s",
              "bytes_per_step": int(gather_bytes)}
    return builder, gather


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def partition_heads(H: int, world: int, rank: int):
    """Heads [h0, h1) of rank `rank` when one layer's H heads are split over
    `world` ranks: contiguous and as even as possible (sizes differ by at
    most one)."""
    if world < 1 or not 0 <= rank < world or world > H:
        raise ValueError(f"cannot split {H} heads over {world} ranks")
    return rank * H // world, (rank + 1) * H // world


def local_workload(w, split: str, world: int, rank: int):
    """(workload of this rank, input seed, head range or None)."""
    import dataclasses
    if world == 1:
        return w, 0, None
    if split == "heads":
        h0, h1 = partition_heads(w.H, world, rank)
        return dataclasses.replace(w, H=h1 - h0), 0, (h0, h1)
    return w, rank, None


def slice_heads(x: dict, heads):
    if heads is None:
        return x
    h0, h1 = heads
    return {n: np.ascontiguousarray(a[:, h0:h1]) for n, a in x.items() if n in ("q", "k", "v")}


def aggregate(local_ms: float, local_units: float, world: int, group=None):
    """Max step time over ranks and total units (all-reduce on the host
    backend; the only collective in the benchmark)."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


# --------------------------------------------------------------- CPU oracle
def oracle_sample(w, x, budget_s: float, threads: int):
    """Times the fp64 oracle (mean-query scores + selection + restricted
    attention) on a growing sample of units until about `budget_s` seconds of
    work; returns (effective TFLOP/s, description, threads)."""
    import oracle
    rows = w.B * w.H * w.G
    rng = np.random.default_rng(7)
    order = rng.permutation(rows)
    n = min(threads, rows)
    spent, pairs, done = 0.0, 0, 0
    while True:
        units = np.sort(order[done:done + n]).astype(np.int64)
        t0 = time.perf_counter()
        lists, _, _ = oracle.build_index(x["q"], x["k"], w.group, w.scale, w.mode, topk=w.topk,
                                         tau=w.threshold, rho=w.mass, units=units, threads=threads)
        counts = np.zeros(rows, dtype=np.int64)
        counts[units] = [len(l) for l in lists]
        row_ptr = np.zeros(rows + 1, dtype=np.int64)
        np.cumsum(counts, out=row_ptr[1:])
        col = np.zeros(row_ptr[-1], dtype=np.int32)
        for u, l in zip(units, lists):
            col[row_ptr[u]:row_ptr[u + 1]] = l
        oracle.forward(x["q"], x["k"], x["v"], w.group, w.scale, row_ptr, col, units, threads)
        spent += time.perf_counter() - t0
        for u, l in zip(units, lists):
            g = u % w.G
            pairs += (min((g + 1) * w.group, w.Nq) - g * w.group) * len(l)
        done += units.size
        if spent >= budget_s or done >= rows:
            break
        n = min(rows - done, max(n, int(n * budget_s / max(spent, 1e-3))))
    tflops = 4.0 * w.d * pairs / spent / 1e12
    desc = f"{done} of {rows} query groups (seeded), full scoring+selection+attention per group"
    return tflops, desc, spent


def run_reference(args, w):
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from video_dit_sparse_gb300 import inputs as I
    threads = oracle.default_threads()
    x = I.make_inputs(w, 0)
    for _ in range(args.warmup):
        oracle_sample(w, x, 0.0, threads)
    times, vals = [], []
    for _ in range(args.steps):
        v, desc, spent = oracle_sample(w, x, args.ref_budget, threads)
        vals.append(v)
        times.append(spent)
    value = float(np.mean(vals))
    ms = 1e3 * float(np.mean(times))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, topk_pairs(w), args.split, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def topk_pairs(w):
    """Kept pairs of a TOPK layer, known without running it: every group keeps
    min(k, Nk) keys for each of its rows.  None for data-dependent rules."""
    if w.mode != "topk":
        return None
    return w.B * w.H * w.Nq * min(w.topk, w.Nk)


def workload_config(w, pairs, split="batch", world=1):
    c = {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
         "group": w.group, "selection": {"topk": f"k={w.topk}", "mass": f"rho={w.mass}",
                                         "threshold": f"tau={w.threshold}",
                                         "cached": f"column max >= {w.threshold:.4g}",
                                         "colsum": f"column sum top k={w.topk}"}[w.mode],
         "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)"}
    if pairs is not None:
        c["kept_pairs"] = pairs
    if world > 1:
        c["parallelism"] = f"{split} split over {world} ranks"
    return c


# --------------------------------------------------------------- GPU arm
def run_ours(args, w):
    import torch
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from video_dit_sparse_gb300 import binding as sa
    from video_dit_sparse_gb300 import inputs as I

    w_layer = w
    w, seed, heads = local_workload(w, args.split, world, rank)
    x = slice_heads(I.make_inputs(w_layer if heads else w, seed), heads)
    dev = torch.device("cuda", local)

    def host(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = host(x["q"]), host(x["k"]), host(x["v"])
    q, k, v = hq.to(dev), hk.to(dev), hv.to(dev)
    stream = torch.cuda.current_stream()
    p = sa.problem(q, k, w.group, w.scale)
    ws = torch.empty(sa.sparse_attn_build_index_workspace_size(p), dtype=torch.uint8, device=dev)
    rows = w.B * w.H * w.G
    cap = rows * (w.topk if w.mode == "topk" else w.Nk)
    col = torch.empty(cap, dtype=torch.int32, device=dev)
    row_ptr = torch.empty(rows + 1, dtype=torch.int64, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sel = sa.sa_select(sa._MODES[w.mode], w.topk, w.threshold, w.mass)
    nnz_box = sa.ctypes.c_int64(0)
    sync_nnz = w.mode != "topk"

    def build():
        st = sa.lib.sparse_attn_build_index(
            sa.ctypes.byref(p), sa.ctypes.byref(sel), sa._ptr(q), sa._ptr(k), sa._ptr(row_ptr),
            sa._ptr(col), cap, sa.ctypes.byref(nnz_box) if sync_nnz else None, sa._ptr(ws),
            ws.numel(), sa._stream(stream))
        if st:
            raise sa.SparseAttnError(st, "build_index")

    def fwd(nnz):
        st = sa.lib.sparse_attn_forward(sa.ctypes.byref(p), sa._ptr(q), sa._ptr(k), sa._ptr(v),
                                        sa._ptr(row_ptr), sa._ptr(col), nnz, sa._ptr(o),
                                        sa._ptr(lse), None, sa._stream(stream))
        if st:
            raise sa.SparseAttnError(st, "forward")

    def nnz_now():
        return nnz_box.value if sync_nnz else rows * w.topk

    for _ in range(max(args.warmup, 1)):
        build()
        fwd(nnz_now())
    torch.cuda.synchronize()
    pairs = kept_pairs(row_ptr.cpu().numpy(), w.B, w.H, w.Nq, w.group)
    flops = 4.0 * w.d * pairs
    _, pairs_total = aggregate(0.0, float(pairs), world)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            build()
            ev[i][1].record(stream)
            fwd(nnz_now())
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_build = [e[0].elapsed_time(e[1]) for e in ev]
    t_fwd = [e[1].elapsed_time(e[2]) for e in ev]
    ms_step = float(np.mean(t_build) + np.mean(t_fwd))
    ms_max, units_total = aggregate(ms_step, float(flops), world)
    value = units_total / (ms_max * 1e-3) / 1e12

    # end to end through the C ABI with host buffers: sparse_attn_layer_from_host
    # overlaps the copies of one chunk of heads with the build + forward of
    # the previous one (pinned host q, k, v in; o and lse out, every step)
    e2e_steps = max(3, min(args.steps, 20))
    layer = sa.HostLayer(w.B, w.H, w.Nq, w.Nk, w.d, group_size=w.group, mode=w.mode, topk=w.topk,
                         threshold=w.threshold, mass=w.mass, device=dev)
    h_o = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    layer(hq, hk, hv, h_o, h_lse, stream=stream)  # warm-up
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(e2e_steps):
        flush.zero_()
        e0.record(stream)
        layer(hq, hk, hv, h_o, h_lse, stream=stream)
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    del layer
    e2e_ms_max, _ = aggregate(float(np.mean(e2e_ms)), 0.0, world)
    e2e_value = units_total / (e2e_ms_max * 1e-3) / 1e12

    if rank != 0:
        return
    pk, pk_kind = peaks()
    fwd_ms = float(np.mean(t_fwd))
    achieved = flops / (fwd_ms * 1e-3) / 1e12
    traffic = recorded_traffic("sa_forward_kernel", w.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                "kernel": "sa_forward_kernel", "peak_source": f"{pk_kind} bf16_tflops (burst)",
                "frac_of_sustained": achieved / pk.get("bf16_tflops_sustained", pk["bf16_tflops"])}
    builder, gather = builder_and_gather(w.B, w.H, w.Nq, w.Nk, w.d, w.group, int(nnz_now()),
                                         float(np.mean(t_build)), fwd_ms, pk["hbm_gbs"], pk_kind)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True,
            "scaling": "strong" if (world > 1 and args.split == "heads") else "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w_layer if heads else w,
                                      int(pairs_total) if heads else pairs, args.split, world),
            "ms_build_index": float(np.mean(t_build)), "ms_forward": fwd_ms,
            "gpu_launches": kernels_per_step(w.mode, w.topk, w.Nk) * args.steps,
            "roofline": roofline, "builder": builder, "gather": gather,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(3 * q.numel() * 2),
                    "d2h_bytes_per_step": int(o.numel() * 2 + lse.numel() * 4),
                    "ms_per_step": e2e_ms_max},
            "clocks": clocks.summary()}
    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        cv, desc, spent = oracle_sample(w, x, args.cpu_budget, threads)
        line["cpu_baseline"] = {"value": cv, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": round(spent, 2)}
    print(json.dumps(line), flush=True)


def run_ours_dense(args, w):
    """Dense-step workloads.  One step = the refresh of a cached mask and the
    sparse work that follows it:
      cached:  dense forward (o, lse) -> column max of the dense probabilities
               >= tau (FG-Attn cached mask) -> sparse forward on those lists;
      colsum:  dense forward (fp32 o, lse) -> column-sum top-k (Chipmunk)
               -> sparse delta writing the cache (o - kept terms) -> sparse
               delta adding the kept terms back (the next step's update).
    value = 4*d*(kept pairs of every attention call) / step time."""
    import torch
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from video_dit_sparse_gb300 import binding as sa
    from video_dit_sparse_gb300 import inputs as I

    x = I.make_inputs(w, 0)
    dev = torch.device("cuda", local)

    def host(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = host(x["q"]), host(x["k"]), host(x["v"])
    q, k, v = hq.to(dev), hk.to(dev), hv.to(dev)
    stream = torch.cuda.current_stream()
    cached = w.mode == "cached"
    p = sa.problem(q, k, w.group, w.scale, torch.bfloat16 if cached else torch.float32)
    ws = torch.empty(sa.sparse_attn_build_index_workspace_size(p), dtype=torch.uint8, device=dev)
    rows = w.B * w.H * w.G
    cap = rows * (w.Nk if cached else w.topk)
    col = torch.empty(cap, dtype=torch.int32, device=dev)
    row_ptr = torch.empty(rows + 1, dtype=torch.int64, device=dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16 if cached else torch.float32, device=dev)
    o2 = torch.empty_like(o)
    cache = torch.empty(q.shape, dtype=torch.float32, device=dev) if not cached else None
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if cached:
        sel = sa.sa_select(sa.SA_SELECT_THRESHOLD, 0, w.threshold, 0.99)
        stat = sa.SA_COLSTAT_MAX
    else:
        sel = sa.sa_select(sa.SA_SELECT_TOPK, w.topk, 0.0, 0.99)
        stat = sa.SA_COLSTAT_SUM
    P, S = sa.ctypes.byref(p), sa._stream(stream)

    def check(st, where):
        if st:
            raise sa.SparseAttnError(st, where)

    def dense():
        check(sa.lib.sparse_attn_forward(P, sa._ptr(q), sa._ptr(k), sa._ptr(v), None, None, 0,
                                         sa._ptr(o), sa._ptr(lse), None, S), "dense forward")

    def build():
        # capacity covers every key, so no synchronisation is needed for nnz
        check(sa.lib.sparse_attn_build_index_dense(P, sa.ctypes.byref(sel), stat, sa._ptr(q),
                                                   sa._ptr(k), sa._ptr(lse), sa._ptr(row_ptr),
                                                   sa._ptr(col), cap, None, sa._ptr(ws),
                                                   ws.numel(), S), "build_index_dense")

    def sparse():
        if cached:
            check(sa.lib.sparse_attn_forward(P, sa._ptr(q), sa._ptr(k), sa._ptr(v), sa._ptr(row_ptr),
                                             sa._ptr(col), cap, sa._ptr(o2), None, None, S),
                  "sparse forward")
        else:
            check(sa.lib.sparse_attn_forward_delta(P, sa._ptr(q), sa._ptr(k), sa._ptr(v),
                                                   sa._ptr(row_ptr), sa._ptr(col), cap, sa._ptr(lse),
                                                   sa._ptr(o), -1.0, sa._ptr(cache), None, S),
                  "delta (cache)")
            check(sa.lib.sparse_attn_forward_delta(P, sa._ptr(q), sa._ptr(k), sa._ptr(v),
                                                   sa._ptr(row_ptr), sa._ptr(col), cap, sa._ptr(lse),
                                                   sa._ptr(cache), 1.0, sa._ptr(o2), None, S),
                  "delta (update)")

    for _ in range(max(args.warmup, 1)):
        dense()
        build()
        sparse()
    torch.cuda.synchronize()
    pairs = kept_pairs(row_ptr.cpu().numpy(), w.B, w.H, w.Nq, w.group)
    dense_pairs = w.B * w.H * w.Nq * w.Nk
    sparse_calls = 1 if cached else 2
    flops = 4.0 * w.d * (dense_pairs + sparse_calls * pairs)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            dense()
            ev[i][1].record(stream)
            build()
            ev[i][2].record(stream)
            sparse()
            ev[i][3].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in ev])
    t_dense, t_build, t_sparse = (float(x) for x in t.mean(axis=0))
    ms_step = t_dense + t_build + t_sparse
    ms_max, units_total = aggregate(ms_step, flops, world)
    value = units_total / (ms_max * 1e-3) / 1e12

    e2e_steps = max(3, min(args.steps, 10))
    h_o = torch.empty(o2.shape, dtype=o2.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(e2e_steps):
        flush.zero_()
        e0.record(stream)
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        dense()
        build()
        sparse()
        h_o.copy_(o2, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_ms_max, _ = aggregate(float(np.mean(e2e_ms)), 0.0, world)
    if rank != 0:
        return
    pk, pk_kind = peaks()
    achieved = 4.0 * w.d * dense_pairs / (t_dense * 1e-3) / 1e12
    cs_flops = 2.0 * w.d * dense_pairs  # the column statistics' QK^T
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(w, pairs),
            "ms_dense_forward": t_dense, "ms_build_index_dense": t_build,
            ("ms_sparse_forward" if cached else "ms_delta_pair"): t_sparse,
            "density": pairs / dense_pairs,
            "gpu_launches": kernels_per_step(w.mode) * args.steps,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": None,
                         "kernel": "sa_forward_kernel (dense mode)",
                         "peak_source": f"{pk_kind} bf16_tflops (burst)"},
            "build_index_dense_tflops": cs_flops / (t_build * 1e-3) / 1e12,
            "e2e": {"value": units_total / (e2e_ms_max * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(3 * q.numel() * 2),
                    "d2h_bytes_per_step": int(o2.numel() * o2.element_size()),
                    "ms_per_step": e2e_ms_max},
            "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def run_layout(args, w):
    """Layout and index-format workloads, bound by HBM bandwidth.  voxel69k:
    one step reorders Q, K and V into voxel order and O back to raster order
    (4 calls); kvwindow_rollingkv: one step appends a chunk to the full 4-slot
    K/V window (the sink stays, the other chunks roll); bitmask69k_top20 /
    blockmask69k_top20: one step converts a keep-mask into CSR lists.
    value = algorithmic bytes read + written per step / step time."""
    import torch
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from video_dit_sparse_gb300 import binding as sa
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def rnd(*shape):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)

    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if w.mode == "layout":
        grid, voxel = w.grid_q, w.voxel
        xs = [rnd(w.B, w.H, w.Nq, w.d) for _ in range(4)]
        ys = [torch.empty_like(x) for x in xs]

        def step():
            for i, (x, y) in enumerate(zip(xs, ys)):
                sa.sparse_attn_voxel_permute(x, grid, voxel, inverse=(i == 3), out=y, stream=stream)

        step_bytes = sum(2 * x.numel() * 2 for x in xs)
        calls, kernel = 4, "sa_voxel_permute_kernel"
    elif w.mode in ("bitmask", "blockmask"):
        rows = w.B * w.H * w.G
        dens = w.keep_pct / 100.0
        if w.mode == "bitmask":
            nw = -(-w.Nk // 32)
            bits_ = torch.rand(rows, nw * 32, generator=g, device=dev) < dens
            weights = (1 << torch.arange(32, device=dev, dtype=torch.int64))
            mask = (bits_.view(rows, nw, 32).to(torch.int64) * weights).sum(-1).to(torch.int64)
            mask = torch.where(mask >= (1 << 31), mask - (1 << 32), mask).to(torch.int32).contiguous()
            nnz_est = int(bits_[:, :w.Nk].sum().item())
            mask_bytes = mask.numel() * 4
        else:
            bk = 128
            mask = (torch.rand(rows, -(-w.Nk // bk), generator=g, device=dev) < dens).to(torch.uint8)
            nnz_est = int(mask.sum().item()) * bk
            mask_bytes = mask.numel()
        cap = rows * w.Nk
        row_ptr = torch.empty(rows + 1, dtype=torch.int64, device=dev)
        col = torch.empty(cap, dtype=torch.int32, device=dev)
        p = sa.sa_problem(w.B, w.H, w.Nq, w.Nk, w.d, w.group, w.scale, 0)

        def step():
            if w.mode == "bitmask":
                st = sa.lib.sparse_attn_index_from_bitmask(sa.ctypes.byref(p), sa._ptr(mask), sa._ptr(row_ptr),
                                                           sa._ptr(col), cap, None, sa._stream(stream))
            else:
                st = sa.lib.sparse_attn_index_from_block_mask(sa.ctypes.byref(p), 128, sa._ptr(mask),
                                                              sa._ptr(row_ptr), sa._ptr(col), cap, None,
                                                              sa._stream(stream))
            if st:
                raise sa.SparseAttnError(st, "index from mask")

        step_bytes = mask_bytes + 4 * nnz_est + 8 * (rows + 1)
        calls, kernel = 3, "sa_fmt_emit_kernel"
    else:
        L = w.Nq  # one chunk: the newest 8 frames
        S = w.Nk // L
        ck, cv = rnd(w.B, w.H, S * L, w.d), rnd(w.B, w.H, S * L, w.d)
        nk, nv = rnd(w.B, w.H, L, w.d), rnd(w.B, w.H, L, w.d)

        def step():
            sa.sparse_attn_kv_window_append(ck, cv, nk, nv, S + 3, stream=stream)

        chunk = nk.numel() * 2
        step_bytes = 2 * (chunk + 2 * (S - 2) * chunk + chunk)  # K and V: new read, rolls read+write, last slot write
        calls, kernel = 1, "sa_kv_window_kernel"
    for _ in range(max(args.warmup, 1)):
        step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    ms_max, bytes_total = aggregate(ms, float(step_bytes), world)
    if rank != 0:
        return
    pk, pk_kind = peaks()
    gbs = bytes_total / (ms_max * 1e-3) / 1e9
    line = {"metric": "GB/s moved by the layout / index-format kernels (bytes read + written)", "value": gbs,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)"},
            "gpu_launches": calls * args.steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": None, "kernel": kernel,
                         "peak_source": f"{pk_kind} hbm_gbs"},
            "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads (smaller ncu captures)")
    ap.add_argument("--split", choices=["batch", "heads"], default="batch",
                    help="N > 1: each rank its own layer (batch) or a share of one layer's heads")
    args = ap.parse_args()
    from video_dit_sparse_gb300 import inputs as I
    w = I.preset(args.workload)
    if args.heads > 0:
        import dataclasses
        w = dataclasses.replace(w, H=args.heads, name=f"{w.name}_h{args.heads}")
    if args.impl == "reference":
        run_reference(args, w)
    elif w.mode in ("cached", "colsum"):
        run_ours_dense(args, w)
    elif w.mode in ("layout", "kvwindow", "bitmask", "blockmask"):
        run_layout(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
