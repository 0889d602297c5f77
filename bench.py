#!/usr/bin/env python3
"""Benchmark: useful TFLOPS of forward + backward block-causal attention on the
packed training-replay workload (16 packed sequences, lengths U[512, 4096]
rounded to 32, block 32, 32 query / 8 KV heads, head_dim 128, bf16).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

One step is one pass of the whole hot path over one batch: the tile plan
(host, copied to the workspace), the forward kernel and the three backward
stages, on inputs already resident in HBM.  `value` counts useful FLOPs only
(4 d Hq pairs forward + 10 d Hq pairs backward, pairs = allowed (query, key)
pairs).  `e2e` repeats the step through the same public API with the inputs
copied from pinned host memory and every output (O, LSE, dQ, dK, dV) copied
back inside the timed region; as in a training loop that prefetches its next
batch, the copies run on two copy streams and overlap the neighbouring steps'
compute (two device buffer sets).  `decode` times the HBM-bound decode step
(32 queries over 2,080 keys, forward only) against the measured copy
bandwidth, and its replay from a captured CUDA graph.  With N > 1 (torchrun, one rank per GPU) the
global batch holds 16 N sequences, sharded whole by longest-first load
balancing with no collective on the data path (weak scaling); the timing is
the max over ranks.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on the host cores.
"""
import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from diffusion_lm_block_bda_b300 import workloads as W  # noqa: E402

METRIC = "useful TFLOPS and % of B300 BF16 peak, fwd+bwd block-causal/staircase attention"
UNIT = "TFLOPS"
WORKLOAD_NAME = "packed block-causal training replay: 16 seqs U[512,4096]/32*32, B=32, Hq=32, Hkv=8, d=128"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-side", action="store_true",
                   help="skip the staircase (c4) and long-sequence (c5) measurements")
    p.add_argument("--stub", action="store_true",
                   help="launcher check without a GPU: every rank shards the batch and reports "
                        "(gloo), no kernel runs")
    return p.parse_args()


# ------------------------------------------------------------ distributed
def free_port():
    import socket
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    return port


def launch_ranks(args):
    """`--gpus N` without an outer launcher: start N ranks (one process per
    GPU) through torch.distributed.run and return its exit status.  Under a
    launcher whose world size differs from --gpus, refuse."""
    world = os.environ.get("WORLD_SIZE")
    if world is not None:
        if int(world) != args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}")
        return None
    if args.gpus <= 1:
        return None
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if args.stub:
            dist.init_process_group("gloo")
        else:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------- workload
def rank_workload(world, rank):
    """Global batch of 16 * world packed sequences (seed 0), LPT-sharded:
    (this rank's workload, its sequence ids, every rank's useful-pair load)."""
    from diffusion_lm_block_bda_b300 import sharding
    gen = torch.Generator().manual_seed(0)
    lens = W.packed_lengths(gen, n=16 * world)
    full = W.Workload("packed_block_causal_16xU512_4096_B32", W.BLOCK_CAUSAL, 32, 32, 8, 128,
                      lens, list(lens))
    if world == 1:
        return full, list(range(len(lens))), None
    costs = sharding.sequence_costs(full)
    shards = sharding.lpt_shard(costs, world)
    loads = [sum(costs[i] for i in sh) for sh in shards]
    return sharding.subset(full, shards[rank], f"_rank{rank}"), shards[rank], loads


def run_stub(args, world, rank):
    """The multi-rank launch path without a GPU: every rank derives its shard
    of the global batch and rank 0 prints what each rank got."""
    w, seq_ids, loads = rank_workload(world, rank)
    shards = [seq_ids]
    if world > 1:
        import torch.distributed as dist
        shards = [None] * world
        dist.all_gather_object(shards, seq_ids)
        dist.barrier()
    if rank == 0:
        print(json.dumps({"stub": True, "n_gpus": world, "gpus_active": world,
                          "global_sequences": 16 * world, "shards": shards,
                          "shard_pairs": loads}), flush=True)


# ------------------------------------------------------------------ clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.f.read())) if len(r) >= 9]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), \
            float(j["hbm_gbs"]), "measured"
    return 1800.0, 1400.0, 6400.0, "fallback"


KERNEL_SOURCES = ("diffusion_lm_block_bda_b300/csrc/bda_bwd.cu",
                  "diffusion_lm_block_bda_b300/csrc/bda_fwd.cu",
                  "diffusion_lm_block_bda_b300/csrc/bda_ptx.cuh",
                  "diffusion_lm_block_bda_b300/csrc/bda_internal.h",
                  "diffusion_lm_block_bda_b300/csrc/bda_kernels.h")


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel="bwd_dkdv"):
    """DRAM bytes per launch of a kernel ("bwd_dkdv" or "fwd") from the
    committed ncu summary; None when absent or taken on a different build of
    the kernels (the summary records a hash of the kernels' sources)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        j = json.load(f)
    if j.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return j.get(f"{kernel}_bytes_per_launch")


# -------------------------------------------------------------- reference
def run_reference(args, world, rank):
    """The fp64 CPU oracle, timed on the host cores: each step is a bounded
    sample (the median-length sequence of the batch, one KV head and its 4
    query heads, forward + backward)."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    w, _, _ = rank_workload(1, 0)
    inp = W.make_inputs(w, seed=0)
    s = int(np.argsort(w.seqlens_q)[len(w.seqlens_q) // 2])
    L = w.seqlens_q[s]
    c = w.cu_seqlens_q
    sl = slice(c[s], c[s + 1])
    pairs = oracle.count_pairs(W.BLOCK_CAUSAL, 32, L, L, L)  # useful work, counted by the oracle
    G = w.hq // w.hkv
    flops = 14.0 * w.head_dim * G * pairs
    times = []
    for i in range(args.warmup + args.steps):
        kvh = i % w.hkv
        t0 = time.perf_counter()
        oracle.fwd_seq(w.kind, 32, L, inp["q"][sl], inp["k"][sl], inp["v"][sl], w.hq, w.hkv,
                       w.softmax_scale, heads=(kvh * G, (kvh + 1) * G))
        oracle.bwd_seq(w.kind, 32, L, inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["dout"][sl],
                       w.hq, w.hkv, w.softmax_scale, kv_heads=(kvh, kvh + 1))
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times)
    value = flops * len(times) / t / 1e12
    sample = (f"sequence {s} (L={L}) of the packed batch, one KV head and its {G} query heads, "
              f"fwd+bwd fp64 per step")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * t / len(times), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16 inputs)",
           "config": {"workload": WORKLOAD_NAME, "sample": sample},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def cpu_baseline(w, inp):
    """The oracle as it stands on one bounded sample: the median-length
    sequence, all heads, fwd+bwd."""
    import numpy as np
    import oracle
    s = int(np.argsort(w.seqlens_q)[len(w.seqlens_q) // 2])
    L = w.seqlens_q[s]
    c = w.cu_seqlens_q
    sl = slice(c[s], c[s + 1])
    pairs = oracle.count_pairs(w.kind, w.block_size, L, L, L)
    t0 = time.perf_counter()
    oracle.fwd_seq(w.kind, w.block_size, L, inp["q"][sl], inp["k"][sl], inp["v"][sl], w.hq,
                   w.hkv, w.softmax_scale)
    oracle.bwd_seq(w.kind, w.block_size, L, inp["q"][sl], inp["k"][sl], inp["v"][sl],
                   inp["dout"][sl], w.hq, w.hkv, w.softmax_scale)
    t = time.perf_counter() - t0
    flops = 14.0 * w.head_dim * w.hq * pairs
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"sequence {s} (L={L}) of the packed batch, all {w.hq} heads, fwd+bwd fp64, "
                      f"{t:.1f} s"}


# ------------------------------------------------------------------ decode
def decode_measurement(bda, dev, stream, hbm_gbs, reps=32, n_rot=16):
    """The decode step (32 new queries over a 2,080-key context: 2,048
    committed tokens + the active block; Hq=32, Hkv=8, d=128; forward only)
    is bound by HBM bandwidth and latency, not by the tensor cores.  Its
    forward runs the split kernel (each query tile's 17 key tiles as 9 chunks,
    x 8 head groups = 72 CTAs) and the combine kernel.  As in a denoising loop, where every
    layer's KV cache has left L2 by the time the layer comes round again
    while the kernels' code stays cached, the timed launches rotate through 16
    copies of Q, K and V (144 MB, more than L2): each launch reads its copy
    from HBM.  The stream is held busy while the host enqueues, so the events
    bracket GPU time only.  `us`: median time of the forward; `achieved` =
    the minimum bytes (Q, K, V read once, O and LSE written) / `us`.
    `graph_us`: one copy's forward captured in a CUDA graph and replayed back
    to back (everything in L2), GPU time per replay.  `fp8`: the same step
    over an e4m3 KV cache (bda_attn_fwd_fp8kv), whose minimum bytes count K
    and V at one byte per element."""
    from diffusion_lm_block_bda_b300 import Problem
    w = W.named("c2")
    pb = Problem.from_workload(w)
    sets, sets8 = [], []
    for i in range(n_rot):
        inp = W.make_inputs(w, seed=i, with_dout=False)
        sets.append(tuple(inp[n].to(dev) for n in ("q", "k", "v")))
    q, k, v = sets[0]
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, pb.total_q), dtype=torch.float32, device=dev)
    ws = torch.zeros(bda.bda_attn_workspace_size(pb, False), dtype=torch.uint8, device=dev)
    host = torch.empty(bda.bda_attn_plan_size(pb), dtype=torch.uint8).pin_memory()
    bda.bda_attn_plan(pb, host, ws, stream)
    k_scale = torch.empty(w.hkv, dtype=torch.float32, device=dev)
    v_scale = torch.empty(w.hkv, dtype=torch.float32, device=dev)
    for (qq, kk, vv) in sets:
        k8 = torch.empty(kk.shape, dtype=torch.uint8, device=dev)
        v8 = torch.empty(vv.shape, dtype=torch.uint8, device=dev)
        bda.bda_kv_fp8_scales(kk, k_scale, stream)
        bda.bda_kv_fp8_scales(vv, v_scale, stream)
        bda.bda_kv_quantize_fp8(kk, k8, k_scale, stream)
        bda.bda_kv_quantize_fp8(vv, v8, v_scale, stream)
        sets8.append((qq, k8, v8))
    nbytes = sum(t.numel() * t.element_size() for t in (q, k, v, o, lse))
    nbytes8 = nbytes - (k.numel() + v.numel())

    def run(i, fp8):
        if fp8:
            bda.bda_attn_fwd_fp8kv(pb, *sets8[i % n_rot], k_scale, v_scale, o, lse, ws, stream)
        else:
            bda.bda_attn_fwd(pb, *sets[i % n_rot], o, lse, ws, stream)

    def timed(fp8):
        for i in range(n_rot):
            run(i, fp8)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for i, (e0, e1) in enumerate(evs):
            torch.cuda._sleep(400000)  # ~0.2 ms of GPU time while the host enqueues the launch
            e0.record(stream)
            run(i, fp8)
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3

    us = timed(False)
    us8 = timed(True)
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        bda.bda_attn_fwd(pb, q, k, v, o, lse, ws, cap)
    for _ in range(10):
        graph.replay()  # replays launch on the current stream, `stream`
    torch.cuda.synchronize()
    rounds = 200
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(4000000)  # ~2 ms of GPU time: the host enqueues every replay meanwhile
    g0.record(stream)
    for _ in range(rounds):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    st = bda.bda_attn_check_status(ws, stream)
    if st != bda.BDA_OK:
        raise RuntimeError(f"device status {st} after the decode measurement")
    achieved = nbytes / (us * 1e-6) / 1e9
    achieved8 = nbytes8 / (us8 * 1e-6) / 1e9
    return {"workload": "decode step: 32 queries over 2,080 keys (2,048 + one block of 32), "
                        "Hq=32, Hkv=8, d=128, forward only",
            "kernels": "split forward (9 chunks of <= 2 key tiles x 8 head groups = 72 CTAs) + combine",
            "bound": "hbm", "bytes": nbytes, "us": us, "achieved": achieved,
            "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
            "l2": f"launches rotate through {n_rot} Q/K/V copies (> L2)",
            "graph_us": g0.elapsed_time(g1) * 1e3 / rounds, "graph_rounds": rounds,
            "fp8": {"bytes": nbytes8, "us": us8, "achieved": achieved8, "peak": hbm_gbs,
                    "unit": "GB/s", "frac": achieved8 / hbm_gbs,
                    "kv": "e4m3 codes, one fp32 scale per KV head"}}


# ---------------------------------------------------------- side workloads
def side_measurement(bda, dev, stream, name, peak_burst, reps):
    """Useful TFLOPS of one more workload of the pages' kind, fwd + bwd, on
    inputs resident in HBM: "staircase" = 8 trajectories of a 1,024-token
    prefix and 16 copies of a 32-token block; "long" = one 32,768-token
    sequence, block 64.  The plan is built once; each rep is the forward and
    the three backward stages, back to back, timed with CUDA events on the
    launching stream (median per stage)."""
    from diffusion_lm_block_bda_b300 import Problem
    w = W.named(name)
    inp = W.make_inputs(w, seed=0)
    pb = Problem.from_workload(w)
    pairs = bda.bda_attn_count_pairs(pb)
    fwd_fl, bwd_fl = 4.0 * w.head_dim * w.hq * pairs, 10.0 * w.head_dim * w.hq * pairs
    q, k, v, dout = (inp[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty((w.hq, pb.total_q), dtype=torch.float32, device=dev)
    ws = torch.zeros(bda.bda_attn_workspace_size(pb, True), dtype=torch.uint8, device=dev)
    host = torch.empty(bda.bda_attn_plan_size(pb), dtype=torch.uint8).pin_memory()

    bda.bda_attn_plan(pb, host, ws, stream)  # the same plan serves every rep

    def rep(ev=None):
        if ev:
            ev[0].record(stream)
        bda.bda_attn_fwd(pb, q, k, v, o, lse, ws, stream)
        if ev:
            ev[1].record(stream)
        bda.bda_attn_bwd_preprocess(pb, o, dout, ws, stream)
        if ev:
            ev[2].record(stream)
        bda.bda_attn_bwd_dkdv(pb, q, k, v, lse, dout, dk, dv, ws, stream)
        if ev:
            ev[3].record(stream)
        bda.bda_attn_bwd_dq_convert(pb, dq, ws, stream)
        if ev:
            ev[4].record(stream)

    for _ in range(3):
        rep()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(reps)]
    for e in evs:
        rep(e)
    torch.cuda.synchronize()
    if bda.bda_attn_check_status(ws, stream) != bda.BDA_OK:
        raise RuntimeError(f"device status reports an error in the {name} measurement")
    med = [statistics.median(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(4)]
    fwd_ms, pre_ms, dkdv_ms, conv_ms = med
    step_ms = sum(med)
    useful = fwd_fl + bwd_fl
    return {"workload": w.note or w.name, "useful_pairs_per_head": pairs,
            "useful_gflop": useful / 1e9, "reps": reps,
            "stages_ms": {"fwd": round(fwd_ms, 4), "bwd_preprocess": round(pre_ms, 4),
                          "bwd_dkdv": round(dkdv_ms, 4), "bwd_dq_convert": round(conv_ms, 4)},
            "ms_per_step": step_ms, "value": useful / (step_ms * 1e-3) / 1e12, "unit": UNIT,
            "frac_of_peak": useful / (step_ms * 1e-3) / 1e12 / peak_burst,
            "fwd_tflops": fwd_fl / (fwd_ms * 1e-3) / 1e12,
            "bwd_dkdv_tflops": bwd_fl / (dkdv_ms * 1e-3) / 1e12,
            "peak": peak_burst, "peak_kind": "bf16 burst (measured)"}


# ------------------------------------------------------------------ native
def main():
    args = parse()
    rc = launch_ranks(args)
    if rc is not None:
        raise SystemExit(rc)
    if args.impl == "reference":
        # CPU-only arm: rank 0 runs the oracle, other ranks have nothing to do.
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup(args)
    if args.stub:
        run_stub(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    import diffusion_lm_block_bda_b300 as bda
    from diffusion_lm_block_bda_b300 import Problem

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w, seq_ids, shard_pairs = rank_workload(world, rank)
    inp = W.make_inputs(w, seed=rank)
    pb = Problem.from_workload(w)
    pairs = bda.bda_attn_count_pairs(pb)
    d, hq = w.head_dim, w.hq
    fwd_flops = 4.0 * d * hq * pairs
    bwd_flops = 10.0 * d * hq * pairs
    step_flops = fwd_flops + bwd_flops

    q, k, v, dout = (inp[n].to(dev) for n in ("q", "k", "v", "dout"))
    o = torch.empty_like(q)
    lse = torch.empty((hq, pb.total_q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.zeros(bda.bda_attn_workspace_size(pb, True), dtype=torch.uint8, device=dev)
    n_plan = bda.bda_attn_plan_size(pb)
    ring = [torch.empty(n_plan, dtype=torch.uint8).pin_memory() for _ in range(4)]
    ring_ev = [None] * len(ring)
    stream = torch.cuda.current_stream()
    step_no = [0]

    def plan():
        b = step_no[0] % len(ring)
        if ring_ev[b] is not None:
            ring_ev[b].synchronize()  # the copy from this host buffer has run
        bda.bda_attn_plan(pb, ring[b], ws, stream)
        ev = torch.cuda.Event()
        ev.record(stream)
        ring_ev[b] = ev
        step_no[0] += 1

    def step(evs=None, io=None):
        i_, o_ = io if io is not None else (dict(q=q, k=k, v=v, dout=dout),
                                            dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv))
        if evs:
            evs[0].record(stream)
        plan()
        if evs:
            evs[1].record(stream)
        bda.bda_attn_fwd(pb, i_["q"], i_["k"], i_["v"], o_["o"], o_["lse"], ws, stream)
        if evs:
            evs[2].record(stream)
        bda.bda_attn_bwd_preprocess(pb, o_["o"], i_["dout"], ws, stream)
        if evs:
            evs[3].record(stream)
        bda.bda_attn_bwd_dkdv(pb, i_["q"], i_["k"], i_["v"], o_["lse"], i_["dout"], o_["dk"],
                              o_["dv"], ws, stream)
        if evs:
            evs[4].record(stream)
        bda.bda_attn_bwd_dq_convert(pb, o_["dq"], ws, stream)
        if evs:
            evs[5].record(stream)

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    clk = Clocks(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or local))
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if bda.bda_attn_check_status(ws, stream) != bda.BDA_OK:
        raise SystemExit("device status reports a timeout during warm-up")

    # ---- device-resident timed region
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk.start()
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    stage_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in evs) / K for j in range(5)]
    gpu_launches = 4 * K

    # ---- end-to-end through the public API with host buffers.  Every step
    # uploads its inputs from pinned host memory and downloads all of its
    # outputs; as a training loop would, the upload of step j+1 and the
    # download of step j-1 run on their own streams while step j computes
    # (two device buffer sets, ordered by events).
    e2e = None
    if not args.no_e2e:
        host_in = {n: inp[n].pin_memory() for n in ("q", "k", "v", "dout")}
        out_like = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
        host_out = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in out_like.items()}
        sets = [({"q": q, "k": k, "v": v, "dout": dout}, out_like)]
        sets.append(({n: torch.empty_like(t) for n, t in sets[0][0].items()},
                     {n: torch.empty_like(t) for n, t in out_like.items()}))
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        in_ready = [torch.cuda.Event() for _ in sets]
        in_free = [torch.cuda.Event() for _ in sets]
        out_free = [torch.cuda.Event() for _ in sets]
        computed = [torch.cuda.Event() for _ in sets]
        for e in in_free + out_free:
            e.record(stream)

        def e2e_step(j):
            b = j % 2
            di, do = sets[b]
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(in_free[b])
                for n, t in host_in.items():
                    di[n].copy_(t, non_blocking=True)
                in_ready[b].record(s_h2d)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            step(io=(di, do))
            computed[b].record(stream)
            in_free[b].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(computed[b])
                for n, t in host_out.items():
                    t.copy_(do[n], non_blocking=True)
                out_free[b].record(s_d2h)

        for j in range(2):
            e2e_step(j)
        torch.cuda.synchronize()
        K2 = max(3, min(K, 20))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        s_h2d.wait_event(e0)
        s_d2h.wait_event(e0)
        for j in range(K2):
            e2e_step(j)
        for e in out_free:
            stream.wait_event(e)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K2, world)
        e2e_flops = sum_over_ranks(step_flops, world)
        e2e = {"value": e2e_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K2,
               "ms_per_step": e2e_ms,
               "overlap": "step j+1 upload and step j-1 download overlap step j (3 streams)"}
    clocks = clk.stop()
    status = bda.bda_attn_check_status(ws, stream)
    if status != bda.BDA_OK:
        raise SystemExit(f"device status {status} after the timed region")

    ms = max_over_ranks(total_ms / K, world)
    total_flops = sum_over_ranks(step_flops, world)
    value = total_flops / (ms * 1e-3) / 1e12
    peak_burst, peak_sust, hbm, peak_kind = measured_peaks()
    stages = dict(zip(["plan", "fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq_convert"],
                      [round(x, 4) for x in stage_ms]))
    # Both tensor-core kernels against the measured bf16 burst peak: the timed
    # region is a fraction of a second of back-to-back steps, not a
    # seconds-long run under the power cap.
    def roofline(kernel, flops, ms_):
        achieved = flops / (ms_ * 1e-3) / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak_burst,
                "unit": "TFLOP/s", "frac": achieved / peak_burst,
                "peak_kind": f"bf16 burst ({peak_kind})", "ms_per_launch": ms_,
                "algorithmic_flops_per_launch": flops}
    rl_dkdv = roofline("bda_bwd_dkdv", bwd_flops, stage_ms[3])
    rl_dkdv["traffic"] = profiled_traffic()
    rl_fwd = roofline("bda_fwd", fwd_flops, stage_ms[1])
    rl_fwd["traffic"] = profiled_traffic("fwd")

    if rank != 0:
        return
    out = {
        "impl": "native",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs)",
        "config": {"workload": WORKLOAD_NAME, "total_tokens": pb.total_q,
                   "seqlens": w.seqlens_q, "useful_pairs_per_head": pairs,
                   "useful_gflop_per_step": step_flops / 1e9,
                   "l2": "inputs larger than L2 (Q, O, dO, dQ 0.3 GB each)",
                   "parallelism": f"dp{world} (whole sequences, LPT-sharded)" if world > 1 else "1 GPU"},
        "frac_of_peak": value / peak_burst,
        "timed_region_ms": total_ms,
        "stages_ms": stages,
        "roofline": rl_dkdv,
        "rooflines": {"bda_bwd_dkdv": rl_dkdv, "bda_fwd": rl_fwd},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if world > 1:
        out["gpus_active"] = world
        out["shard_pairs_per_rank"] = shard_pairs
    out["fwd_tflops"] = fwd_flops / (stage_ms[1] * 1e-3) / 1e12
    out["bwd_tflops"] = bwd_flops / (sum(stage_ms[2:]) * 1e-3) / 1e12
    if e2e is not None:
        out["e2e"] = e2e
    # The side measurements and the CPU baseline belong to the one-GPU line;
    # a multi-GPU line carries the data-parallel step only.
    if not args.no_decode and world == 1:
        try:
            out["decode"] = decode_measurement(bda, dev, stream, hbm)
        except Exception as e:  # a side measurement: the main line is printed regardless
            torch.cuda.synchronize()
            out["decode"] = {"error": f"{type(e).__name__}: {e}"}
    if not args.no_side and world == 1:
        for key, name, reps in (("staircase", "c4", 20), ("long", "c5", 5)):
            try:
                out[key] = side_measurement(bda, dev, stream, name, peak_burst, reps)
            except Exception as e:  # a side measurement: the main line is printed regardless
                torch.cuda.synchronize()
                out[key] = {"error": f"{type(e).__name__}: {e}"}
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
