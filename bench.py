#!/usr/bin/env python3
"""Benchmark of one paged-KV decode step on GB300.

A step is one pass of the hot path over one batch: ``pa_reshape_and_cache``
writes each sequence's new K/V token into its slot, then ``pa_decode``
attends every sequence over its paged cache (split-K partitions + log-sum-exp
reduce where a sequence spans several partitions).

Default workload: LLaMA-style GQA decode -- 256 sequences, 32 query heads,
8 KV heads, head_dim 128, bf16, block_size 16, context lengths U{1..4096},
blocks scattered over a pool 1.25x the size needed (2.7 GB, far larger than
L2, so no step re-reads the previous step's data from L2).

Output: one JSON line (rank 0).  ``value`` is achieved HBM GB/s of the whole
step: algorithmic bytes (valid K/V rows once per kv head + Q + out + tables
+ lengths for the decode, new rows + slots for the cache write) over device
time.  ``--impl reference`` times the CPU oracle instead, on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak) and tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(source: str) -> str:
    import hashlib
    src = os.path.join(ROOT, "paged_kv_cache_224_gb300", "csrc", source)
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def load_traffic(kernel_key: str, sources):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if
    it was taken on the current sources: an entry lists the hash of every
    source file the kernel is built from, comma-separated, and each of
    `sources` must be among them."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = [source_hash(s) for s in sources]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel_key and all(h in parts[1].split(",") for h in want):
            return float(parts[2])
    return None


# The files each kernel is compiled from (its own source and the device
# headers it includes), for the traffic entries' hashes.
DECODE_SOURCES = ["pa_decode.cuh", "pa_device.cuh"]
DECODE_TC_SOURCES = ["pa_decode_tc.cuh", "pa_decode_tc.cu", "pa_tcgen05.cuh", "pa_device.cuh"]
PREFILL_SOURCES = ["pa_prefill.cu", "pa_prefill.cuh", "pa_tcgen05.cuh", "pa_device.cuh"]
MIXED_SOURCES = ["pa_mixed.cuh", "pa_mixed_bf16.cu", "pa_prefill.cuh", "pa_decode_tc.cuh", "pa_tcgen05.cuh",
                 "pa_device.cuh"]


def decode_kernel_of(group: int, head_dim: int):
    """The decode kernel the library runs for a head group, and its sources."""
    if group == 8 and head_dim == 128:
        return "decode_tc_kernel", DECODE_TC_SOURCES
    return "decode_kernel", DECODE_SOURCES


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""
        return False

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def make_case(name: str, seed_offset: int):
    from paged_kv_cache_224_gb300 import workload as wl
    if name == "tiny":
        return wl.tiny_case()
    if name == "llama_gqa":
        return wl.llama_gqa_case(seed=1002 + seed_offset)
    if name == "opt13b_mha":
        return wl.opt13b_case(seed=1001 + seed_offset)
    if name == "long_context":
        return wl.long_context_case(block_size=16, seed=1004 + seed_offset)
    if name == "long_context_bs32":
        return wl.long_context_case(block_size=32, seed=1004 + seed_offset)
    if name in ("shared_prefix", "shared_prefix_grouped"):
        return wl.shared_prefix_case(seed=1003 + seed_offset)
    raise SystemExit(f"unknown workload {name}")


def cpu_oracle_sample(case, tensors, nseq: int, threads: int):
    """Time the CPU oracle on the first ``nseq`` sequences of the step.
    Returns (seconds, algorithmic bytes of the sample)."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from tests.helpers import oracle_inputs
    oracle.build()
    seqs = list(range(min(nseq, case.num_seqs)))
    inp = oracle_inputs(case, tensors, seqs)
    kc, vc = inp["k_cache"], inp["v_cache"]
    lens = inp["context_lens"]
    t0 = time.perf_counter()
    oracle.reshape_and_cache(inp["new_key"], inp["new_value"], kc, vc, inp["slot_mapping"], case.block_size)
    oracle.decode(inp["query"], kc, vc, inp["block_tables"], lens, case.scale, case.dtype,
                  num_threads=threads)
    dt = time.perf_counter() - t0
    el = 2
    kv = int(lens.astype(np.int64).sum()) * 2 * case.num_kv_heads * case.head_dim * el
    q = len(seqs) * case.num_heads * case.head_dim * el
    return dt, kv + 2 * q


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step is one oracle decode
    over a bounded sample of the workload's sequences."""
    if rank != 0:
        return
    if args.workload in ("chunked_prefill", "prefill_batch", "mixed"):
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the CPU oracle's "
                              "decode step; run it on a decode workload"}), flush=True)
        return
    case = make_case(args.workload, 0)
    tensors = case.materialize("cpu")
    threads = os.cpu_count() or 1
    nseq = args.ref_seqs
    for _ in range(args.warmup):
        cpu_oracle_sample(case, tensors, nseq, threads)
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        dt, b = cpu_oracle_sample(case, tensors, nseq, threads)
        total_t += dt
        total_b += b
    gbs = total_b / total_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total_t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "sample_seqs": min(nseq, case.num_seqs)},
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {min(nseq, case.num_seqs)} of {case.num_seqs} sequences "
                                       f"of {case.name}, cache write + decode, per step"},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill_bench(args, world, rank, local, dev, stream):
    """One chunked-prefill step: write the chunk's K/V (pa_reshape_and_cache),
    then attend the 512-row chunk over its 8192-token paged prefix."""
    import paged_kv_cache_224_gb300 as pa
    from paged_kv_cache_224_gb300 import workload as wl
    batch = args.workload == "prefill_batch"
    case = wl.prefill_batch_case(seed=1005 + rank) if batch else wl.chunked_prefill_case(seed=1004 + rank)
    t = case.materialize(dev)
    slots = torch.as_tensor(case.slot_mapping, device=dev)
    bt = torch.as_tensor(case.block_tables if batch else case.block_table, device=dev)
    out = torch.empty_like(t["query"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # stream-K over one CTA per SM (partials in the workspace), or one CTA per unit
    stream_k = args.prefill_schedule == "stream_k"
    ws = pa.prefill_workspace(t["query"], case.num_kv_heads, len(case.chunk_lens) if batch else 1) if stream_k else None

    def prefill():
        if batch:
            pa.pa_prefill_batch(out, t["query"], t["k_cache"], t["v_cache"], bt, case.prefix_lens, case.chunk_lens,
                                case.scale, d_err=err, workspace=ws)
        else:
            pa.pa_prefill_chunk(out, t["query"], t["k_cache"], t["v_cache"], bt, case.prefix_len, case.scale,
                                d_err=err, workspace=ws)

    def step():
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)
        prefill()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"device error flags {int(err.item()):#x}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    flops = case.flops()
    total = sum_over_ranks(float(flops) * args.steps, world, dev)
    tflops = total / (elapsed_ms / 1e3) / 1e12
    pf_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    achieved = flops / (pf_ms / 1e3) / 1e12
    peak, kind = FALLBACK_BF16_TFLOPS, "fallback"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        peak, kind = float(json.load(open(path))["bf16_tflops"]), "measured"
    if rank == 0:
        line = {"metric": "chunked prefill attention: achieved TFLOP/s (% of bf16 dense peak)",
                "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
                "data": "synthetic",
                "config": {"workload": case.name,
                           "prefix_len": case.prefix_lens.tolist() if batch else case.prefix_len,
                           "chunk_len": case.chunk_lens.tolist() if batch else case.chunk_len,
                           "num_heads": case.num_heads, "num_kv_heads": case.num_kv_heads,
                           "head_dim": case.head_dim, "block_size": case.block_size,
                           "step": "pa_reshape_and_cache (chunk K/V) + "
                                   + ("pa_prefill_batch (one launch)" if batch else "pa_prefill_chunk"),
                           "schedule": ("stream-K: one CTA per SM over equal shares of the key tiles, "
                                        "log-sum-exp merge of split units" if stream_k else "one CTA per unit"),
                           "l2": "each kv head's KV is reused from L2 by its row tiles"},
                "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                             "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                             "traffic": load_traffic(case.name, PREFILL_SOURCES),
                             "kernel": "prefill_tc_kernel", "flops_per_launch": flops, "avg_ms": round(pf_ms, 5),
                             "peak_kind": f"{kind} (bf16 dense, burst)"},
                "gpu_launches": 2 * args.steps, "clocks": clk.summary()}
        print(json.dumps(line), flush=True)


def run_mixed_bench(args, world, rank, local, dev, stream):
    """One continuous-batching step of a 64/8-head model: write the step's new
    K/V (one decode token for each of 256 sequences, a 512-token prompt chunk),
    then pa_mixed_step (the chunk's prefill and the decodes, concurrently).
    The same step with the two calls one after the other is timed beside it."""
    import paged_kv_cache_224_gb300 as pa
    from paged_kv_cache_224_gb300 import workload as wl
    case = wl.mixed_case(seed=1006 + rank)
    t = case.materialize(dev)
    slots = torch.as_tensor(case.slot_mapping, device=dev)
    pbt = torch.as_tensor(case.prefill_tables, device=dev)
    dbt = torch.as_tensor(case.decode_tables, device=dev)
    lens = torch.as_tensor(case.context_lens, device=dev)
    pout = torch.empty_like(t["prefill_query"])
    dout = torch.empty_like(t["decode_query"])
    ws = pa.decode_workspace(t["decode_query"], case.num_kv_heads, case.block_size, case.max_context_len,
                             args.partition_tokens)
    # one launch (prefill CTAs and persistent decode CTAs in one grid) needs the mixed-step workspace
    ws_one = pa.mixed_workspace(t["prefill_query"], t["decode_query"], case.num_kv_heads, case.block_size,
                                len(case.chunk_lens), case.max_context_len, args.partition_tokens)
    ws_pf = pa.prefill_workspace(t["prefill_query"], case.num_kv_heads, len(case.chunk_lens))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    part = pa.pa_decode_partition_tokens(case.num_seqs, case.num_heads, case.num_kv_heads, case.block_size,
                                         case.max_context_len, args.partition_tokens)

    def write():
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)

    def one_launch():
        pa.pa_mixed_step(pout, t["prefill_query"], pbt, case.prefix_lens, case.chunk_lens, dout, t["decode_query"],
                         dbt, lens, t["k_cache"], t["v_cache"], case.scale, case.max_context_len,
                         partition_tokens=args.partition_tokens, workspace=ws_one, d_err=err)

    def concurrent():
        pa.pa_mixed_step(pout, t["prefill_query"], pbt, case.prefix_lens, case.chunk_lens, dout, t["decode_query"],
                         dbt, lens, t["k_cache"], t["v_cache"], case.scale, case.max_context_len,
                         partition_tokens=args.partition_tokens, workspace=ws, d_err=err)

    def sequential():
        pa.pa_prefill_batch(pout, t["prefill_query"], t["k_cache"], t["v_cache"], pbt, case.prefix_lens,
                            case.chunk_lens, case.scale, d_err=err, workspace=ws_pf)
        pa.pa_decode(dout, t["decode_query"], t["k_cache"], t["v_cache"], dbt, lens, case.scale,
                     case.max_context_len, partition_tokens=args.partition_tokens, workspace=ws, d_err=err)

    def timed(body):
        for _ in range(args.warmup):
            write()
            body()
        torch.cuda.synchronize()
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            a.record(stream)
            for _ in range(args.steps):
                write()
                body()
            b.record(stream)
            torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(a.elapsed_time(b), world, dev) / args.steps, clk

    ms_mixed, clk = timed(one_launch)
    ms_two, _ = timed(concurrent)
    ms_seq, _ = timed(sequential)
    if int(err.item()) != 0:
        raise SystemExit(f"device error flags {int(err.item()):#x}")
    peak, peak_kind = load_peaks()
    dec_gbs = case.decode_bytes() / (ms_mixed / 1e3) / 1e9
    if rank == 0:
        line = {"metric": "mixed continuous-batching step (512-token prompt chunk + 256 decodes): ms per step",
                "value": round(ms_mixed, 5), "unit": "ms", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_mixed, 5), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": case.dtype, "data": "synthetic",
                "config": {"workload": case.name, "num_decode": case.num_seqs, "context_lens": "U{1..4096}",
                           "prefix_len": case.prefix_lens.tolist(), "chunk_len": case.chunk_lens.tolist(),
                           "num_heads": case.num_heads, "num_kv_heads": case.num_kv_heads,
                           "head_dim": case.head_dim, "block_size": case.block_size, "partition_tokens": part,
                           "step": "pa_reshape_and_cache (all new K/V) + pa_mixed_step (one launch)",
                           "l2": "inputs larger than L2: %.2f GB of decode KV per step" % (case.decode_bytes() / 1e9)},
                "two_launches_ms_per_step": round(ms_two, 5),
                "sequential_ms_per_step": round(ms_seq, 5),
                "overlap_gain": round(ms_seq / ms_mixed - 1.0, 4),
                "prefill_tflops_in_step": round(case.prefill_flops() / (ms_mixed / 1e3) / 1e12, 2),
                "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
                             "frac": round(dec_gbs / peak, 4), "traffic": load_traffic(case.name, MIXED_SOURCES),
                             "kernel": "the decode half's KV streamed per step while the prompt chunk runs",
                             "bytes_per_launch": case.decode_bytes(), "avg_ms": round(ms_mixed, 5),
                             "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
                "gpu_launches": 2 * args.steps, "clocks": clk.summary()}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama_gqa", choices=["tiny", "llama_gqa", "opt13b_mha", "long_context", "long_context_bs32",
                             "shared_prefix", "shared_prefix_grouped", "chunked_prefill", "prefill_batch", "mixed"])
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--prefill-schedule", default="stream_k", choices=["stream_k", "per_unit"],
                    help="prefill workloads: with a workspace (stream-K) or without (one CTA per unit)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seqs", type=int, default=64, help="sequences in the CPU-baseline sample")
    ap.add_argument("--ref-seqs", type=int, default=2, help="sequences per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", action="store_true",
                    help="decode workloads: before every timed step write a 256 MB buffer (twice L2), then read "
                         "another, so no line of the previous step survives and the written lines are evicted "
                         "before the step; the step time is the sum of per-step events, which exclude the flush")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import paged_kv_cache_224_gb300 as pa
    from paged_kv_cache_224_gb300 import build as pa_build
    pa_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    if args.workload in ("chunked_prefill", "prefill_batch", "mixed"):
        (run_mixed_bench if args.workload == "mixed" else run_prefill_bench)(args, world, rank, local, dev, stream)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    case = make_case(args.workload, rank)
    t = case.materialize(dev)
    tensors_host_copy_needed = rank == 0 and not args.no_cpu_baseline
    cpu_sample = None
    if tensors_host_copy_needed:
        # the oracle reads the pre-step pool: take its sample before any kernel runs
        cpu_sample = cpu_oracle_sample(case, t, args.cpu_seqs, os.cpu_count() or 1)
        cpu_seqs_1 = max(4, args.cpu_seqs // 8)
        cpu_sample_1 = cpu_oracle_sample(case, t, cpu_seqs_1, 1)

    slots = torch.as_tensor(case.slot_mapping, device=dev)
    bt = torch.as_tensor(case.block_tables, device=dev)
    lens = torch.as_tensor(case.context_lens, device=dev)
    out = torch.empty_like(t["query"])
    pt = args.partition_tokens
    # shared_prefix_grouped: the same workload, decoded with the shared-prefix
    # entry point (each group's prefix blocks read once)
    grouped = args.workload == "shared_prefix_grouped"
    if grouped:
        n = pa.pa_decode_shared_prefix_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim,
                                                       case.block_size, case.max_context_len,
                                                       case.shared_blocks, pt)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    else:
        ws = pa.decode_workspace(t["query"], case.num_kv_heads, case.block_size, case.max_context_len, pt)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    part = pa.pa_decode_partition_tokens(case.num_seqs, case.num_heads, case.num_kv_heads, case.block_size,
                                         case.max_context_len, pt)
    max_parts = -(-case.max_context_len // part)
    pairs = torch.as_tensor(case.cow_pairs, device=dev) if case.cow_pairs.shape[0] else None
    cow_ws = (torch.empty(pa.pa_copy_blocks_workspace_bytes(pairs.shape[0]), dtype=torch.uint8, device=dev)
              if pairs is not None else None)
    # copy-on-write: clear, count and copy kernels
    launches_per_step = (3 if pairs is not None else 0) + 1 + (3 if grouped else 1 + (1 if max_parts > 1 else 0))

    def decode(q, bt_, lens_):
        if grouped:
            pa.pa_decode_shared_prefix(out, q, t["k_cache"], t["v_cache"], bt_, lens_, case.scale,
                                       case.max_context_len, case.group_size, case.shared_blocks,
                                       partition_tokens=pt, workspace=ws, d_err=err)
        else:
            pa.pa_decode(out, q, t["k_cache"], t["v_cache"], bt_, lens_, case.scale,
                         case.max_context_len, partition_tokens=pt, workspace=ws, d_err=err)

    def cow():
        # copy-on-write of shared blocks before the tails are written (idempotent across steps)
        if pairs is not None:
            pa.pa_copy_blocks(t["k_cache"], t["v_cache"], pairs, d_err=err, workspace=cow_ws)

    def step():
        cow()
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)
        decode(t["query"], bt, lens)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"device error flags {int(err.item()):#x}")

    # ---- device-timed region: K steps, inputs resident in HBM
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    flush = torch.zeros((2, 256 << 20), dtype=torch.uint8, device=dev) if args.l2_flush else None
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)
    st_ev = [(torch.cuda.Event(enable_timing=True),) for _ in range(args.steps)] if flush is not None else None
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                # write 2x L2, then read another 2x L2 so the written lines are
                # evicted (and written back) here, not inside the next step
                flush[0].fill_(i & 0xff)
                flush_sink.add_(flush[1].sum(dtype=torch.int64))
                st_ev[i][0].record(stream)
            cow()
            pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)
            ev[i][0].record(stream)
            decode(t["query"], bt, lens)
            ev[i][1].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    if flush is not None:
        # flushes fall between steps: the step time is the sum of its own events
        elapsed_ms = sum(a.elapsed_time(b[1]) for a, b in zip((e[0] for e in st_ev), ev))
    else:
        elapsed_ms = start.elapsed_time(stop)
    decode_ms = [a.elapsed_time(b) for a, b in ev]
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    step_bytes = case.decode_bytes() + case.reshape_bytes() + case.copy_bytes()
    total_bytes = sum_over_ranks(float(step_bytes) * args.steps, world, dev)
    gbs = total_bytes / (elapsed_ms / 1e3) / 1e9
    ms_per_step = elapsed_ms / args.steps
    tokens_per_s = sum_over_ranks(float(case.num_seqs), world, dev) / (ms_per_step / 1e3)

    peak, peak_kind = load_peaks()
    dec_avg_ms = statistics.mean(decode_ms)
    dec_achieved = case.decode_bytes() / (dec_avg_ms / 1e3) / 1e9
    G = case.num_heads // case.num_kv_heads
    kname, ksrc = decode_kernel_of(G, case.head_dim)
    if grouped:
        # three kernels (prefix pass, tail pass, reduce): the traffic entry is
        # their sum, valid while both decode sources are unchanged
        pre_src = decode_kernel_of(G * case.group_size, case.head_dim)[1]
        traffic = load_traffic(f"decode_{case.name}_grouped", sorted(set(pre_src) | set(ksrc)))
    else:
        traffic = load_traffic(f"decode_{case.name}", ksrc)

    # ---- end to end through the C ABI's host-input step: every step copies
    # its inputs from pinned host memory (queries, new K/V, slots, copy pairs,
    # block tables, lengths), runs the step and copies the output back
    pin = lambda x: x.cpu().pin_memory()  # noqa: E731
    h_q, h_nk, h_nv = pin(t["query"]), pin(t["new_key"]), pin(t["new_value"])
    h_slots, h_bt, h_lens = pin(slots), pin(bt), pin(lens)
    h_pairs = pin(pairs) if pairs is not None else None
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_nk, h_nv, h_slots, h_bt, h_lens, h_pairs)
              if x is not None)
    d2h = h_out.numel() * h_out.element_size()
    staging = torch.empty(max(1, pa.pa_decode_step_host_staging_bytes(
        case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim, case.block_size, h_bt.shape[1],
        case.max_context_len, h_nk.shape[0], 0 if h_pairs is None else h_pairs.shape[0],
        case.group_size if grouped else 0, case.shared_blocks if grouped else 0, pt)), dtype=torch.uint8, device=dev)

    def e2e_step():
        pa.pa_decode_step_host(h_out, h_q, h_nk, h_nv, h_slots, h_bt, h_lens, t["k_cache"], t["v_cache"],
                               case.scale, case.max_context_len, pairs=h_pairs,
                               group_size=case.group_size if grouped else 0,
                               prefix_blocks=case.shared_blocks if grouped else 0, partition_tokens=pt,
                               staging=staging, d_err=err)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.e2e_steps
    e2e_bytes = sum_over_ranks(float(step_bytes), world, dev)
    e2e_gbs = e2e_bytes / (e2e_ms / 1e3) / 1e9
    if int(err.item()) != 0:
        raise SystemExit(f"device error flags {int(err.item()):#x}")

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
            "data": "synthetic",
            "config": {"workload": case.name, "num_seqs": case.num_seqs, "num_heads": case.num_heads,
                       "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
                       "block_size": case.block_size, "context_lens": "uniform, see workload",
                       "max_context_len": case.max_context_len, "partition_tokens": part,
                       "pool_blocks": case.num_blocks,
                       "l2": ("L2 flushed before every step (256 MB written, then 256 MB read, outside the step's events); " if flush is not None
                              else "") + "inputs larger than L2: KV pool %.2f GB, %.2f GB read per step" % (
                           2 * case.num_blocks * case.num_kv_heads * case.block_size * case.head_dim * 2 / 1e9,
                           case.kv_bytes() / 1e9),
                       "step": ("pa_copy_blocks + " if pairs is not None else "")
                               + f"pa_reshape_and_cache ({case.num_new_tokens} tokens) + "
                               + ("pa_decode_shared_prefix (groups of %d, %d shared blocks)" % (
                                   case.group_size, case.shared_blocks) if grouped else "pa_decode"),
                       "unique_kv_bytes": case.unique_kv_bytes(),
                       "parallelism": f"replicas x{world}, sequences sharded, no collective"},
            "pct_of_peak": round(100 * gbs / peak, 2),
            "tokens_per_s": round(tokens_per_s, 1),
            "context_tokens_per_s": round(float(case.context_lens.sum()) * world / (ms_per_step / 1e3), 1),
            "roofline": {"bound": "hbm", "achieved": round(dec_achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(dec_achieved / peak, 4), "traffic": traffic,
                         "kernel": "pa_decode_shared_prefix (%s prefix pass + %s tail pass + decode_reduce_kernel)" % (
                                   decode_kernel_of(G * case.group_size, case.head_dim)[0], kname)
                                   if grouped else "pa_decode (%s + decode_reduce_kernel)" % kname,
                         "bytes_per_launch": case.decode_bytes(), "avg_ms": round(dec_avg_ms, 5),
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback"},
            "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "api": "pa_decode_step_host (C ABI, pinned host buffers)",
                    "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        }
        if cpu_sample is not None:
            dt, b = cpu_sample
            line["cpu_baseline"] = {"value": round(b / dt / 1e9, 4), "unit": "GB/s",
                                    "cores": os.cpu_count() or 1, "kind": "oracle",
                                    "sample": f"first {min(args.cpu_seqs, case.num_seqs)} of {case.num_seqs} "
                                              f"sequences of {case.name}: cache write + decode, fp64",
                                    "single_thread": {
                                        "value": round(cpu_sample_1[1] / cpu_sample_1[0] / 1e9, 4), "cores": 1,
                                        "sample": f"first {min(cpu_seqs_1, case.num_seqs)} sequences, same step"}}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
