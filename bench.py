#!/usr/bin/env python3
"""Decode-attention benchmark: KV-cache HBM GB/s of one tree-attention decode step.

One step = one ``tree_attn_decode`` call (split-KV kernel + tree combine) for
one attention layer of the Llama-3.1-8B-shaped decode workload (B1, 32 query /
8 KV heads, d128, 131072 BF16 KV tokens).  Metric: algorithmic KV bytes
(every valid K and V element once) per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--num-splits P] [--kernel auto|mma|fma]

Rank 0 prints one JSON line.  For N > 1 (torchrun, one rank per GPU) every
rank runs its own replica -- the path has no cross-GPU step -- and the value is
the bytes all ranks processed divided by the slowest rank's time.
``--impl reference`` times the float64 CPU oracle instead, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention KV HBM GB/s (fraction of GB300 peak) and us/step vs context len"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per launch of the dominant kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by kernel family and
# workload, with the SHA-256 of the kernel source it was taken on; reported
# only while that source is unchanged.
NCU_TRAFFIC = {
    # warp-level tensor-core kernel, BF16 cache, 8B-shaped layer of 131072 tokens, 19 splits
    ("mma", "llama3.1-8b-decode-layer", 1): {
        "bytes_per_launch": 537316608 + 2760192, "num_splits": 19,
        "src_sha256": "59386695fba4fc9262837d650de324d47d9e706eacf4aa39fcf9eb83df155df7"},
    # tcgen05 kernel, the same layer with 8 and 16 queries per row (32 and 64 columns per KV head)
    ("tc05", "llama3.1-8b-decode-layer", 8): {
        "bytes_per_launch": 537053696 + 2923008, "num_splits": 19,
        "src_sha256": "7b2271b50877b0922013af7bf995687381b9919b45172c56d16581a9ad887131"},
    ("tc05", "llama3.1-8b-decode-layer", 16): {
        "bytes_per_launch": 537125632 + 3222016, "num_splits": 19,
        "src_sha256": "7b2271b50877b0922013af7bf995687381b9919b45172c56d16581a9ad887131"},
    # tcgen05 FP8 kernel, the same layer's E4M3 cache with 8 queries per row (32 columns per KV head)
    ("fp8tc05", "llama3.1-8b-decode-layer", 8): {
        "bytes_per_launch": 268646656 + 3003904, "num_splits": 19,
        "src_sha256": "5e686e4a74a3e0766f61d2ad2a9009fcea89ac37da8bc5e2c0252ec89b010c34"},
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3.1-8b-decode-layer")
    ap.add_argument("--num-splits", type=int, default=0, help="<= 0: the library's heuristic")
    ap.add_argument("--kernel", choices=["auto", "mma", "fma", "tc05"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=8192,
                    help="reference arm: tokens per row in each step's sample")
    ap.add_argument("--sweep-splits", default="",
                    help="comma list of split counts: print one JSON line per count and kernel, then exit")
    ap.add_argument("--sweep-context", default="",
                    help="comma list of context lengths for the workload's head shape (heuristic splits): "
                         "print one JSON line per length, then exit")
    ap.add_argument("--sweep-kernels", default="mma,fma")
    ap.add_argument("--sweep-len", type=int, default=0,
                    help="split sweep: context length per row instead of the workload's (0: the workload's)")
    ap.add_argument("--paged", type=int, default=0,
                    help="run through the paged-KV entry point with this page size (pages shuffled in a pool)")
    ap.add_argument("--queries", type=int, default=1,
                    help="queries per sequence (causal over the last positions, as when verifying draft tokens)")
    ap.add_argument("--paged-order", choices=["shuffled", "sequential"], default="shuffled",
                    help="physical page order: a random permutation of the pool, or each row's pages in order")
    ap.add_argument("--paged-layout", choices=["NHD", "HND"], default="NHD",
                    help="page layout: [pages][page][heads][d] (NHD) or [pages][heads][page][d] (HND)")
    ap.add_argument("--graph", action="store_true",
                    help="sweeps: capture the timed steps in one CUDA graph (removes the host's per-call cost)")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 E4M3 caches (the workload's K and V rounded with one scale per KV head)")
    ap.add_argument("--cluster-merge", action="store_true",
                    help="each row's (2..8) blocks merge through a thread-block cluster's shared memory")
    ap.add_argument("--merge", choices=["auto", "ticket", "cluster"], default="auto",
                    help="context sweep: the library's choice of split count and merge (auto), the "
                         "heuristic's split count merged by the last-arriving block (ticket), or "
                         "--cluster-merge (cluster)")
    ap.add_argument("--deterministic", action="store_true",
                    help="fixed chunk assignment (bitwise reproducible) instead of run-time balancing")
    return ap.parse_args(argv)


# --------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


_WARP_LEVEL = ("common.cuh", "emit.cuh", "kernels.h", "sched.cuh", "warp_mma.cuh")
_TCGEN05 = ("common.cuh", "kernels.h", "sched.cuh", "tc05.cuh")
# Per kernel family: its own source first, then every header it includes
# (directly or through another header), under softmax_tree_reduction_gb300/csrc.
KERNEL_SOURCES = {"mma": ("split_kv_mma.cu",) + _WARP_LEVEL,
                  "fp8": ("split_kv_fp8.cu",) + _WARP_LEVEL,
                  "fma": ("split_kv_fma.cuh", "common.cuh", "emit.cuh", "kernels.h", "sched.cuh"),
                  "tc05": ("split_kv_tc05.cu",) + _TCGEN05,
                  "fp8tc05": ("split_kv_tc05_fp8.cu",) + _TCGEN05}


def kernel_source_hash(kernel):
    """SHA-256 of the sources a kernel family is compiled from (its own file and
    the headers it includes) and of the host code that configures its launch."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel] + ("api.cu",):
        with open(os.path.join(ROOT, "softmax_tree_reduction_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None, interval_ms=50):
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
               f"-lms={self.interval_ms}"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for r in rows if self.t_start and self.t_stop and self.t_start <= r[0] <= self.t_stop + 0.05]
        used = inside if inside else rows[-3:]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in used if num(p[1]) is not None]
        mx = [num(p[2]) for _, p in used if num(p[2]) is not None]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for _, p in used:
            for name, val in zip(names, p[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(used),
                "samples_inside_timed_region": len(inside)}


def gpu_uuid(device):
    import torch
    try:
        u = torch.cuda.get_device_properties(device).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def max_over_ranks(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


L2_BYTES = 126.5 * 2**20   # GB300 L2 (the device reports its own size; this is the default)


def l2_note(kv_bytes, copies):
    try:
        import torch
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    except Exception:
        l2 = L2_BYTES
    mib = kv_bytes / 2**20
    if kv_bytes > l2:
        return (f"inputs larger than L2: {copies} K+V copies of {mib:.0f} MiB alternated step to step "
                f"(L2 {l2 / 2**20:.0f} MiB)")
    return (f"inputs fit in L2 ({copies} x {mib:.1f} MiB K+V vs {l2 / 2**20:.0f} MiB L2, not flushed): "
            "a latency figure, not an HBM one")


# ------------------------------------------------------------- CPU oracle
def oracle_baseline(w, inp, target_s, max_s=30.0, kv_bytes=None):
    """Time the float64 oracle as it stands on the host's cores.

    Sample: the whole workload (every head, every token), repeated until
    ``target_s`` seconds of CPU work; value = KV bytes processed / time.
    With ``k_scale`` in ``inp`` the caches are E4M3 codes (the FP8 oracle)."""
    import oracle
    threads = oracle.max_threads()
    if kv_bytes is None:
        kv_bytes = w.kv_bytes(inp["seqlens"])
    reps, elapsed = 0, 0.0
    while elapsed < target_s and elapsed < max_s:
        t0 = time.perf_counter()
        if "k_scale" in inp:
            oracle.attention_e4m3(inp["q"], inp["k"], inp["v"], inp["k_scale"], inp["v_scale"],
                                  inp["seqlens"], scale=w.softmax_scale, threads=threads)
        else:
            oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], w.softmax_scale, threads=threads)
        elapsed += time.perf_counter() - t0
        reps += 1
        if reps == 1 and elapsed * 2 > max_s:
            break
    return {"value": kv_bytes * reps / elapsed / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"whole workload ({w.name}), {reps} pass(es), {elapsed:.1f} s, float64 C oracle "
                      f"with {threads} OpenMP threads on {os.cpu_count()} host cores"}


def _clone_view(t):
    """A copy with the same strides (clone() of a permuted view keeps its layout)."""
    return t.clone(memory_format=torch_preserve_format())


def torch_preserve_format():
    import torch
    return torch.preserve_format


# ------------------------------------------------------------ our GPU arm
def run_ours(args, rank, world, local):
    import torch
    import softmax_tree_reduction_gb300 as ta
    from softmax_tree_reduction_gb300 import workloads

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ta.load()
    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(w)
    if args.queries > 1:
        gq = torch.Generator().manual_seed(w.seed + 1)
        inp["q"] = torch.randn(w.batch, w.num_q_heads, args.queries, w.head_dim, generator=gq).to(w.q_dtype)
    kv_names = ("q", "k", "v", "seqlens")
    if args.fp8:
        import dataclasses
        inp["k"], inp["k_scale"] = workloads.quantize_e4m3(inp["k"])
        inp["v"], inp["v_scale"] = workloads.quantize_e4m3(inp["v"])
        w = dataclasses.replace(w, kv_dtype=torch.float8_e4m3fn)
        kv_names = kv_names + ("k_scale", "v_scale")
    kv_bytes = w.kv_bytes(inp["seqlens"])
    dev = {k: inp[k].cuda() for k in kv_names}
    scales = dict(k_scale=dev.get("k_scale"), v_scale=dev.get("v_scale"), cluster_merge=args.cluster_merge)
    if args.paged:
        kp, vp, bt = workloads.page_pool(inp["k"], inp["v"], inp["seqlens"], args.paged, seed=w.seed,
                                         layout=args.paged_layout, shuffle=args.paged_order == "shuffled")
        dev.update(k=kp.cuda(), v=vp.cuda(), block_table=bt.cuda())
        del kp, vp
    # two copies of the KV cache, alternated step to step (each far larger than L2)
    copies = [dev, dict(dev, k=_clone_view(dev["k"]), v=_clone_view(dev["v"]))]
    shape = (ta.make_shape(dev["q"] if args.queries == 1 else dev["q"][:, :, 0], inp["k"]) if not args.paged else
             ta.TaShape(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_seqlen,
                        ta.TA_BF16 if w.q_dtype == torch.bfloat16 else ta.TA_F32,
                        ta.TA_E4M3 if args.fp8 else ta.TA_BF16 if w.kv_dtype == torch.bfloat16
                        else ta.TA_F32, 0.0,
                        dev["k"].stride(0), dev["k"].stride(2), dev["k"].stride(1)))
    if args.queries > 1:  # each (head, query) pair counts as a query head
        shape = ta.TaShape.from_buffer_copy(shape)
        shape.num_q_heads *= args.queries
    # the workload's row lengths are known on the host, as a serving engine knows its sequences'
    P = (args.num_splits if args.num_splits > 0
         else ta.tree_attn_pick_splits(shape, inp["seqlens"], page_size=args.paged))
    if args.cluster_merge and args.num_splits <= 0:
        P = min(P, 8)  # one cluster per row: at most 8 blocks
    kernel_used = args.kernel
    if args.fp8:
        # the library's choice for E4M3 caches: tcgen05 above 16 columns per KV
        # head (not with the cluster merge), else the warp-level FP8 kernel
        cols = w.group * args.queries
        tc = args.kernel == "tc05" or (args.kernel == "auto" and cols > 16 and not args.cluster_merge)
        kernel_used = "fp8tc05" if tc else "fp8"
    elif kernel_used == "auto":
        # the library's choice: warp-level tensor cores for BF16 with up to 16
        # columns per KV head; tcgen05 for 17..64 columns at head_dim 128 (the
        # warp-level kernel when the cluster merge is asked for)
        cols = w.group * args.queries
        bf16 = w.kv_dtype == torch.bfloat16 and w.q_dtype == torch.bfloat16
        if bf16 and 16 < cols <= 64 and w.head_dim == 128:
            kernel_used = "mma" if args.cluster_merge else "tc05"
        else:
            kernel_used = "mma" if (bf16 and cols <= 16) else "fma"
    B, Hq, d = dev["q"].shape[0], dev["q"].shape[1], dev["q"].shape[-1]
    out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(dev["q"].shape[:-1], dtype=torch.float32, device="cuda")
    nbytes = ta.tree_attn_workspace_bytes(shape, P)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i, events=None):
        c = copies[i & 1]
        if args.queries > 1:
            ta.tree_attn_decode_multi(c["q"], c["k"], c["v"], c["seqlens"], causal=True,
                                      block_table=c.get("block_table"), out=out, lse=lse, num_splits=P,
                                      workspace=ws, kernel=args.kernel, deterministic=args.deterministic,
                                      max_seqlen=w.max_seqlen if args.paged else None, **scales)
            return
        if args.paged:
            ta.tree_attn_decode_paged(c["q"], c["k"], c["v"], c["block_table"], c["seqlens"], out=out,
                                      lse=lse, num_splits=P, workspace=ws, kernel=args.kernel,
                                      deterministic=args.deterministic, max_seqlen=w.max_seqlen, **scales)
            return
        ta.tree_attn_decode(c["q"], c["k"], c["v"], c["seqlens"], out=out, lse=lse, num_splits=P,
                            workspace=ws, kernel=args.kernel, split_events=events,
                            deterministic=args.deterministic, **scales)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    assert ta.tree_attn_get_device_error() == 0

    sampler = ClockSampler(gpu_uuid(local))
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    # ---- timed region A: the API call as a user makes it
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark_start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    barrier(world)
    elapsed_ms = e0.elapsed_time(e1)
    launches = ta.tree_attn_launch_count(shape, P, args.kernel, args.deterministic)
    if launches == 1 or args.paged or args.queries > 1:
        # the step is the split-KV kernel alone: its launch duration is the step time
        split_ms = elapsed_ms / args.steps
    else:
        # ---- timed region B: same steps, split-KV kernel bracketed by events
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            step(i, events=evs[i])
        torch.cuda.synchronize()
        barrier(world)
        split_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # ---- per-step spread: each step bracketed by its own events (outside the timed regions)
    n_dist = min(args.steps, 1000)
    dev_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_dist)]
    torch.cuda.synchronize()
    for i in range(n_dist):
        dev_evs[i][0].record(stream)
        step(i)
        dev_evs[i][1].record(stream)
    torch.cuda.synchronize()
    per_step = sorted(a.elapsed_time(b) * 1e3 for a, b in dev_evs)
    dist = {"p10": round(per_step[n_dist // 10], 3), "p50": round(statistics.median(per_step), 3),
            "p90": round(per_step[min(n_dist - 1, (9 * n_dist) // 10)], 3), "steps": n_dist,
            "unit": "us", "how": "after the timed region, one event pair around each step "
                   "(which keeps it from overlapping its neighbours, so each is a standalone call)"}
    if rank == 0:
        time.sleep(0.1)
        sampler.stop()
    assert ta.tree_attn_get_device_error() == 0

    elapsed_ms = max_over_ranks(elapsed_ms, world)
    split_ms_max = max_over_ranks(split_ms, world)
    ms_per_step = elapsed_ms / args.steps
    value = kv_bytes * args.steps * world / (elapsed_ms / 1e3) / 1e9

    # ---- end to end: pinned host inputs -> device, decode, results -> host
    e2e = None
    if not args.no_e2e:
        n_e2e = max(1, min(args.e2e_steps, args.steps))
        host = {k: (dev[k].cpu() if args.paged and k in ("k", "v", "block_table") else inp[k]).pin_memory()
                for k in (kv_names + ("block_table",) if args.paged else kv_names)}
        dbuf = {k: torch.empty_like(host[k], device="cuda") for k in host}
        dscales = dict(k_scale=dbuf.get("k_scale"), v_scale=dbuf.get("v_scale"), cluster_merge=args.cluster_merge)
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = h_out.numel() * 4 + h_lse.numel() * 4

        def e2e_step():
            for k in host:
                dbuf[k].copy_(host[k], non_blocking=True)
            if args.queries > 1:
                ta.tree_attn_decode_multi(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["seqlens"], causal=True,
                                          block_table=dbuf.get("block_table"), out=out, lse=lse,
                                          num_splits=P, workspace=ws, kernel=args.kernel,
                                          max_seqlen=w.max_seqlen if args.paged else None, **dscales)
            elif args.paged:
                ta.tree_attn_decode_paged(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["block_table"],
                                          dbuf["seqlens"], out=out, lse=lse, num_splits=P, workspace=ws,
                                          kernel=args.kernel, max_seqlen=w.max_seqlen, **dscales)
            else:
                ta.tree_attn_decode(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["seqlens"], out=out, lse=lse,
                                    num_splits=P, workspace=ws, kernel=args.kernel, **dscales)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b), world)
        e2e = {"value": kv_bytes * n_e2e * world / (e2e_ms / 1e3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "ms_per_step": e2e_ms / n_e2e}
        del dbuf, host

    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    achieved = kv_bytes / (split_ms_max / 1e3) / 1e9
    tr = NCU_TRAFFIC.get((kernel_used, w.name, args.queries))
    traffic = None
    if (tr and tr.get("src_sha256") == kernel_source_hash(kernel_used) and tr.get("num_splits") == P
            and not args.paged and not args.deterministic):
        traffic = tr["bytes_per_launch"]
    cpu = None
    if not args.no_cpu_baseline:
        cpu = oracle_baseline(w, inp, args.cpu_seconds, kv_bytes=kv_bytes)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_step": round(ms_per_step * 1e3, 3),
        "us_per_step_dist": dist,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV, bf16 q, f16 mma / f32 accumulate" if args.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) Llama-shaped KV cache; no weights or datasets)"
                + ("; K and V rounded to E4M3 with one scale per KV head" if args.fp8 else ""),
        "config": {"workload": f"{w.name}: {w.description}", "batch": w.batch,
                   "seq_len": int(max(inp['seqlens'])), "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "num_splits": P,
                   "kernel": kernel_used, "deterministic": args.deterministic,
                   "cluster_merge": args.cluster_merge,
                   "kv_dtype": "e4m3 (per-KV-head scales)" if args.fp8 else str(w.kv_dtype).replace("torch.", ""),
                   "queries_per_sequence": args.queries,
                   "kv_layout": f"paged ({args.paged_layout}), {args.paged}-token pages "
                                f"{'shuffled in' if args.paged_order == 'shuffled' else 'in row order in'} a pool"
                   if args.paged
                   else "dense [B][Hkv][S][d]",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": l2_note(kv_bytes, len(copies))},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": "split_kv_tc05_fp8" if kernel_used == "fp8tc05" else f"split_kv_{kernel_used}",
                     # time per launch over the timed region, steps back to back: a launch
                     # starts its L2 prefetch while the previous one merges, so launches overlap
                     "launch_us_back_to_back": round(split_ms_max * 1e3, 3),
                     # one call on its own (an event pair around each step keeps it
                     # from overlapping its neighbours): the single-call figure
                     "standalone": {"us_p50": dist["p50"],
                                    "achieved": round(kv_bytes / (dist["p50"] / 1e6) / 1e9, 1),
                                    "frac": round(kv_bytes / (dist["p50"] / 1e6) / 1e9 / peak, 4)},
                     "bytes_per_launch": int(kv_bytes), "traffic": traffic,
                     "frac_of_8TBps": round(achieved / 8000.0, 4)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(args.steps * launches),
        "clocks": sampler.summary(),
    }


# ----------------------------------------------------------------- sweeps
def _time_steps(ta, torch, copies, P, kernel, steps, warmup, out, lse, ws, deterministic=False,
                graph=False, cluster_merge=False):
    """(ms per step, split-kernel ms) over ``steps`` decode calls; when the step
    is a single kernel the two are the same number.  With ``graph`` the steps
    are captured once in a CUDA graph and the replay is timed."""
    def step(i, events=None):
        c = copies[i % len(copies)]
        ta.tree_attn_decode(c["q"], c["k"], c["v"], c["seqlens"], out=out, lse=lse, num_splits=P,
                            workspace=ws, kernel=kernel, split_events=events,
                            deterministic=deterministic, k_scale=c.get("k_scale"), v_scale=c.get("v_scale"),
                            cluster_merge=cluster_merge)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                step(i)
        g.replay()
        torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    if graph:
        g.replay()
    else:
        for i in range(steps):
            step(i)
    b.record(s)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    if graph:
        assert ta.tree_attn_get_device_error() == 0
        return ms, ms
    shape = ta.make_shape(copies[0]["q"], copies[0]["k"])
    if ta.tree_attn_launch_count(shape, P, kernel, deterministic) == 1:
        assert ta.tree_attn_get_device_error() == 0
        return ms, ms
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        step(i, events=evs[i])
    torch.cuda.synchronize()
    split = statistics.mean(x.elapsed_time(y) for x, y in evs)
    assert ta.tree_attn_get_device_error() == 0
    return ms, split


def run_sweeps(args):
    """Sweep modes: seeded inputs drawn on the device (timing only; parity is
    covered by the tests), two KV copies alternated when they fit."""
    import torch
    import softmax_tree_reduction_gb300 as ta
    from softmax_tree_reduction_gb300 import workloads

    torch.cuda.set_device(0)
    ta.load()
    w = workloads.WORKLOADS[args.workload]
    if args.fp8:
        import dataclasses
        w = dataclasses.replace(w, kv_dtype=torch.float8_e4m3fn)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed)

    def draw(N):
        B, Hq, Hkv, d = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
        q = torch.randn(B, Hq, d, generator=gen, device="cuda").to(w.q_dtype)
        copies = []
        per_copy = 2 * B * Hkv * N * d * torch.empty((), dtype=w.kv_dtype).element_size()
        n_copies = 2 if per_copy <= (8 << 30) else 1
        for _ in range(n_copies):
            c = {"q": q, "seqlens": torch.full((B,), N, dtype=torch.int32, device="cuda")}
            if args.fp8:  # rounded to E4M3 with one scale per KV head
                c["k"], c["k_scale"] = workloads.quantize_e4m3(
                    (torch.randn(B, Hkv, N, d, generator=gen, device="cuda") * w.k_scale).to(torch.bfloat16))
                c["v"], c["v_scale"] = workloads.quantize_e4m3(
                    torch.randn(B, Hkv, N, d, generator=gen, device="cuda").to(torch.bfloat16))
            else:
                c["k"] = (torch.randn(B, Hkv, N, d, generator=gen, device="cuda") * w.k_scale).to(w.kv_dtype)
                c["v"] = torch.randn(B, Hkv, N, d, generator=gen, device="cuda").to(w.kv_dtype)
            copies.append(c)
        return copies

    peak, _ = load_peaks()
    lines = []
    if args.sweep_splits:
        n_tok = args.sweep_len if args.sweep_len > 0 else w.max_seqlen
        copies = draw(n_tok)
        shape = ta.make_shape(copies[0]["q"], copies[0]["k"])
        kv_bytes = w.kv_bytes(np.full(w.batch, n_tok))
        B, Hq, d = copies[0]["q"].shape
        out = torch.empty(B, Hq, d, device="cuda")
        lse = torch.empty(B, Hq, device="cuda")
        heur = ta.tree_attn_pick_splits(shape)
        for kern in (["auto"] if args.fp8 else args.sweep_kernels.split(",")):
            for P in [int(x) for x in args.sweep_splits.split(",")]:
                ws = torch.empty(max(16, ta.tree_attn_workspace_bytes(shape, P)), dtype=torch.uint8,
                                 device="cuda")
                ms, split = _time_steps(ta, torch, copies, P, kern, args.steps, args.warmup, out, lse, ws,
                                        args.deterministic, args.graph)
                lines.append({"sweep": "splits", "workload": w.name, "kernel": "fp8" if args.fp8 else kern,
                              "context": n_tok, "num_splits": P,
                              "deterministic": args.deterministic, "graph": args.graph,
                              "heuristic": P == heur, "us_per_step": round(ms * 1e3, 3),
                              "split_kernel_us": round(split * 1e3, 3),
                              "step_gbs": round(kv_bytes / (ms / 1e3) / 1e9, 1),
                              "kernel_gbs": round(kv_bytes / (split / 1e3) / 1e9, 1),
                              "frac_of_measured_peak": round(kv_bytes / (split / 1e3) / 1e9 / peak, 4)})
                print(json.dumps(lines[-1]), flush=True)
        del copies
        torch.cuda.empty_cache()
    if args.sweep_context:
        for N in [int(x) for x in args.sweep_context.split(",")]:
            copies = draw(N)
            shape = ta.make_shape(copies[0]["q"], copies[0]["k"])
            P = ta.tree_attn_pick_splits(shape)
            merge = "cluster" if args.cluster_merge else args.merge
            if merge == "cluster":
                P = min(P, 8)  # one cluster per row: at most 8 blocks
            kv_bytes = w.kv_bytes(np.full(w.batch, N))
            B, Hq, d = copies[0]["q"].shape
            out = torch.empty(B, Hq, d, device="cuda")
            lse = torch.empty(B, Hq, device="cuda")
            ws = torch.empty(max(16, ta.tree_attn_workspace_bytes(shape, P)), dtype=torch.uint8,
                             device="cuda")
            ms, split = _time_steps(ta, torch, copies, 0 if merge == "auto" else P, args.kernel, args.steps,
                                    args.warmup, out, lse, ws, args.deterministic, args.graph,
                                    merge == "cluster")
            lines.append({"sweep": "context", "workload": w.name, "kv": "e4m3" if args.fp8 else "bf16",
                          "merge": merge,
                          "context": N, "num_splits": P,
                          "graph": args.graph, "l2": "fits" if w.kv_bytes(np.full(w.batch, N)) * len(copies)
                          < L2_BYTES else "exceeds",
                          "us_per_step": round(ms * 1e3, 3), "split_kernel_us": round(split * 1e3, 3),
                          "step_gbs": round(kv_bytes / (ms / 1e3) / 1e9, 1),
                          "frac_of_measured_peak": round(kv_bytes / (ms / 1e3) / 1e9 / peak, 4)})
            print(json.dumps(lines[-1]), flush=True)
            del copies
            torch.cuda.empty_cache()
    return lines


# ------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return None
    import numpy as np
    import torch
    import oracle
    from softmax_tree_reduction_gb300 import workloads

    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(w)
    n = min(args.ref_tokens, int(inp["seqlens"].min()))
    sub_len = torch.full_like(inp["seqlens"], n)
    kv_bytes = w.kv_bytes(sub_len)
    threads = oracle.max_threads()
    k_sub = inp["k"][:, :, :n].contiguous()
    v_sub = inp["v"][:, :, :n].contiguous()

    def step():
        oracle.attention(inp["q"], k_sub, v_sub, sub_len, w.softmax_scale, threads=threads)

    for _ in range(max(args.warmup, 3)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = kv_bytes * args.steps / el / 1e9
    sample = (f"first {n} tokens of every (row, head) of {w.name} per step; float64 C oracle, "
              f"{threads} OpenMP threads on {os.cpu_count()} host cores")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Llama-shaped KV cache)",
        "config": {"workload": f"{w.name}: {w.description}", "batch": w.batch, "seq_len": n,
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.sweep_splits or args.sweep_context:
        run_sweeps(args)
        return 0
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
