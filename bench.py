#!/usr/bin/env python
"""Throughput of the packed, document-masked, chunked causal attention path
on GB300 ("ByteScale: Communication-Efficient Scaling of LLM Training with a
2048K Context Length on 16384 GPUs", research digest, sections 2-3.2).

One step = the whole hot path on one micro-batch resident in HBM:
  plan (scans, chunk/block tables, best-fit shards, heaviest-first work list)
  -> attention forward (FUSED: partials merged by the online softmax)
  -> per-shard FLOPs.
Metric: useful causal-attention TFLOP/s, 4*d*Hq*sum_i s_i(s_i+1)/2 per step,
and its fraction of the bf16 dense tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload seq2m]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

The default workload is the largest single-GPU one: one 2,097,152-token
sequence, C = 8,192 (256 chunks, 32,896 causal blocks), Hq = 32, Hkv = 8,
d = 128.  After it, the 131,072-token sequence is timed in FUSED and SPLIT
mode as extra entries of the same line.

Prints ONE JSON line (rank 0).  With --gpus N > 1 the script starts N ranks
itself (torchrun, one per GPU) unless it already runs under torchrun; every
rank runs an independent replica (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "varlen causal attention fwd useful TFLOP/s and fraction of GB300 BF16 peak"
L2_BYTES = 129 * 10**6
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
ATTN_SRC = os.path.join(ROOT, "packed_varlen_attention_aware_gb300", "csrc", "attn_fwd.cu")


def useful_flops(lengths, d, hq) -> int:
    return sum(4 * d * hq * s * (s + 1) // 2 for s in lengths)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            out = {}
            for key in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs"):
                v = j.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                out[key] = float(v) if v is not None else FALLBACK_PEAKS[key]
            return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def attn_kernel_source_sha256() -> str:
    """Hash of the attention kernel's device code (the part of attn_fwd.cu
    before its host-side section, plus the PTX wrapper header), with comments
    and blank lines left out so that documentation edits keep it."""
    src = open(ATTN_SRC).read()
    cut = src.index("// ---------------------------------------------------------------- host side")
    ptx = open(os.path.join(os.path.dirname(ATTN_SRC), "sm103_ptx.cuh")).read()
    code = []
    for line in (src[:cut] + ptx).splitlines():
        line = re.sub(r"//.*", "", line).rstrip()
        if line:
            code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()


# DRAM bytes per attention launch (dram__bytes_read.sum + dram__bytes_write.sum)
# from the ncu captures summarised under profiles/, keyed by (workload, mode).
# A figure is reported only while the attention kernel's device source hashes
# to the value it was captured with.
PROFILED_TRAFFIC = {
    ("seq128k", "fused"): {
        "kernel_source_sha256": "4e86f2afb84c3505bc11a8646696fcb7da983bd40007f35eb8ab557c4695ac66",
        "dram_bytes_per_launch": 7911812352 + 1073514496,
        "source": "ncu capture summarised in profiles/attn_fwd_seq128k.md",
    },
    ("seq2m", "fused"): {
        "kernel_source_sha256": "4e86f2afb84c3505bc11a8646696fcb7da983bd40007f35eb8ab557c4695ac66",
        "dram_bytes_per_launch": 950496080640 + 17950700288,
        "source": "single-pass ncu capture (DRAM bytes only) summarised in profiles/attn_fwd_seq2m_traffic.md",
    },
}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        rows = []
        try:
            for line in open(self.out.name):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_median": statistics.median(float(r[3]) for r in rows)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(times, flops, ws, device):
    """Replicas (weak scaling: every rank runs its own micro-batch, no data-path
    collective): the job's times are the slowest rank's, its useful FLOPs the
    sum over ranks.  Returns (list of max times, summed FLOPs)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x) for x in times], dtype=torch.float64, device=device)
    f = torch.tensor([float(flops)], dtype=torch.float64, device=device)
    if ws > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return t.tolist(), f.item()


def job_throughput(job_flops: float, steps: int, ms: float) -> float:
    """Whole-job useful TFLOP/s: the FLOPs every rank did in `steps` steps over
    the slowest rank's time for them."""
    return job_flops * steps / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(w, q, k, v, seconds: float, seed: int):
    """Time the fp64 oracle on a bounded sample of (token, head) rows of the
    workload; returns (useful FLOPs of the sample, seconds, rows, threads)."""
    import oracle
    from packed_varlen_attention_aware_gb300 import workloads as wl

    lengths = np.array(w.lengths, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    rng = np.random.default_rng(seed)
    doc_of = np.repeat(np.arange(len(lengths)), lengths)
    kh, vh = wl.bf16_bits(k), wl.bf16_bits(v)
    qh = np.zeros((T, w.hq, w.d), np.uint16)

    def run(nrows):
        toks = rng.integers(0, T, nrows)
        heads = rng.integers(0, w.hq, nrows).astype(np.int32)
        uniq = np.unique(toks)
        import torch

        qh[uniq] = wl.bf16_bits(q[torch.as_tensor(uniq, device=q.device)])
        pos = toks - cu[doc_of[toks]]
        flops = int(np.sum(4 * w.d * (pos + 1)))
        t0 = time.perf_counter()
        oracle.attention_rows(qh, kh, vh, cu, w.hq, w.hkv, w.d, w.scale, toks, heads)
        return flops, time.perf_counter() - t0

    f0, t0 = run(64)  # calibration
    rate = f0 / max(t0, 1e-6)
    n = max(64, int(64 * seconds * rate / max(f0, 1)))
    f1, t1 = run(n)
    return f1, t1, n, oracle.num_threads()


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def reference_arm(args, rank):
    """The fp64 oracle as it stands, on the host cores, on our workload."""
    if rank != 0:
        return 0
    import torch

    from packed_varlen_attention_aware_gb300 import workloads as wl

    w = wl.workload(args.workload, args.seed)
    # the same seeded bytes as our arm: large workloads are drawn by the GPU's
    # generator (input generation only; the timed work is the CPU oracle)
    big = w.total_tokens > (1 << 17)
    q, k, v = wl.qkv(w, device="cuda" if big and torch.cuda.is_available() else "cpu")
    per_step = args.ref_step_seconds or max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, per_step, args.seed + 1000)
    flops, secs, rows = 0, 0.0, 0
    threads = 1
    for i in range(args.steps):
        f, t, n, threads = oracle_sample(w, q, k, v, per_step, args.seed + i)
        flops, secs, rows = flops + f, secs + t, rows + n
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args, "oracle"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} random (token, head) rows of {w.name} over {args.steps} steps, "
                                   f"~{per_step:.1f} s each, fp64 C oracle with OpenMP on {cpu_model()}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, args, mode):
    T = w.total_tokens
    in_bytes = T * (w.hq + 2 * w.hkv) * w.d * 2
    return {
        "workload": f"{w.name}: {len(w.lengths)} documents packed into {T} tokens, Hq={w.hq}, Hkv={w.hkv}, "
                    f"d={w.d}, capacity C={w.capacity}, seed {w.seed}",
        "tokens": T, "documents": len(w.lengths), "max_doc": max(w.lengths), "hq": w.hq, "hkv": w.hkv, "d": w.d,
        "capacity": w.capacity, "seed": w.seed, "mode": mode,
        "useful_flops_per_step": useful_flops(w.lengths, w.d, w.hq),
        "l2": f"inputs larger than L2: Q/K/V {in_bytes / 2**20:.0f} MiB vs 129 MB L2" if in_bytes > L2_BYTES
        else f"L2 flushed between steps (inputs {in_bytes / 2**20:.1f} MiB)",
    }


# ---------------------------------------------------------------- our arm

def gpu_numa_node(dev_index: int):
    """The host NUMA node nearest the GPU (its PCI device's numa_node), or None."""
    import torch

    try:
        p = torch.cuda.get_device_properties(dev_index)
        bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        node = int(open(f"/sys/bus/pci/devices/{bdf}/numa_node").read().strip())
        return node if node >= 0 else None
    except Exception:
        return None


def bind_to_numa_node(node):
    """Run this process on the CPUs of `node`, so pinned host buffers it
    allocates afterwards are placed (first touch) in that node's memory.
    Returns the CPU count bound to, or None when nothing was changed."""
    if node is None:
        return None
    try:
        cpus = set()
        for part in open(f"/sys/devices/system/node/node{node}/cpulist").read().strip().split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return len(cpus)
    except Exception:
        return None


def shard_report(shard_flops, nshards: int):
    """Per-shard useful FLOPs of the step (hdp_flops_per_shard) and their
    max/mean imbalance."""
    f = [int(x) for x in shard_flops[:nshards].cpu().tolist()]
    mean = sum(f) / max(1, len(f))
    out = {"num_shards": nshards, "max": max(f), "mean": mean, "max_over_mean": max(f) / mean if mean else None}
    if nshards <= 512:
        out["flops"] = f
    return out


def flops_spread(name: str, seeds, dev):
    """Useful FLOPs of the workload's micro-batch for each seed, from the
    library's per-shard FLOPs (the lengths differ by seed)."""
    import torch

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import workloads as wl

    per_seed = []
    for sd in seeds:
        w = wl.workload(name, sd)
        dl = torch.tensor(w.lengths, dtype=torch.int32, device=dev)
        with pkg.hdp_plan_create(dl, w.capacity) as plan:
            f = torch.empty(plan.view.num_shards, dtype=torch.int64, device=dev)
            pkg.hdp_flops_per_shard(plan, w.d, w.hq, f)
            per_seed.append(int(f.sum().item()))
    return {"seeds": list(seeds), "useful_flops": per_seed, "min": min(per_seed), "max": max(per_seed),
            "max_over_min": max(per_seed) / min(per_seed)}


def attention_only(name: str, mode_name: str, seed: int, warmup: int, steps: int, dev, peaks):
    """CUDA-event time of the attention call alone (plan made once) on another
    named workload, for the extra timed entries of the line."""
    import torch

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import workloads as wl

    w = wl.workload(name, seed)
    mode = pkg.HDP_MODE_SPLIT if mode_name == "split" else pkg.HDP_MODE_FUSED
    q, k, v = wl.qkv(w, device=str(dev))
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, w.total_tokens), dtype=torch.float32, device=dev)
    dl = torch.tensor(w.lengths, dtype=torch.int32, device=dev)
    plan = pkg.hdp_plan_create(dl, w.capacity)
    wsb = pkg.hdp_attention_workspace_bytes(plan, w.hq, w.d, mode)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
    stream = torch.cuda.current_stream()
    times = []
    with ClockSampler(dev.index or 0) as clocks:
        for it in range(warmup + steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, mode, ws, o, lse, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= warmup:
                times.append(e0.elapsed_time(e1))
    pkg.hdp_device_status()
    plan.destroy()
    flops = useful_flops(w.lengths, w.d, w.hq)
    ms = statistics.mean(times)
    achieved = flops / (ms * 1e-3) / 1e12
    out = {"workload": workload_config(w, None, mode_name)["workload"], "mode": mode_name, "warmup": warmup,
           "steps": steps, "attn_ms": ms, "attn_ms_min": min(times), "achieved": achieved, "unit": "TFLOP/s",
           "frac": achieved / peaks["bf16_tflops"], "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
           "kernel": "k_attn_fwd" + (" + k_merge_blocks" if mode_name == "split" else ""),
           "clocks": clocks.summary()}
    prof = PROFILED_TRAFFIC.get((name, mode_name))
    if prof and prof["kernel_source_sha256"] == attn_kernel_source_sha256():
        out["traffic"] = prof["dram_bytes_per_launch"]
        out["traffic_source"] = prof["source"]
    del q, k, v, o, lse, ws
    torch.cuda.empty_cache()
    return out


def our_arm(args, ws, rank, local):
    import torch
    import torch.distributed as dist

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import build as native_build
    from packed_varlen_attention_aware_gb300 import workloads as wl

    native_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    numa_node = gpu_numa_node(local)
    numa_cpus = bind_to_numa_node(numa_node)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = wl.workload(args.workload, args.seed + rank)
    mode = pkg.HDP_MODE_SPLIT if args.mode == "split" else pkg.HDP_MODE_FUSED
    q, k, v = wl.qkv(w, device=str(dev))
    T = w.total_tokens
    lengths_d = torch.tensor(w.lengths, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, T), dtype=torch.float32, device=dev)
    flops_step = useful_flops(w.lengths, w.d, w.hq)
    in_bytes = q.numel() * 2 + k.numel() * 2 + v.numel() * 2
    flush = None if in_bytes > L2_BYTES else torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    probe = pkg.hdp_plan_create(lengths_d, w.capacity, flags=pkg.HDP_PLAN_NO_SPLIT)
    nshards = probe.view.num_shards
    ws_bytes = pkg.hdp_attention_workspace_bytes(probe, w.hq, w.d, mode)
    probe.destroy()
    shard_flops = torch.empty(max(nshards, 1), dtype=torch.int64, device=dev)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    attn_events = []

    # neither attention mode walks the plan's SPLIT work list
    plan_flags = pkg.HDP_PLAN_NO_SPLIT

    def step(record=False):
        plan = pkg.hdp_plan_create(lengths_d, w.capacity, flags=plan_flags, stream=stream)
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, mode, workspace, o, lse, stream=stream)
        if record:
            e1.record(stream)
            attn_events.append((e0, e1))
        pkg.hdp_flops_per_shard(plan, w.d, w.hq, shard_flops, stream=stream)
        plan.destroy()
        if flush is not None:
            flush.zero_()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pkg.hdp_device_status()
    assert int(shard_flops[:nshards].sum().item()) == flops_step, "per-shard FLOPs do not sum to the total"

    launches0 = pkg.hdp_kernel_launch_count()
    with ClockSampler(local) as clocks:
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step(record=True)
        t1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
    launches = pkg.hdp_kernel_launch_count() - launches0
    pkg.hdp_device_status()
    ms = t0.elapsed_time(t1)
    attn_ms = sum(a.elapsed_time(b) for a, b in attn_events) / len(attn_events)
    clk = clocks.summary()
    shards = shard_report(shard_flops, nshards)

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs from pinned host memory, runs the path and reads its
    # outputs back; step i+1's upload and step i-1's download run on their own
    # streams while step i computes (two device buffer sets).  Steps of more
    # than a second (the 2M-token sequence) run this leg over fewer steps.
    long_step = ms / args.steps > 1000.0
    e2e_steps = min(args.steps, 3) if long_step else args.steps
    e2e_warm = 1 if long_step else max(2, args.warmup // 2)

    def run_e2e():
        """The end-to-end leg; returns ((e2e_ms, h2d, d2h, rates), None), or
        (None, reason) when the pinned host buffers cannot be had on every rank."""
        def pinned_like(t):
            return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)

        err = None
        try:
            qh, kh, vh = pinned_like(q), pinned_like(k), pinned_like(v)
            qh.copy_(q)
            kh.copy_(k)
            vh.copy_(v)
            lh = torch.tensor(w.lengths, dtype=torch.int32).pin_memory()
            oh, lseh, fh = pinned_like(o), pinned_like(lse), pinned_like(shard_flops)
        except RuntimeError as exc:
            err = "pinned host buffers: " + str(exc).splitlines()[0][:160]
        flag = torch.tensor([0 if err else 1], dtype=torch.int32, device=dev)
        if ws > 1:
            dist.all_reduce(flag, op=dist.ReduceOp.MIN)
        if int(flag.item()) == 0:
            return None, err or "another rank could not pin its host buffers"
        qd = [q, torch.empty_like(q)]
        kd = [k, torch.empty_like(k)]
        vd = [v, torch.empty_like(v)]
        ld = [torch.empty_like(lengths_d), torch.empty_like(lengths_d)]
        od = [o, torch.empty_like(o)]
        lsed = [lse, torch.empty_like(lse)]
        fd = [shard_flops, torch.empty_like(shard_flops)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        def upload(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[b])  # the slot's inputs are no longer read: its last compute is done
                qd[b].copy_(qh, non_blocking=True)
                kd[b].copy_(kh, non_blocking=True)
                vd[b].copy_(vh, non_blocking=True)
                ld[b].copy_(lh, non_blocking=True)
                ev_in[b].record(s_in)

        def compute_and_download(i):
            b = i & 1
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])  # the slot's previous outputs are home before they are overwritten
            plan = pkg.hdp_plan_create(ld[b], w.capacity, flags=plan_flags, stream=stream)
            pkg.hdp_attention_fwd(plan, qd[b], kd[b], vd[b], w.hq, w.hkv, w.d, w.scale, mode, workspace, od[b], lsed[b],
                                  stream=stream)
            pkg.hdp_flops_per_shard(plan, w.d, w.hq, fd[b], stream=stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                oh.copy_(od[b], non_blocking=True)
                lseh.copy_(lsed[b], non_blocking=True)
                fh.copy_(fd[b], non_blocking=True)
                ev_out[b].record(s_out)
            plan.destroy()

        def e2e_run(steps):
            upload(0)
            for i in range(steps):
                if i + 1 < steps:
                    upload(i + 1)
                compute_and_download(i)

        for b in range(2):
            ev_out[b].record(s_out)
            ev_done[b].record(stream)
        e2e_run(e2e_warm)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)
        e2e_run(e2e_steps)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        pkg.hdp_device_status()
        h2d = in_bytes + lh.numel() * 4
        d2h = oh.numel() * 2 + lseh.numel() * 4 + fh.numel() * 8
        # the host link alone, per direction: one step's uploads, then its downloads
        rates = {}
        for direction in ("h2d", "d2h"):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(s_in)
            with torch.cuda.stream(s_in):
                if direction == "h2d":
                    qd[1].copy_(qh, non_blocking=True)
                    kd[1].copy_(kh, non_blocking=True)
                    vd[1].copy_(vh, non_blocking=True)
                else:
                    oh.copy_(od[1], non_blocking=True)
                    lseh.copy_(lsed[1], non_blocking=True)
            c1.record(s_in)
            torch.cuda.synchronize()
            nbytes = in_bytes if direction == "h2d" else oh.numel() * 2 + lseh.numel() * 4
            rates[direction] = nbytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
        del qh, kh, vh, oh, lseh, qd, kd, vd, od, lsed
        return (e2e_ms, h2d, d2h, rates), None

    e2e_result, e2e_error = run_e2e()
    e2e_ms, h2d, d2h, rates = e2e_result if e2e_result else (0.0, 0, 0, {})

    (ms, e2e_ms, attn_ms_max), job_flops = aggregate_over_ranks([ms, e2e_ms, attn_ms], flops_step, ws, dev)

    peaks, src = load_peaks()
    extras = {}
    if rank == 0 and ws == 1 and not args.no_extras:
        del o, lse, workspace
        if args.workload == "seq2m":
            q = k = v = None  # room for the 128K workload's SPLIT partials
        torch.cuda.empty_cache()
        if args.workload == "seq2m":
            for m in ("fused", "split"):
                extras[f"seq128k_{m}"] = attention_only("seq128k", m, args.seed, 3, 10, dev, peaks)
        if args.workload == "mb32k":
            extras["mb32k_useful_flops_by_seed"] = flops_spread("mb32k", range(10), dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        if q is None:
            q, k, v = wl.qkv(w, device=str(dev))
        f, secs, rows, threads = oracle_sample(w, q, k, v, args.cpu_seconds, args.seed + 7)
        cpu = {"value": f / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} random (token, head) rows of {w.name}, {secs:.1f} s, fp64 C oracle with "
                         f"OpenMP on {cpu_model()}"}
    if rank == 0:
        achieved = flops_step / (attn_ms * 1e-3) / 1e12
        value = job_throughput(job_flops, args.steps, ms)
        prof = PROFILED_TRAFFIC.get((args.workload, args.mode))
        traffic = None
        if prof and prof["kernel_source_sha256"] == attn_kernel_source_sha256():
            traffic = prof["dram_bytes_per_launch"]
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(w, args, args.mode), shards=shards),
            "frac_of_bf16_peak": value / (peaks["bf16_tflops"] * ws),
            "roofline": {"bound": "tensor", "kernel": "k_attn_fwd", "achieved": achieved,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                         "peak_source": f"{src} bf16 dense burst",
                         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "attn_ms": attn_ms, "traffic": traffic,
                         "traffic_note": prof["source"] if traffic is not None else
                         "no ncu capture of the current kernel source on this workload"},
            "cpu_baseline": cpu,
            "e2e": ({"value": job_throughput(job_flops, e2e_steps, e2e_ms), "unit": "TFLOP/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / e2e_steps,
                     "steps": e2e_steps, "warmup": e2e_warm,
                     "pipeline": "step i+1 upload and step i-1 download overlap step i compute",
                     "copy_gbs": rates, "numa_node": numa_node, "numa_cpus_bound": numa_cpus}
                    if e2e_error is None else
                    {"value": None, "unit": "TFLOP/s", "error": e2e_error, "numa_node": numa_node}),
            "gpu_launches": launches,
            "clocks": clk,
        }
        if extras:
            line["extra"] = extras
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def attn_only_mode(args):
    """The attention call alone on --workload / --mode, plan made once: W
    warm-up and K timed launches (CUDA events), one JSON line.  Small enough
    to run under ncu on the 128K sequence."""
    import torch

    from packed_varlen_attention_aware_gb300 import build as native_build

    native_build.build()
    torch.cuda.set_device(0)
    peaks, _ = load_peaks()
    out = attention_only(args.workload, args.mode, args.seed, args.warmup, args.steps, torch.device("cuda", 0), peaks)
    out["mode_of_run"] = "attn-only"
    print(json.dumps(out), flush=True)
    return 0


def kernels_mode(args):
    """Secondary kernels: the plan on 2^24 random lengths and the LSE merge on
    16 partials of 2^20 rows (d = 128).  CUDA-event times per call; the merge
    also as HBM GB/s of its algorithmic bytes."""
    import torch

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import build as native_build

    native_build.build()
    torch.cuda.set_device(0)
    peaks, src = load_peaks()
    out = {"mode": "kernels", "peak_source": src}
    g = torch.Generator(device="cuda").manual_seed(args.seed)
    # plan stress
    n = 1 << 24
    lengths = torch.randint(1, 100, (n,), generator=g, device="cuda", dtype=torch.int32)
    times = []
    for it in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        plan = pkg.hdp_plan_create(lengths, 64, flags=pkg.HDP_PLAN_NO_SHARDS)
        e1.record()
        torch.cuda.synchronize()
        if it:
            times.append(e0.elapsed_time(e1))
        v = plan.view
        plan.destroy()
    scan_bytes = 4 * n * 2 + (n + 1) * (4 + 4 + 8 + 8 + 8) + 8 * v.num_tiles_fused * 4
    out["plan_stress"] = {"docs": n, "capacity": 64, "ms_per_call": statistics.median(times),
                          "num_chunks": v.num_chunks, "num_blocks": v.num_blocks,
                          "note": "whole hdp_plan_create incl. host sync, allocation and the work-list sort; "
                                  "per-kernel HBM rates come from the ncu launch list"}
    # merge
    m, rows, d = 16, 1 << 20, 128
    o_parts = torch.randn(m, rows, d, generator=g, device="cuda", dtype=torch.float32)
    lse_parts = torch.randn(m, rows, generator=g, device="cuda", dtype=torch.float32) * 2
    o = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    times = []
    for it in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkg.hdp_lse_merge_rows(o_parts, lse_parts, o, lse)
        e1.record()
        torch.cuda.synchronize()
        if it:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    nbytes = m * rows * (4 * d + 4) + rows * (2 * d + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["lse_merge"] = {"m": m, "rows": rows, "d": d, "ms_per_call": ms, "algorithmic_bytes": nbytes,
                        "achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"]}
    del o_parts, lse_parts, o, lse
    # the SPLIT partials of the 131,072-token sequence (136 blocks), merged by
    # hdp_lse_merge: per (row, head) m (4d + 4) bytes read and 2d + 4 written,
    # m = q chunk + 1
    from packed_varlen_attention_aware_gb300 import workloads as wl

    w = wl.workload("seq128k", args.seed)
    q, k, v = wl.qkv(w, device="cuda")
    dl = torch.tensor(w.lengths, dtype=torch.int32, device="cuda")
    plan = pkg.hdp_plan_create(dl, w.capacity)
    wsb = pkg.hdp_attention_workspace_bytes(plan, w.hq, w.d, pkg.HDP_MODE_SPLIT)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(w.hq, w.total_tokens, dtype=torch.float32, device="cuda")
    pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, pkg.HDP_MODE_SPLIT, ws, o, lse)
    rows_total = plan.view.num_blocks * w.capacity
    o_part = ws[: rows_total * w.hq * w.d * 4].view(torch.float32)
    lse_off = (rows_total * w.hq * w.d * 4 + 255) // 256 * 256
    lse_part = ws[lse_off: lse_off + rows_total * w.hq * 4].view(torch.float32)
    times = []
    for it in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkg.hdp_lse_merge(plan, o_part, lse_part, w.hq, w.d, o, lse)
        e1.record()
        torch.cuda.synchronize()
        if it:
            times.append(e0.elapsed_time(e1))
    pkg.hdp_device_status()
    nch = plan.view.num_chunks
    read = sum(w.capacity * w.hq * (qc + 1) * (4 * w.d + 4) for qc in range(nch))
    written = w.total_tokens * w.hq * (2 * w.d + 4)
    ms = statistics.median(times)
    gbs = (read + written) / (ms * 1e-3) / 1e9
    out["lse_merge_seq128k_split"] = {"blocks": plan.view.num_blocks, "ms_per_call": ms, "bytes_read": read,
                                      "bytes_written": written, "achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"],
                                      "frac": gbs / peaks["hbm_gbs"]}
    plan.destroy()
    print(json.dumps(out), flush=True)
    return 0


def cost_model_mode(args):
    """Calibrates the cost models of the research digest (sections 3.2-3.3) on
    this GPU: times the attention of one document of s tokens (Hq = 32,
    Hkv = 8, d = 128, FUSED) for several s, fits T(s) = alpha1 s^2 + beta1 s +
    gamma with the library's hdp_fit_cost_model (weights 1/T^2: relative
    error, the times span five orders of magnitude), and derives the time of one
    full C x C block, t_blk = 2 alpha1 C^2 (a causal document of s tokens has
    about s^2/2 query-key pairs, a full block C^2).  It then applies the ring
    model (hdp_ring_step_compute / hdp_ring_attention_time) with this t_blk
    and the pages' measured transfer t_x = 1.5 ms: the static 256-rank ring's
    shortest hidden length, and whether an HDP ring of one long sequence hides
    its transfers.  One JSON line."""
    import torch

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import build as native_build

    native_build.build()
    torch.cuda.set_device(0)
    hq, hkv, d, C = 32, 8, 128, 8192
    lengths = [4096, 8192, 16384, 32768, 65536, 131072]
    g = torch.Generator(device="cuda").manual_seed(args.seed)
    points = []
    for s in lengths:
        q = torch.randn(s, hq, d, generator=g, device="cuda").to(torch.bfloat16)
        k = torch.randn(s, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn(s, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
        dl = torch.tensor([s], dtype=torch.int32, device="cuda")
        plan = pkg.hdp_plan_create(dl, C)
        o = torch.empty_like(q)
        lse = torch.empty(hq, s, dtype=torch.float32, device="cuda")
        times = []
        for it in range(3 + 5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pkg.hdp_attention_fwd(plan, q, k, v, hq, hkv, d, 1.0 / math.sqrt(d), pkg.HDP_MODE_FUSED, None, o, lse)
            e1.record()
            torch.cuda.synchronize()
            if it >= 3:
                times.append(e0.elapsed_time(e1))
        pkg.hdp_device_status()
        plan.destroy()
        ms = statistics.median(times)
        flops = 4 * d * hq * s * (s + 1) // 2
        points.append({"s": s, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12})
        del q, k, v, o, lse
    x = [p["s"] for p in points]
    y = [p["ms"] for p in points]
    coef = pkg.hdp_fit_cost_model(x, y, 2, w=[1.0 / (t * t) for t in y])  # relative errors
    alpha1, beta1, gamma = float(coef[2]), float(coef[1]), float(coef[0])
    t_blk = 2.0 * alpha1 * C * C
    t_x = 1.5
    N, s_max = 256, 256 * C
    # static ring: packs of equal lengths that divide S_max
    hidden = [s for s in (1 << e for e in range(10, 22))
              if pkg.hdp_ring_step_compute([s] * (s_max // s), N, C, t_blk) >= t_x]
    hdp_t_c = pkg.hdp_ring_step_compute([39 * C], 39, C, t_blk)
    out = {"mode": "cost_model", "unit": "ms", "workload": f"one document of s tokens, Hq={hq}, Hkv={hkv}, "
           f"d={d}, FUSED, bf16", "points": points,
           "fit": {"alpha1": alpha1, "beta1": beta1, "gamma": gamma,
                   "max_rel_residual": max(abs(alpha1 * p["s"] ** 2 + beta1 * p["s"] + gamma - p["ms"]) / p["ms"]
                                           for p in points)},
           "t_blk_ms": t_blk, "capacity": C,
           "ring_model_at_t_x_1.5ms": {
               "static_256_ring_shortest_hidden_pow2_length": min(hidden) if hidden else None,
               "static_256_ring_shortest_hidden_length_closed_form": t_x / t_blk * s_max,
               "hdp_39_rank_ring_t_c_ms": hdp_t_c,
               "hdp_39_rank_ring_T_attn_ms": pkg.hdp_ring_attention_time(39, hdp_t_c, t_x),
               "hdp_ring_hides": t_blk >= t_x}}
    print(json.dumps(out), flush=True)
    return 0


def balance_mode(args):
    """Balance scheduler (research digest, section 3.4) on the 1M-token skewed
    mixture: plan and per-shard FLOPs on the GPU (hdp_plan_create,
    hdp_flops_per_shard), then hdp_balance_schedule on the host for several
    worker counts.  Reports each schedule's slowest-worker load over the mean
    (1.0 = perfect) for equal micro-batch counts (an infinite threshold),
    DP-Balance (delta = 0, 4 buckets) and PP-Balance, and the host time of
    one call.  One JSON line."""
    import time

    import numpy as np
    import torch

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import build as native_build
    from packed_varlen_attention_aware_gb300 import workloads as wl

    native_build.build()
    torch.cuda.set_device(0)
    w = wl.workload("mix1m", args.seed)
    dl = torch.tensor(w.lengths, dtype=torch.int32, device="cuda")
    plan = pkg.hdp_plan_create(dl, w.capacity)
    flops = torch.empty(plan.view.num_shards, dtype=torch.int64, device="cuda")
    pkg.hdp_flops_per_shard(plan, w.d, w.hq, flops)
    costs = flops.cpu().numpy()
    pkg.hdp_device_status()
    plan.destroy()
    rows = []
    for R in (8, 16, 32, 64):
        res = {"workers": R}
        for label, delta, mode in (("equal_counts", (1 << 62), pkg.HDP_BALANCE_DP), ("dp_balance", 0,
                                   pkg.HDP_BALANCE_DP), ("pp_balance", 0, pkg.HDP_BALANCE_PP)):
            t0 = time.perf_counter()
            reps = 20
            for _ in range(reps):
                _, load, _ = pkg.hdp_balance_schedule(costs, R, 4, delta, mode)
            us = (time.perf_counter() - t0) / reps * 1e6
            res[label] = {"max_over_mean": float(load.max() / load.mean()), "host_us_per_call": us}
        rows.append(res)
    out = {"mode": "balance", "workload": f"mix1m seed {args.seed}: {len(w.lengths)} sequences, "
           f"{len(costs)} micro-batches of C = {w.capacity} tokens", "cost": "useful FLOPs per micro-batch "
           "(hdp_flops_per_shard)", "max_over_mean_micro_batch_flops": float(costs.max() / costs.mean()),
           "schedules": rows}
    print(json.dumps(out), flush=True)
    return 0


def backward_mode(args):
    """Backward pass (dq, dk, dv) after the forward of the same micro-batch,
    on --workload.  CUDA events around each call; the backward's useful FLOPs
    are 2.5 x the forward's (five products of the forward's shape instead of
    two: S, dP, dV, dK, dQ).  One JSON line."""
    import torch

    import packed_varlen_attention_aware_gb300 as pkg
    from packed_varlen_attention_aware_gb300 import build as native_build
    from packed_varlen_attention_aware_gb300 import workloads as wl

    native_build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = wl.workload(args.workload, args.seed)
    q, k, v = wl.qkv(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(args.seed + 1)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    T = w.total_tokens
    lengths_d = torch.tensor(w.lengths, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    plan = pkg.hdp_plan_create(lengths_d, w.capacity)
    ws = torch.empty(pkg.hdp_attention_bwd_workspace_bytes(plan, w.hq, w.d), dtype=torch.uint8, device=dev)
    flops_fwd = useful_flops(w.lengths, w.d, w.hq)
    flops_bwd = flops_fwd * 5 // 2
    peaks, src = load_peaks()
    fwd_ms, bwd_ms = [], []
    with ClockSampler(0) as clocks:
        for it in range(args.warmup + args.steps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, pkg.HDP_MODE_FUSED, None, o, lse)
            e[1].record()
            pkg.hdp_attention_bwd(plan, q, k, v, o, lse, dout, w.hq, w.hkv, w.d, w.scale, ws, dq, dk, dv)
            e[2].record()
            torch.cuda.synchronize()
            if it >= args.warmup:
                fwd_ms.append(e[0].elapsed_time(e[1]))
                bwd_ms.append(e[1].elapsed_time(e[2]))
    pkg.hdp_device_status()
    plan.destroy()
    fm, bm = statistics.median(fwd_ms), statistics.median(bwd_ms)
    bw = flops_bwd / (bm * 1e-3) / 1e12
    out = {"mode": "backward", "workload": workload_config(w, args, "fused")["workload"], "steps": args.steps, "warmup": args.warmup,
           "fwd_ms": fm, "bwd_ms": bm, "fwd_tflops": flops_fwd / (fm * 1e-3) / 1e12, "bwd_tflops": bw,
           "step_tflops": (flops_fwd + flops_bwd) / ((fm + bm) * 1e-3) / 1e12,
           "roofline": {"bound": "tensor", "kernel": "whole backward: k_bwd_delta, k_attn_bwd (dK, dV), k_attn_bwd_dq (dQ)", "achieved": bw,
                        "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": bw / peaks["bf16_tflops"],
                        "peak_source": src},
           "clocks": clocks.summary()}
    print(json.dumps(out), flush=True)
    return 0


def free_port() -> int:
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launcher_command(argv, gpus: int, port: int):
    """torchrun command that runs this script with the same arguments as
    `gpus` ranks on this node (one process per GPU)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="seq2m", choices=["tiny", "mb32k", "seq128k", "mix1m", "seq2m"])
    ap.add_argument("--mode", choices=["fused", "split"], default="fused")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the extra entries (128K FUSED/SPLIT after seq2m, the FLOP spread of mb32k)")
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="reference arm: CPU seconds per step (default: about 150 s over all steps)")
    ap.add_argument("--kernels", action="store_true", help="time the plan stress input and the LSE merge")
    ap.add_argument("--attn-only", action="store_true", help="time the attention call alone on --workload")
    ap.add_argument("--cost-model", action="store_true",
                    help="calibrate T(s) and t_blk on this GPU and apply the ring model")
    ap.add_argument("--balance", action="store_true",
                    help="balance scheduler on the per-shard FLOPs of the 1M-token mixture")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (after the forward) on --workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the ranks here
        return subprocess.call(launcher_command(argv, args.gpus, free_port()))
    ws, rank, local = dist_setup()
    if ws != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {ws}")
    if args.kernels:
        return kernels_mode(args) if rank == 0 else 0
    if args.attn_only:
        return attn_only_mode(args) if rank == 0 else 0
    if args.cost_model:
        return cost_model_mode(args) if rank == 0 else 0
    if args.balance:
        return balance_mode(args) if rank == 0 else 0
    if args.backward:
        return backward_mode(args) if rank == 0 else 0
    if args.impl == "reference":
        return reference_arm(args, rank)
    return our_arm(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
