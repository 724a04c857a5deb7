#!/usr/bin/env python
"""Benchmark of the fused ZeRO shard step on one GB300 (or N replicas).

One step = one fused zero_step over rank 0's 842M-element shard of the
LLaMA-7B flat group (8 virtual ranks, 50M-element buckets, one launch per
bucket): reduce-scatter of the 8 bf16 gradient slices, AdamW on the fp32
master/m/v shard, bf16 cast and the write of the rank's slot of the flat
parameter buffer.  It is the largest group of the path that fits one GPU.
The same line carries `per_config`: the other groups (the tiny MLP back to
back and with L2 flushed, BERT-base, the round-robin ToyModel, the 40-layer
LLaMA-13B ZeRO-3 stream) measured in the same run.

Prints one JSON line (rank 0).  `value` is whole-job params/s with inputs
resident in HBM; `e2e` is the same metric through the public API with the
gradients copied from pinned host memory and the updated parameters copied
back every step; `roofline` relates the kernel's algorithmic bytes to the
measured HBM copy bandwidth; `cpu_baseline` times the CPU oracle on a bounded
sample.  `--impl reference` times the oracle alone (the reference arm).

Multi-GPU (`torchrun --nproc-per-node N bench.py --gpus N`): every rank runs
its own full replica of the workload (the virtual ranks live inside one GPU;
there is no data-path collective), timing is max-over-ranks, value sums the
work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "llama7b_rank0"
METRIC = "fused ZeRO shard step: params/s and HBM GB/s (fraction of GB300 peak)"
UNIT = "params/s"
KERNEL_PREFIX = "k_step"


# ----------------------------------------------------------------------------
# distributed plumbing (host side; no data-path collective)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is None:
        return
    if device is not None:
        dist.barrier(device_ids=[device])
    else:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest `value` over all ranks (timing only)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=f"cuda:{device}" if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []  # (host time, fields)
        self.proc = None
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError) as e:
            self.error = f"nvidia-smi unavailable: {e}"
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.error:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": self.error}
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = None
        if not win:
            win = [p for (_, p) in self.samples]
            note = "no sample fell inside the timed region; all samples of the run"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        reasons = sorted({name for p in win for name, val in zip(self.REASONS, p[5:9])
                          if val.lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(win)}
        if note:
            out["note"] = note
        return out


# ----------------------------------------------------------------------------
# helpers


# The files that define the kernels and their launch shape; host-only code
# (argument checks, the plan, other entry points) does not change them.
KERNEL_FILES = ("zero_internal.h", "zero_kernels.cuh", "zero_kernels_bf16.cu",
                "zero_kernels_fp16.cu", "zero_launch.cu")


def kernel_source_hash() -> str:
    csrc = os.path.join(ROOT, "zero_sharded_optimizer_flatten_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_FILES:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_src_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def step_bytes(phi_padded: int, n_ranks: int, n16_out: int = 1) -> int:
    """Algorithmic HBM bytes of one fused step: per element N 16-bit gradient
    reads, master/m/v read + write (24 B), and n16_out 16-bit parameter writes
    (1: the gathered buffer or, in the ZeRO-3 layout, the rank's shard; 2: both)."""
    return (2 * n_ranks + 24 + 2 * n16_out) * phi_padded


# ----------------------------------------------------------------------------
# the oracle as a CPU baseline


class OracleSample:
    """The CPU oracle's element step on the first n elements of the workload
    (all gradient replicas), inputs drawn once on the CPU; step(t) times one
    oracle call, nothing else."""

    def __init__(self, w, n_elems: int):
        import numpy as np
        import torch

        import oracle
        from zero_sharded_optimizer_flatten_gb300 import workloads as W
        torch.set_num_threads(1)
        self.oracle, self.w, self.n = oracle, w, n_elems
        self.dt = oracle.FP16 if w.dtype == "fp16" else oracle.BF16
        self.op = oracle.AVG if w.op == "avg" else oracle.SUM
        p16 = W.fill(w, "param", 0, 0, 0, n_elems, torch.empty(n_elems, dtype=w.torch_dtype))
        self.grads = np.stack([W.grads16(w, 1, q, "cpu", 0, n_elems).view(torch.int16).numpy()
                               .view(np.uint16) for q in range(w.n_ranks)])
        self.master = oracle.to_f32(p16.view(torch.int16).numpy().view(np.uint16), self.dt)
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.out = np.zeros(n_elems, np.uint16)
        self.hp = oracle.hparams()

    def step(self, t: int) -> float:
        t0 = time.perf_counter()
        self.oracle.update_elements(self.grads, self.master, self.m, self.v, self.dt, self.op,
                                    self.hp, t, out16=self.out)
        return time.perf_counter() - t0

    def step_threads(self, t: int, k: int) -> float:
        """The same oracle call over k contiguous element ranges on k host
        threads (the C oracle runs with the interpreter lock released); the
        per-thread copies of the gradient columns are made before timing."""
        import concurrent.futures as cf

        import numpy as np
        if getattr(self, "_parts_k", None) != k:
            cut = [min(self.n, (self.n * i // k) // 8 * 8) for i in range(k)] + [self.n]
            self._parts = [(np.ascontiguousarray(self.grads[:, a:b]), a, b)
                           for a, b in zip(cut[:-1], cut[1:]) if b > a]
            self._parts_k = k
        with cf.ThreadPoolExecutor(len(self._parts)) as pool:
            t0 = time.perf_counter()
            futs = [pool.submit(self.oracle.update_elements, g, self.master[a:b], self.m[a:b],
                                self.v[a:b], self.dt, self.op, self.hp, t, self.out[a:b])
                    for g, a, b in self._parts]
            for f in futs:
                f.result()
            return time.perf_counter() - t0


def oracle_rate(w, n_elems: int):
    el = OracleSample(w, n_elems).step(1)
    return n_elems / el, el


def host_available_bytes():
    """MemAvailable of this host in bytes (None if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def host_cpu() -> dict:
    """The host the oracle runs on: its logical CPU count and model name."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "processor name") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:  # Arm hosts list no model name in /proc/cpuinfo
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "model": model}


def cpu_baseline(w, budget_s: float = 10.0, whole_bucket: bool = True):
    """The oracle on a bounded sample of the workload: one whole bucket for a
    bucketed group (the unit one launch of the step processes), else about
    `budget_s` seconds of single-threaded work."""
    if w.bucket_elems and whole_bucket:
        n = int(min(w.phi, w.bucket_elems))
        what = f"one whole {n}-element bucket (the first) of the {w.key} group"
    else:
        rate, _ = oracle_rate(w, 1 << 16)
        n = int(min(w.phi, max(1 << 16, rate * budget_s)))
        what = f"{n} elements of the {w.key} group"
    n -= n % 8
    sample = OracleSample(w, n)
    el = sample.step(1)
    out = {"value": n / el, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
           "sample": f"{what} (all {w.n_ranks} gradient replicas), one step of the "
                     f"single-threaded C oracle, {el:.1f} s"}
    # the same plain oracle over all host cores (element ranges split evenly)
    k = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
            else os.cpu_count() or 1)
    if k > 1:
        sample.step_threads(2, k)                       # warm the pool's threads
        el_k = min(sample.step_threads(3 + i, k) for i in range(2))
        out["all_cores"] = {"value": n / el_k, "unit": UNIT, "cores": k, "kind": "oracle",
                            "sample": f"the same {n} elements split over {k} host threads, "
                                      f"best of 2 steps, {el_k:.2f} s"}
    return out


# ----------------------------------------------------------------------------
# arms


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle timed on the host cores."""
    if rank != 0:
        return 0
    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    rate, _ = oracle_rate(w, 1 << 16)
    n = int(rate * args.ref_budget / max(1, args.steps + args.warmup))
    n = max(4096, min(n, w.phi))
    n -= n % 8
    sample = OracleSample(w, n)
    t = 0
    for _ in range(args.warmup):
        t += 1
        sample.step(t)
    els = []
    for _ in range(args.steps):
        t += 1
        els.append(sample.step(t))
    tot = sum(els)
    value = n * args.steps / tot
    # the elements one step of the GPU arm updates: the masked ranks' shards
    # (the oracle's own plan)
    import oracle
    mode = oracle.FLAT if w.mode == "flat" else oracle.ROUND_ROBIN
    units = sum(oracle.shard_len(list(w.numel), w.n_ranks, mode, w.align, r)
                for r in range(w.n_ranks) if (w.mask >> r) & 1)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.title, "phi": w.phi, "elements_per_step": units,
                   "virtual_ranks": w.n_ranks, "sample_elements_per_step": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "host": host_cpu(),
                         "sample": f"the first {n} of the {units} elements one step updates "
                                   "(all gradient replicas), single-threaded C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class FlatRunner:
    """One fused step over the masked ranks of a flat or round-robin group
    (bucketed if the workload says so).  Gradient buffers hold only the flat
    range the masked ranks own."""

    def __init__(self, w, dev, grad_sets, amp=None, offload=False, from_shards=False,
                 reduced=False):
        import torch

        import zero_sharded_optimizer_flatten_gb300 as Z
        from zero_sharded_optimizer_flatten_gb300 import workloads as W
        self.Z, self.w, self.dev = Z, w, dev
        self.plan = plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
        self.mask = w.mask
        self.ext = ext = plan.flat_extent(self.mask)
        self.hp = Z.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
        p16 = W.fill(w, "param", 0, 0, 0, ext, torch.empty(ext, dtype=w.torch_dtype, device=dev))
        self.full16 = torch.zeros_like(p16)
        S = [plan.shard_len(r) if (self.mask >> r) & 1 else 0 for r in range(w.n_ranks)]
        # offload: the fp32 optimizer state lives in pinned host memory and the
        # kernels stream it across the host link
        self.offload = offload

        def state(n):
            if offload:
                return torch.empty(n, dtype=torch.float32, pin_memory=True)
            return torch.empty(n, dtype=torch.float32, device=dev)
        self.master = [state(n) for n in S]
        self.m = [state(n) for n in S]
        self.v = [state(n) for n in S]
        Z.zero_init_shards(plan, p16, self.master, self.m, self.v, rank_mask=self.mask)
        del p16
        self.grads = [[W.grads16(w, s + 1, q, dev, 0, ext) for q in range(w.n_ranks)]
                      for s in range(grad_sets)]
        self.elems = sum(S)                       # work units per step
        self.padded = plan.padded
        # offload: the kernels read and write master/m/v across the host link
        self.link_bytes_per_step = 24 * self.elems if offload else 0
        if amp is None:
            self.calls = [Z.ZeroStep(plan, g, w.op, self.master, self.m, self.v, self.full16,
                                     None, self.hp, rank_mask=self.mask,
                                     bucket_elems=w.bucket_elems) for g in self.grads]
            self.bytes_per_step = step_bytes(self.elems, w.n_ranks)
            self.kernel = KERNEL_PREFIX
        else:
            # mixed-precision controls: fp32 gradient shards, device state, workspace
            self.gsh = [torch.empty(n, dtype=torch.float32, device=dev) for n in S]
            self.state = Z.amp_state_tensor(dev)
            Z.zero_amp_init(self.state, amp)
            self.ws_bucket = w.bucket_elems
            if reduced and not self.ws_bucket:
                # the reductions that write the partials go bucket by bucket;
                # a group without buckets is one bucket of the whole buffer
                self.ws_bucket = plan.padded
            self.ws = torch.empty(max(16, Z.zero_amp_workspace_bytes(plan, self.mask,
                                                                      self.ws_bucket)),
                                  dtype=torch.uint8, device=dev)

            def make(g):
                return lambda t: Z.zero_step_amp(plan, g, w.op, self.gsh, self.master, self.m,
                                                 self.v, self.full16, None, self.hp, amp,
                                                 self.state, self.ws, rank_mask=self.mask,
                                                 bucket_elems=w.bucket_elems)
            self.calls = [make(g) for g in self.grads]
            # reduction pass 2N + 4 B, update pass 4 + 24 + 2 B per element
            self.bytes_per_step = (2 * w.n_ranks + 34) * self.elems
            self.kernel = "k_stats + k_amp_finalize + k_adamw_amp"
        if amp is not None and from_shards:
            # the gradients arrive reduce-scattered (as a training loop's
            # overlapped bucket reductions leave them): reduce once, untimed
            Z.zero_reduce_scatter(plan, self.grads[0], w.op, self.gsh, rank_mask=self.mask,
                                  bucket_elems=w.bucket_elems)

            def step_shards(t):
                Z.zero_step_amp_shards(plan, self.gsh, self.master, self.m, self.v, self.full16,
                                       None, self.hp, amp, self.state, self.ws,
                                       rank_mask=self.mask, bucket_elems=w.bucket_elems)
            self.calls = [step_shards]
            # shard read 4 B, update pass 4 + 24 + 2 B per element
            self.bytes_per_step = 34 * self.elems
            self.kernel = "k_shard_stats + k_amp_finalize + k_adamw_amp"
        if amp is not None and reduced:
            # the bucket reductions of a training loop already wrote the fp32
            # shards and their tiles' sums of squares (untimed, once)
            B = self.ws_bucket
            red = Z.ReduceScatterBucketAmp(plan, self.grads[0], w.op, self.gsh, self.hp,
                                           self.state, self.ws, rank_mask=self.mask,
                                           bucket_elems=B)
            for b in range(-(-plan.padded // B)):
                red(b)

            def step_reduced(t):
                Z.zero_step_amp_reduced(plan, self.gsh, self.master, self.m, self.v, self.full16,
                                        None, self.hp, amp, self.state, self.ws,
                                        rank_mask=self.mask, bucket_elems=B)
            self.calls = [step_reduced]
            # update pass only: 4 + 24 + 2 B per element
            self.bytes_per_step = 30 * self.elems
            self.kernel = "k_amp_finalize + k_adamw_amp"

    def step(self, t, events=None):
        if events is not None:
            events[0].record()
        self.calls[t % len(self.calls)](t)
        if events is not None:
            events[1].record()

    def e2e(self, t0, steps):
        """The public API with host buffers: the step's gradient replicas
        arrive in pinned host memory and its updated 16-bit parameters must
        end up in pinned host memory.  Two ways, both timed:
          direct -- zero_step is given the host buffers; its kernel reads the
                    replicas and writes the parameters across the host link;
          copies -- copy the replicas to HBM, zero_step, copy the result back.
        A third timing, "h2d_only", copies the replicas to HBM and does nothing
        else: the host link's own rate, the bound the two paths are held to.
        Returns {"direct": s, "copies": s, "h2d_only": s} per step and the
        bytes moved."""
        import torch
        w, Z = self.w, self.Z
        host_g = [torch.empty(self.ext, dtype=w.torch_dtype, pin_memory=True)
                  for _ in range(w.n_ranks)]
        for q in range(w.n_ranks):
            host_g[q].copy_(self.grads[0][q])
        host_out = torch.empty(self.ext, dtype=w.torch_dtype, pin_memory=True)
        dev_g = self.grads[0]

        def direct(t):
            Z.zero_step(self.plan, host_g, w.op, self.master, self.m, self.v, host_out, None,
                        self.hp, t, rank_mask=self.mask, bucket_elems=w.bucket_elems)

        def copies(t):
            for q in range(w.n_ranks):
                dev_g[q].copy_(host_g[q], non_blocking=True)
            Z.zero_step(self.plan, dev_g, w.op, self.master, self.m, self.v, self.full16, None,
                        self.hp, t, rank_mask=self.mask, bucket_elems=w.bucket_elems)
            host_out.copy_(self.full16, non_blocking=True)

        def h2d_only(t):
            for q in range(w.n_ranks):
                dev_g[q].copy_(host_g[q], non_blocking=True)

        out = {}
        t = t0
        for name, one in (("direct", direct), ("copies", copies), ("h2d_only", h2d_only)):
            for _ in range(2):
                t += 1
                one(t)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                t += 1
                one(t)
            e1.record()
            torch.cuda.synchronize()
            out[name] = e0.elapsed_time(e1) / 1e3 / steps
        return out, w.n_ranks * self.ext * 2, self.ext * 2


class FloorRunner:
    """zero_floor_probe with a FlatRunner's plan and buffers: the step's grid
    and memory accesses without its arithmetic (kind 0: launch only; 1: the
    loads; 2: the loads and stores), timed like the step."""

    def __init__(self, run, kind):
        self.Z, self.w, self.run, self.kind = run.Z, run.w, run, kind
        self.bytes_per_step = run.bytes_per_step
        self.elems = run.elems
        self.kernel = "k_floor"
        self.call = run.Z.FloorProbe(run.plan, kind, run.grads[0], run.master, run.m, run.v,
                                     run.full16, rank_mask=run.mask,
                                     bucket_elems=run.w.bucket_elems)

    def step(self, t, events=None):
        if events is not None:
            events[0].record()
        self.call()
        if events is not None:
            events[1].record()


def floors(run, dev, steps, warmup, graph, flush_l2):
    """Per-step time (us) of the step's launch shape alone, with its loads,
    and with its loads and stores, next to the step itself, in one harness."""
    out = {}
    for kind, name in ((0, "launch_only_us"), (1, "loads_us"), (2, "loads_and_stores_us")):
        r = time_steps(FloorRunner(run, kind), dev, steps, warmup, graph, flush_l2)
        out[name] = 1e6 * r["kernel_s"]
    out["step_us"] = 1e6 * time_steps(run, dev, steps, warmup, graph, flush_l2, t=10 ** 6)[
        "kernel_s"]
    out["note"] = ("zero_floor_probe: the step's grid, job table and memory accesses over the "
                   "same buffers without its arithmetic, timed in the same harness")
    return out


class Zero3Runner:
    """The ZeRO-3 layer stream: per layer, all-gather the 8 ranks' 16-bit
    shards into the layer buffer, then the fused step writing each rank's
    shard (the next gather's source).  One gradient set is shared by all
    layers (the backward pass refills one buffer per layer)."""

    def __init__(self, w, dev, layer_states, prefetch=0, offload=False):
        import torch

        import zero_sharded_optimizer_flatten_gb300 as Z
        from zero_sharded_optimizer_flatten_gb300 import workloads as W
        self.Z, self.w, self.dev = Z, w, dev
        # offload: every layer's 16-bit shards and fp32 master/m/v live in
        # pinned host memory; the gathers and steps stream them across the
        # host link (the replicas and the layer buffers stay in HBM)
        self.offload = offload
        self.plan = plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
        self.hp = Z.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
        L = plan.padded
        S = [plan.shard_len(r) for r in range(w.n_ranks)]
        self.layer_buf = torch.empty(L, dtype=w.torch_dtype, device=dev)
        self.grads = [W.grads16(w, 1, q, dev, 0, L) for q in range(w.n_ranks)]
        self.n_states = min(w.layers, layer_states)
        self.shards, self.calls, self.states = [], [], []
        def state(n, dtype):
            if offload:
                return torch.empty(n, dtype=dtype, pin_memory=True)
            return torch.empty(n, dtype=dtype, device=dev)
        for layer in range(self.n_states):
            p16 = W.params16(w, dev, L, layer=layer)
            sh = [state(S[r], w.torch_dtype) for r in range(w.n_ranks)]
            for r in range(w.n_ranks):
                sh[r].copy_(p16[sum(S[:r]):sum(S[:r]) + S[r]])
            master = [state(n, torch.float32) for n in S]
            m = [state(n, torch.float32) for n in S]
            v = [state(n, torch.float32) for n in S]
            Z.zero_init_shards(plan, p16, master, m, v)
            del p16
            self.shards.append(sh)
            self.states.append((master, m, v))
            self.calls.append(Z.ZeroStep(plan, self.grads, w.op, master, m, v, None, sh, self.hp))
        self.layers = w.layers
        self.prefetch = prefetch
        if prefetch:
            if w.layers % self.n_states:
                raise SystemExit("--prefetch needs the layer count to be a multiple of "
                                 "--layer-states")
            layers = [{"grads": self.grads, "master": st[0], "m": st[1], "v": st[2],
                       "shards16": self.shards[k]} for k, st in enumerate(self.states)]
            bufs = [self.layer_buf] + [torch.empty_like(self.layer_buf)
                                       for _ in range(prefetch - 1)]
            self.passes = Z.Zero3Pass(plan, layers, bufs, w.op, self.hp)
            self.gather_stream = torch.cuda.Stream(dev)
        self.elems = w.layers * plan.padded
        self.bytes_per_step = w.layers * (step_bytes(plan.padded, w.n_ranks) + 4 * plan.padded)
        self.kernel_bytes = step_bytes(plan.padded, w.n_ranks)  # per k_step launch
        self.kernel = KERNEL_PREFIX
        # across the host link per element and layer: the gather reads the
        # 16-bit shard, the step reads and writes master/m/v and writes it
        self.link_bytes_per_step = 28 * self.elems if offload else 0

    def step(self, t, events=None):
        if self.prefetch:
            # the native layer stream: gathers on their own stream run ahead
            if events is not None:
                events[0][0].record()
            for k in range(self.layers // self.n_states):
                self.passes(t, gather_stream=self.gather_stream)
            if events is not None:
                events[0][1].record()
            return
        for layer in range(self.layers):
            k = layer % self.n_states
            self.Z.zero_allgather(self.plan, self.shards[k], self.layer_buf)
            if events is not None:
                events[layer][0].record()
            self.calls[k](t)
            if events is not None:
                events[layer][1].record()


# The other groups, measured in the same run as the headline and reported in
# its `per_config` object: (key, workload, regime, options).  The tiny group
# fits in L2, so it is reported twice: back to back from a CUDA graph (its
# 36 MB stay in L2 between steps) and with L2 flushed before every step.
PER_CONFIG = (
    ("tiny_mlp/back_to_back", "tiny_mlp",
     "back to back: the K steps captured in one CUDA graph and replayed once; the step's "
     "36 MB stay in L2 between steps", dict(steps=2000, warmup=20)),
    ("tiny_mlp/l2_flushed", "tiny_mlp",
     "L2 flushed: a 256 MB buffer is read before every step, outside the step's events; "
     "each step timed by its own events", dict(steps=300, warmup=5, flush_l2=True)),
    ("bert_base", "bert_base",
     "the K steps captured in one CUDA graph and replayed once; inputs larger than L2",
     dict(steps=500, warmup=10)),
    ("toy_rr", "toy_rr",
     "the K steps captured in one CUDA graph and replayed once; inputs larger than L2",
     dict(steps=500, warmup=10)),
    ("llama13b_layer", "llama13b_layer",
     "one step = one pass over the 40 layers through zero_zero3_pass (3 layer buffers, "
     "gathers on a second stream); 40 distinct layer states; inputs larger than L2",
     dict(steps=3, warmup=3, prefetch=3)),
)


def make_runner(w, dev, grad_sets=2, amp=None, offload=False, from_shards=False,
                layer_states=40, prefetch=0, reduced=False):
    if w.zero3:
        return Zero3Runner(w, dev, layer_states, prefetch, offload)
    return FlatRunner(w, dev, grad_sets, amp, offload, from_shards, reduced)


def time_steps(run, dev, steps, warmup, graph=True, flush_l2=False, dist=None, local=0, t=0):
    """Warm up, then time `steps` steps of `run` on the current stream.

    Flat groups: the timed steps are captured in one CUDA graph (each with its
    own step number) and replayed once, unless `flush_l2`, which reads a
    256 MB buffer before every step (outside the step's own events).  ZeRO-3
    streams are launched step by step with events per layer (or per pass).
    Returns the wall-clock window of the timed region and the timings."""
    import torch
    Z = run.Z
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        t += 1
        run.step(t)
    torch.cuda.synchronize(dev)

    def pair():
        return (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    zero3 = run.w.zero3
    if zero3:
        ev = [[pair() for _ in range(1 if run.prefetch else run.layers)] for _ in range(steps)]
    else:
        ev = [pair() for _ in range(steps)]
    graph_obj = None
    graph_launches = 0
    use_graph = graph and not flush_l2 and not zero3
    if use_graph:
        graph_obj = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        n0 = Z.zero_launch_count()
        with torch.cuda.graph(graph_obj, stream=cap):
            for k in range(steps):
                run.step(t + 1 + k)
        graph_launches = Z.zero_launch_count() - n0   # kernel nodes the replay runs
        torch.cuda.synchronize(dev)
    flush = flush_sink = None
    if flush_l2:
        # twice the size of L2, read (not written, which would leave dirty
        # lines to be written back during the step) before every step
        flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        flush_sink = torch.empty((), dtype=torch.float32, device=dev)
    barrier(dist, local)
    torch.cuda.synchronize(dev)
    launches0 = Z.zero_launch_count()
    wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if flush is not None:
        # the steps are enqueued one Python call at a time and timed by their
        # own events: hold the GPU for a while first, so that the host is
        # ahead of it and no step's events include time the GPU spends
        # waiting for the host to enqueue it
        torch.cuda._sleep(int(5e5 * steps))
    start.record(stream)
    if graph_obj is not None:
        graph_obj.replay()
        t += steps
    else:
        for k in range(steps):
            t += 1
            if flush is not None:
                torch.sum(flush, dim=0, out=flush_sink)
            run.step(t, ev[k])
    stop.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    launches = Z.zero_launch_count() - launches0 + graph_launches
    barrier(dist, local)
    elapsed = start.elapsed_time(stop) / 1e3
    if flush is not None:
        # the flushes are not part of the step: time the steps by their events
        elapsed = sum(a.elapsed_time(b) for a, b in ev) / 1e3
    elapsed = max_over_ranks(dist, elapsed, local)
    if zero3 and run.prefetch:
        # events bracket whole passes: the pass's bytes (gathers + steps)
        kernel_s = statistics.fmean(a.elapsed_time(b) for st in ev for a, b in st) / 1e3
        bytes_per_launch = run.bytes_per_step
    elif zero3:
        kernel_s = statistics.fmean(a.elapsed_time(b) for st in ev for a, b in st) / 1e3
        bytes_per_launch = run.kernel_bytes
    elif graph_obj is not None:
        kernel_s = elapsed / steps   # graph replay: launches back to back
        bytes_per_launch = run.bytes_per_step
    else:
        kernel_s = statistics.fmean(a.elapsed_time(b) for a, b in ev) / 1e3
        bytes_per_launch = run.bytes_per_step
    del graph_obj, flush
    return {"elapsed": elapsed, "kernel_s": kernel_s, "bytes_per_launch": bytes_per_launch,
            "launches": launches, "t": t, "use_graph": use_graph, "window": (wall0, wall1)}


def flushed_marginal(run, dev, steps, t=0, reps=3):
    """Per-step time after an L2 flush, without per-step events: a CUDA graph
    of `steps` (flush, step) pairs and one of `steps` flushes alone are each
    replayed between two events; the difference over `steps` is what a step
    adds after a flush (the median of `reps` pairs of replays).  The flush
    reads a 256 MB buffer, twice the L2, so every step starts from DRAM."""
    import torch
    stream = torch.cuda.current_stream(dev)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def capture(with_step):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for k in range(steps):
                torch.sum(flush, dim=0, out=sink)
                if with_step:
                    run.step(t + 1 + k)
        torch.cuda.synchronize(dev)
        return g
    both, alone = capture(True), capture(False)
    both.replay()
    alone.replay()
    torch.cuda.synchronize(dev)
    per = []
    for _ in range(reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        both.replay()
        ev[1].record(stream)
        alone.replay()
        ev[2].record(stream)
        torch.cuda.synchronize(dev)
        per.append((ev[0].elapsed_time(ev[1]) - ev[1].elapsed_time(ev[2])) / 1e3 / steps)
    del both, alone, flush
    return statistics.median(per)


def regime_text(run, use_graph, flush_l2):
    if flush_l2:
        return (f"flushed: a 256 MB buffer is read before every timed step, outside the "
                f"step's events ({run.bytes_per_step / 1e6:.1f} MB touched per step)")
    if use_graph:
        return (f"back to back in a CUDA graph; {run.bytes_per_step / 1e6:.1f} MB touched per "
                f"step ({'fits' if run.bytes_per_step < 120e6 else 'larger than'} L2)")
    return f"inputs larger than L2: {run.bytes_per_step / 1e9:.2f} GB touched per step"


def per_config(args, dev, clocks, peak):
    """Every other group of the path, one after another on the same GPU."""
    import gc

    import torch

    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    out = {}
    seen = set()
    for key, wkey, regime, opt in PER_CONFIG:
        if wkey == args.workload and not opt.get("flush_l2"):
            continue
        w = W.WORKLOADS[wkey]
        try:
            out[key] = one_config(args, dev, clocks, peak, w, regime, opt)
        except Exception as e:  # one record's failure must not lose the line
            out[key] = {"workload": w.title, "error": f"{type(e).__name__}: {e}"}
        gc.collect()
        torch.cuda.empty_cache()
        if not args.no_cpu_baseline and wkey not in seen and "error" not in out[key]:
            # the oracle on a bounded sample of this group (about a second)
            out[key]["cpu_baseline"] = cpu_baseline(w, args.per_config_cpu_budget,
                                                    whole_bucket=False)
            seen.add(wkey)
    return out


def zero3_layer_states(w, dev, want: int) -> int:
    """Distinct layer states of the ZeRO-3 pass that fit the device's free
    memory (each holds fp32 master/m/v and a 16-bit shard: 14 B per element;
    the gradient replicas and 3 layer buffers are shared): the largest
    divisor of the layer count up to `want` that fits in 85 % of it."""
    import torch
    free, _ = torch.cuda.mem_get_info(dev)
    per = 14 * w.phi
    fixed = (2 * w.n_ranks + 2 * 3) * w.phi
    fit = int((0.85 * free - fixed) // per)
    for k in range(min(want, w.layers), 0, -1):
        if w.layers % k == 0 and k <= fit:
            return k
    return 1


def one_config(args, dev, clocks, peak, w, regime, opt):
    """One per_config record: the group's runner, timed as the options say."""
    import torch
    want = 40
    states = zero3_layer_states(w, dev, want) if w.zero3 else want
    run = make_runner(w, dev, prefetch=opt.get("prefetch", 0), layer_states=states)
    torch.cuda.synchronize(dev)
    r = time_steps(run, dev, opt["steps"], opt["warmup"], graph=True,
                   flush_l2=opt.get("flush_l2", False))
    sec = r["elapsed"] / opt["steps"]
    gbs = r["bytes_per_launch"] / r["kernel_s"] / 1e9
    rec = {
        "workload": w.title, "regime": regime, "steps": opt["steps"],
        "warmup": opt["warmup"], "ms_per_step": 1e3 * sec,
        "params_per_s": run.elems / sec, "elements_per_step": run.elems,
        "bytes_per_step": run.bytes_per_step,
        "gbs": gbs, "frac": gbs / peak,
        "kernel": ("zero_zero3_pass (k_allgather + k_step per layer)"
                   if getattr(run, "prefetch", 0) else run.kernel),
        "gpu_launches": r["launches"],
        "clocks": clocks.summary(*r["window"]),
    }
    if w.zero3:
        rec.update({"layers": run.layers, "layer_states": run.n_states,
                    "bytes_per_element": 46})
        if run.n_states < want:
            rec["note"] = (f"{run.n_states} distinct layer states cycled over the {run.layers} "
                           f"layers: the device's free memory does not hold {want}")
    if opt.get("flush_l2"):
        rec["floor"] = floors(run, dev, opt["steps"], opt["warmup"], True, True)
        # the same regime without per-step events (see flushed_marginal)
        mg = {"step_us": 1e6 * flushed_marginal(run, dev, opt["steps"], t=2 * 10 ** 6)}
        for kind, name in ((0, "launch_only_us"), (2, "loads_and_stores_us")):
            mg[name] = 1e6 * flushed_marginal(FloorRunner(run, kind), dev, opt["steps"])
        mg["frac"] = run.bytes_per_step / (mg["step_us"] * 1e-6) / 1e9 / peak
        mg["note"] = ("a CUDA graph of K (L2 flush, step) pairs replayed between two events, "
                      "minus a graph of K flushes alone, over K: what a step adds after a "
                      "flush, without per-step event records")
        rec["graph_marginal"] = mg
    del run
    return rec


def run_gpu(args, world, rank, local):
    import gc

    import torch

    import zero_sharded_optimizer_flatten_gb300 as Z
    from zero_sharded_optimizer_flatten_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm has no CPU fallback)")
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    w = W.WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    amp = None
    if args.amp and not w.zero3:
        amp = Z.AmpConfig(init_scale=1.0, min_scale=1.0, window=1000, hysteresis=2,
                          max_norm=args.max_norm)
    run = make_runner(w, dev, args.grad_sets, amp, args.offload, args.from_shards,
                      args.layer_states, args.prefetch, args.reduced)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    r = time_steps(run, dev, args.steps, args.warmup, args.graph, args.flush_l2, dist, local)
    elapsed, kernel_s = r["elapsed"], r["kernel_s"]
    bytes_per_launch, t = r["bytes_per_launch"], r["t"]

    e2e = None
    pinned_need = (w.n_ranks + 1) * run.ext * 2 if hasattr(run, "ext") else 0
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    host_free = host_available_bytes()
    if (not w.zero3 and not args.amp and not args.offload and args.e2e_steps > 0
            and host_free is not None and pinned_need * local_world > 0.6 * host_free):
        # every rank on this node would pin its own copy of the replicas
        e2e = {"value": None, "unit": UNIT,
               "skipped": f"the e2e leg pins {pinned_need / 1e9:.1f} GB of host memory per rank "
                          f"({local_world} ranks on this node); only {host_free / 1e9:.0f} GB "
                          f"are available"}
    elif not w.zero3 and not args.amp and not args.offload and args.e2e_steps > 0:
        e2e_steps = max(3, min(args.steps, args.e2e_steps))
        per_step, h2d, d2h = run.e2e(t, e2e_steps)
        link_s = per_step.pop("h2d_only")
        best = min(per_step, key=per_step.get)
        sec = max_over_ranks(dist, per_step[best], local)
        e2e = {"value": run.elems * world / sec, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "path": best,
               "ms_per_step": {k: 1e3 * v for k, v in per_step.items()},
               # the inputs must cross the host link: the copy engine's rate for
               # the same replicas (nothing else), next to the rate the direct
               # path's kernel loads and stores reach across it
               "link": {"h2d_copy_gbs": h2d / link_s / 1e9, "h2d_copy_ms": 1e3 * link_s,
                        "direct_gbs": (h2d + d2h) / per_step["direct"] / 1e9},
               "note": "direct: zero_step reads the pinned host replicas and writes the pinned "
                       "host parameters across NVLink-C2C; copies: cudaMemcpyAsync in, "
                       "zero_step, cudaMemcpyAsync out"}

    peak, peak_src = measured_peaks()
    achieved = bytes_per_launch / kernel_s / 1e9
    line = {
        "impl": "gb300",
        "metric": METRIC,
        "value": run.elems * args.steps * world / elapsed,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": w.title,
            "phi": w.phi,
            "elements_per_step": run.elems,
            "virtual_ranks": w.n_ranks,
            "storage": f"{w.dtype} params and gradients, fp32 master/m/v",
            "parallelism": f"{world} independent replica(s); {w.n_ranks} virtual ranks each",
            "l2": regime_text(run, r["use_graph"], args.flush_l2),
            "hbm_gbs_per_step": run.bytes_per_step / (elapsed / args.steps) / 1e9,
            "launch": ("the K timed steps captured in one CUDA graph (each with its own step "
                       "number), replayed once" if r["use_graph"] else
                       "one Python call per step through the binding"),
        },
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": (recorded_traffic(args.workload)
                        if not (args.amp or args.offload or w.zero3) else None),
            "kernel": run.kernel,
            "bytes_per_launch": bytes_per_launch,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                           else "fallback 6.8 TB/s",
        },
        "e2e": e2e,
        "gpu_launches": r["launches"],
        "clocks": clocks.summary(*r["window"]),
    }
    if w.bucket_elems and not (args.amp or args.offload):
        # one k_step launch per bucket: the algorithmic bytes of one full
        # bucket's launch sit beside its measured DRAM traffic; `achieved` is
        # the step's bytes over the step's time (the launches' average)
        nb = -(-run.elems // w.bucket_elems)
        line["roofline"].update({
            "bytes_per_launch": step_bytes(w.bucket_elems, w.n_ranks),
            "launches_per_step": nb,
            "achieved_from": "bytes of the step's launches / their back-to-back time"})
    if args.offload:
        link = run.link_bytes_per_step
        line["config"]["offload"] = {
            "state": ("every layer's 16-bit shards and fp32 master/m/v in pinned host memory, "
                      "streamed by the gathers and steps" if w.zero3 else
                      "fp32 master/m/v in pinned host memory, streamed by the kernels"),
            "host_link_bytes_per_step": link,
            "hbm_bytes_per_step": run.bytes_per_step - link,
        }
        # the step is bound by the host link, not by HBM
        line["roofline"].update({
            "bound": "host-link", "achieved": link / kernel_s / 1e9, "peak": None, "frac": None,
            "bytes_per_launch": link,
            "peak_source": "no measured host-link peak in MEASURED_PEAKS.json; one-direction "
                           "copies measured about 210 GB/s in and 193 GB/s out"})
    if args.amp:
        line["config"]["amp"] = {"max_norm": args.max_norm, "init_scale": 1.0,
                                 "note": "loss-scale check, global-norm clipping, skip on overflow"}
    if w.zero3:
        if run.prefetch:
            line["roofline"]["kernel"] = "zero_zero3_pass (k_allgather + k_step per layer)"
            line["config"]["prefetch_layer_buffers"] = run.prefetch
        line["config"]["layer_states"] = run.n_states
        line["config"]["layers"] = run.layers
    if args.floor and not (w.zero3 or args.amp or args.offload):
        line["floor"] = floors(run, dev, args.steps, args.warmup, args.graph, args.flush_l2)
    del run
    gc.collect()
    torch.cuda.empty_cache()
    if world == 1 and args.per_config and not (args.amp or args.offload):
        line["per_config"] = per_config(args, dev, clocks, peak)
    clocks.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_offload_cpu(args, world, rank, local):
    """ZeRO-Offload with the CPU optimizer: per step the GPU reduce-scatters
    the replicas into pinned host fp32 shards, host threads run AdamW + cast on
    the host-resident state, the GPU all-gathers the host 16-bit shards into
    HBM.  Timed two ways on the host clock (part of the step runs on the CPU):
    the three calls one after another (with each phase's time), and
    zero_offload_step, which overlaps them chunk by chunk."""
    import torch

    import zero_sharded_optimizer_flatten_gb300 as Z
    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
    S = [plan.shard_len(r) for r in range(w.n_ranks)]
    p16 = W.params16(w, dev, plan.padded)
    full16 = torch.zeros_like(p16)
    dm = [torch.empty(n, dtype=torch.float32, device=dev) for n in S]
    Z.zero_init_shards(plan, p16, dm, [torch.empty_like(x) for x in dm],
                       [torch.empty_like(x) for x in dm])
    torch.cuda.synchronize(dev)
    master = [x.cpu().pin_memory() for x in dm]
    del dm
    pin = lambda n, dt: torch.zeros(n, dtype=dt, pin_memory=True)  # noqa: E731
    m = [pin(n, torch.float32) for n in S]
    v = [pin(n, torch.float32) for n in S]
    gsh = [pin(n, torch.float32) for n in S]
    s16 = [pin(n, w.torch_dtype) for n in S]
    grads = [W.grads16(w, 1, q, dev, 0, plan.padded) for q in range(w.n_ranks)]
    hp = Z.AdamW()
    dt = Z.ZERO_BF16 if w.dtype == "bf16" else Z.ZERO_FP16
    chunk = args.chunk if args.chunk >= 0 else max(1, -(-plan.padded // 8))
    phases = {"reduce": 0.0, "cpu_adamw": 0.0, "gather": 0.0}

    def serial(t, acc=None):
        t0 = time.perf_counter()
        Z.zero_reduce_scatter(plan, grads, w.op, gsh)
        Z.zero_sync()
        t1 = time.perf_counter()
        Z.zero_cpu_adamw_shard_step(plan, master, m, v, gsh, s16, hp, t, dt,
                                    n_threads=args.threads)
        t2 = time.perf_counter()
        Z.zero_allgather(plan, s16, full16)
        Z.zero_sync()
        t3 = time.perf_counter()
        if acc is not None:
            acc["reduce"] += t1 - t0
            acc["cpu_adamw"] += t2 - t1
            acc["gather"] += t3 - t2

    amp = None
    if args.amp:
        # the mixed-precision form: the device reduces, sums the squares and
        # decides; the host applies the decision (scale 1, clipping active)
        amp = Z.AmpConfig(init_scale=1.0, min_scale=1.0, window=1000, hysteresis=2,
                          max_norm=args.max_norm)
        state = Z.amp_state_tensor(dev)
        Z.zero_amp_init(state, amp)
        ws = torch.empty(max(16, Z.zero_amp_workspace_bytes(plan)), dtype=torch.uint8,
                         device=dev)

    def pipelined(t, acc=None):
        if amp is not None:
            Z.zero_offload_step_amp(plan, grads, w.op, gsh, master, m, v, s16, full16, hp, amp,
                                    state, ws, chunk_elems=chunk, n_threads=args.threads)
        else:
            Z.zero_offload_step(plan, grads, w.op, gsh, master, m, v, s16, full16, hp, t,
                                chunk_elems=chunk, n_threads=args.threads)
        Z.zero_sync()

    t = 0

    def timed(one, acc=None):
        nonlocal t
        for _ in range(args.warmup):
            t += 1
            one(t)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            t += 1
            one(t, acc)
        return time.perf_counter() - t0
    el_serial = timed(serial, phases)
    el = timed(pipelined)
    ncpu = os.cpu_count() or 1
    threads = {"pipelined": args.threads if args.threads > 0 else max(1, ncpu - 1),
               "serial": args.threads if args.threads > 0 else ncpu}
    line = {"impl": "gb300", "metric": METRIC, "value": plan.phi * args.steps / el, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.title, "phi": plan.phi,
                       "offload": "CPU optimizer: fp32 state in pinned host memory, AdamW + cast "
                                  "on host threads, GPU reduce-scatter and all-gather across the "
                                  f"host link, overlapped in chunks of {chunk} flat elements "
                                  + ("(zero_offload_step_amp: mixed-precision controls decided on "
                                     "the device, clipping active)" if amp is not None
                                     else "(zero_offload_step)"),
                       "host_threads": threads,
                       "serial": {"ms_per_step": 1e3 * el_serial / args.steps,
                                  "ms_per_phase": {k: 1e3 * x / args.steps
                                                   for k, x in phases.items()},
                                  "calls": "zero_reduce_scatter, zero_sync, "
                                           "zero_cpu_adamw_shard_step, zero_allgather, zero_sync"},
                       "host_bytes_per_element": 30,
                       "timing": "host clock around each step, device synchronised at its end"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_unfused(args, world, rank, local):
    """The three unfused calls of one step (zero_reduce_scatter,
    zero_adamw_shard_step with 16-bit shard output, zero_allgather), each
    timed by its own CUDA events, with its algorithmic bytes per element:
    reduce 2N + 4, AdamW 4 + 24 + 2, gather 2 + 2."""
    import torch

    import zero_sharded_optimizer_flatten_gb300 as Z
    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
    mask, bucket = w.mask, w.bucket_elems
    S = [plan.shard_len(r) if (mask >> r) & 1 else 0 for r in range(w.n_ranks)]
    ext = plan.flat_extent(mask)
    p16 = W.fill(w, "param", 0, 0, 0, ext, torch.empty(ext, dtype=w.torch_dtype, device=dev))
    full = torch.zeros_like(p16)
    master = [torch.empty(n, dtype=torch.float32, device=dev) for n in S]
    m = [torch.empty_like(x) for x in master]
    v = [torch.empty_like(x) for x in master]
    Z.zero_init_shards(plan, p16, master, m, v, rank_mask=mask)
    gsh = [torch.empty(n, dtype=torch.float32, device=dev) for n in S]
    s16 = [torch.empty(n, dtype=w.torch_dtype, device=dev) for n in S]
    grads = [W.grads16(w, 1, q, dev, 0, ext) for q in range(w.n_ranks)]
    hp = Z.AdamW()
    E = sum(S)          # elements of the masked shards
    per = {"k_reduce_scatter": 2 * w.n_ranks + 4, "k_adamw": 30, "k_allgather": 4}

    def pair():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = {k: [pair() for _ in range(args.steps)] for k in per}
    t = 0
    for k in range(args.warmup + args.steps):
        t += 1
        rec = k >= args.warmup
        i = k - args.warmup
        if rec:
            ev["k_reduce_scatter"][i][0].record()
        Z.zero_reduce_scatter(plan, grads, w.op, gsh, rank_mask=mask, bucket_elems=bucket)
        if rec:
            ev["k_reduce_scatter"][i][1].record()
            ev["k_adamw"][i][0].record()
        Z.zero_adamw_shard_step(plan, master, m, v, gsh, s16, hp, t, rank_mask=mask)
        if rec:
            ev["k_adamw"][i][1].record()
            ev["k_allgather"][i][0].record()
        Z.zero_allgather(plan, s16, full, rank_mask=mask)
        if rec:
            ev["k_allgather"][i][1].record()
    torch.cuda.synchronize(dev)
    peak, _ = measured_peaks()
    kernels = {}
    total = 0.0
    for k, b in per.items():
        sec = statistics.fmean(a.elapsed_time(c) for a, c in ev[k]) / 1e3
        total += sec
        kernels[k] = {"us": 1e6 * sec, "bytes": b * E, "GB/s": b * E / sec / 1e9,
                      "frac": b * E / sec / 1e9 / peak}
    line = {"impl": "gb300", "metric": METRIC, "value": E / total, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.title, "phi": plan.phi, "elements_per_step": E,
                       "path": "unfused: reduce-scatter, AdamW + cast, all-gather",
                       "kernels": kernels,
                       "bytes_per_element": sum(per.values())}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_gather_all(args, world, rank, local):
    """zero_allgather of every rank's 16-bit shard into the whole flat buffer
    (the all-gather row at full size; for the LLaMA-7B group 6.74 G elements,
    4 B each: 26.95 GB per call).  Flat groups only: the shards are views of
    one flat parameter buffer, and the gathered buffer must equal it."""
    import torch

    import zero_sharded_optimizer_flatten_gb300 as Z
    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    if w.mode != "flat":
        raise SystemExit("--gather-all: flat groups only")
    plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
    src = W.params16(w, dev, plan.padded)
    shards = [src[off:off + n] for off, n in plan.shards]
    full = torch.zeros_like(src)
    E = plan.padded
    for _ in range(args.warmup):
        Z.zero_allgather(plan, shards, full)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    for a, b in ev:
        a.record()
        Z.zero_allgather(plan, shards, full)
        b.record()
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clocks.stop()
    assert torch.equal(full, src), "the gathered buffer differs from the shards' source"
    sec = statistics.fmean(a.elapsed_time(b) for a, b in ev) / 1e3
    peak, peak_src = measured_peaks()
    gbs = 4 * E / sec / 1e9
    line = {"impl": "gb300", "metric": METRIC, "value": E / sec, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sec, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": w.title + ": all-gather of every rank's shard",
                       "elements_per_call": E, "bytes_per_call": 4 * E,
                       "l2": f"inputs larger than L2: {4 * E / 1e6:.1f} MB per call"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": None, "kernel": "k_allgather",
                         "bytes_per_launch": 4 * E, "peak_source": peak_src},
            "gpu_launches": args.steps, "clocks": clocks.summary(t0, t1)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_engine(args, world, rank, local):
    """A training iteration of the ToyModel group (hidden 1024, 12 layers,
    round-robin over 4 virtual ranks) through the autograd-driven engine:
    4 x (forward + backward on the rank's micro-batch) + step, timed with and
    without overlapping the bucket reduce-scatters with the backward pass."""
    import torch

    import zero_sharded_optimizer_flatten_gb300 as Z
    from zero_sharded_optimizer_flatten_gb300.engine import ZeroEngine
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def toy():
        torch.manual_seed(0)
        layers = []
        for _ in range(12):
            layers += [torch.nn.Linear(1024, 4096), torch.nn.GELU(), torch.nn.Linear(4096, 1024)]
        layers.append(torch.nn.Linear(1024, 10))
        return torch.nn.Sequential(*layers).to(dev, torch.bfloat16)

    N = 4
    xs = [torch.randn(args.tokens, 1024, device=dev, dtype=torch.bfloat16) for _ in range(N)]
    out = {}
    amp = (Z.AmpConfig(init_scale=1.0, min_scale=1.0, window=1000, hysteresis=2,
                       max_norm=args.max_norm) if args.amp else None)
    for overlap in (False, True):
        model = toy()
        eng = ZeroEngine(model.parameters(), N, mode="round_robin", op="sum",
                         bucket_elems=args.bucket, overlap_comm=overlap, amp=amp,
                         offload=args.engine_offload, host_threads=args.threads)

        def iteration():
            for q in range(N):
                eng.backward(model(xs[q]).float().pow(2).mean(), q)
            eng.step()
        for _ in range(args.warmup):
            iteration()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            iteration()
        e1.record()
        torch.cuda.synchronize(dev)
        out["overlap" if overlap else "serial"] = e0.elapsed_time(e1) / args.steps
        out["launched_during_backward"] = eng.launched_during_backward
        phi = eng.plan.phi
        del eng, model
        torch.cuda.empty_cache()
    line = {"impl": "gb300", "metric": "ZeRO engine training iteration (4 virtual ranks)",
            "value": 1e3 / out["overlap"], "unit": "iterations/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": out["overlap"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "ToyModel hidden 1024 x12 + Linear(1024,10), round-robin N=4"
                                   + (", mixed precision (loss scale, clipping)" if amp else "")
                                   + (f", optimizer offload {args.engine_offload}"
                                      if args.engine_offload else ""),
                       "phi": phi, "tokens_per_rank": args.tokens, "bucket_elems": args.bucket,
                       "ms_per_iteration": {"serial": out["serial"], "overlap": out["overlap"]},
                       "bucket_launches_during_backward": out["launched_during_backward"]}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline object")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-config-cpu-budget", type=float, default=1.0,
                    help="seconds of oracle work for each per_config record's cpu_baseline")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the other groups' records (per_config) after the headline")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="parameter group to time (the reported line uses the default)")
    ap.add_argument("--grad-sets", type=int, default=2,
                    help="distinct gradient sets resident in HBM, alternated per step")
    ap.add_argument("--amp", action="store_true",
                    help="time the mixed-precision step (norm check + clipping) instead")
    ap.add_argument("--max-norm", type=float, default=1.0)
    ap.add_argument("--from-shards", action="store_true",
                    help="--amp: the step from already reduce-scattered fp32 gradient shards "
                         "(zero_step_amp_shards)")
    ap.add_argument("--reduced", action="store_true",
                    help="--amp: the step after bucket reductions that also wrote the sums of "
                         "squares (zero_reduce_scatter_bucket_amp, then zero_step_amp_reduced)")
    ap.add_argument("--offload", action="store_true",
                    help="keep the fp32 optimizer state in pinned host memory (ZeRO-Offload "
                         "over the host link)")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="ZeRO-3 stream through zero_zero3_pass with this many layer buffers "
                         "(gathers on a second stream); 0 = serial Python loop")
    ap.add_argument("--flush-l2", action="store_true",
                    help="read a 256 MB buffer before every timed step (for groups that fit "
                         "in L2); the steps are then timed by their own events")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch every timed step from Python instead of replaying the "
                         "steps captured in one CUDA graph (the default for flat groups)")
    ap.add_argument("--floor", action="store_true",
                    help="flat groups: also time the step's launch shape without arithmetic "
                         "(launch only, loads, loads + stores) in the same harness")
    ap.add_argument("--unfused", action="store_true",
                    help="time the three unfused calls of a step separately")
    ap.add_argument("--gather-all", action="store_true",
                    help="time the all-gather of every rank's shard into the whole flat "
                         "buffer (flat groups)")
    ap.add_argument("--offload-cpu", action="store_true",
                    help="ZeRO-Offload with the CPU optimizer (host threads run AdamW)")
    ap.add_argument("--threads", type=int, default=0,
                    help="--offload-cpu: host threads (0 = all hardware threads)")
    ap.add_argument("--chunk", type=int, default=-1,
                    help="--offload-cpu: flat elements per pipelined chunk (-1: an eighth of "
                         "the buffer; 0: one chunk)")
    ap.add_argument("--engine", action="store_true",
                    help="time a training iteration through the autograd-driven engine")
    ap.add_argument("--tokens", type=int, default=4096, help="--engine: tokens per rank")
    ap.add_argument("--engine-offload", choices=["cpu", "host_state"], default=None,
                    help="--engine: optimizer state in pinned host memory (cpu: host AdamW; "
                         "host_state: GPU AdamW across the host link)")
    ap.add_argument("--bucket", type=int, default=5_000_000, help="--engine: bucket elements")
    ap.add_argument("--layer-states", type=int, default=40,
                    help="ZeRO-3 stream: distinct layer states kept (cycled if fewer than layers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.engine:
        return run_engine(args, world, rank, local)
    if args.offload_cpu:
        return run_offload_cpu(args, world, rank, local)
    if args.unfused:
        return run_unfused(args, world, rank, local)
    if args.gather_all:
        return run_gather_all(args, world, rank, local)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
