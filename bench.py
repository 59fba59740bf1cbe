#!/usr/bin/env python3
"""Benchmark of the fused data-parallel step on GB300.

One step = the whole hot path on the BERT-large parameter list (336,226,108
parameters, 398 tensors) with R = 8 emulated replicas: the slab laid out in
reverse layer order by the bucket planner, then the fused reduce + AdamW +
redistribute kernel launched bucket by bucket (25 MiB buckets) through the
C ABI.  Printed as one JSON line (rank 0):

  value      parameters per second, device-timed (CUDA events, inputs
             resident in HBM, inputs 14.8 GB >> 129 MB L2 so no flush)
  e2e        the same step through the C ABI with the gradients copied in
             from pinned host memory and the updated bf16 parameters copied
             back every step
  roofline   achieved HBM GB/s of the fused kernel (algorithmic bytes
             (4R + 24) per parameter) against the measured copy bandwidth
  overlap    the step-time decomposition of the bucketed step behind a
             proxy backward of bf16 GEMMs: T_bwd, T_comm, overlapped and
             sequential step times, exposed ms
  gpt2_slice_r4  the same step on 24 GPT-2 8.3B layers (2.7B parameters)
             at R=4, 76 GB resident
  launch_floor  the small L2-resident case (R=2, 1M parameters): single
             launches after an L2 flush, back to back, and in a CUDA graph
  cpu_baseline  the oracle (single-threaded C) on a bounded sample, and
             split over every host core

`--impl reference` times the oracle alone on the host cores (the reference
arm).  Under torchrun (N > 1) the ranks run the real multi-GPU form with
R = N (one replica per GPU, the optimizer state sharded, per bucket a
ReduceScatter over NCCL, the fused rank step, an AllGather); the JSON
reports the parameters stepped per second against the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused DP step params/s and HBM GB/s (% of ~8 TB/s) at R=8; exposed ms/step"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = [os.path.join(ROOT, "gradient_reduce_optimizer_gb300", "csrc", f)
                  for f in ("cc_dp_kernels.cu", "cc_dp_device.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_step_kernel_traffic.json")


# ---------------------------------------------------------------------------
# Process group (replicas only) and cross-rank reductions
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str, timeout_s: float = 300.0):
    """The process group, with a limit on every collective: an exchange that
    stalls (a rank that died or never joined) ends with an error on the
    others instead of holding their GPUs."""
    import datetime
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend,
                                timeout=datetime.timedelta(seconds=timeout_s))
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_scalar(x: float, world: int, op: str, device="cpu") -> float:
    """Max or sum of a float over ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(ms_per_step: float, units_per_step: float, world: int,
              device="cpu"):
    """Whole-job throughput: units of all ranks over the slowest rank."""
    slowest = reduce_scalar(ms_per_step, world, "max", device)
    total_units = reduce_scalar(units_per_step, world, "sum", device)
    return slowest, total_units / (slowest * 1e-3)


# ---------------------------------------------------------------------------
# Peaks, profile figures and clocks
# ---------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 TFLOP/s of a cuBLAS GEMM timed alone (burst), if measured."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return None


def kernel_sha() -> str:
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic_per_param(R: int):
    """DRAM bytes per parameter of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source and this R."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_sha") != kernel_sha() or int(d.get("R", -1)) != R:
        return None
    return float(d["dram_bytes"]) / float(d["elements"])


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]),
                                 power=float(parts[3]), hw=parts[5], hwt=parts[6],
                                 swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 250.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# Workload
# ---------------------------------------------------------------------------

def build_workload(device, R_override=None, bucket_mib=25, preset=None):
    """Device slabs of a planned workload (BERT-large R=8 unless `preset`
    names another): gradients scaled per layer where the preset says so,
    pre-multiplied by its loss scale, zero on padding."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi
    from gradient_reduce_optimizer_gb300 import workloads as wl

    w = preset or wl.bert_large_r8(bucket_bytes=bucket_mib * wl.MiB)
    if R_override:
        w.R = R_override
    numel, layer_of = w.numel(), w.layer_of()
    offsets, buckets, n_slab = capi.cc_plan_buckets(numel, w.bucket_bytes)
    lay = wl.element_layer_map(numel, layer_of, offsets, n_slab, device=device)
    scale = None
    if w.layer_scale is not None:
        per_layer = wl.layer_scales(max(layer_of) + 1, *w.layer_scale, device=device)
        scale = per_layer[lay.clamp(min=0).long()]
    grads = wl.make_grads(w.R, n_slab, w.grad_sigma, device=device,
                          elem_scale=scale, mask=lay >= 0, premultiply=w.grad_scale)
    del lay, scale
    master, m, v = wl.make_state(n_slab, w.step, w.grad_sigma,
                                 master_sigma=w.master_sigma, device=device)
    outs = [torch.empty(n_slab, dtype=torch.bfloat16, device=device)
            for _ in range(w.R)]
    torch.cuda.synchronize()
    return dict(w=w, numel=numel, layer_of=layer_of, offsets=offsets,
                buckets=buckets, n_slab=n_slab, grads=grads, master=master,
                m=m, v=v, outs=outs)


def build_small_workload(device, n, R=8):
    """A flat R-replica slab of n elements with the same value recipe (one
    bucket): the small case for profiler captures."""
    import torch
    from gradient_reduce_optimizer_gb300 import workloads as wl

    w = wl.bert_large_r8(bucket_bytes=0)
    w.R, w.n, w.tensors = R, n, None
    grads = wl.make_grads(R, n, w.grad_sigma, device=device)
    master, m, v = wl.make_state(n, w.step, w.grad_sigma, device=device)
    outs = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(R)]
    torch.cuda.synchronize()
    return dict(w=w, numel=[n], layer_of=[0], offsets=[0], buckets=[(0, n)],
                n_slab=n, grads=grads, master=master, m=m, v=v, outs=outs)


def step_args(wk, step):
    w = wk["w"]
    return dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                weight_decay=w.weight_decay, step=step, grad_scale=w.grad_scale)


def uniform_buckets(n_slab, bucket_bytes):
    """The cut cc_fused_dp_step makes: floor(bucket_bytes/16)*8 elements."""
    per = max(8, bucket_bytes // 16 * 8) if bucket_bytes else n_slab
    return [(b, min(n_slab, b + per)) for b in range(0, n_slab, per)]


def launches_per_step(n_slab, bucket_bytes):
    per = max(8, bucket_bytes // 16 * 8) if bucket_bytes else n_slab
    return (n_slab + per - 1) // per


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_inputs(R, sample, seed_offset=0):
    """The first `sample` slab elements of the BERT-large R-replica workload,
    generated on the host with the same recipe (layer scales, padding)."""
    import numpy as np
    import torch
    import oracle
    from gradient_reduce_optimizer_gb300 import workloads as wl

    w = wl.bert_large_r8()
    numel, layer_of = w.numel(), w.layer_of()
    offsets, _, n_slab = oracle.plan_buckets(numel, w.bucket_bytes)
    sample = min(sample, n_slab)
    lay = torch.full((sample,), -1, dtype=torch.int32)
    for t, (k, l) in enumerate(zip(numel, layer_of)):
        lo, hi = offsets[t], min(offsets[t] + k, sample)
        if lo < sample:
            lay[lo:hi] = l
    per_layer = wl.layer_scales(max(layer_of) + 1, *w.layer_scale)
    scale = per_layer[lay.clamp(min=0).long()]
    grads = wl.make_grads(R, sample, w.grad_sigma, elem_scale=scale, mask=lay >= 0)
    master, m, v = wl.make_state(sample, w.step, w.grad_sigma)
    g16 = [g.view(torch.int16).numpy().view(np.uint16).copy() for g in grads]
    st = [x.numpy().copy() for x in (master, m, v)]
    hp = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
              weight_decay=w.weight_decay, step=w.step, grad_scale=w.grad_scale)
    return g16, st, hp, sample


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleRunner:
    """The oracle's step over a sample, on one thread or split into
    contiguous element chunks over `threads` host threads.  Each chunk is
    one unchanged oracle call (the step is elementwise, so the bits do not
    depend on the split); ctypes releases the GIL for the C call, so the
    chunks run in parallel."""

    def __init__(self, g16, st, hp, threads: int):
        self.hp, self.threads = hp, max(1, threads)
        n = st[0].size
        cuts = [n * k // self.threads // 8 * 8 for k in range(self.threads)] + [n]
        self.chunks = [([g[a:b] for g in g16], [x[a:b] for x in st])
                       for a, b in zip(cuts, cuts[1:]) if b > a]
        self.pool = None
        if len(self.chunks) > 1:
            from concurrent.futures import ThreadPoolExecutor
            self.pool = ThreadPoolExecutor(max_workers=len(self.chunks))

    def step(self):
        import oracle
        if self.pool is None:
            for g, st in self.chunks:
                oracle.fused_dp_step(g, *st, **self.hp)
            return
        futs = [self.pool.submit(oracle.fused_dp_step, g, *st, **self.hp)
                for g, st in self.chunks]
        for f in futs:
            f.result()

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def time_oracle(R, sample, min_seconds, max_seconds, threads=1):
    g16, st, hp, sample = oracle_sample_inputs(R, sample)
    runner = OracleRunner(g16, st, hp, threads)
    runner.step()                                  # warm the pool and pages
    passes, t0 = 0, time.perf_counter()
    while True:
        runner.step()
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or el >= max_seconds:
            break
    runner.close()
    return sample * passes / el, sample, passes, el


def host_bytes_available() -> int:
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


def to_host_inputs(grads, state):
    """Host copies (bf16 bits as uint16, fp32) of device inputs drawn by the
    workload generators."""
    import numpy as np
    import torch
    g16 = [g.view(torch.int16).cpu().numpy().view(np.uint16) for g in grads]
    st = [x.cpu().numpy() for x in state]
    return g16, st


def time_full_steps(g16, st, hp, threads, min_passes=1, min_seconds=0.0):
    """The oracle's step over whole slabs: one untimed pass when more than
    one thread runs (to start the pool), then timed passes until both
    min_passes and min_seconds are met.  Returns (seconds per step, passes,
    threads used)."""
    runner = OracleRunner(g16, st, hp, threads)
    if len(runner.chunks) > 1:
        runner.step()
    passes, t0 = 0, time.perf_counter()
    while True:
        runner.step()
        passes += 1
        el = time.perf_counter() - t0
        if passes >= min_passes and el >= min_seconds:
            break
    runner.close()
    return el / passes, passes, len(runner.chunks)


def run_cpu_baseline(args, wk, dev):
    """The oracle (single-threaded C, as it stands) timed on the host's cores
    on whole steps: the headline workload's full step (336,226,120 slab
    elements, R = 8) on one core and on every core, the small flat case
    (1,048,576 elements, R = 2) in full, and the 2.7B GPT-2 slice (R = 4) on
    one eighth of its slab, extrapolated.  Inputs are drawn by the same
    seeded generators on the device and copied to the host; the gradient
    slabs are the headline step's own (kernels only read them), master/m/v
    are drawn afresh.  Also the bounded 4M-element sample of earlier runs."""
    import torch
    from gradient_reduce_optimizer_gb300 import workloads as wl

    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    cores = host_cores()
    hp = step_args(wk, w.step)
    out = {"unit": UNIT, "kind": "oracle", "host_cores": cores}

    # C2, the headline step, whole
    need = n_slab * (2 * R + 12 + 2 * R) * 2          # inputs, outputs, slack
    avail = host_bytes_available()
    if avail and avail < need:
        out["headline_full_step"] = {"skipped": f"host memory: {avail} B free, {need} B needed"}
    else:
        state = wl.make_state(n_slab, w.step, w.grad_sigma, master_sigma=w.master_sigma,
                              device=dev)
        g16, st = to_host_inputs(wk["grads"], state)
        del state
        torch.cuda.empty_cache()
        t1, p1, _ = time_full_steps(g16, st, hp, 1)
        tn, pn, used = time_full_steps(g16, st, hp, cores, min_passes=3)
        out["headline_full_step"] = {
            "workload": f"BERT-large list, R={R}, {n_slab:,} slab elements (one whole step)",
            "one_core": {"s_per_step": round(t1, 3), "params_per_s": round(w.n / t1),
                         "passes": p1},
            "all_cores": {"s_per_step": round(tn, 4), "params_per_s": round(w.n / tn),
                          "passes": pn, "cores": used}}
        del g16, st

    # C1, the small flat case, whole
    c1 = wl.flat_1m_r2()
    grads = wl.make_grads(c1.R, c1.n, c1.grad_sigma, device=dev)
    state = wl.make_state(c1.n, c1.step, c1.grad_sigma, device=dev)
    g16, st = to_host_inputs(grads, state)
    hp1 = dict(lr=c1.lr, beta1=c1.beta1, beta2=c1.beta2, eps=c1.eps,
               weight_decay=c1.weight_decay, step=c1.step, grad_scale=c1.grad_scale)
    t1, p1, _ = time_full_steps(g16, st, hp1, 1, min_seconds=1.0)
    tn, pn, used = time_full_steps(g16, st, hp1, cores, min_seconds=1.0)
    out["flat_1m_r2_full_step"] = {
        "one_core": {"ms_per_step": round(1e3 * t1, 3), "params_per_s": round(c1.n / t1),
                     "passes": p1},
        "all_cores": {"ms_per_step": round(1e3 * tn, 3), "params_per_s": round(c1.n / tn),
                      "passes": pn, "cores": used}}
    del grads, state, g16, st

    # C3, one eighth of the GPT-2 slice (every tensor is a multiple of 8
    # elements, so the slab has no padding), extrapolated to the whole
    c3 = wl.gpt2_slice_r4()
    part = c3.n // 8 // 8 * 8
    need3 = part * (2 * c3.R + 12 + 2 * c3.R) * 2
    if avail and avail < need3:
        out["gpt2_slice_eighth"] = {"skipped": f"host memory: {avail} B free, {need3} B needed"}
    else:
        grads = wl.make_grads(c3.R, part, c3.grad_sigma, device=dev, premultiply=c3.grad_scale)
        state = wl.make_state(part, c3.step, c3.grad_sigma, device=dev)
        g16, st = to_host_inputs(grads, state)
        del grads, state
        torch.cuda.empty_cache()
        hp3 = dict(lr=c3.lr, beta1=c3.beta1, beta2=c3.beta2, eps=c3.eps,
                   weight_decay=c3.weight_decay, step=c3.step, grad_scale=c3.grad_scale)
        t1, p1, _ = time_full_steps(g16, st, hp3, 1)
        tn, pn, used = time_full_steps(g16, st, hp3, cores, min_passes=3)
        scale = c3.n / part
        out["gpt2_slice_eighth"] = {
            "workload": (f"GPT-2 slice recipe, R={c3.R}, first {part:,} of {c3.n:,} "
                         "elements; whole-step seconds extrapolated x8 (elementwise step)"),
            "one_core": {"s_per_eighth": round(t1, 3),
                         "s_per_step_extrapolated": round(t1 * scale, 2),
                         "params_per_s": round(part / t1), "passes": p1},
            "all_cores": {"s_per_eighth": round(tn, 4),
                          "s_per_step_extrapolated": round(tn * scale, 3),
                          "params_per_s": round(part / tn), "passes": pn, "cores": used}}
        del g16, st

    # the bounded sample of earlier runs, kept beside the whole steps
    v, sample, passes, el = time_oracle(R, args.cpu_sample, 3.0, 10.0)
    out["sample_4m"] = {"params_per_s": round(v), "cores": 1,
                        "sample": f"first {sample:,} slab elements, {passes} passes in {el:.1f} s"}

    full = out.get("headline_full_step", {})
    if "one_core" in full:
        out["value"] = full["one_core"]["params_per_s"]
        out["cores"] = 1
        out["sample"] = (f"one whole step of the same workload ({n_slab:,} slab elements, "
                         f"R={R}), single-threaded C oracle, {full['one_core']['passes']} "
                         f"pass(es) of {full['one_core']['s_per_step']} s")
    else:
        out["value"], out["cores"] = round(v), 1
        out["sample"] = (f"first {sample:,} slab elements of the same workload (R={R}), "
                         f"{passes} passes in {el:.1f} s, single-threaded C oracle")
    return out


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def headline_config(args, R, world, n_params, n_slab, bucket_bytes):
    """The `config` of the headline line, shared by both arms."""
    return {
        "workload": (f"BERT-large parameter list (336,226,108 params, 398 tensors), "
                     f"R={R} emulated replicas, {args.bucket_mib} MiB buckets in "
                     "reverse layer order, AdamW wd=0.01 step>=10, bf16 grads "
                     "N(0,1e-3) x U(0.5,2) per layer"),
        "R": R, "n_params": n_params, "n_slab": n_slab,
        "bucket_bytes": bucket_bytes,
        "launches_per_step": launches_per_step(n_slab, bucket_bytes),
        "parallelism": f"replicas x{world} (R={R} emulated per GPU)",
        "l2": "inputs 14.8 GB per GPU, larger than the 129 MB L2: no flush",
    }


def run_dist(args):
    """The real multi-GPU form under torchrun: R = world size ranks, one
    replica per GPU.  Each rank holds its replica's gradient and parameter
    slabs of the BERT-large list and the optimizer state of its shards only;
    per bucket (25 MiB, reverse layer order) a ReduceScatter of the bf16
    gradients over NCCL into local staging, the library's rank step, and an
    AllGather of the bf16 parameters.  Units: parameters stepped per second
    (each of the n parameters once per step), over the slowest rank."""
    import torch
    from gradient_reduce_optimizer_gb300 import build as gbuild
    from gradient_reduce_optimizer_gb300 import capi
    from gradient_reduce_optimizer_gb300 import workloads as wl
    from gradient_reduce_optimizer_gb300.dist import ShardedStep

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    if local == 0:
        gbuild.build()
    barrier(world)
    capi.lib()
    w = wl.bert_large_r8(bucket_bytes=args.bucket_mib * wl.MiB)
    numel, layer_of = w.numel(), w.layer_of()
    step = ShardedStep(numel, w.bucket_bytes, rank=rank, world=world, device=dev,
                       layer_of=layer_of)
    n_slab = step.n_slab
    lay = wl.element_layer_map(numel, layer_of, step.offsets, n_slab, device=dev)
    per_layer = wl.layer_scales(max(layer_of) + 1, *w.layer_scale, device=dev)
    scale = per_layer[lay.clamp(min=0).long()]
    # replica `rank`'s gradient: the emulated workload's seed for replica r
    g = wl._randn(n_slab, wl.SEED_GRAD + rank, dev).mul_(w.grad_sigma).mul_(scale)
    g.masked_fill_(lay < 0, 0.0)
    grads = g.to(torch.bfloat16)
    del g, lay, scale
    master, m, v = wl.make_state(n_slab, w.step, w.grad_sigma, master_sigma=w.master_sigma,
                                 device=dev)
    # this rank's shards of the state, packed in launch order
    st = [torch.empty(step.state_elems, device=dev) for _ in range(3)]
    for (lo, hi), (a, b) in step.shard_state_ranges():
        for dst, src in zip(st, (master, m, v)):
            dst[a:b] = src[lo:hi]
    del master, m, v
    params = torch.empty(n_slab, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def one(i):
        step.step(grads, *st, params, stream=stream, **step_args({"w": w}, w.step + i))

    for i in range(args.warmup):
        one(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        one(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_local = e0.elapsed_time(e1) / args.steps
    # every rank steps its shards: the units of all ranks add up to n
    mine = sum(b - a for _, (a, b) in step.shard_state_ranges())
    ms, value = aggregate(ms_local, float(mine) * w.n / n_slab, world, device=dev)
    result = {
        "metric": METRIC, "value": round(value), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": (f"BERT-large parameter list (336,226,108 params, 398 tensors), "
                         f"R={world} real ranks (one replica per GPU), {args.bucket_mib} MiB "
                         "buckets in reverse layer order: per bucket a ReduceScatter of "
                         "bf16 gradients (NCCL send/recv), the fused AdamW rank step, an "
                         "AllGather of bf16 parameters"),
            "R": world, "n_params": w.n, "n_slab": n_slab, "bucket_bytes": w.bucket_bytes,
            "num_buckets": len(step.buckets), "state_elems_per_rank": step.state_elems,
            "parallelism": f"dp{world}, optimizer state sharded",
            "l2": "inputs larger than the 129 MB L2: no flush"},
        "clocks": clk,
        "gpu_launches": len(step.buckets) * args.steps,
    }
    if not args.no_overlap:
        result["overlap_ready_driven"] = run_dist_overlap(args, step, grads, st, params, w,
                                                          layer_of, world, dev)
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_dist_overlap(args, step, grads, st, params, w, layer_of, world, dev):
    """The real multi-GPU form behind a proxy backward (the model's compute:
    per layer 3 bf16 GEMMs, M=8192, N=K=1024, as in cc_overlap_bench), in
    the two schedules: every bucket after the backward (step()), and DDP's
    ready-driven one (begin / layer_ready / end: each bucket's exchanges go
    out as soon as the backward has produced it).  Exposed = T_step - T_bwd,
    slowest rank, median over iterations."""
    import torch

    L = max(layer_of) + 1
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    a = torch.randn(8192, 1024, generator=g, device=dev).to(torch.bfloat16)
    bs = [torch.randn(1024, 1024, generator=g, device=dev).to(torch.bfloat16)
          for _ in range(3)]
    c = torch.empty(8192, 1024, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    # one layer's GEMMs captured once and replayed: the proxy runs at the
    # GPU's pace, not at the pace Python issues three launches
    for b_ in bs:
        torch.matmul(a, b_, out=c)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for b_ in bs:
            torch.matmul(a, b_, out=c)
    torch.cuda.synchronize()

    def layer(l):
        graph.replay()

    def backward():
        for l in range(L - 1, -1, -1):
            layer(l)

    def after(i):
        backward()
        step.step(grads, *st, params, stream=stream, **step_args({"w": w}, w.step + i))

    def ready(i):
        step.begin(grads, *st, params, stream=stream, **step_args({"w": w}, w.step + i))
        for l in range(L - 1, -1, -1):
            layer(l)
            step.layer_ready(l)
        step.end()

    iters = max(3, min(args.overlap_iters, 20))

    def med_ms(fn):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        barrier(world)
        times = []
        for i in range(iters):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(3 + i)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        barrier(world)
        return reduce_scalar(statistics.median(times), world, "max", device=dev)

    t_bwd = med_ms(lambda i: backward())
    t_after = med_ms(after)
    t_ready = med_ms(ready)
    return {"layers": L, "gemm": "3 per layer, 8192 x 1024 x 1024 bf16 (torch.matmul, one "
                                  "CUDA graph per layer)",
            "buckets": len(step.buckets), "iters": iters,
            "t_bwd_ms": round(t_bwd, 4), "t_step_after_backward_ms": round(t_after, 4),
            "t_step_ready_driven_ms": round(t_ready, 4),
            "exposed_after_backward_ms": round(t_after - t_bwd, 4),
            "exposed_ready_driven_ms": round(t_ready - t_bwd, 4)}
    return result


def run_ours(args):
    import torch
    from gradient_reduce_optimizer_gb300 import build as gbuild
    from gradient_reduce_optimizer_gb300 import capi

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    # one process per node compiles (if the library is stale); the others
    # wait, so that no two ranks write the same objects
    if local == 0:
        gbuild.build()
    barrier(world)
    capi.lib()

    if args.small:
        wk = build_small_workload(dev, args.small)
        args.no_e2e = args.no_overlap = args.no_cpu_baseline = True
        args.no_unfused = args.no_tp = args.no_launch_floor = True
        args.no_gpt2_slice = args.no_accum = args.no_bulk_rates = True
    else:
        wk = build_workload(dev, bucket_mib=args.bucket_mib)
    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    n_params = w.n
    bb = w.bucket_bytes
    stream = torch.cuda.current_stream()

    cuts = uniform_buckets(n_slab, bb)
    acc = None
    if args.small and (args.reducing or args.micro):
        # fp32 accumulators that stand for three earlier micro-steps
        acc = [g.float() * 3.0 for g in wk["grads"]]
        torch.cuda.synchronize()

    ws = None
    if args.small and args.unfused:
        ws = torch.empty(n_slab, dtype=torch.float32, device=dev)

    def one_step(step):
        if args.small and args.rank_step:
            # profile case: one rank's compute of the multi-GPU form over the
            # whole flat slab (R gradient slices in, the parameters out once)
            capi.cc_fused_dp_rank_step(wk["grads"], wk["master"], wk["m"], wk["v"],
                                       wk["outs"][0], n_slab, R, stream=stream,
                                       **step_args(wk, step))
        elif ws is not None:
            # profile case: the unfused schedule (reduce, AdamW, R-1 copies)
            capi.cc_unfused_dp_step(wk["grads"], wk["master"], wk["m"], wk["v"], wk["outs"],
                                    ws, ws.numel() * 4, n_slab, R, bb, stream=stream,
                                    **step_args(wk, step))
        elif args.small and args.micro:
            # profile case: one local micro-step (acc = g, or acc += g)
            capi.cc_accumulate_local(wk["grads"], acc, n_slab, R, args.micro == "first",
                                     stream=stream)
        elif acc is not None:
            capi.cc_fused_dp_step_accum(wk["grads"], acc, wk["master"], wk["m"], wk["v"],
                                        wk["outs"], n_slab, R, bb, accum_k=4,
                                        stream=stream, **step_args(wk, step))
        elif args.engine_ctas > 0:
            # a budget of SMs, bucket by bucket: the wide-CTA kernel, or the
            # bulk-copy engine
            flags = ((capi.CC_ARITH_FAST if args.fast_arith else 0) |
                     (capi.CC_ENGINE_BULK_COPY if args.bulk_copy else 0))
            for b, e in cuts:
                capi.cc_fused_dp_bucket_ex(wk["grads"], None, wk["master"], wk["m"],
                                           wk["v"], wk["outs"], n_slab, R, b, e,
                                           max_ctas=args.engine_ctas, arith_flags=flags,
                                           stream=stream, **step_args(wk, step))
        else:
            capi.cc_fused_dp_step(wk["grads"], wk["master"], wk["m"], wk["v"],
                                  wk["outs"], n_slab, R, bb, stream=stream,
                                  **step_args(wk, step))

    for i in range(args.warmup):
        one_step(w.step + i)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        one_step(w.step + args.warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms, value = aggregate(ms_local, float(n_params), world, device=dev)

    bytes_per_param = (2 * R + 26 if args.small and args.rank_step else
                       6 * R + 30 if ws is not None else
                       4 * R + 24 if acc is None else
                       (6 * R if args.micro == "first" else 10 * R) if args.micro else
                       8 * R + 24)
    launches = launches_per_step(n_slab, bb)
    per_launch_elems = n_slab / launches
    launch_ms = ms_local / launches           # launches run back to back
    achieved = bytes_per_param * per_launch_elems / (launch_ms * 1e-3) / 1e9
    peak, peak_src = measured_hbm_peak()
    tpp = (profiled_traffic_per_param(R)
           if args.engine_ctas == 0 and acc is None and ws is None and not args.rank_step
           else None)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": (round(tpp * per_launch_elems) if tpp else None),
                "peak_source": peak_src,
                "algorithmic_bytes_per_launch": round(bytes_per_param * per_launch_elems),
                "kernel": (f"fused_step_kernel<R={R}, one output> (rank step)"
                           if args.small and args.rank_step else
                           "reduce_kernel + adamw_kernel + copies" if ws is not None else
                           f"accumulate_kernel<R={R}, first={args.micro == 'first'}>"
                           if args.micro else
                           f"fused_step_kernel<R={R}, accumulators>" if acc is not None else
                           (f"fused_step_bulk_kernel<R={R}> on {args.engine_ctas} SMs"
                            if args.bulk_copy else
                            f"fused_step_kernel<R={R}, wide CTAs> on {args.engine_ctas} SMs")
                           if args.engine_ctas > 0 else f"fused_step_kernel<R={R}>"),
                "launches_per_step": launches}

    result = {
        "metric": METRIC, "value": round(value), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(args, R, world, n_params, n_slab, bb)
        if not args.small else {
            "workload": (f"profile case: flat slab of {n_slab} elements, R={R}, one bucket"
                         + (", unfused schedule" if ws is not None else
                            f", {args.micro} local micro-step" if args.micro else
                            ", reducing step with fp32 accumulators" if acc is not None else "")),
            "R": R, "n_slab": n_slab, "bucket_bytes": 0},
        "hbm_gbs": round(bytes_per_param * n_slab / (ms * 1e-3) / 1e9, 1),
        "hbm_pct_of_8tbs": round(100 * bytes_per_param * n_slab / (ms * 1e-3) / 8e12, 2),
        "roofline": roofline,
        "clocks": clk,
        "gpu_launches": launches * args.steps * (2 if ws is not None else 1),
    }

    if not args.no_unfused and not args.small:
        result["unfused"] = run_unfused(args, wk, stream, ms)
    if not args.small and not args.no_bulk_rates:
        result["bulk_engine_per_sm"] = run_bulk_rates(args, wk, stream)
    if not args.no_tp and not args.small:
        result["tp_matmul_allreduce"] = run_tp(args, dev)
    if not args.no_launch_floor and not args.small:
        result["launch_floor"] = run_launch_floor(args, dev)
    if not args.no_gpt2_slice and not args.small:
        result["gpt2_slice_r4"] = run_gpt2_slice(args, dev)
    if not args.no_accum and not args.small:
        result["accumulation"] = run_accumulation(args, wk, stream)
    if not args.no_unfused and not args.small:
        result["rank_step"] = run_rank_step(args, wk, stream)
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, wk, stream, world, dev)
    if args.small and args.overlap_small:
        # profile case: the overlap bench on the flat slab cut into 4 layers
        # (the proxy GEMM is the full-size one; a few GB resident)
        swk = small_overlap_workload(wk, 4)
        result["overlap_small"] = run_overlap(args, swk, dev, [1], num_layers=4)
    if not args.no_overlap:
        result["overlap"] = run_overlap(args, wk, dev, [args.bucket_mib])
        result["overlap_rank_share"] = run_overlap(args, wk, dev, [args.bucket_mib],
                                                   rank_share=True)
        # the overlapped arm on a static SM partition (green contexts), at the
        # partition sizes measured best for each mode
        result["overlap_partitioned"] = {
            "all_replicas_96_sms": run_overlap(args, wk, dev, [args.bucket_mib], comm_sms=96),
            "rank_share_48_sms": run_overlap(args, wk, dev, [args.bucket_mib],
                                             rank_share=True, comm_sms=48)}
        if not args.no_sweep:
            sweep = {}
            for share in (False, True):
                rows = run_overlap(args, wk, dev, [1, 4, 25, 100, 500], rank_share=share)
                sweep["rank_share" if share else "all_replicas"] = [
                    {k: r[k] for k in OVERLAP_KEEP} for r in rows]
            sweep["tuned_bucket_mib"] = {mode: next(r["bucket_mib"] for r in rows
                                                    if r["tuner_choice"])
                                         for mode, rows in list(sweep.items())}
            result["overlap_sweep"] = sweep
        # the rank share with the opt-in fast arithmetic: fewer instructions
        # per element, so the reduction takes less SM time beside the GEMMs
        result["overlap_rank_share_fast"] = [
            {k: r[k] for k in OVERLAP_KEEP + ("mode",)}
            for r in run_overlap(args, wk, dev, [25, 100], rank_share=True,
                                 arith_flags=capi.CC_ARITH_FAST)]
        if not args.no_accum:
            # the reducing k-th step of accumulation (k = 4) behind the same
            # backward: accumulators that stand for three earlier micro-steps
            acc = [torch.empty(n_slab, dtype=torch.float32, device=dev) for _ in range(R)]
            for j in range(3):
                capi.cc_accumulate_local(wk["grads"], acc, n_slab, R, j == 0, stream=stream)
            torch.cuda.synchronize()
            red = {}
            for share in (False, True):
                rows = run_overlap(args, wk, dev, [1, 4, 25, 100, 500], rank_share=share,
                                   acc=acc)
                red["rank_share" if share else "all_replicas"] = [
                    {k: r[k] for k in OVERLAP_KEEP} for r in rows]
            red["tuned_bucket_mib"] = {mode: next(r["bucket_mib"] for r in rows
                                                  if r["tuner_choice"])
                                       for mode, rows in list(red.items())}
            result["overlap_reducing_step"] = red
            del acc
            torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = run_cpu_baseline(args, wk, dev)
    if rank == 0:
        print(json.dumps(result), flush=True)
    return result


def run_gpt2_slice(args, dev, steps=20):
    """The fused step on 24 GPT-2 8.3B layers (2,718,867,456 parameters, 288
    tensors) at R = 4 with loss scale 65536 and 25 MiB buckets: (4R + 24) =
    40 bytes per parameter, 108.8 GB per step, 76 GB resident in HBM."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi
    from gradient_reduce_optimizer_gb300 import workloads as wl

    wk = build_workload(dev, preset=wl.gpt2_slice_r4())
    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    stream = torch.cuda.current_stream()

    def step(i):
        capi.cc_fused_dp_step(wk["grads"], wk["master"], wk["m"], wk["v"], wk["outs"],
                              n_slab, R, w.bucket_bytes, stream=stream,
                              **step_args(wk, w.step + i))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    bpp = 4 * R + 24
    peak, src = measured_hbm_peak()
    gbs = bpp * n_slab / (ms * 1e-3) / 1e9
    out = {"workload": ("24 GPT-2 8.3B layers (hidden 3072, FFN 12288), R=4, "
                        "loss scale 65536, 25 MiB buckets in reverse layer order"),
           "n_params": w.n, "n_slab": n_slab, "R": R,
           "launches_per_step": launches_per_step(n_slab, w.bucket_bytes),
           "ms_per_step": round(ms, 3), "params_per_s": round(w.n / (ms * 1e-3)),
           "bytes_per_param": bpp, "hbm_gbs": round(gbs, 1),
           "frac": round(gbs / peak, 4), "peak_source": src, "steps": steps}
    del wk
    torch.cuda.empty_cache()
    return out


def run_launch_floor(args, dev, reps=100, samples=50):
    """The small flat case: R = 2, 1,048,576 parameters, one bucket, step 1
    from m = v = 0.  Its 33.5 MB per step ((4R + 24) bytes per parameter)
    fit in the 129 MB L2, so this measures the launch and L2 floor, three
    ways:
      flushed  one launch at a time, a 512 MiB write before each (the
               step's inputs come from HBM, and its loads evict the
               flush's dirty lines), median over `samples`
      flushed_clean  the same with a 512 MiB read after the write (the L2
               holds clean lines only: the step's own traffic alone)
      warm     `reps` launches back to back from the stream (L2-resident)
      graph    the same `reps` launches captured once in a CUDA graph and
               replayed, median over `samples` replays."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi
    from gradient_reduce_optimizer_gb300 import workloads as wl

    w = wl.flat_1m_r2()
    R, n = w.R, w.n
    grads = wl.make_grads(R, n, w.grad_sigma, device=dev)
    master, m, v = wl.make_state(n, w.step, w.grad_sigma, device=dev)
    outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    hp = {k: getattr(w, k) for k in ("lr", "beta1", "beta2", "eps",
                                     "weight_decay", "step", "grad_scale")}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    step_bytes = (4 * R + 24) * n

    def step(stream):
        capi.cc_fused_dp_step(grads, master, m, v, outs, n, R, 0, stream=stream, **hp)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step(stream)
    torch.cuda.synchronize()

    pairs = []
    for _ in range(samples):
        capi.cc_l2_flush(flush, flush.numel(), stream=stream)
        e0, e1 = ev(), ev()
        e0.record(stream)
        step(stream)
        e1.record(stream)
        pairs.append((e0, e1))
    torch.cuda.synchronize()
    flushed_us = statistics.median(a.elapsed_time(b) for a, b in pairs) * 1e3

    # the same after a read of another 512 MiB: the flush's dirty lines are
    # written back before the launch, so the step pays only for its own
    # traffic from HBM
    clean = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean.fill_(1)
    pairs = []
    for _ in range(samples):
        capi.cc_l2_flush(flush, flush.numel(), stream=stream)
        clean.max()
        e0, e1 = ev(), ev()
        e0.record(stream)
        step(stream)
        e1.record(stream)
        pairs.append((e0, e1))
    torch.cuda.synchronize()
    clean_us = statistics.median(a.elapsed_time(b) for a, b in pairs) * 1e3
    del clean

    e0, e1 = ev(), ev()
    e0.record(stream)
    for _ in range(reps):
        step(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    warm_us = e0.elapsed_time(e1) * 1e3 / reps

    out = {"workload": f"flat slab of {n:,} parameters, R={R}, one bucket, step 1, "
                       "m = v = 0, wd 0",
           "bytes_per_step": step_bytes,
           "flushed_us": round(flushed_us, 2),
           "flushed_gbs": round(step_bytes / (flushed_us * 1e-6) / 1e9, 1),
           "flushed_clean_us": round(clean_us, 2),
           "flushed_clean_gbs": round(step_bytes / (clean_us * 1e-6) / 1e9, 1),
           "warm_us": round(warm_us, 2),
           "warm_gbs": round(step_bytes / (warm_us * 1e-6) / 1e9, 1),
           "reps": reps}
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream()
            for _ in range(reps):
                step(cap)
        graph.replay()
        torch.cuda.synchronize()
        pairs = []
        for _ in range(samples):
            e0, e1 = ev(), ev()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            pairs.append((e0, e1))
        torch.cuda.synchronize()
        graph_us = statistics.median(a.elapsed_time(b) for a, b in pairs) * 1e3 / reps
        out.update(graph_us=round(graph_us, 2),
                   graph_gbs=round(step_bytes / (graph_us * 1e-6) / 1e9, 1))
        del graph
    except RuntimeError as e:        # capture refused: report, keep the run
        out["graph_error"] = str(e).splitlines()[0][:200]
    return out


def run_tp(args, dev, R=8, m=8192, n=3072, k=12288, chunk_list=(1, 2, 4, 8, 16)):
    """The tensor-parallel MatMul-then-AllReduce of a GPT-2 8.3B MLP output
    projection (row-parallel: k = 12288 -> n = 3072 over m = 8192 tokens) at
    tensor-parallel degree R = 8, sequential and overlapped in chunks of rows
    ("LIT-735", Key takeaways: chunked overlap of the two, reported to hide
    most of the MatMul's time)."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    kr = k // R
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    # each operand one buffer cut into R equal shards (batched GEMM per chunk)
    x = list(torch.randn(R * m * kr, generator=g, device=dev).to(torch.bfloat16).view(R, -1))
    w = list((torch.randn(R * kr * n, generator=g, device=dev) * 0.02)
             .to(torch.bfloat16).view(R, -1))
    partials = list(torch.empty(R, m * n, device=dev))
    outs = [torch.empty(m * n, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    rows = []
    for chunks in chunk_list:
        t = capi.cc_tp_overlap_bench(R=R, m=m, n=n, k=k, chunks=chunks, x=x, w=w,
                                     partials=partials, out=outs, warmup=args.warmup,
                                     iters=args.overlap_iters,
                                     stream_priority=args.stream_priority)
        hidden = (t["t_sequential_ms"] - t["t_overlap_ms"]) / t["t_allreduce_ms"]
        rows.append({"chunks": chunks, **{key: round(v, 4) for key, v in t.items()},
                     "allreduce_hidden_pct": round(100 * hidden, 1),
                     "speedup_vs_sequential": round(t["t_sequential_ms"] / t["t_overlap_ms"], 3)})
    ar = rows[0]["t_allreduce_ms"]
    tflops = 2 * m * n * k / (rows[0]["t_gemm_ms"] * 1e-3) / 1e12
    bf16_peak = measured_bf16_peak()
    del partials
    fused = run_tp_fused(args, dev, x, w, outs, R, m, n, k,
                         sequential_ms=rows[0]["t_sequential_ms"])
    return {"shape": {"R": R, "m": m, "n": n, "k": k},
            "gemm_tflops": round(tflops, 1),
            "gemm_frac_of_measured_bf16": round(tflops / bf16_peak, 3) if bf16_peak else None,
            "allreduce_bytes": 6 * R * m * n,
            "allreduce_hbm_gbs": round(6 * R * m * n / (ar * 1e-3) / 1e9, 1),
            "chunks": rows, "fused_tcgen05": fused}


def run_tp_fused(args, dev, x, w, outs, R, m, n, k, sequential_ms=None, reps=20):
    """The same layer through cc_tp_matmul_allreduce: one tcgen05 kernel that
    keeps the R partial products in TMEM and writes only the R bf16 outputs.
    The weight shards are given K-contiguous (n x k/R, a linear layer's
    layout): the transposes of the shards the cuBLAS arm reads."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    kr = k // R
    wt = [wr.view(kr, n).t().contiguous() for wr in w]
    stream = torch.cuda.current_stream()
    ws_bytes = capi.cc_tp_matmul_allreduce_workspace(m, n, k, R)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def timed(call):
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    # the last wave split over every CTA pair (the workspace form), and
    # every group of output tiles whole (no workspace)
    ms = timed(lambda: capi.cc_tp_matmul_allreduce_ex(x, wt, outs, None, m, n, k, R, ws,
                                                      ws_bytes, 0, stream=stream))
    ms_whole = timed(lambda: capi.cc_tp_matmul_allreduce(x, wt, outs, None, m, n, k, R,
                                                         stream=stream))
    status = capi.cc_device_status(clear=True)
    tflops = 2 * m * n * k / (ms * 1e-3) / 1e12
    bf16_peak = measured_bf16_peak()
    out = {"kernel": "tp_fused_pair_kernel (tcgen05 cta_group::2, TMA, TMEM accumulators)",
           "ms": round(ms, 4), "tflops": round(tflops, 1),
           "frac_of_measured_bf16": round(tflops / bf16_peak, 3) if bf16_peak else None,
           "workspace_bytes": ws_bytes, "ms_without_workspace": round(ms_whole, 4),
           "hbm_bytes_algorithmic": 2 * (m * k + n * k) + 2 * R * m * n,
           "status_word": status, "launches": 2 * reps}
    if sequential_ms:
        out["speedup_vs_cublas_then_allreduce"] = round(sequential_ms / ms, 3)
    del wt, ws
    return out


def run_bulk_rates(args, wk, stream, elems=1 << 25, ctas_list=(16, 32, 64, 96), reps=5):
    """What one SM streams under a CTA budget, exact and fast arithmetic,
    on both budget engines: the wide-CTA kernel (the default) and the TMA
    bulk-copy engine (CC_ENGINE_BULK_COPY).  The first 2^25 slab elements of
    the headline workload stepped on 16..96 SMs.  GB/s of the step's
    (4R + 24) algorithmic bytes per parameter, in total and per SM."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    elems = min(elems, n_slab) // 8 * 8
    bpp = 4 * R + 24
    rows = []
    for ctas in ctas_list:
        row = {"ctas": ctas}
        for name, flags in (("exact", 0), ("fast", capi.CC_ARITH_FAST),
                            ("bulk_copy_exact", capi.CC_ENGINE_BULK_COPY),
                            ("bulk_copy_fast", capi.CC_ENGINE_BULK_COPY | capi.CC_ARITH_FAST)):
            def one(i):
                capi.cc_fused_dp_bucket_ex(wk["grads"], None, wk["master"], wk["m"], wk["v"],
                                           wk["outs"], n_slab, R, 0, elems, max_ctas=ctas,
                                           arith_flags=flags, stream=stream,
                                           **step_args(wk, w.step + i))
            one(0)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(reps):
                one(1 + i)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            gbs = bpp * elems / (ms * 1e-3) / 1e9
            row[name] = {"ms": round(ms, 4), "gbs": round(gbs, 1),
                         "gbs_per_sm": round(gbs / ctas, 1)}
        rows.append(row)
    assert capi.cc_device_status(clear=True) == 0
    return {"elements": elems, "bytes_per_param": bpp, "rows": rows}


def run_accumulation(args, wk, stream, k=4):
    """Gradient accumulation with k micro-steps on the same workload: k-1
    local micro-steps (first: acc = g, 6R bytes per parameter; later:
    acc += g, 10R) and the reducing step, the fused kernel with the
    accumulators (8R + 24).  The reducing step, not a typical micro-step,
    is the one the accumulation paragraph of Overlapping Communication and
    Computation says to profile."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    acc = [torch.empty(n_slab, dtype=torch.float32, device=wk["master"].device)
           for _ in range(R)]
    reps = max(3, min(args.steps, 20))

    def timed(fn):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(reps):
            fn(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / reps

    def micro(first):
        return lambda i: capi.cc_accumulate_local(wk["grads"], acc, n_slab, R, first,
                                                  stream=stream)

    def reducing(i):
        capi.cc_fused_dp_step_accum(wk["grads"], acc, wk["master"], wk["m"], wk["v"],
                                    wk["outs"], n_slab, R, w.bucket_bytes,
                                    accum_k=k, stream=stream, **step_args(wk, w.step + i))

    def whole(i):
        for j in range(k - 1):
            micro(j == 0)(i)
        reducing(i)

    out = {"accum_k": k}
    for name, fn, bpp in (("micro_first", micro(True), 6 * R),
                          ("micro_later", micro(False), 10 * R),
                          ("reducing_step", reducing, 8 * R + 24)):
        ms = timed(fn)
        out[name] = {"ms": round(ms, 4), "bytes_per_param": bpp,
                     "hbm_gbs": round(bpp * n_slab / (ms * 1e-3) / 1e9, 1)}
    ms = timed(whole)
    total = 6 * R + (k - 2) * 10 * R + 8 * R + 24
    out["optimizer_step"] = {"ms": round(ms, 4), "bytes_per_param": total,
                             "hbm_gbs": round(total * n_slab / (ms * 1e-3) / 1e9, 1),
                             "params_per_s": round(w.n / (ms * 1e-3))}
    del acc
    torch.cuda.empty_cache()
    return out


def run_rank_step(args, wk, stream):
    """One rank's compute in the real multi-GPU form, on this GPU: rank 0's
    shard of every planned bucket of the headline slab (cc_shard_plan over
    R ranks), its R gradient slices read straight from the replica slabs
    (where the ReduceScatter would have put them), its state shard packed
    in launch order, its bf16 parameters written once.  (2R + 24 + 2)
    algorithmic bytes per shard element; the exchanges themselves need
    several GPUs and are not in this figure."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w, R = wk["w"], wk["w"].R
    shards, state_off, elems = capi.cc_shard_plan(wk["buckets"], R)
    n0 = elems[0]
    dev = wk["master"].device
    master = wk["master"][:n0].clone()
    m = wk["m"][:n0].clone()
    v = wk["v"][:n0].clone()
    # the views each launch takes, built once
    calls = [([g[lo:hi] for g in wk["grads"]], master[o:o + hi - lo], m[o:o + hi - lo],
              v[o:o + hi - lo], wk["outs"][0][lo:hi], hi - lo)
             for (lo, hi), o in ((row[0], off[0]) for row, off in zip(shards, state_off))
             if hi > lo]

    def one(step, strm):
        hp = step_args(wk, step)
        for sl, ms_, mm_, vv_, out, length in calls:
            capi.cc_fused_dp_rank_step(sl, ms_, mm_, vv_, out, length, R, stream=strm, **hp)

    def timed(fn, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for i in range(3):
        one(w.step + i, stream)
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 20))
    # issued from Python, one call per bucket (host-bound at these sizes)
    host_ms = timed(lambda i: one(w.step + 3 + i, stream), reps)
    # the same launches captured once in a CUDA graph and replayed: the
    # device's own time for the step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        one(w.step, torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    ms = timed(lambda i: graph.replay(), reps)
    del graph
    bpp = 2 * R + 26
    gbs = bpp * n0 / (ms * 1e-3) / 1e9
    peak, _ = measured_hbm_peak()
    del master, m, v, calls
    return {"workload": f"rank 0 of {R}: its shard of each of the {len(shards)} planned buckets",
            "shard_elements": n0, "ms": round(ms, 4), "timing": "CUDA graph of one step",
            "bytes_per_element": bpp, "hbm_gbs": round(gbs, 1),
            "frac_of_measured_copy": round(gbs / peak, 3),
            "launches_per_step": len(shards), "ms_issued_from_python": round(host_ms, 4)}


def run_unfused(args, wk, stream, fused_ms):
    """The same step in the unfused schedule (reduce into a workspace, AdamW,
    broadcast copies): the separate-kernel baseline the fused step is
    compared against.  Same workload, buckets and timing rules."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    bb = w.bucket_bytes
    per = max(8, bb // 16 * 8) if bb else n_slab
    ws = torch.empty(min(per, n_slab), dtype=torch.float32, device=wk["master"].device)

    def step(i):
        capi.cc_unfused_dp_step(wk["grads"], wk["master"], wk["m"], wk["v"],
                                wk["outs"], ws, ws.numel() * 4, n_slab, R, bb,
                                stream=stream, **step_args(wk, w.step + i))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 100))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    buckets = launches_per_step(n_slab, bb)
    return {"ms_per_step": round(ms, 4), "value": round(w.n / (ms * 1e-3)),
            "unit": UNIT, "steps": steps,
            "bytes_per_param": 6 * R + 30,
            "hbm_gbs": round((6 * R + 30) * n_slab / (ms * 1e-3) / 1e9, 1),
            "launches_per_step": buckets * 2, "copies_per_step": buckets * (R - 1),
            "fused_speedup": round(ms / fused_ms, 3)}


def run_e2e(args, wk, stream, world, dev):
    """The step through the C ABI with HOST buffers, the GB300 way: the R
    gradient slabs and one parameter replica live in pinned host memory and
    the fused kernel reads and writes them directly over NVLink-C2C, so the
    host->device traffic (R x 2n bytes of gradients) and the device->host
    result (2n bytes of parameters) move inside the timed step with no
    staging copy.  master/m/v stay in HBM, as across real training steps."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    host_grads = [g.cpu().pin_memory() for g in wk["grads"]]
    host_out = torch.empty(n_slab, dtype=torch.bfloat16).pin_memory()
    outs = [host_out] + wk["outs"][1:]
    steps = max(3, min(args.steps, args.e2e_steps))

    def e2e_step(step):
        capi.cc_fused_dp_step(host_grads, wk["master"], wk["m"], wk["v"], outs,
                              n_slab, R, w.bucket_bytes, stream=stream,
                              **step_args(wk, step))

    for i in range(args.warmup):
        e2e_step(w.step + i)
    torch.cuda.synchronize()
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        e2e_step(w.step + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_local = ev0.elapsed_time(ev1) / steps
    ms, value = aggregate(ms_local, float(w.n), world, device=dev)
    staged = run_e2e_staged(args, wk, stream, world, dev, host_grads, host_out)
    return {"value": round(value), "unit": UNIT,
            "h2d_bytes_per_step": 2 * R * n_slab, "d2h_bytes_per_step": 2 * n_slab,
            "ms_per_step": round(ms, 3), "steps": steps,
            "how": "gradients and replica 0 in pinned host memory, read/written by "
                   "the fused kernel over NVLink-C2C",
            "c2c_gbs": round(2 * (R + 1) * n_slab / (ms * 1e-3) / 1e9, 1),
            "staged": staged}


def run_e2e_staged(args, wk, stream, world, dev, host_grads, host_out):
    """For comparison: the same step with explicit staging -- every step
    copies the R gradient slabs in from pinned host memory and the updated
    bf16 parameters (one replica; the others are bit-identical) back out."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w, n_slab, R = wk["w"], wk["n_slab"], wk["w"].R
    steps = max(3, min(args.steps, args.e2e_steps))

    def e2e_step(step):
        for h, d in zip(host_grads, wk["grads"]):
            d.copy_(h, non_blocking=True)
        capi.cc_fused_dp_step(wk["grads"], wk["master"], wk["m"], wk["v"],
                              wk["outs"], n_slab, R, w.bucket_bytes,
                              stream=stream, **step_args(wk, step))
        host_out.copy_(wk["outs"][0], non_blocking=True)

    for i in range(args.warmup):
        e2e_step(w.step + i)
    torch.cuda.synchronize()
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        e2e_step(w.step + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_local = ev0.elapsed_time(ev1) / steps
    ms, value = aggregate(ms_local, float(w.n), world, device=dev)
    return {"value": round(value), "unit": UNIT,
            "h2d_bytes_per_step": 2 * R * n_slab, "d2h_bytes_per_step": 2 * n_slab,
            "ms_per_step": round(ms, 3), "steps": steps}


def run_overlap(args, wk, dev, mibs, rank_share=False, comm_sms=0, acc=None,
                num_layers=24, arith_flags=0):
    """Exposed time of the bucketed step behind a proxy backward of
    num_layers x 3 bf16 GEMMs (M=8192, N=K=1024); buckets planned at each
    size.

    rank_share=False: one GPU carries all R replicas' traffic (the emulated
    step).  rank_share=True: one rank's share of the sharded step -- each
    bucket shrinks to rank 0's 1/R shard: it reads the R replicas' gradients
    of the shard, updates the shard's master/m/v and writes the shard's
    parameters to all R replica slabs, (4 + 24/R) bytes per parameter.
    acc: the R fp32 accumulators of gradient accumulation, which makes every
    bucket the reducing k-th step ((8R + 24) bytes per parameter; a rank's
    share (8 + 24/R)): with accumulation, the reducing step must hide the
    whole model's gradient traffic behind only its own backward
    (Overlapping Communication and Computation, the accumulation
    paragraph)."""
    import torch
    from gradient_reduce_optimizer_gb300 import capi

    w = wk["w"]
    M, N, K = 8192, 1024, 1024
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    A = torch.randn(M * K, generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn(K * N, generator=g, device=dev).to(torch.bfloat16)
    C = torch.empty(M * N, dtype=torch.bfloat16, device=dev)
    # every size through the library's tuner: it plans each cap (and rank
    # 0's shard of each bucket), times it and names the shortest step
    _, _, n_slab = capi.cc_plan_buckets(wk["numel"], 0)
    assert n_slab == wk["n_slab"]
    best, results = capi.cc_tune_bucket_bytes(
        numel=wk["numel"], layer_of=wk["layer_of"], candidates=[mib << 20 for mib in mibs],
        rank=0 if rank_share else -1,
        grads=wk["grads"], master=wk["master"], m=wk["m"], v=wk["v"],
        params_out=wk["outs"], n=n_slab, R=w.R, num_layers=num_layers, gemms_per_layer=3,
        gemm_m=M, gemm_n=N, gemm_k=K, gemm_a=A, gemm_b=B, gemm_c=C,
        warmup=args.warmup, iters=args.overlap_iters,
        max_ctas=args.overlap_ctas, stream_priority=args.stream_priority,
        comm_sms=comm_sms, gemm_algo=args.overlap_gemm_algo,
        budget_buckets=args.overlap_budget_buckets, acc=acc, arith_flags=arith_flags,
        **step_args(wk, w.step))
    out = []
    for mib, r in zip(mibs, results):
        r = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()}
        r["bucket_mib"] = mib
        r["tuner_choice"] = (mib << 20) == best
        r["mode"] = (("rank share (1/R of each bucket)" if rank_share else "all R replicas")
                     + (", reducing step with fp32 accumulators" if acc is not None else "")
                     + (", fast arithmetic" if arith_flags else ""))
        r["exposed_pct_of_bwd"] = round(100 * r["exposed_ms"] / r["t_bwd_ms"], 1)
        r["bwd_tflops"] = round(num_layers * 3 * 2 * M * N * K / (r["t_bwd_ms"] * 1e-3) / 1e12,
                                1)
        bf16_peak = measured_bf16_peak()
        r["bwd_frac_of_measured_bf16"] = (round(r["bwd_tflops"] / bf16_peak, 3)
                                          if bf16_peak else None)
        out.append(r)
    return out[0] if len(out) == 1 else out


OVERLAP_KEEP = ("bucket_mib", "tuner_choice", "num_buckets", "t_bwd_ms", "t_comm_ms",
                "t_step_overlap_ms", "t_step_seq_ms", "exposed_ms", "exposed_bound_ms",
                "t_overlap_ms", "overlap_eff")


def small_overlap_workload(wk, num_layers):
    """The profile case's flat slab seen as num_layers equal tensors (one
    per layer), so that the overlap bench has buckets that become ready
    layer by layer, with few GB resident."""
    n = wk["n_slab"]
    per = n // num_layers // 8 * 8
    numel = [per] * (num_layers - 1) + [n - per * (num_layers - 1)]
    wk = dict(wk)
    wk["numel"], wk["layer_of"] = numel, list(range(num_layers))
    from gradient_reduce_optimizer_gb300 import capi
    offsets, _, n_slab = capi.cc_plan_buckets(numel, 0)
    assert n_slab == n
    wk["offsets"] = offsets
    return wk


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1:
        # rank 0 runs the oracle for minutes before the closing barrier
        dist_init(world, "gloo", timeout_s=1800.0)
    if rank != 0:
        barrier(world)
        return None
    from oracle import build as obuild
    obuild.build()
    import oracle
    from gradient_reduce_optimizer_gb300 import workloads as wl
    w = wl.bert_large_r8(bucket_bytes=args.bucket_mib * wl.MiB)
    R = w.R
    _, _, n_slab = oracle.plan_buckets(w.numel(), w.bucket_bytes)
    threads = args.ref_threads or host_cores()
    g16, st, hp, sample = oracle_sample_inputs(R, args.ref_sample)
    runner = OracleRunner(g16, st, hp, threads)
    for _ in range(args.warmup):
        runner.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        runner.step()
    el = time.perf_counter() - t0
    runner.close()
    threads = len(runner.chunks)
    value = sample * args.steps / el
    desc = (f"first {sample:,} slab elements of the BERT-large R=8 workload per "
            + ("step, single-threaded C oracle" if threads == 1 else
               f"step, split into {threads} contiguous chunks, one C oracle call "
               "per chunk on its own host thread"))
    result = {
        "metric": METRIC, "value": round(value), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "impl": "reference",
        "config": headline_config(args, R, world, w.n, n_slab, w.bucket_bytes),
        "cpu_baseline": {"value": round(value), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    barrier(world)
    return result


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--bucket-mib", type=int, default=25)
    p.add_argument("--engine-ctas", type=int, default=0,
                   help="run each bucket on a budget of this many SMs "
                        "(cc_fused_dp_bucket max_ctas: the wide-CTA kernel); 0 = the "
                        "plain kernel over the whole GPU")
    p.add_argument("--rank-step", action="store_true",
                   help="with --small: one rank's compute of the multi-GPU form "
                        "(cc_fused_dp_rank_step over the flat slab)")
    p.add_argument("--bulk-copy", action="store_true",
                   help="with --engine-ctas: the TMA bulk-copy engine (CC_ENGINE_BULK_COPY)")
    p.add_argument("--small", type=int, default=0,
                   help="profile case: a flat R=8 slab of this many elements, "
                        "one bucket, device timing only")
    p.add_argument("--reducing", action="store_true",
                   help="with --small: time the reducing step with fp32 accumulators")
    p.add_argument("--unfused", action="store_true",
                   help="with --small: time the unfused schedule (reduce, AdamW, copies)")
    p.add_argument("--micro", choices=("first", "later"), default=None,
                   help="with --small: time one local micro-step (acc = g, or acc += g)")
    p.add_argument("--dist", action="store_true",
                   help="the real multi-GPU form (one replica per rank, NCCL exchanges); "
                        "the default under torchrun with more than one rank")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--tp-only", type=int, default=0,
                   help="profile case: only the tensor-parallel path, with this many rows")
    p.add_argument("--no-tp", action="store_true",
                   help="skip the tensor-parallel MatMul-then-AllReduce overlap")
    p.add_argument("--no-gpt2-slice", action="store_true",
                   help="skip the 2.7B-parameter GPT-2 slice at R=4 (76 GB)")
    p.add_argument("--no-launch-floor", action="store_true",
                   help="skip the small L2-resident case (single launches, CUDA graph)")
    p.add_argument("--no-accum", action="store_true",
                   help="skip timing gradient accumulation (k=4)")
    p.add_argument("--no-bulk-rates", action="store_true",
                   help="skip the bulk engine's per-SM rates (exact and fast arithmetic)")
    p.add_argument("--fast-arith", action="store_true",
                   help="with --small --engine-ctas: the opt-in fast arithmetic")
    p.add_argument("--no-unfused", action="store_true",
                   help="skip timing the unfused (reduce, AdamW, copies) schedule")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-overlap", action="store_true")
    p.add_argument("--overlap-small", action="store_true",
                   help="with --small: the overlap bench on the flat slab cut into 4 "
                        "layers (profile case for the proxy GEMM)")
    p.add_argument("--overlap-iters", type=int, default=20)
    p.add_argument("--overlap-ctas", type=int, default=0)
    p.add_argument("--overlap-budget-buckets", type=int, default=0,
                   help="overlap: only the first this-many buckets take --overlap-ctas; "
                        "the rest wait for the backward and take the whole GPU")
    p.add_argument("--overlap-gemm-algo", type=int, default=0,
                   help="overlap: 0 = the proxy GEMMs through cublasGemmEx; k > 0 = "
                        "through cuBLASLt with its k-th heuristic candidate")
    p.add_argument("--stream-priority", type=int, default=2, choices=(0, 1, 2),
                   help="overlap: 0 equal, 1 side stream high, 2 compute high")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the 1/4/25/100/500 MiB bucket-size sweep")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample", type=int, default=1 << 22)
    p.add_argument("--ref-sample", type=int, default=1 << 22)
    p.add_argument("--ref-threads", type=int, default=0,
                   help="reference arm: host threads (0 = every core this process may use)")
    a = p.parse_args(argv)
    a.warmup = max(3, a.warmup)     # at least 3 untimed warm-up steps
    return a


def main(argv=None):
    args = parse_args(argv)
    if args.tp_only:
        # profile case: the tensor-parallel path alone, m rows
        import torch
        torch.cuda.set_device(0)
        from gradient_reduce_optimizer_gb300 import build as gbuild
        gbuild.build()
        print(json.dumps({"tp_matmul_allreduce": run_tp(args, torch.device("cuda", 0),
                                                        m=args.tp_only, chunk_list=(1, 4))}),
              flush=True)
        return
    _, world, _ = dist_env()
    if args.impl == "reference":
        run_reference(args)
    elif world > 1 or args.dist:
        run_dist(args)
    else:
        run_ours(args)
    _, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
