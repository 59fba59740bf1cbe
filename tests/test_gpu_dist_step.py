"""The real multi-GPU form of the step on the GPU: the rank step kernel
(cc_fused_dp_rank_step: R gradient slices in, one parameter shard out) and
the package's ShardedStep over NCCL.

This run has one GPU, so (a) R ranks are played one after another in one
process -- each rank's slices are views of the R replica slabs, which is
what the ReduceScatter exchange delivers -- with the AllGather done by
copies, and the result must equal the oracle's emulated step bit for bit;
(b) ShardedStep runs over a real NCCL process group of one rank.  The
exchanges between ranks are covered over gloo on the host
(tests/test_sharded_step_gloo.py)."""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gradient_reduce_optimizer_gb300 import workloads as wl
from gpu_common import DEV, compare_all, host_copy, new_slabs, oracle_step, u16

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=4,
          grad_scale=2.0)


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    capi.lib()


def small_model():
    t = wl.bert_large_tensors(layers=2, hidden=64, ffn=256, vocab=101, positions=16)
    return [x[1] for x in t]


def seeded(n, R, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    grads = [(torch.randn(n, generator=g, device=DEV) * 2e-3).to(torch.bfloat16)
             for _ in range(R)]
    master = torch.randn(n, generator=g, device=DEV) * 0.02
    m = torch.randn(n, generator=g, device=DEV) * 1e-4
    v = (torch.randn(n, generator=g, device=DEV) * 1e-3) ** 2
    return grads, master, m, v


@pytest.mark.parametrize("R,bucket_bytes", [(1, 4096), (2, 4096), (3, 1000), (8, 0),
                                            (16, 2048)])
def test_ranks_played_in_turn_equal_the_emulated_step(R, bucket_bytes):
    numel = small_model()
    _, buckets, n = capi.cc_plan_buckets(numel, bucket_bytes)
    shards, state_off, elems = capi.cc_shard_plan(buckets, R)
    grads, master, m, v = seeded(n, R, seed=60 + R)
    ref = new_slabs(grads, master.clone(), m.clone(), v.clone())
    h_grads, h_state, _ = host_copy(ref)
    ref_outs = oracle_step(h_grads, h_state, HP)
    params = [torch.full((n,), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
              for _ in range(R)]
    states = []
    for q in range(R):                       # rank q's packed state of its shards
        st = [torch.empty(elems[q], device=DEV) for _ in range(3)]
        for b, row in enumerate(shards):
            lo, hi = row[q]
            o = state_off[b][q]
            for dst, src in zip(st, (master, m, v)):
                dst[o:o + hi - lo] = src[lo:hi]
        states.append(st)
    for b, row in enumerate(shards):
        for q in range(R):                   # every rank's update of bucket b
            lo, hi = row[q]
            o = state_off[b][q]
            slices = [grads[p][lo:hi] for p in range(R)]
            capi.cc_fused_dp_rank_step(slices, *(s[o:o + hi - lo] for s in states[q]),
                                       params[q][lo:hi], hi - lo, R, **HP)
        for q in range(R):                   # the AllGather, by copies
            lo, hi = row[q]
            for p in range(R):
                if p != q:
                    params[p][lo:hi].copy_(params[q][lo:hi])
    torch.cuda.synchronize()
    for p in range(R):
        np.testing.assert_array_equal(u16(params[p]), ref_outs[p], err_msg=f"params[{p}]")
    for q in range(R):
        for b, row in enumerate(shards):
            lo, hi = row[q]
            o = state_off[b][q]
            for got, want in zip(states[q], h_state):
                a = got[o:o + hi - lo].cpu().numpy()
                np.testing.assert_array_equal(a.view(np.uint32), want[lo:hi].view(np.uint32))


def test_sharded_step_over_nccl_world_one():
    import torch.distributed as dist
    from gradient_reduce_optimizer_gb300.dist import ShardedStep

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                            world_size=1)
    try:
        numel = small_model()
        step = ShardedStep(numel, 4096, rank=0, world=1, device=DEV)
        n = step.n_slab
        assert step.state_elems == n
        grads, master, m, v = seeded(n, 1, seed=70)
        params = torch.full((n,), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        st = [master.clone(), m.clone(), v.clone()]
        # world 1: the packed state is the slab's own order
        ref = new_slabs(grads, master, m, v)
        h_grads, h_state, _ = host_copy(ref)
        for t in range(2):
            step.step(grads[0], *st, params, **dict(HP, step=HP["step"] + t))
            ref_outs = oracle_step(h_grads, h_state, dict(HP, step=HP["step"] + t))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(u16(params), ref_outs[0])
        for got, want in zip(st, h_state):
            np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32),
                                          want.view(np.uint32))
    finally:
        dist.destroy_process_group()


def test_ready_driven_schedule_over_nccl_waits_for_each_layer():
    """ShardedStep's ready-driven schedule (begin / layer_ready / end) over
    a one-rank NCCL group.  The gradient slab starts with every tensor NaN;
    a stand-in backward on the caller's stream restores each layer's
    gradients, from the last layer down, after a ~50 us spin, and reports
    the layer.  A bucket's update ordered before its layer's gradients would
    read NaN: two steps must equal the oracle's, bit for bit."""
    import torch.distributed as dist
    from gradient_reduce_optimizer_gb300.dist import ShardedStep

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                            world_size=1)
    try:
        t = wl.bert_large_tensors(layers=2, hidden=64, ffn=256, vocab=101, positions=16)
        numel, layer_of = [x[1] for x in t], [x[2] for x in t]
        step = ShardedStep(numel, 4096, rank=0, world=1, device=DEV, layer_of=layer_of)
        n = step.n_slab
        grads, master, m, v = seeded(n, 1, seed=71)
        real = grads[0]
        params = torch.full((n,), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        st = [master.clone(), m.clone(), v.clone()]
        ref = new_slabs(grads, master, m, v)
        h_grads, h_state, _ = host_copy(ref)
        stream = torch.cuda.current_stream()
        for k in range(2):
            hp = dict(HP, step=HP["step"] + k)
            g = real.clone()
            for off, cnt in zip(step.offsets, numel):
                g[off:off + cnt] = float("nan")
            step.begin(g, *st, params, stream=stream, **hp)
            went = 0
            for layer in range(max(layer_of), -1, -1):
                torch.cuda._sleep(100_000)       # a slow layer of the backward
                for ti, (off, cnt) in enumerate(zip(step.offsets, numel)):
                    if layer_of[ti] == layer:
                        g[off:off + cnt].copy_(real[off:off + cnt])
                went += step.layer_ready(layer)
            assert went == len(step.buckets)
            step.end()
            ref_outs = oracle_step(h_grads, h_state, hp)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(u16(params), ref_outs[0])
        for got, want in zip(st, h_state):
            np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32),
                                          want.view(np.uint32))
    finally:
        dist.destroy_process_group()


def test_bench_real_form_runs_at_world_one():
    """bench.py's real multi-GPU form (the line a torchrun launch prints),
    forced at one rank with --dist: the step after the backward and the
    ready-driven schedule behind the proxy backward both run and report."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--dist", "--steps", "3",
                        "--warmup", "3", "--overlap-iters", "3"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 1 and d["config"]["parallelism"].startswith("dp1")
    assert d["value"] > 0 and d["gpu_launches"] == 3 * d["config"]["num_buckets"]
    o = d["overlap_ready_driven"]
    assert o["buckets"] == d["config"]["num_buckets"]
    assert o["t_bwd_ms"] > 0 and o["t_step_ready_driven_ms"] > 0
    assert o["t_step_after_backward_ms"] > o["t_bwd_ms"]
