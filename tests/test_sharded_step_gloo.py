"""The sharded form of the step across real ranks, on the CPU over gloo.

CoCoNet's data-parallel schedule ("LIT-735", Key takeaways) reduce-scatters
the gradient, runs the optimizer on each rank's shard and all-gathers the
parameters.  Here two ranks each hold one gradient replica; for every
planned bucket rank k gathers all replicas' values of its 1/R shard (so the
sum keeps the fixed replica order), applies the oracle's AdamW to that
shard of master/m/v, and the bf16 parameter shards are all-gathered.  The
result must equal the single-process emulated step bit for bit: the
decomposition changes where work runs, not the values.  (This run has one
GPU, so the multi-GPU form is exercised on the host; the shard rule is the
one bench.py uses for one rank's share.)
"""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=7,
          grad_scale=1.0)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def inputs(R):
    sys.path.insert(0, ROOT)
    import oracle
    from gradient_reduce_optimizer_gb300 import workloads as wl
    t = wl.bert_large_tensors(layers=2, hidden=64, ffn=256, vocab=101, positions=16)
    numel = [x[1] for x in t]
    offsets, buckets, n = oracle.plan_buckets(numel, 4096)
    rng = np.random.default_rng(5)
    grads = [oracle.bf16_round((rng.standard_normal(n) * 1e-3).astype(np.float32))
             for _ in range(R)]
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = ((rng.standard_normal(n) * 1e-3) ** 2).astype(np.float32)
    return buckets, n, grads, master, m, v


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    buckets, n, grads, master, m, v = inputs(world)
    mine = torch.from_numpy(oracle.bf16_widen(grads[rank]))   # this rank's replica only
    params = np.empty(n, dtype=np.uint16)
    for b, e in buckets:
        shards = [bench.shard_range(b, e, world, k) for k in range(world)]
        # every rank's gradient values of every shard (fp32, exact widening)
        seen = [torch.empty(e - b) for _ in range(world)]
        dist.all_gather(seen, mine[b:e].contiguous())
        lo, hi = shards[rank]
        g_shard = [oracle.bf16_round(x[lo - b:hi - b].numpy()) for x in seen]
        st = [a[lo:hi].copy() for a in (master, m, v)]
        out = oracle.fused_dp_step(g_shard, *st, **HP)[0]
        for a, new in zip((master, m, v), st):
            a[lo:hi] = new
        got = [torch.empty(hi2 - lo2, dtype=torch.int32) for lo2, hi2 in shards]
        dist.all_gather(got, torch.from_numpy(out.astype(np.int32)))
        for (lo2, hi2), g in zip(shards, got):
            params[lo2:hi2] = g.numpy().astype(np.uint16)
    lo_all = [bench.shard_range(b, e, world, rank) for b, e in buckets]
    q.put((rank, params, [(lo, hi, master[lo:hi].copy(), m[lo:hi].copy(),
                           v[lo:hi].copy()) for lo, hi in lo_all]))
    dist.destroy_process_group()


def test_sharded_step_equals_emulated_step():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict((r, (p_, s)) for r, p_, s in (q.get(timeout=300) for _ in range(world)))
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    sys.path.insert(0, ROOT)
    import oracle
    buckets, n, grads, master, m, v = inputs(world)
    ref_out = oracle.fused_dp_step(grads, master, m, v, **HP)[0]
    for rank in range(world):
        params, shards = results[rank]
        np.testing.assert_array_equal(params, ref_out)          # every rank, all params
        for lo, hi, ms, mm, vv in shards:                       # its shard of the state
            np.testing.assert_array_equal(ms, master[lo:hi])
            np.testing.assert_array_equal(mm, m[lo:hi])
            np.testing.assert_array_equal(vv, v[lo:hi])
