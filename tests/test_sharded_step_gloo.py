"""The real multi-GPU form of the step -- per bucket a ReduceScatter, AdamW
on each rank's shard, an AllGather -- across real ranks on the CPU over
gloo ("LIT-735" (CoCoNet), Key takeaways: the fused ReduceScatter-
optimizer-AllGather with sharded optimizer state).

Each rank holds one gradient replica.  The library plans who owns what
(cc_shard_plan, host code, no GPU needed) and the package's exchange code
(gradient_reduce_optimizer_gb300.dist: the point-to-point ReduceScatter into
a staging buffer and the AllGather into the parameter slab) moves the bf16
bytes, exactly as on GPUs over NCCL.  Only the per-shard arithmetic, which
on a GPU is the library's kernel, is the oracle here.  Every rank's
parameters and each rank's shard of master/m/v must equal the single-process
emulated step bit for bit: the decomposition changes where work runs, not
the values.  World sizes 2 and 3 (uneven shards, empty shards)."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

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
    return numel, buckets, n, grads, master, m, v


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    from gradient_reduce_optimizer_gb300 import capi
    from gradient_reduce_optimizer_gb300 import dist as gdist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    numel, buckets, n, grads, master, m, v = inputs(world)
    # the library's plan of the slab and of the shards
    _, lib_buckets, n_lib = capi.cc_plan_buckets(numel, 4096)
    assert lib_buckets == buckets and n_lib == n
    shards, state_off, elems = capi.cc_shard_plan(buckets, world)
    # this rank's replica and its state shards, packed in launch order
    g = torch.from_numpy(grads[rank].view(np.int16).copy())        # bf16 bits
    params = torch.full((n,), -1, dtype=torch.int16)
    st = [np.empty(elems[rank], dtype=np.float32) for _ in range(3)]
    for b, row in enumerate(shards):
        lo, hi = row[rank]
        o = state_off[b][rank]
        for dst, src in zip(st, (master, m, v)):
            dst[o:o + hi - lo] = src[lo:hi]
    longest = max(r[rank][1] - r[rank][0] for r in shards)
    staging = torch.empty(world * gdist.staging_stride(longest), dtype=torch.int16)
    for b, row in enumerate(shards):
        slices, ops = gdist.reduce_scatter_ops(g, staging, row, rank, world)
        gdist.finish(gdist.start(ops))
        lo, hi = row[rank]
        o = state_off[b][rank]
        shard_state = [a[o:o + hi - lo] for a in st]
        if hi > lo:
            got = [s_.numpy().view(np.uint16).copy() for s_ in slices]
            out = oracle.fused_dp_step(got, *shard_state, **HP)[0]
            params[lo:hi] = torch.from_numpy(out.view(np.int16))
        gdist.finish(gdist.start(gdist.all_gather_ops(params, row, rank, world)))
    q.put((rank, params.numpy().view(np.uint16).copy(), st, shards, state_off))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_step_equals_emulated_step(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {r: rest for r, *rest in (q.get(timeout=300) for _ in range(world))}
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    sys.path.insert(0, ROOT)
    import oracle
    numel, buckets, n, grads, master, m, v = inputs(world)
    ref_out = oracle.fused_dp_step(grads, master, m, v, **HP)[0]
    for rank in range(world):
        params, st, shards, state_off = results[rank]
        np.testing.assert_array_equal(params, ref_out)           # every rank, all params
        for b, row in enumerate(shards):                         # its shards of the state
            lo, hi = row[rank]
            o = state_off[b][rank]
            for got, want in zip(st, (master, m, v)):
                np.testing.assert_array_equal(got[o:o + hi - lo], want[lo:hi])
