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


def small_tensors():
    sys.path.insert(0, ROOT)
    from gradient_reduce_optimizer_gb300 import workloads as wl
    return wl.bert_large_tensors(layers=2, hidden=64, ffn=256, vocab=101, positions=16)


def inputs(R):
    sys.path.insert(0, ROOT)
    import oracle
    numel = [x[1] for x in small_tensors()]
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


def oracle_update(slices, master, m, v, out, length, R, *, stream=None, **hp):
    """The shard's arithmetic on the host: the oracle in place of the GPU
    kernel (master/m/v are updated through their numpy views)."""
    import oracle
    import torch
    got = [s_.numpy().view(np.uint16).copy() for s_ in slices]
    res = oracle.fused_dp_step(got, master.numpy(), m.numpy(), v.numpy(), **hp)[0]
    out.copy_(torch.from_numpy(res.view(np.int16)))


def packed_state(shards, state_off, elems, rank, master, m, v):
    import torch
    st = [torch.empty(elems[rank], dtype=torch.float32) for _ in range(3)]
    for b, row in enumerate(shards):
        lo, hi = row[rank]
        o = state_off[b][rank]
        for dst, src in zip(st, (master, m, v)):
            dst[o:o + hi - lo] = torch.from_numpy(src[lo:hi])
    return st


def _rank_class(rank, world, port, q):
    """The package's ShardedStep itself, both schedules, over gloo."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from gradient_reduce_optimizer_gb300 import dist as gdist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    numel, buckets, n, grads, master, m, v = inputs(world)
    layer_of = [x[2] for x in small_tensors()]
    step = gdist.ShardedStep(numel, 4096, rank=rank, world=world, layer_of=layer_of,
                             update=oracle_update, dtype=torch.int16)
    assert step.buckets == buckets
    _, _, elems = capi_shard_plan(step)
    out = {}
    for mode in ("after the backward", "ready-driven"):
        st = packed_state(step.shards, step.state_offsets, elems, rank, master, m, v)
        params = torch.full((n,), -1, dtype=torch.int16)
        g = torch.from_numpy(grads[rank].view(np.int16).copy())
        if mode == "after the backward":
            step.step(g, *st, params, **HP)
        else:
            step.begin(g, *st, params, **HP)
            for layer in range(max(layer_of), -1, -1):
                step.layer_ready(layer)
            step.end()
        out[mode] = (params.numpy().view(np.uint16).copy(), [a.numpy().copy() for a in st])
    q.put((rank, out, step.shards, step.state_offsets))
    dist.destroy_process_group()


def capi_shard_plan(step):
    from gradient_reduce_optimizer_gb300 import capi
    return capi.cc_shard_plan(step.buckets, step.world)


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_step_class_both_schedules(world):
    """ShardedStep.step() and the ready-driven begin()/layer_ready()/end()
    over gloo: every rank's parameters and state shards equal the emulated
    step bit for bit, in either schedule."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_class, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {r: rest for r, *rest in (q.get(timeout=300) for _ in range(world))}
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    import oracle
    numel, buckets, n, grads, master, m, v = inputs(world)
    ref_out = oracle.fused_dp_step(grads, master, m, v, **HP)[0]
    for rank in range(world):
        out, shards, state_off = results[rank]
        for mode, (params, st) in out.items():
            np.testing.assert_array_equal(params, ref_out, err_msg=mode)
            for b, row in enumerate(shards):
                lo, hi = row[rank]
                o = state_off[b][rank]
                for got, want in zip(st, (master, m, v)):
                    np.testing.assert_array_equal(got[o:o + hi - lo], want[lo:hi],
                                                  err_msg=mode)


def test_ready_driven_schedule_issues_each_bucket_once_its_layer_is_done():
    """One rank, no process group (world 1 has nothing to exchange): after
    layer l is reported, exactly the buckets whose every tensor is at layer
    l or above have gone out, in plan order; the result is the oracle's
    step; calls out of order are refused."""
    import torch
    import oracle
    from gradient_reduce_optimizer_gb300 import capi
    from gradient_reduce_optimizer_gb300 import dist as gdist
    numel, buckets, n, grads, master, m, v = inputs(1)
    layer_of = [x[2] for x in small_tensors()]
    step = gdist.ShardedStep(numel, 4096, rank=0, world=1, layer_of=layer_of,
                             update=oracle_update, dtype=torch.int16)
    offsets = step.offsets
    # the bucket of each tensor, and from it the buckets complete after each layer
    complete_after = {}
    for layer in range(max(layer_of), -1, -1):
        done = {t for t in range(len(numel)) if layer_of[t] >= layer}
        count = 0
        for b, (lo, hi) in enumerate(buckets):
            members = [t for t, off in enumerate(offsets) if lo <= off < hi]
            if all(t in done for t in members):
                count = b + 1
            else:
                break
        complete_after[layer] = count
    assert complete_after[0] == len(buckets)
    assert 0 < complete_after[max(layer_of)] < len(buckets)   # some go out before the end
    st = [torch.from_numpy(a.copy()) for a in (master, m, v)]
    params = torch.full((n,), -1, dtype=torch.int16)
    g = torch.from_numpy(grads[0].view(np.int16).copy())
    with pytest.raises(RuntimeError):
        step.layer_ready(0)                      # no step open
    step.begin(g, *st, params, **HP)
    with pytest.raises(RuntimeError):
        step.begin(g, *st, params, **HP)         # already open
    with pytest.raises(RuntimeError):
        step.step(g, *st, params, **HP)          # the other schedule while one is open
    issued = 0
    for layer in range(max(layer_of), -1, -1):
        issued += step.layer_ready(layer)
        assert issued == complete_after[layer], layer
        if layer == 1:
            with pytest.raises(RuntimeError):
                step.end()                       # layer 0's buckets are still out
    assert step.layer_ready(0) == 0              # nothing twice
    step.end()
    ref = oracle.fused_dp_step(grads, master.copy(), m.copy(), v.copy(), **HP)[0]
    np.testing.assert_array_equal(params.numpy().view(np.uint16), ref)
    with pytest.raises(ValueError):
        gdist.ShardedStep(numel, 4096, rank=0, world=1, update=oracle_update,
                          dtype=torch.int16).begin(g, *st, params, **HP)
