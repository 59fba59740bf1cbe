"""The real multi-GPU form of the fused step: per bucket, a ReduceScatter of
the bf16 gradients, the AdamW step on each rank's shard, and an AllGather of
the bf16 parameters ("LIT-735: Breaking the Computation and Communication
Abstraction Barrier in Distributed Machine Learning Workloads" (CoCoNet),
Key takeaways: the fused ReduceScatter-optimizer-AllGather, with the
optimizer state sharded; "Communication Optimization › Communication
Overlap": one collective per DDP bucket, in reverse layer order).

One process per GPU; rank p holds replica p's gradient and parameter slabs
(the same layout as the single-GPU emulation: cc_plan_buckets' slab in
reverse layer order) and the optimizer state of its shards only.  The
library decides who owns what (cc_shard_plan) and does every step of the
arithmetic (cc_fused_dp_rank_step); torch.distributed moves the bytes:

  ReduceScatter  rank p sends its gradient of shard q to rank q and receives
                 every other rank's gradient of shard p into a staging
                 buffer in local memory.  The exchange moves bf16 values
                 unchanged (point-to-point sends, not a reducing collective,
                 whose sum would be in bf16 and in the library's own order):
                 the sum is the kernel's, in fp32 and in rank order.
  update         cc_fused_dp_rank_step reads the R slices of the shard,
                 takes the AdamW step on the rank's state and writes the
                 shard's bf16 parameters into the rank's own slab.
  AllGather      rank p sends its shard's parameters to every rank and
                 receives every other shard into its slab.

Kernels only ever read local memory.  The exchanges are queued on the
communication backend's own stream: bucket b+1's ReduceScatter is issued
before bucket b's update, so it runs while the update computes.

Two schedules.  step() runs every bucket once the whole backward is done.
begin() / layer_ready() / end() is DDP's ready-driven schedule ("Communication
Optimization > Communication Overlap": a bucket's collective starts as soon as
the backward has produced its last gradient, the last layer's bucket first):
the caller reports each finished layer, from the last down, and every bucket
that is then complete goes out at once -- its exchange, update and AllGather
on a side stream ordered after the caller's gradients -- while the backward
computes the layers below.  Both give the same values.

The exchange helpers take plain tensors and a process group, so the same
code runs over NCCL on GPUs and over gloo on host tensors.
"""
from __future__ import annotations

import contextlib
from typing import Callable, List, Optional, Sequence, Tuple

from . import capi

Range = Tuple[int, int]


def staging_stride(length: int) -> int:
    """Elements between staging slices: the shard length rounded up to 8, so
    that every slice starts 16-byte aligned."""
    return (length + 7) // 8 * 8


def reduce_scatter_ops(grads, staging, shards: Sequence[Range], rank: int, world: int,
                       group=None):
    """The ReduceScatter exchange of one bucket: point-to-point operations
    and the R gradient slices of this rank's shard in rank order (this
    rank's own slice is a view of its gradient slab; the others are staging
    slices that the receives fill).  Empty shards are neither sent nor
    received (every rank knows the plan)."""
    import torch.distributed as dist

    lo, hi = shards[rank]
    length = hi - lo
    stride = staging_stride(length)
    slices, ops = [], []
    for q in range(world):
        if q == rank:
            slices.append(grads[lo:hi])
        else:
            slices.append(staging[q * stride:q * stride + length])
    for q in range(world):
        if q == rank:
            continue
        qlo, qhi = shards[q]
        if qhi > qlo:
            ops.append(dist.P2POp(dist.isend, grads[qlo:qhi], q, group))
        if length > 0:
            ops.append(dist.P2POp(dist.irecv, slices[q], q, group))
    return slices, ops


def all_gather_ops(params, shards: Sequence[Range], rank: int, world: int, group=None):
    """The AllGather exchange of one bucket: this rank's shard of the
    parameters to every rank, every other shard into this rank's slab."""
    import torch.distributed as dist

    lo, hi = shards[rank]
    ops = []
    for q in range(world):
        if q == rank:
            continue
        if hi > lo:
            ops.append(dist.P2POp(dist.isend, params[lo:hi], q, group))
        qlo, qhi = shards[q]
        if qhi > qlo:
            ops.append(dist.P2POp(dist.irecv, params[qlo:qhi], q, group))
    return ops


def start(ops) -> list:
    import torch.distributed as dist
    return dist.batch_isend_irecv(ops) if ops else []


def finish(works) -> None:
    for w in works:
        w.wait()


def library_update(slices, master, m, v, out, length: int, R: int, *, stream=None, **hp):
    """One rank's update of one bucket shard: the library's rank step."""
    capi.cc_fused_dp_rank_step(slices, master, m, v, out, length, R, stream=stream, **hp)


class ShardedStep:
    """The sharded fused step of one rank over a planned slab.

    numel: tensor sizes in forward (layer) order; bucket_bytes: the DDP
    bucket cap; layer_of: each tensor's layer, for the ready-driven
    schedule.  The rank's gradient and parameter slabs are bf16 tensors of
    n_slab elements laid out by cc_plan_buckets; its master/m/v are fp32
    tensors of state_elems elements, its shards of every bucket in launch
    order (state_offsets gives each one's place).  update: the arithmetic of
    one shard (library_update, the GPU kernel; host tests pass their own).
    dtype: of the gradient slab and the staging buffers.
    """

    def __init__(self, numel: Sequence[int], bucket_bytes: int, rank: int, world: int,
                 group=None, device=None, layer_of: Optional[Sequence[int]] = None,
                 update: Callable = library_update, dtype=None):
        import torch

        self.rank, self.world, self.group = rank, world, group
        self.update = update
        self.offsets, self.buckets, self.n_slab = capi.cc_plan_buckets(list(numel),
                                                                       bucket_bytes)
        self.shards, self.state_offsets, elems = capi.cc_shard_plan(self.buckets, world)
        self.state_elems = elems[rank]
        # the layer after whose backward each bucket is complete (non-increasing)
        self.ready = (capi.cc_bucket_ready_layers(list(numel), list(layer_of), self.offsets,
                                                  self.buckets)
                      if layer_of is not None else None)
        longest = max((hi - lo for b in self.shards for lo, hi in [b[rank]]), default=0)
        # two staging buffers: bucket b+1's slices arrive while b computes
        self.staging = [torch.empty(world * staging_stride(longest),
                                    dtype=dtype or torch.bfloat16, device=device)
                        for _ in range(2)]
        self._run = None
        self._side_streams = {}

    def shard_state_ranges(self) -> List[Tuple[Range, Range]]:
        """(slab range, state range) of each of this rank's shards."""
        out = []
        for b, shards in enumerate(self.shards):
            lo, hi = shards[self.rank]
            o = self.state_offsets[b][self.rank]
            out.append(((lo, hi), (o, o + hi - lo)))
        return out

    def step(self, grads, master, m, v, params, *, lr: float, beta1: float, beta2: float,
             eps: float, weight_decay: float, step: int, grad_scale: float,
             stream=None) -> None:
        """One optimizer step: every bucket's ReduceScatter, update and
        AllGather.  Returns once everything is queued; the parameters are
        complete when the stream (and the backend's) reach this point."""
        if self._run is not None:
            raise RuntimeError("step() while a ready-driven step is open: end() it first")
        hp = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay,
                  step=step, grad_scale=grad_scale)
        B = len(self.buckets)
        if B == 0:
            return
        rs = [None] * B
        rs[0] = reduce_scatter_ops(grads, self.staging[0], self.shards[0], self.rank,
                                   self.world, self.group)
        pending = start(rs[0][1])
        gathers = []
        for b in range(B):
            slices, _ = rs[b]
            finish(pending)                      # slices of bucket b are in place
            if b + 1 < B:                        # next bucket's exchange runs meanwhile
                rs[b + 1] = reduce_scatter_ops(grads, self.staging[(b + 1) % 2],
                                               self.shards[b + 1], self.rank, self.world,
                                               self.group)
                pending = start(rs[b + 1][1])
            self._update(b, slices, master, m, v, params, stream, hp)
            gathers += start(all_gather_ops(params, self.shards[b], self.rank, self.world,
                                            self.group))
            rs[b] = None
        finish(gathers)

    def _update(self, b, slices, master, m, v, params, stream, hp) -> None:
        lo, hi = self.shards[b][self.rank]
        if hi == lo:
            return
        o = self.state_offsets[b][self.rank]
        self.update(slices, master[o:o + hi - lo], m[o:o + hi - lo], v[o:o + hi - lo],
                    params[lo:hi], hi - lo, self.world, stream=stream, **hp)

    # ---- the ready-driven schedule -------------------------------------

    def begin(self, grads, master, m, v, params, *, lr: float, beta1: float, beta2: float,
              eps: float, weight_decay: float, step: int, grad_scale: float,
              stream=None, side_stream=None) -> None:
        """Start a step whose buckets go out as the backward produces them.
        stream: the caller's (the backward's) stream, default the current
        one; side_stream: where the buckets' exchanges and updates are
        ordered (CUDA tensors only; default one stream of this object's,
        made on first use)."""
        import torch

        if self.ready is None:
            raise ValueError("the ready-driven schedule needs layer_of")
        if self._run is not None:
            raise RuntimeError("begin() while a step is open: end() it first")
        cuda = grads.is_cuda
        if cuda:
            stream = stream or torch.cuda.current_stream(grads.device)
            if side_stream is None:
                # one side stream per device, made once and reused by every step
                own = self._side_streams.get(grads.device)
                if own is None:
                    own = self._side_streams[grads.device] = torch.cuda.Stream(
                        device=grads.device)
                side_stream = own
        self._run = dict(grads=grads, state=(master, m, v), params=params, next=0,
                         gathers=[], stream=stream, side=side_stream, cuda=cuda,
                         hp=dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps,
                                 weight_decay=weight_decay, step=step,
                                 grad_scale=grad_scale))

    def _side(self):
        import torch
        run = self._run
        return torch.cuda.stream(run["side"]) if run["cuda"] else contextlib.nullcontext()

    def layer_ready(self, layer: int) -> int:
        """The backward has written every gradient of `layer` (and, since it
        runs from the last layer down, of every later one) on the caller's
        stream.  Each bucket that is now complete goes out, in plan order:
        its ReduceScatter, update and AllGather, ordered after those
        gradients.  Returns how many buckets went out."""
        import torch

        run = self._run
        if run is None:
            raise RuntimeError("layer_ready() outside begin() / end()")
        B = len(self.buckets)
        if run["next"] >= B or self.ready[run["next"]] < layer:
            return 0
        if run["cuda"]:
            done = torch.cuda.Event()
            done.record(run["stream"])
            run["side"].wait_event(done)
        count = 0
        with self._side():
            while run["next"] < B and self.ready[run["next"]] >= layer:
                b = run["next"]
                slices, ops = reduce_scatter_ops(run["grads"], self.staging[b % 2],
                                                 self.shards[b], self.rank, self.world,
                                                 self.group)
                finish(start(ops))               # the slices of bucket b are in place
                self._update(b, slices, *run["state"], run["params"], run["side"], run["hp"])
                run["gathers"] += start(all_gather_ops(run["params"], self.shards[b],
                                                       self.rank, self.world, self.group))
                run["next"] += 1
                count += 1
        return count

    def end(self) -> None:
        """Close the step: every bucket must have gone out (layer_ready(0)
        was called); if not, this raises and the step stays open, to be
        closed once the remaining layers are reported.  The caller's stream
        waits for the last AllGather, so the parameters are complete when it
        reaches this point."""
        run = self._run
        if run is None:
            raise RuntimeError("end() without begin()")
        left = len(self.buckets) - run["next"]
        if left:
            raise RuntimeError(f"{left} bucket(s) never became ready: report every layer "
                               "down to layer 0 before end()")
        with self._side():
            finish(run["gathers"])
        if run["cuda"]:
            run["stream"].wait_stream(run["side"])
        self._run = None
