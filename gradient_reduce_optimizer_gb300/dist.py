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

The exchange helpers take plain tensors and a process group, so the same
code runs over NCCL on GPUs and over gloo on host tensors.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

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


class ShardedStep:
    """The sharded fused step of one rank over a planned slab.

    numel: tensor sizes in forward (layer) order; bucket_bytes: the DDP
    bucket cap.  The rank's gradient and parameter slabs are bf16 tensors of
    n_slab elements laid out by cc_plan_buckets; its master/m/v are fp32
    tensors of state_elems elements, its shards of every bucket in launch
    order (state_offsets gives each one's place).
    """

    def __init__(self, numel: Sequence[int], bucket_bytes: int, rank: int, world: int,
                 group=None, device=None):
        import torch

        self.rank, self.world, self.group = rank, world, group
        self.offsets, self.buckets, self.n_slab = capi.cc_plan_buckets(list(numel),
                                                                       bucket_bytes)
        self.shards, self.state_offsets, elems = capi.cc_shard_plan(self.buckets, world)
        self.state_elems = elems[rank]
        longest = max((hi - lo for b in self.shards for lo, hi in [b[rank]]), default=0)
        # two staging buffers: bucket b+1's slices arrive while b computes
        self.staging = [torch.empty(world * staging_stride(longest), dtype=torch.bfloat16,
                                    device=device) for _ in range(2)]

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
            lo, hi = self.shards[b][self.rank]
            o = self.state_offsets[b][self.rank]
            capi.cc_fused_dp_rank_step(slices, master[o:o + hi - lo], m[o:o + hi - lo],
                                       v[o:o + hi - lo], params[lo:hi], hi - lo, self.world,
                                       stream=stream, **hp)
            gathers += start(all_gather_ops(params, self.shards[b], self.rank, self.world,
                                            self.group))
            rs[b] = None
        finish(gathers)
