"""The oracle: plain, slow, obviously correct CPU versions of the fused
data-parallel step.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``gradient_reduce_optimizer_gb300``) never imports it, and this package
never imports the product.

Contents
--------
* ``fused_dp_step`` / ``accumulate_local`` / ``bf16_round`` / ``bf16_widen``:
  thin ctypes wrappers over ``cc_oracle.c`` (single-threaded C, binary32,
  no FMA contraction).  See that file's header for the arithmetic and the
  passages it follows.
* ``plan_buckets`` / ``bucket_ready_layers``: the bucket planner and the
  readiness rule in plain Python loops.
* ``shard_plan``: the shards of every bucket in the sharded (multi-GPU)
  form.

Sources: "Communication Optimization › Communication Overlap"
(mbrenndoerfer.com), the paragraphs on reverse-order readiness, on DDP
bucketing (fixed-size buckets, default 25 MB, each launched once all its
gradients are ready) and on bucket ordering (the last layer's bucket goes
first); "Overlapping Communication and Computation" (praveentn.live), the
paragraph on bucket size (a very large single tensor is not split and can
defeat the pipelining).

Every function here is pinned by ``tests/test_oracle_pins.py`` and
``tests/test_planner.py`` against closed forms, torch's CPU AdamW, exact
integer arithmetic, hand-counted plans and brute force.  No function is
parity unpinned.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from . import build as _build

__all__ = [
    "bf16_round",
    "bf16_widen",
    "fused_dp_step",
    "accumulate_local",
    "plan_buckets",
    "bucket_ready_layers",
    "shard_plan",
    "tp_allreduce",
    "MAX_R",
]

MAX_R = 16
_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(_build.build())
        vp, sz, f, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float, ctypes.c_int
        lib.oracle_bf16_round_array.argtypes = [vp, vp, sz]
        lib.oracle_bf16_round_array.restype = None
        lib.oracle_bf16_widen_array.argtypes = [vp, vp, sz]
        lib.oracle_bf16_widen_array.restype = None
        lib.oracle_accumulate_local.argtypes = [vp, vp, sz, i, i]
        lib.oracle_accumulate_local.restype = i
        lib.oracle_fused_dp_step.argtypes = [
            vp, vp, vp, vp, vp, vp, sz, i, f, f, f, f, f, i, f]
        lib.oracle_fused_dp_step.restype = i
        lib.oracle_tp_allreduce.argtypes = [vp, vp, sz, i]
        lib.oracle_tp_allreduce.restype = i
        _LIB = lib
    return _LIB


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _ptr_array(arrays: Sequence[np.ndarray]):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _check(a: np.ndarray, dtype, n: int, name: str) -> None:
    if a.dtype != dtype or a.ndim != 1 or a.size != n or not a.flags.c_contiguous:
        raise ValueError(f"{name}: want contiguous 1-D {np.dtype(dtype)}[{n}], "
                         f"got {a.dtype}{list(a.shape)}")


def bf16_round(x: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    _lib().oracle_bf16_round_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_widen(h: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> binary32 (exact)."""
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(h.size, dtype=np.float32)
    _lib().oracle_bf16_widen_array(_ptr(h), _ptr(out), h.size)
    return out


def accumulate_local(grads: Sequence[np.ndarray], acc: Sequence[np.ndarray],
                     first: bool) -> None:
    """One local micro-step: ``acc[r] (+)= float(grads[r])``, in place."""
    R = len(grads)
    if R != len(acc) or not 1 <= R <= MAX_R:
        raise ValueError("need 1..16 replicas and one accumulator each")
    n = grads[0].size
    for r in range(R):
        _check(grads[r], np.uint16, n, f"grads[{r}]")
        _check(acc[r], np.float32, n, f"acc[{r}]")
    rc = _lib().oracle_accumulate_local(_ptr_array(grads), _ptr_array(acc),
                                        n, R, int(bool(first)))
    if rc != 0:
        raise ValueError("oracle_accumulate_local rejected its arguments")


def fused_dp_step(grads: Sequence[np.ndarray], master: np.ndarray,
                  m: np.ndarray, v: np.ndarray, *, lr: float, beta1: float,
                  beta2: float, eps: float, weight_decay: float, step: int,
                  grad_scale: float,
                  acc: Optional[Sequence[np.ndarray]] = None) -> list:
    """Reduce R bf16 gradient replicas, take one AdamW step, redistribute.

    ``grads`` are R uint16 (bf16 bit) arrays; ``master``, ``m``, ``v`` are
    float32 and are updated in place.  Returns R uint16 arrays, the bf16
    parameters written to every replica.  ``acc`` (optional) are the R
    per-replica fp32 accumulators of the earlier micro-steps.
    """
    R = len(grads)
    if not 1 <= R <= MAX_R:
        raise ValueError("R must be in 1..16")
    n = master.size
    for r in range(R):
        _check(grads[r], np.uint16, n, f"grads[{r}]")
    for a, name in ((master, "master"), (m, "m"), (v, "v")):
        _check(a, np.float32, n, name)
    acc_arg = None
    if acc is not None:
        if len(acc) != R:
            raise ValueError("one accumulator per replica")
        for r in range(R):
            _check(acc[r], np.float32, n, f"acc[{r}]")
        acc_arg = _ptr_array(acc)
    outs = [np.empty(n, dtype=np.uint16) for _ in range(R)]
    rc = _lib().oracle_fused_dp_step(
        _ptr_array(grads), acc_arg, _ptr(master), _ptr(m), _ptr(v),
        _ptr_array(outs), n, R, lr, beta1, beta2, eps, weight_decay,
        int(step), grad_scale)
    if rc != 0:
        raise ValueError("oracle_fused_dp_step rejected its arguments")
    return outs


def tp_allreduce(partials: Sequence[np.ndarray]) -> list:
    """The tensor-parallel AllReduce of R fp32 partial products: their sum
    in rank order, rounded to bf16, one uint16 array per rank."""
    R = len(partials)
    if not 1 <= R <= MAX_R:
        raise ValueError("R must be in 1..16")
    n = partials[0].size
    for r in range(R):
        _check(partials[r], np.float32, n, f"partials[{r}]")
    outs = [np.empty(n, dtype=np.uint16) for _ in range(R)]
    if _lib().oracle_tp_allreduce(_ptr_array(partials), _ptr_array(outs), n, R) != 0:
        raise ValueError("oracle_tp_allreduce rejected its arguments")
    return outs


# --------------------------------------------------------------------------
# Bucket planner, in plain Python.
# --------------------------------------------------------------------------

PAD_ELEMS = 8      # 16 bytes of bf16: every tensor starts on a 16-byte line
GRAD_BYTES = 2     # bf16 gradient element


def plan_buckets(numel: Sequence[int], bucket_bytes: int):
    """Lay tensors out in reverse layer order and cut them into buckets.

    ``numel`` lists tensor sizes in forward (layer) order.  Backward produces
    gradients from the last layer to the first, so the slab holds the last
    tensor first.  Each tensor's span is padded up to a multiple of 8
    elements.  Tensors join the open bucket in that order; once the open
    bucket holds at least ``bucket_bytes`` bytes of bf16 gradient (padded
    spans) it is closed.  A tensor is never split, so one tensor may exceed
    the cap on its own.  ``bucket_bytes == 0`` means a single bucket.  A
    bucket with no elements is not emitted.

    Returns ``(offsets, buckets, n_padded)``: ``offsets[t]`` is tensor t's
    first slab element (t in forward order), ``buckets`` a list of
    ``(begin, end)`` element ranges in launch order.
    """
    T = len(numel)
    offsets = [0] * T
    buckets = []
    cursor = 0
    open_begin = 0
    open_bytes = 0
    for t in range(T - 1, -1, -1):
        if numel[t] < 0:
            raise ValueError("negative tensor size")
        offsets[t] = cursor
        span = (numel[t] + PAD_ELEMS - 1) // PAD_ELEMS * PAD_ELEMS
        cursor += span
        open_bytes += span * GRAD_BYTES
        if bucket_bytes > 0 and open_bytes >= bucket_bytes:
            if cursor > open_begin:
                buckets.append((open_begin, cursor))
            open_begin = cursor
            open_bytes = 0
    if cursor > open_begin:
        buckets.append((open_begin, cursor))
    return offsets, buckets, cursor


def shard_plan(buckets, world: int):
    """Who owns what in the sharded form of the step: every bucket is cut
    into ``world`` shards in rank order, rank q reducing, updating and
    gathering shard q ("LIT-735" (CoCoNet), Key takeaways: ReduceScatter,
    the optimizer on each rank's shard, AllGather; one collective per DDP
    bucket).  Cut in 8-element units (16 bytes of bf16): of a bucket's u
    whole units, rank q holds units floor(u q / W) .. floor(u (q + 1) / W)
    - 1 (an even split, sizes differing by at most one unit); the last rank
    also takes any ragged tail.  Rank q's optimizer state holds its shards
    of every bucket one after the other, in launch order.

    Returns ``(shards, state_offsets, state_elems)``: ``shards[b][q] =
    (begin, end)``, ``state_offsets[b][q]`` where that shard starts in rank
    q's state, ``state_elems[q]`` the length of rank q's state.
    """
    shards, offsets = [], []
    used = [0] * world
    for begin, end in buckets:
        units = (end - begin) // PAD_ELEMS
        row, offs = [], []
        for q in range(world):
            first_unit = (units * q) // world
            stop_unit = (units * (q + 1)) // world
            lo = begin + PAD_ELEMS * first_unit
            hi = begin + PAD_ELEMS * stop_unit
            if q == world - 1:
                hi = end                     # the ragged tail, if any
            row.append((lo, hi))
            offs.append(used[q])
            used[q] += hi - lo
        shards.append(row)
        offsets.append(offs)
    return shards, offsets, used


def bucket_ready_layers(numel: Sequence[int], layer_of: Sequence[int],
                        offsets: Sequence[int], buckets) -> list:
    """The backward layer after which each bucket's gradients are complete.

    Backward runs layers from the highest index down to 0, and a bucket can
    launch once every tensor in it has its gradient, i.e. after the lowest
    layer among its (non-empty) tensors has finished.  Returns one layer
    index per bucket.
    """
    ready = []
    for begin, end in buckets:
        lowest = None
        for t in range(len(numel)):
            if numel[t] > 0 and begin <= offsets[t] < end:
                if lowest is None or layer_of[t] < lowest:
                    lowest = layer_of[t]
        if lowest is None:
            raise ValueError("bucket with no tensor")
        ready.append(lowest)
    return ready
