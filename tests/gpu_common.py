"""Helpers shared by the GPU parity tests: device slabs, host copies, and
NaN-aware bit comparisons.  The oracle is always fed the exact bytes the
CUDA path read."""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
from gradient_reduce_optimizer_gb300 import capi
from gradient_reduce_optimizer_gb300 import workloads as wl

DEV = "cuda"


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


def same_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Elementwise: identical bits, or both NaN (NaN payloads may differ)."""
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))


def same_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = np.asarray(a, np.uint16)
    b = np.asarray(b, np.uint16)
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return (a == b) | (nan_a & nan_b)


def assert_bits(name: str, got, want, kind: str) -> None:
    ok = same_f32(got, want) if kind == "f32" else same_bf16(got, want)
    if not ok.all():
        bad = np.flatnonzero(~ok)
        i = bad[0]
        raise AssertionError(f"{name}: {bad.size} of {ok.size} elements differ; "
                             f"first at {i}: got {got[i]!r} want {want[i]!r}")


@dataclass
class Slabs:
    grads: List[torch.Tensor]
    master: torch.Tensor
    m: torch.Tensor
    v: torch.Tensor
    outs: List[torch.Tensor]
    acc: Optional[List[torch.Tensor]] = None

    @property
    def R(self) -> int:
        return len(self.grads)

    @property
    def n(self) -> int:
        return self.master.numel()


def new_slabs(grads, master, m, v, with_acc=False) -> Slabs:
    R, n = len(grads), master.numel()
    outs = [torch.full((n,), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            for _ in range(R)]
    acc = ([torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(R)]
           if with_acc else None)
    return Slabs(grads, master, m, v, outs, acc)


def host_copy(s: Slabs, idx: Optional[torch.Tensor] = None):
    """(grads u16 list, master, m, v, acc list or None) on the host, for all
    elements or the sampled indices."""
    pick = (lambda t: t) if idx is None else (lambda t: t[idx])
    grads = [u16(pick(g)) for g in s.grads]
    st = [f32(pick(x)).copy() for x in (s.master, s.m, s.v)]
    acc = [f32(pick(a)).copy() for a in s.acc] if s.acc is not None else None
    return grads, st, acc


HP_KEYS = ("lr", "beta1", "beta2", "eps", "weight_decay", "step", "grad_scale")


def hp_of(w: wl.Workload) -> dict:
    return {k: getattr(w, k) for k in HP_KEYS}


def gpu_step(s: Slabs, hp: dict, bucket_bytes: int = 0, accum_k: int = 1,
             use_acc: bool = False) -> None:
    if use_acc:
        capi.cc_fused_dp_step_accum(s.grads, s.acc, s.master, s.m, s.v, s.outs,
                                    s.n, s.R, bucket_bytes, accum_k=accum_k, **hp)
    else:
        capi.cc_fused_dp_step(s.grads, s.master, s.m, s.v, s.outs, s.n, s.R,
                              bucket_bytes, **hp)


def oracle_step(grads, state, hp: dict, acc=None):
    master, m, v = state
    outs = oracle.fused_dp_step(grads, master, m, v, acc=acc, **hp)
    return outs


def compare_all(s: Slabs, state_ref, outs_ref, idx=None, label="") -> None:
    pick = (lambda t: t) if idx is None else (lambda t: t[idx])
    for name, t, ref in zip(("master", "m", "v"), (s.master, s.m, s.v), state_ref):
        assert_bits(f"{label}{name}", f32(pick(t)), ref, "f32")
    for r, (t, ref) in enumerate(zip(s.outs, outs_ref)):
        assert_bits(f"{label}params_out[{r}]", u16(pick(t)), ref, "bf16")


def random_inputs(R: int, n: int, seed: int, sigma: float = 1e-3,
                  step: int = 1, premultiply: float = 1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    grads = [(torch.randn(n, generator=g, device=DEV) * sigma * premultiply)
             .to(torch.bfloat16) for _ in range(R)]
    master = torch.randn(n, generator=g, device=DEV) * 0.02
    if step == 1:
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
    else:
        m = torch.randn(n, generator=g, device=DEV) * 0.1 * sigma
        v = (torch.randn(n, generator=g, device=DEV) * sigma) ** 2
    return grads, master, m, v


def workload_grads(w: wl.Workload, offsets, n_slab: int, micro: int = 0):
    """R bf16 gradient slabs of a planned workload: scaled per layer,
    pre-multiplied by the loss scale, zero on padding."""
    numel, layer_of = w.numel(), w.layer_of()
    lay = wl.element_layer_map(numel, layer_of, offsets, n_slab, device=DEV)
    mask = lay >= 0
    scale = None
    if w.layer_scale is not None:
        per_layer = wl.layer_scales(max(layer_of) + 1, *w.layer_scale, device=DEV)
        scale = per_layer[lay.clamp(min=0).long()]
    del lay
    return wl.make_grads(w.R, n_slab, w.grad_sigma, micro=micro, device=DEV,
                         elem_scale=scale, mask=mask, premultiply=w.grad_scale)


def planned_workload_slabs(w: wl.Workload, micro: int = 0, with_acc=False):
    """Device slabs for a workload laid out by the oracle's planner (reverse
    layer order, 8-element padding)."""
    offsets, _, n_slab = oracle.plan_buckets(w.numel(), w.bucket_bytes)
    grads = workload_grads(w, offsets, n_slab, micro)
    master, m, v = wl.make_state(n_slab, w.step, w.grad_sigma,
                                 master_sigma=w.master_sigma, device=DEV)
    return new_slabs(grads, master, m, v, with_acc=with_acc), offsets, n_slab
