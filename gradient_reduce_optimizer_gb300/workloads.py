"""Seeded synthetic inputs and parameter-shape lists.

This module holds no arithmetic of the method: it lists tensor shapes of the
model families the fused step is measured on, and draws seeded random
gradients and optimizer state.  The tests feed the same bytes to the CUDA
path and to the oracle; the benchmark uses them as its workload.

Shapes only (no weights, no data): BERT-large (24 layers, hidden 1024,
FFN 4096, vocabulary 30522, 336,226,108 parameters, 398 tensors) and a
24-layer slice of an 8.3B GPT-2 (hidden 3072, FFN 12288, 2,718,867,456
parameters, 288 tensors).  The data-parallel result being reproduced is
measured on BERT training with Adam ("LIT-735: Breaking the Computation and
Communication Abstraction Barrier in Distributed Machine Learning
Workloads", Key takeaways).

Seeds: gradient of replica r at micro-step j = 1000 + 100*j + r; master = 1;
per-layer gradient scales = 2; m = 3; v = 4.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

MiB = 1 << 20

SEED_GRAD = 1000
SEED_MASTER = 1
SEED_LAYER_SCALE = 2
SEED_M = 3
SEED_V = 4

# (name, numel, layer) in forward order.
Tensor = Tuple[str, int, int]


def bert_large_tensors(layers: int = 24, hidden: int = 1024, ffn: int = 4096,
                       vocab: int = 30522, positions: int = 512,
                       types: int = 2) -> List[Tensor]:
    """BERT-large parameter list in forward order.

    Embeddings belong to layer 0 and the heads to the last layer (their
    gradients are produced with that layer's in backward).  The MLM decoder
    weight is tied to the word embedding, so only its bias is listed.
    """
    h = hidden
    out: List[Tensor] = [
        ("emb.word", vocab * h, 0),
        ("emb.position", positions * h, 0),
        ("emb.token_type", types * h, 0),
        ("emb.ln.weight", h, 0),
        ("emb.ln.bias", h, 0),
    ]
    for l in range(layers):
        p = f"layer{l}."
        for proj in ("q", "k", "v", "attn_out"):
            out.append((p + proj + ".weight", h * h, l))
            out.append((p + proj + ".bias", h, l))
        out += [
            (p + "ln1.weight", h, l), (p + "ln1.bias", h, l),
            (p + "ffn_in.weight", h * ffn, l), (p + "ffn_in.bias", ffn, l),
            (p + "ffn_out.weight", ffn * h, l), (p + "ffn_out.bias", h, l),
            (p + "ln2.weight", h, l), (p + "ln2.bias", h, l),
        ]
    last = layers - 1
    out += [
        ("pooler.weight", h * h, last), ("pooler.bias", h, last),
        ("mlm.transform.weight", h * h, last), ("mlm.transform.bias", h, last),
        ("mlm.ln.weight", h, last), ("mlm.ln.bias", h, last),
        ("mlm.decoder.bias", vocab, last),
        ("nsp.weight", 2 * h, last), ("nsp.bias", 2, last),
    ]
    return out


def gpt2_slice_tensors(layers: int = 24, hidden: int = 3072,
                       ffn: int = 12288) -> List[Tensor]:
    """Transformer layers of GPT-2 8.3B (pre-LN), without embeddings."""
    h = hidden
    out: List[Tensor] = []
    for l in range(layers):
        p = f"layer{l}."
        out += [
            (p + "ln1.weight", h, l), (p + "ln1.bias", h, l),
            (p + "qkv.weight", h * 3 * h, l), (p + "qkv.bias", 3 * h, l),
            (p + "proj.weight", h * h, l), (p + "proj.bias", h, l),
            (p + "ln2.weight", h, l), (p + "ln2.bias", h, l),
            (p + "fc1.weight", h * ffn, l), (p + "fc1.bias", ffn, l),
            (p + "fc2.weight", ffn * h, l), (p + "fc2.bias", h, l),
        ]
    return out


@dataclass
class Workload:
    """One measured configuration of the fused step."""
    name: str
    R: int
    tensors: Optional[List[Tensor]]   # None: one flat tensor of n elements
    n: int                            # parameters (sum of numel)
    grad_sigma: float                 # std of the unscaled gradient
    layer_scale: Optional[Tuple[float, float]]  # U(lo, hi) per layer, or None
    grad_scale: float
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    step: int = 1
    bucket_bytes: int = 0
    accum_k: int = 1
    master_sigma: float = 0.02
    notes: str = field(default="")

    def numel(self) -> List[int]:
        return [t[1] for t in self.tensors] if self.tensors else [self.n]

    def layer_of(self) -> List[int]:
        return [t[2] for t in self.tensors] if self.tensors else [0]


def flat_1m_r2() -> Workload:
    """R=2, one flat tensor of 1,048,576 parameters, one bucket, step 1."""
    return Workload("flat-1M-R2", R=2, tensors=None, n=1 << 20,
                    grad_sigma=1e-3, layer_scale=None, grad_scale=1.0,
                    lr=1e-3, weight_decay=0.0, step=1, bucket_bytes=0)


def bert_large_r8(accum_k: int = 1, bucket_bytes: int = 25 * MiB) -> Workload:
    """R=8 on the BERT-large parameter list, 25 MiB buckets, step 10."""
    t = bert_large_tensors()
    return Workload("bert-large-R8", R=8, tensors=t, n=sum(x[1] for x in t),
                    grad_sigma=1e-3, layer_scale=(0.5, 2.0), grad_scale=1.0,
                    lr=1e-3, weight_decay=0.01, step=10,
                    bucket_bytes=bucket_bytes, accum_k=accum_k)


def gpt2_slice_r4() -> Workload:
    """R=4 on 24 GPT-2 8.3B layers, loss scale 65536, 25 MiB buckets."""
    t = gpt2_slice_tensors()
    return Workload("gpt2-8.3B-24L-R4", R=4, tensors=t,
                    n=sum(x[1] for x in t), grad_sigma=1e-4, layer_scale=None,
                    grad_scale=65536.0, lr=1.5e-4, weight_decay=0.01,
                    step=10, bucket_bytes=25 * MiB)


# ---------------------------------------------------------------------------
# Seeded generators
# ---------------------------------------------------------------------------

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(n: int, seed: int, device, chunk: int = 1 << 28) -> torch.Tensor:
    """n standard normals from one seeded stream, drawn in bounded chunks."""
    g = _gen(device, seed)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=g, device=device,
                               dtype=torch.float32)
    return out


def layer_scales(num_layers: int, lo: float, hi: float,
                 device="cpu") -> torch.Tensor:
    """One U(lo, hi) draw per layer, shared by every replica."""
    g = _gen(device, SEED_LAYER_SCALE)
    u = torch.rand(num_layers, generator=g, device=device, dtype=torch.float32)
    return lo + (hi - lo) * u


def element_layer_map(numel: Sequence[int], layer_of: Sequence[int],
                      offsets: Sequence[int], n_slab: int,
                      device="cpu") -> torch.Tensor:
    """Layer index of every slab element; -1 on padding.

    ``offsets`` is where each tensor starts in the slab (whichever layout the
    caller uses).
    """
    lay = torch.full((n_slab,), -1, dtype=torch.int32, device=device)
    for t, (k, l) in enumerate(zip(numel, layer_of)):
        o = offsets[t]
        lay[o:o + k] = l
    return lay


def make_grads(R: int, n_slab: int, sigma: float, *, micro: int = 0,
               device="cpu", elem_scale: Optional[torch.Tensor] = None,
               mask: Optional[torch.Tensor] = None,
               premultiply: float = 1.0) -> List[torch.Tensor]:
    """R bf16 gradient slabs: bf16(premultiply * sigma * N(0,1) * scale).

    ``elem_scale`` (per element, fp32) and ``mask`` (bool, False on padding)
    are optional.  Replica r of micro-step j uses seed 1000 + 100*j + r.
    """
    out = []
    for r in range(R):
        z = _randn(n_slab, SEED_GRAD + 100 * micro + r, device)
        z.mul_(sigma * premultiply)
        if elem_scale is not None:
            z.mul_(elem_scale)
        if mask is not None:
            z.masked_fill_(~mask, 0.0)
        out.append(z.to(torch.bfloat16))
        del z
    return out


def make_state(n_slab: int, step: int, grad_sigma: float, *,
               master_sigma: float = 0.02, device="cpu"):
    """fp32 master ~ N(0, master_sigma); m = v = 0 at step 1, otherwise
    m = 0.1*sigma*z1 and v = (sigma*z2)^2 (a plausible mid-training state)."""
    master = _randn(n_slab, SEED_MASTER, device).mul_(master_sigma)
    if step <= 1:
        m = torch.zeros(n_slab, dtype=torch.float32, device=device)
        v = torch.zeros(n_slab, dtype=torch.float32, device=device)
    else:
        m = _randn(n_slab, SEED_M, device).mul_(0.1 * grad_sigma)
        v = _randn(n_slab, SEED_V, device).mul_(grad_sigma).square_()
    return master, m, v


def integer_grads(R: int, n: int, lo: int = -8, hi: int = 8, *, micro: int = 0,
                  device="cpu") -> List[torch.Tensor]:
    """Integer-valued bf16 gradients in [lo, hi] (sums of them are exact)."""
    out = []
    for r in range(R):
        g = _gen(device, SEED_GRAD + 100 * micro + r)
        x = torch.randint(lo, hi + 1, (n,), generator=g, device=device)
        out.append(x.to(torch.bfloat16))
    return out
