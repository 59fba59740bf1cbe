"""Guard bands: every slab an entry point reads or writes sits between two
256-byte bands of a sentinel pattern, and after each entry point has run on
ragged sizes (partial last vector, buckets, shards, the bulk engine) the
bands are unchanged.  A stand-in for a memory checker: a write one element
past a slab's end, or before its start, changes a band."""
import pytest
import torch

from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 256            # bytes on each side; keeps the slab 16-byte aligned
SENTINEL = 0xA5
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=4,
          grad_scale=2.0)


@pytest.fixture(scope="module", autouse=True)
def library():
    gbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return capi.lib()


class Guarded:
    """A slab of n elements with a sentinel band on either side."""

    def __init__(self, n, dtype, name, fill=None):
        esz = torch.empty(0, dtype=dtype).element_size()
        g = GUARD // esz
        self.name, self.n, self.esz = name, n, esz
        self.buf = torch.empty(n + 2 * g, dtype=dtype, device=DEV)
        self.buf.view(torch.uint8).fill_(SENTINEL)
        self.t = self.buf[g:g + n]
        if fill is not None:
            self.t.copy_(fill)

    def check(self):
        b = self.buf.view(torch.uint8)
        head, tail = b[:GUARD], b[GUARD + self.n * self.esz:]
        assert bool((head == SENTINEL).all()), f"{self.name}: band before the slab changed"
        assert bool((tail == SENTINEL).all()), f"{self.name}: band after the slab changed"


def randn(n, gen, scale):
    return torch.randn(n, generator=gen, device=DEV) * scale


@pytest.mark.parametrize("n", [7, 8, 4099, 8 * 1000 + 5])
@pytest.mark.parametrize("R", [1, 3, 8])
def test_guard_bands_around_every_slab_stay_intact(R, n):
    gen = torch.Generator(device=DEV).manual_seed(1000 * R + n)
    slabs = []

    def guarded(dtype, name, fill=None, length=n):
        s = Guarded(length, dtype, name, fill)
        slabs.append(s)
        return s.t

    grads = [guarded(torch.bfloat16, f"grads[{r}]", randn(n, gen, 1e-3)) for r in range(R)]
    outs = [guarded(torch.bfloat16, f"params_out[{r}]") for r in range(R)]
    acc = [guarded(torch.float32, f"acc[{r}]", randn(n, gen, 1e-3)) for r in range(R)]
    master = guarded(torch.float32, "master", randn(n, gen, 0.02))
    m = guarded(torch.float32, "m", randn(n, gen, 1e-4))
    v = guarded(torch.float32, "v", randn(n, gen, 1e-3) ** 2)
    work = guarded(torch.float32, "workspace")
    partials = [guarded(torch.float32, f"partials[{r}]", randn(n, gen, 1.0)) for r in range(R)]

    capi.cc_fused_dp_step(grads, master, m, v, outs, n, R, 2048, **HP)
    capi.cc_fused_dp_step_accum(grads, acc, master, m, v, outs, n, R, 2048, accum_k=3, **HP)
    for use_acc in (None, acc):
        for ctas, flags in ((0, 0), (7, 0), (7, capi.CC_ENGINE_BULK_COPY)):
            capi.cc_fused_dp_bucket_ex(grads, use_acc, master, m, v, outs, n, R, 0, n,
                                       max_ctas=ctas, arith_flags=flags, **HP)
    cut = n // 16 * 8
    for b, e in ((0, cut), (cut, n)):
        shard = [guarded(torch.float32, f"{nm} shard [{b}, {e})", t[b:e], length=e - b)
                 for nm, t in (("master", master), ("m", m), ("v", v))]
        capi.cc_fused_dp_shard(grads, acc, *shard, outs, n, R, b, e, 1024, **HP)
    capi.cc_accumulate_local(grads, acc, n, R, True)
    capi.cc_accumulate_local(grads, acc, n, R, False)
    capi.cc_unfused_dp_step(grads, master, m, v, outs, work, 4 * n, n, R, 2048, **HP)
    capi.cc_unfused_dp_step_noalloc(grads, master, m, v, outs, n, R, 2048, **HP)
    capi.cc_tp_allreduce(partials, outs, n, R)
    torch.cuda.synchronize()
    for s in slabs:
        s.check()
    assert capi.cc_device_status() == 0
