"""Randomised parity sweep: 120 random configurations of the step through
the C ABI, each bit-identical to the oracle.  Every case draws R, a ragged
n, a bucket size, an engine (fused step, fused bucket on a CTA budget --
the bulk-copy engine --, the unfused schedule, the accumulated reducing
step), hyper-parameters (loss scales that are and are not powers of two)
and slab base offsets of 0 or 16 bytes past a 32-byte boundary."""
import random

import numpy as np
import pytest
import torch

import oracle
from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gpu_common import DEV, compare_all, host_copy, oracle_step, Slabs

pytestmark = pytest.mark.gpu


def placed(t: torch.Tensor, offset_elems: int) -> torch.Tensor:
    """A copy of t whose data starts offset_elems past a fresh allocation."""
    buf = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device=DEV)
    view = buf[offset_elems:]
    view.copy_(t)
    return view


@pytest.fixture(scope="module", autouse=True)
def library():
    gbuild.build()
    return capi.lib()


@pytest.mark.parametrize("case", range(120))
def test_random_configuration(case):
    rnd = random.Random(7000 + case)
    R = rnd.choice([1, 2, 3, 4, 5, 8, 11, 16])
    n = rnd.choice([rnd.randint(1, 100), rnd.randint(100, 5000), rnd.randint(5000, 300_000)])
    engine = rnd.choice(["step", "bucket_bulk", "unfused", "accum"])
    bucket_bytes = rnd.choice([0, 16, 48, 1024, 65536, 1 << 20])
    step = rnd.randint(1, 2000)
    hp = dict(lr=rnd.choice([0.0, 1e-4, 1e-3, 3e-2]), beta1=rnd.choice([0.0, 0.5, 0.9]),
              beta2=rnd.choice([0.0, 0.95, 0.999]), eps=rnd.choice([0.0, 1e-8, 1e-3]),
              weight_decay=rnd.choice([0.0, 0.01, 0.3]), step=step,
              grad_scale=rnd.choice([1.0, 1024.0, 3.0, 0.5]))
    g = torch.Generator(device=DEV)
    g.manual_seed(case)
    bf_off = lambda: rnd.choice([0, 8])     # 0 or 16 bytes for bf16
    f_off = lambda: rnd.choice([0, 4])      # 0 or 16 bytes for fp32
    grads = [placed((torch.randn(n, generator=g, device=DEV) * 1e-3 * hp["grad_scale"])
                    .to(torch.bfloat16), bf_off()) for _ in range(R)]
    master = placed(torch.randn(n, generator=g, device=DEV) * 0.02, f_off())
    m = placed(torch.randn(n, generator=g, device=DEV) * 1e-4, f_off())
    v = placed((torch.randn(n, generator=g, device=DEV) * 1e-3) ** 2, f_off())
    outs = [placed(torch.zeros(n, dtype=torch.bfloat16, device=DEV), bf_off())
            for _ in range(R)]
    acc = ([placed(torch.randn(n, generator=g, device=DEV) * 1e-3, f_off()) for _ in range(R)]
           if engine == "accum" else None)
    s = Slabs(grads, master, m, v, outs, acc)
    grads_h, state, acc_h = host_copy(s)
    if engine == "step":
        capi.cc_fused_dp_step(grads, master, m, v, outs, n, R, bucket_bytes, **hp)
    elif engine == "bucket_bulk":
        per = max(8, bucket_bytes // 16 * 8) if bucket_bytes else n
        ctas = rnd.choice([1, 3, 16, 152])
        flags = rnd.choice([0, capi.CC_ENGINE_BULK_COPY])   # wide CTAs or bulk copies
        for b in range(0, n, per):
            capi.cc_fused_dp_bucket_ex(grads, None, master, m, v, outs, n, R, b,
                                       min(n, b + per), max_ctas=ctas, arith_flags=flags,
                                       **hp)
    elif engine == "unfused":
        per = max(8, bucket_bytes // 16 * 8) if bucket_bytes else n
        ws = torch.empty(min(per, n), dtype=torch.float32, device=DEV)
        capi.cc_unfused_dp_step(grads, master, m, v, outs, ws, 4 * ws.numel(), n, R,
                                bucket_bytes, **hp)
    else:
        capi.cc_fused_dp_step_accum(grads, acc, master, m, v, outs, n, R, bucket_bytes,
                                    accum_k=rnd.randint(2, 6), **hp)
    torch.cuda.synchronize()
    ref = oracle_step(grads_h, state, hp, acc=acc_h if engine == "accum" else None)
    compare_all(s, state, ref, label=f"case {case} ({engine}, R={R}, n={n}) ")
    assert capi.cc_device_status() == 0
