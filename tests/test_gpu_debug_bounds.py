"""The debug build (CC_DEBUG_BOUNDS=1): the fused tensor-parallel kernel's
epilogue and the bulk-copy engine check every computed offset against the
buffer or range their arguments describe, and an access outside it is
skipped and reported (status code 128) instead of made -- a sanitizer
stand-in on a pool where compute-sanitizer is closed.  The debug library is
built beside the release one and exercised in a child process (one CUDA
runtime per process): across shapes, schedules and budgets no check fires
and every result stays exact."""
import os
import subprocess
import sys

import pytest

from gradient_reduce_optimizer_gb300 import build as gbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEBUG_DIR = os.path.join(ROOT, "_build_debug")
DEBUG_LIB = os.path.join(DEBUG_DIR, "libcc_dp.so")

CHILD = r'''
import os, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, os.path.join(sys.argv[1], "tests"))
import numpy as np, torch
from gradient_reduce_optimizer_gb300 import capi
capi.LIBRARY = sys.argv[2]; capi._LIB = None
assert capi.lib()._name == sys.argv[2]          # the debug build, not the release one
import oracle
from gpu_common import DEV, compare_all, host_copy, new_slabs, oracle_step, random_inputs
capi.cc_device_status(clear=True)
hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=4, grad_scale=1.0)
# the bulk-copy engine: ragged sizes, accumulators, budgets
for R, n, ctas, use_acc in ((1, 1025, 3, False), (8, 300_007, 7, False), (16, 9_001, 5, True),
                            (8, 1 << 22, 152, False), (2, 64 * 1024 + 29, 2, True)):
    s = new_slabs(*random_inputs(R, n, seed=R + n % 97, step=4), with_acc=use_acc)
    if use_acc:
        for a in s.acc:
            a.copy_(torch.randn(n, device=DEV) * 1e-3)
    grads, state, acc = host_copy(s)
    capi.cc_fused_dp_bucket_ex(s.grads, s.acc if use_acc else None, s.master, s.m, s.v, s.outs,
                               n, R, 0, n, max_ctas=ctas, arith_flags=capi.CC_ENGINE_BULK_COPY,
                               **hp)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0, ("bulk", R, n)
    compare_all(s, state, oracle_step(grads, state, hp, acc=acc if use_acc else None))
# the fused tensor-parallel kernel: whole and split waves, budgets, partials
for R, m, n, k, ctas, split in ((2, 256, 256, 256, 0, True), (8, 256, 384, 1024, 32, True),
                                (3, 2560, 1280, 192, 12, True), (4, 512, 640, 256, 16, True),
                                (8, 8192, 3072, 12288, 0, True), (5, 2304, 384, 1280, 4, False)):
    kr = k // R
    x = [torch.randint(-3, 4, (m, kr), device=DEV).to(torch.bfloat16) for _ in range(R)]
    w = [torch.randint(-3, 4, (n, kr), device=DEV).to(torch.bfloat16) for _ in range(R)]
    outs = [torch.empty(m, n, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    parts = [torch.empty(m, n, device=DEV) for _ in range(R)] if m * n <= 1 << 22 else None
    wsb = capi.cc_tp_matmul_allreduce_workspace(m, n, k, R, ctas) if split else 0
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV) if split else None
    capi.cc_tp_matmul_allreduce_ex(x, w, outs, parts, m, n, k, R, ws, wsb, ctas)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0, ("tp", R, m, n, k, ctas)
    rows = torch.arange(0, m, max(1, m // 64), device=DEV)
    total = sum(x_[rows].double() @ w_.double().T for x_, w_ in zip(x, w))
    want = total.float().to(torch.bfloat16).view(torch.int16)
    for o in outs:
        assert torch.equal(o[rows].view(torch.int16), want), ("tp out", R, m, n, k)
print("debug bounds: no check fired")
'''


def test_debug_bounds_build_fires_no_check():
    gbuild.build(extra_flags=["-DCC_DEBUG_BOUNDS=1"], build_dir=DEBUG_DIR, library=DEBUG_LIB)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, DEBUG_LIB], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "no check fired" in r.stdout
