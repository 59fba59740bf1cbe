"""The allocation-free entry point, cc_unfused_dp_step_noalloc.

It serves callers that cannot allocate device memory themselves (their
memory belongs to a framework's caching allocator, an allocation would stall
a hot loop, or they are handed buffers with no right to allocate): instead
of a caller-provided workspace it uses a fixed scratch array inside the
library.  This checks, through the C ABI, that two calls in a row give the
same bits as the workspace entry point, and that a bucket larger than the
fixed array is refused.  It lives in its own file, collected last, and
needs nothing from the other tests.
"""
import pytest
import torch

from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gpu_common import DEV, new_slabs, random_inputs

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
          grad_scale=1.0)


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    gbuild.build()
    capi.lib()
    R, n, bucket_bytes = 4, 2 * 1024 * 1024 + 13, 1 << 20   # 5 buckets, ragged tail
    per = bucket_bytes // 16 * 8
    _, master, m, v = random_inputs(R, n, seed=31, step=3)
    a = new_slabs([None] * R, master.clone(), m.clone(), v.clone())
    b = new_slabs([None] * R, master.clone(), m.clone(), v.clone())
    workspace = torch.empty(per, dtype=torch.float32, device=DEV)
    for call in range(2):
        grads = random_inputs(R, n, seed=100 + call, step=1)[0]
        a.grads = b.grads = grads
        hp = dict(HP, step=3 + call)
        capi.cc_unfused_dp_step(a.grads, a.master, a.m, a.v, a.outs, workspace,
                                workspace.numel() * 4, n, R, bucket_bytes, **hp)
        capi.cc_unfused_dp_step_noalloc(b.grads, b.master, b.m, b.v, b.outs, n, R,
                                        bucket_bytes, **hp)
        torch.cuda.synchronize()
        for x, y in zip([a.master, a.m, a.v] + a.outs, [b.master, b.m, b.v] + b.outs):
            assert torch.equal(bits(x), bits(y)), f"call {call}"


def test_noalloc_fills_its_whole_scratch():
    """A bucket of exactly CC_NOALLOC_SCRATCH_ELEMS elements (bucket_bytes of
    32 MiB, and also 15 bytes past it, which floor to the same bucket) uses
    the last element of the fixed array; a ragged second bucket follows.
    Two calls in a row, bit for bit against the workspace entry point."""
    gbuild.build()
    R = 2
    cap = capi.CC_NOALLOC_SCRATCH_ELEMS
    n = cap + 4096 + 5
    _, master, m, v = random_inputs(R, n, seed=41, step=2)
    a = new_slabs([None] * R, master.clone(), m.clone(), v.clone())
    b = new_slabs([None] * R, master.clone(), m.clone(), v.clone())
    workspace = torch.empty(cap, dtype=torch.float32, device=DEV)
    for call, bucket_bytes in enumerate((2 * cap, 2 * cap + 15)):
        grads = random_inputs(R, n, seed=200 + call, step=1)[0]
        a.grads = b.grads = grads
        hp = dict(HP, step=2 + call)
        capi.cc_unfused_dp_step(a.grads, a.master, a.m, a.v, a.outs, workspace,
                                workspace.numel() * 4, n, R, bucket_bytes, **hp)
        capi.cc_unfused_dp_step_noalloc(b.grads, b.master, b.m, b.v, b.outs, n, R,
                                        bucket_bytes, **hp)
        torch.cuda.synchronize()
        for x, y in zip([a.master, a.m, a.v] + a.outs, [b.master, b.m, b.v] + b.outs):
            assert torch.equal(bits(x), bits(y)), f"call {call}"


def test_noalloc_refuses_buckets_beyond_its_scratch():
    gbuild.build()
    R, n = 2, 4096
    s = new_slabs(*random_inputs(R, n, seed=7, step=1))
    too_many = 16 * 1024 * 1024 + 8          # one bucket past the fixed array
    with pytest.raises(capi.CCError) as ei:
        capi.cc_unfused_dp_step_noalloc(s.grads, s.master, s.m, s.v, s.outs, too_many,
                                        R, 0, step=1, **HP)
    assert ei.value.status == capi.CC_ERR_INVALID
    assert "scratch" in ei.value.reason and "n=" in ei.value.reason
    # the same refusal when bucket_bytes sets the size (16 bytes past the
    # edge, on a slab longer than one bucket)
    longer = capi.CC_NOALLOC_SCRATCH_ELEMS + 1000
    big = torch.empty(longer, dtype=torch.float32, device=DEV)
    with pytest.raises(capi.CCError) as ei:
        capi.cc_unfused_dp_step_noalloc([big] * R, big, big, big, [big] * R, longer, R,
                                        2 * capi.CC_NOALLOC_SCRATCH_ELEMS + 16,
                                        step=1, **HP)
    assert ei.value.status == capi.CC_ERR_INVALID
    assert "bucket_bytes=" in ei.value.reason
