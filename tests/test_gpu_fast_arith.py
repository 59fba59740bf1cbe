"""The opt-in fast arithmetic of the bucket kernels (CC_ARITH_FAST), through
the C ABI, against the oracle's exact step.

The method's tolerance for floating point is a relative 1e-5 on the fp32
master weights and moments and one bf16 ulp on the parameters.  The fast form
keeps the replica sum, m and v exact (bit for bit), so only the parameter
moves: by a few ulp of the update.  Worst case, in units of 2^-24 relative:
m^ and v^ are products by reciprocals rounded on the host (3 each, instead of
one correctly rounded division), the square root halves v^'s error and
rounds (2.5), the sum with eps rounds (1), the fast division adds 2 ulp (4),
the quotient and the product by lr round (2): 16 * 2^-24 of the update in
all, plus one ulp of the parameter for the final rounding.  That is inside 1e-5 of the parameter wherever the update does
not cancel the parameter; the test checks both.  Replica identity stays
exact.  Both engines, with and without accumulators, ragged sizes."""
import numpy as np
import pytest
import torch

from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gpu_common import DEV, f32, host_copy, new_slabs, oracle_step, random_inputs, u16

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, grad_scale=4.0)


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    capi.lib()


def ordered(bits16):
    """bf16 bit patterns as integers in the order of their values."""
    b = bits16.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - b, b)


BULK = capi.CC_ENGINE_BULK_COPY


@pytest.mark.parametrize("R,n,max_ctas,use_acc,step,engine", [
    (1, 4099, 0, False, 1, 0), (3, 100_003, 0, False, 7, 0), (8, 100_003, 0, True, 10, 0),
    (3, 100_003, 16, False, 7, 0), (8, 262_147, 16, True, 10, 0), (16, 9_001, 5, False, 2, 0),
    (3, 100_003, 16, False, 7, BULK), (8, 262_147, 16, True, 10, BULK),
    (16, 9_001, 5, False, 2, BULK)])
def test_fast_step_within_the_bound(R, n, max_ctas, use_acc, step, engine):
    grads, master, m, v = random_inputs(R, n, seed=90 + R, sigma=1e-3, step=step,
                                        premultiply=4.0)
    s = new_slabs(grads, master, m, v, with_acc=use_acc)
    if use_acc:
        for a, g in zip(s.acc, grads):
            a.copy_(g.float() * 2.0)
    h_grads, h_state, h_acc = host_copy(s)
    before = h_state[0].copy()
    hp = dict(HP, step=step)
    capi.cc_fused_dp_bucket_ex(s.grads, s.acc, s.master, s.m, s.v, s.outs, n, R, 0, n,
                               max_ctas=max_ctas, arith_flags=capi.CC_ARITH_FAST | engine,
                               **hp)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0
    ref_outs = oracle_step(h_grads, h_state, hp, acc=h_acc)
    ref_p, ref_m, ref_v = h_state
    # the sum, m and v: exact
    np.testing.assert_array_equal(f32(s.m).view(np.uint32), ref_m.view(np.uint32))
    np.testing.assert_array_equal(f32(s.v).view(np.uint32), ref_v.view(np.uint32))
    # the parameter: within 16 * 2^-24 of its update plus one ulp of itself
    got = f32(s.master).astype(np.float64)
    want = ref_p.astype(np.float64)
    decayed = (before * np.float32(1.0 - hp["lr"] * hp["weight_decay"])).astype(np.float64)
    update = np.abs(decayed - want)
    bound = 16 * 2.0 ** -24 * update + 2.0 ** -23 * np.abs(want) + 1e-45
    err = np.abs(got - want)
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"
    no_cancel = update < np.abs(want)
    rel = err[no_cancel] / np.abs(want[no_cancel])
    assert rel.max() <= 1e-5
    # bf16 parameters: at most one bf16 ulp; every replica identical
    out0 = u16(s.outs[0])
    assert np.abs(ordered(out0) - ordered(ref_outs[0])).max() <= 1
    for r in range(1, R):
        np.testing.assert_array_equal(u16(s.outs[r]), out0)


def test_fast_integer_gradients_keep_the_exact_sum():
    """Integer-valued gradients: the replica sum is exact in either mode, so m
    and v (which see only the sum) are bit-identical to the exact kernel."""
    from gradient_reduce_optimizer_gb300 import workloads as wl
    R, n = 8, 50_001
    grads = wl.integer_grads(R, n, device=DEV)
    _, master, m, v = random_inputs(R, n, seed=5, step=3)
    a = new_slabs(grads, master.clone(), m.clone(), v.clone())
    b = new_slabs(grads, master.clone(), m.clone(), v.clone())
    hp = dict(HP, step=3)
    capi.cc_fused_dp_bucket_ex(a.grads, None, a.master, a.m, a.v, a.outs, n, R, 0, n, **hp)
    capi.cc_fused_dp_bucket_ex(b.grads, None, b.master, b.m, b.v, b.outs, n, R, 0, n,
                               arith_flags=capi.CC_ARITH_FAST, **hp)
    torch.cuda.synchronize()
    assert torch.equal(a.m.view(torch.int32), b.m.view(torch.int32))
    assert torch.equal(a.v.view(torch.int32), b.v.view(torch.int32))


def test_unknown_arith_flags_rejected():
    R, n = 2, 64
    s = new_slabs(*random_inputs(R, n, seed=1))
    for bad in (4, 8, 1 << 31):
        with pytest.raises(capi.CCError) as ei:
            capi.cc_fused_dp_bucket_ex(s.grads, None, s.master, s.m, s.v, s.outs, n, R, 0, n,
                                       arith_flags=bad, step=1, **HP)
        assert ei.value.status == capi.CC_ERR_INVALID
