"""The bulk-copy engine's bounded waits, made to run out on the GPU without
any fault: cc_inject_bulk_stall tells the next bulk launch's producer to
skip one tile and bounds that launch's waits by a few milliseconds.  The
consumers waiting for the tile give up, the producer gives up when it comes
back to the tile's stage, both report through the status word, the launch
returns, and what the stalled CTA did not step is left as it was.  The next
call runs normally and matches the oracle bit for bit."""
import time

import numpy as np
import pytest
import torch

from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gpu_common import compare_all, f32, host_copy, new_slabs, oracle_step, random_inputs, u16

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=2,
          grad_scale=1.0)
TILE = 1024          # the engine's tile at R = 2 (16 KB stages)
BULK = capi.CC_ENGINE_BULK_COPY


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    capi.lib()


def test_skipped_tile_runs_out_and_reports():
    R, n = 2, 64 * TILE + 29          # 65 tiles (the last partial) + a 5-element tail
    capi.cc_device_status(clear=True)
    s = new_slabs(*random_inputs(R, n, seed=77, step=2))
    grads, state, _ = host_copy(s)
    outs0 = [u16(o) for o in s.outs]
    capi.cc_inject_bulk_stall(0, 20000)          # CTA 0 never gets its first tile
    t0 = time.perf_counter()
    capi.cc_fused_dp_bucket_ex(s.grads, None, s.master, s.m, s.v, s.outs, n, R, 0, n,
                               max_ctas=2, arith_flags=BULK, **HP)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = capi.cc_device_status(clear=True)
    assert status == 1 | 2, status               # consumers and producer gave up
    assert capi.cc_device_status() == 0
    assert elapsed < 10.0

    # Every tile is either stepped exactly or left exactly as it was.  The
    # skipped tile (CTA 0's first) is untouched; CTA 1, which owns the odd
    # tiles, stepped all of them and, as the last CTA, the tail.  How many of
    # CTA 0's later tiles other consumers stepped before the producer gave up
    # depends on the engine's stage ring, not on the contract.
    ref_state = [x.copy() for x in state]
    ref_outs = oracle_step(grads, ref_state, HP)
    got_state = [f32(t) for t in (s.master, s.m, s.v)]
    got_outs = [u16(o) for o in s.outs]
    tiled = n // 8 * 8

    def matches(lo, hi, st, outs):
        return (all(np.array_equal(g[lo:hi].view(np.uint32), w[lo:hi].view(np.uint32))
                    for g, w in zip(got_state, st)) and
                all(np.array_equal(g[lo:hi], w[lo:hi]) for g, w in zip(got_outs, outs)))

    num_tiles = (tiled + TILE - 1) // TILE
    stepped = []
    for t in range(num_tiles):
        lo, hi = t * TILE, min(tiled, (t + 1) * TILE)
        done = matches(lo, hi, ref_state, ref_outs)
        assert done or matches(lo, hi, state, outs0), f"tile {t} partly stepped"
        stepped.append(done)
    assert not stepped[0]
    assert all(stepped[1::2]), "CTA 1 gave up"
    assert matches(tiled, n, ref_state, ref_outs), "the tail"

    # the next call, with nothing armed, is whole and exact
    s2 = new_slabs(*random_inputs(R, n, seed=78, step=2))
    grads2, state2, _ = host_copy(s2)
    capi.cc_fused_dp_bucket_ex(s2.grads, None, s2.master, s2.m, s2.v, s2.outs, n, R, 0, n,
                               max_ctas=2, arith_flags=BULK, **HP)
    torch.cuda.synchronize()
    compare_all(s2, state2, oracle_step(grads2, state2, HP))
    assert capi.cc_device_status() == 0


def test_stall_on_a_last_tile_lets_the_producer_finish():
    """A skipped tile among the producer's last S leaves it nothing to wait
    for: only the consumers give up (code 1), and the producer still waits
    for every copy it issued before the CTA exits."""
    R, n = 2, 16 * TILE
    capi.cc_device_status(clear=True)
    s = new_slabs(*random_inputs(R, n, seed=79, step=2))
    capi.cc_inject_bulk_stall(15, 20000)         # CTA 0's last tile (grid 1)
    capi.cc_fused_dp_bucket_ex(s.grads, None, s.master, s.m, s.v, s.outs, n, R, 0, n,
                               max_ctas=1, arith_flags=BULK, **HP)
    torch.cuda.synchronize()
    assert capi.cc_device_status(clear=True) == 1
    # tiles 0..14 were stepped
    grads, state, _ = host_copy(s)               # (state already stepped: check outs only)
    out0 = u16(s.outs[0])
    assert (out0[:15 * TILE] != 0xFFFF).all()
    assert (out0[15 * TILE:] == 0xFFFF).all()

