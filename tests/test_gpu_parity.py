"""Parity of the CUDA path (through the C ABI) with the oracle.

Bar: bit-identical master/m/v and bf16 parameters on every case (NaN
payloads excepted: a NaN must meet a NaN).  The operation order is fixed in
include/cc_dp.h and both sides round every binary32 operation separately, so
the looser floating-point bar (1e-5 relative on fp32 state, 1 bf16 ulp on
parameters) is never needed; bit equality is asserted instead.

Element by element at sizes the oracle finishes in seconds (spanning many
thread blocks, grid-stride rounds and a ragged tail), and on sampled
elements at the full workload sizes in the launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gradient_reduce_optimizer_gb300 import workloads as wl
from gpu_common import (DEV, assert_bits, compare_all, f32, gpu_step, host_copy,
                        hp_of, new_slabs, oracle_step, planned_workload_slabs,
                        random_inputs, u16, workload_grads)

pytestmark = pytest.mark.gpu

HP1 = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
           step=1, grad_scale=1.0)
HP10 = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
            step=10, grad_scale=1.0)


@pytest.fixture(scope="module", autouse=True)
def library():
    gbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return capi.lib()


def check_full(s, hp, bucket_bytes=0, label=""):
    grads, state, _ = host_copy(s)
    gpu_step(s, hp, bucket_bytes)
    torch.cuda.synchronize()
    outs = oracle_step(grads, state, hp)
    compare_all(s, state, outs, label=label)


# ---------------------------------------------------------------------------
# Element-by-element parity
# ---------------------------------------------------------------------------

def test_flat_1m_r2_step1():
    """R=2, n=1,048,576, one bucket, step 1, m=v=0: every element."""
    w = wl.flat_1m_r2()
    grads = wl.make_grads(2, w.n, w.grad_sigma, device=DEV)
    master, m, v = wl.make_state(w.n, 1, w.grad_sigma, device=DEV)
    check_full(new_slabs(grads, master, m, v), hp_of(w))


@pytest.mark.parametrize("n", list(range(1, 65)))
def test_small_n_r8(n):
    check_full(new_slabs(*random_inputs(8, n, seed=n, step=3)),
               dict(HP10, step=3), label=f"n={n} ")


@pytest.mark.parametrize("R", [1, 2, 3, 5, 7, 12, 16])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 15, 17, 63, 2049])
def test_small_n_all_r(R, n):
    check_full(new_slabs(*random_inputs(R, n, seed=100 * R + n, step=7)),
               dict(HP10, step=7), label=f"R={R} n={n} ")


@pytest.mark.parametrize("R", [1, 4, 8, 16])
def test_many_blocks_ragged_tail(R):
    """Several grid-stride rounds over all SMs plus a 5-element tail."""
    n = 8 * 256 * 152 * 3 + 8 * 37 + 5
    s = new_slabs(*random_inputs(R, n, seed=R, step=5, premultiply=1024.0))
    check_full(s, dict(HP10, step=5, grad_scale=1024.0))


def test_bucket_cut_does_not_change_values():
    n = 3 * 1024 * 1024 + 5
    base = random_inputs(4, n, seed=7, step=4)
    ref = None
    for bb in (0, 16, 48, 4096, 1 << 20, 4 << 20, 25 << 20, 100 << 20, 500 << 20):
        s = new_slabs([g.clone() for g in base[0]], *[t.clone() for t in base[1:]])
        gpu_step(s, dict(HP10, step=4), bucket_bytes=bb)
        torch.cuda.synchronize()
        got = ([f32(t) for t in (s.master, s.m, s.v)] + [u16(o) for o in s.outs])
        if ref is None:
            ref = got
            grads, state, _ = host_copy(new_slabs(*base))
            outs = oracle_step(grads, state, dict(HP10, step=4))
            compare_all(s, state, outs, label="bucket 0 ")
        else:
            for a, b in zip(got, ref):
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), bb


@pytest.mark.parametrize("max_ctas", [0, 1, 7, 152])
def test_bucket_entry_point_over_planned_buckets(max_ctas):
    """cc_fused_dp_bucket over a planned layout, bucket by bucket."""
    t = wl.bert_large_tensors(layers=2, hidden=256, ffn=1024, vocab=999,
                              positions=64)
    numel = [x[1] for x in t]
    offsets, buckets, n_slab = oracle.plan_buckets(numel, 64 * 1024)
    assert len(buckets) > 4
    s = new_slabs(*random_inputs(3, n_slab, seed=11, step=2))
    grads, state, _ = host_copy(s)
    hp = dict(HP10, step=2)
    for b, e in buckets:
        capi.cc_fused_dp_bucket(s.grads, None, s.master, s.m, s.v, s.outs, n_slab,
                                3, b, e, max_ctas=max_ctas, **hp)
    torch.cuda.synchronize()
    compare_all(s, state, oracle_step(grads, state, hp))


@pytest.mark.parametrize("R,n,use_acc", [(4, 100_003, False), (8, 1 << 20, True),
                                         (3, 8 * 1000 + 5, False), (16, 4099, True),
                                         (2, 7, False)])
def test_sharded_state_ranks_partition_the_step(R, n, use_acc):
    """Each of R ranks owns only its shard of master/m/v (arrays of the
    shard's length) and calls cc_fused_dp_shard on its range of the replica
    slabs.  Together they give the single fused step bit for bit: every
    replica's parameters, and each rank's state shard."""
    s = new_slabs(*random_inputs(R, n, seed=40 + R, step=6), with_acc=use_acc)
    if use_acc:
        g = torch.Generator(device=DEV).manual_seed(41)
        for a in s.acc:
            a.copy_(torch.randn(n, generator=g, device=DEV) * 3e-3)
    grads, state, acc = host_copy(s)
    hp = dict(HP10, step=6)
    units = n // 8
    cuts = [8 * (units * k // R) for k in range(R)] + [n]
    owned = []
    for k in range(R):
        b, e = cuts[k], cuts[k + 1]
        shard = [t[b:e].clone() for t in (s.master, s.m, s.v)]
        capi.cc_fused_dp_shard(s.grads, s.acc, *shard, s.outs, n, R, b, e, 64 << 10, **hp)
        owned.append((b, e, shard))
    torch.cuda.synchronize()
    outs = oracle_step(grads, state, hp, acc=acc)
    for r, (t, ref) in enumerate(zip(s.outs, outs)):
        assert_bits(f"params_out[{r}]", u16(t), ref, "bf16")
    for k, (b, e, shard) in enumerate(owned):
        for name, t, ref in zip(("master", "m", "v"), shard, state):
            assert_bits(f"rank {k} {name}", f32(t), ref[b:e], "f32")


def test_fifty_consecutive_steps_do_not_drift():
    """Steps t = 1..50 from m = v = 0, fresh gradients every step, the GPU
    state and the oracle state each fed back into itself: still the same
    bits after 50 steps (a single differently rounded operation anywhere
    would compound)."""
    R, n = 4, 262_147
    s = new_slabs(*random_inputs(R, n, seed=77, step=1))
    _, state, _ = host_copy(s)
    gen = torch.Generator(device=DEV).manual_seed(78)
    for t in range(1, 51):
        for gr in s.grads:
            gr.copy_((torch.randn(n, generator=gen, device=DEV) * 1e-3).to(torch.bfloat16))
        host_grads = [u16(gr) for gr in s.grads]
        hp = dict(HP10, step=t)
        gpu_step(s, hp, bucket_bytes=96 << 10)
        outs = oracle_step(host_grads, state, hp)
    torch.cuda.synchronize()
    compare_all(s, state, outs, label="step 50 ")


def test_consecutive_steps_captured_in_a_cuda_graph():
    """Two consecutive multi-bucket steps captured in one CUDA graph and
    replayed twice: inside a step the buckets chain by programmatic launch,
    and a step's first bucket waits for all of the previous step.  Same bits
    as four oracle steps."""
    n = 1024 * 1024 + 8 * 13 + 3
    s = new_slabs(*random_inputs(4, n, seed=31, step=2))
    hp = dict(HP10, step=2)
    gpu_step(s, hp, bucket_bytes=256 << 10)      # per-device state set up
    torch.cuda.synchronize()
    grads, state, _ = host_copy(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in (3, 4):
            gpu_step(s, dict(hp, step=t), bucket_bytes=256 << 10)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for t in (3, 4, 3, 4):
        outs = oracle_step(grads, state, dict(hp, step=t))
    compare_all(s, state, outs, label="graph ")


@pytest.mark.parametrize("graph", [False, True])
def test_back_to_back_single_bucket_steps(graph):
    """Twenty one-bucket steps of the same slab with nothing between them
    (the launch-bound small case: R = 2, 1,048,576 parameters): each step's
    kernel may become resident while the previous one finishes, but reads
    master/m/v only after it has completed.  Same bits as twenty oracle
    steps, from the stream and from a CUDA graph."""
    R, n, steps = 2, 1 << 20, 20
    s = new_slabs(*random_inputs(R, n, seed=33, step=3))
    hp = dict(HP10, step=3)
    grads, state, _ = host_copy(s)
    if graph:
        gpu_step(s, hp)                          # per-device state set up
        torch.cuda.synchronize()
        grads, state, _ = host_copy(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(steps // 2):
                gpu_step(s, hp)
        for _ in range(2):
            g.replay()
    else:
        for _ in range(steps):
            gpu_step(s, hp)
    torch.cuda.synchronize()
    for _ in range(steps):
        outs = oracle_step(grads, state, hp)
    compare_all(s, state, outs, label="graph " if graph else "stream ")


@pytest.mark.parametrize("R", [1, 2, 3, 8, 16])
def test_integer_gradients_sum_exactly(R):
    n = 100_003
    grads = wl.integer_grads(R, n, device=DEV)
    master = torch.ones(n, device=DEV)
    m = torch.full((n,), 7.0, device=DEV)
    v = torch.full((n,), 3.0, device=DEV)
    s = new_slabs(grads, master, m, v)
    hp = dict(lr=0.0, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.0, step=1,
              grad_scale=1.0)
    gpu_step(s, hp)
    torch.cuda.synchronize()
    exact = sum(g.float().cpu().numpy().astype(np.int64) for g in grads)
    assert np.array_equal(f32(s.m), exact.astype(np.float32))
    assert np.array_equal(f32(s.v), (exact * exact).astype(np.float32))
    # integer gradients under the normal hyper-parameters: bit-exact too
    s2 = new_slabs(wl.integer_grads(R, n, device=DEV), *random_inputs(1, n, 3, step=10)[1:])
    check_full(s2, HP10)


def test_replicas_bit_identical():
    s = new_slabs(*random_inputs(16, 1 << 20, seed=5, step=2))
    gpu_step(s, dict(HP10, step=2))
    torch.cuda.synchronize()
    ref = s.outs[0].view(torch.int16)
    for o in s.outs[1:]:
        assert torch.equal(o.view(torch.int16), ref)


def test_special_values_propagate_like_the_oracle():
    vals = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), float("nan"),
                         1e-40, -1e-40, 3e38, -3e38, 1e-3, 65504.0, 2.0 ** -133],
                        dtype=torch.float32)
    n = 4096 + 3
    g = torch.Generator().manual_seed(9)
    pick = lambda: vals[torch.randint(0, vals.numel(), (n,), generator=g)]
    grads = [pick().to(torch.bfloat16).to(DEV) for _ in range(3)]
    master = pick().to(DEV)
    m = pick().to(DEV)
    v = pick().abs().to(DEV)
    check_full(new_slabs(grads, master, m, v), dict(HP10, step=2))


@pytest.mark.parametrize("hp", [
    dict(lr=0.0, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, step=1, grad_scale=1.0),
    dict(lr=1e-2, beta1=0.5, beta2=0.75, eps=1e-3, weight_decay=0.5, step=1000, grad_scale=3.0),
    dict(lr=1.5e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=2, grad_scale=65536.0),
])
def test_hyper_parameter_corners(hp):
    check_full(new_slabs(*random_inputs(4, 50_001, seed=3, step=2,
                                        premultiply=hp["grad_scale"])), hp)


@pytest.mark.parametrize("R,k", [(1, 2), (3, 3), (8, 4), (16, 2)])
def test_accumulation_matches_oracle(R, k):
    n = 200_003
    grads0, master, m, v = random_inputs(R, n, seed=R * 10 + k, step=6)
    s = new_slabs(grads0, master, m, v, with_acc=True)
    hp = dict(HP10, step=6)
    ref_acc = [np.empty(n, np.float32) for _ in range(R)]
    for j in range(k - 1):
        gj = [t for t in random_inputs(R, n, seed=1000 + j, step=1)[0]]
        capi.cc_accumulate_local(gj, s.acc, n, R, j == 0)
        oracle.accumulate_local([u16(t) for t in gj], ref_acc, first=(j == 0))
    torch.cuda.synchronize()
    for r in range(R):
        assert_bits(f"acc[{r}]", f32(s.acc[r]), ref_acc[r], "f32")
    grads, state, acc = host_copy(s)
    gpu_step(s, hp, bucket_bytes=1 << 20, accum_k=k, use_acc=True)
    torch.cuda.synchronize()
    compare_all(s, state, oracle_step(grads, state, hp, acc=acc))


def test_accumulation_equals_single_step_on_summed_integer_grads():
    R, n, k = 8, 65_536 + 3, 4
    micro = [wl.integer_grads(R, n, micro=j, device=DEV) for j in range(k)]
    _, master, m, v = random_inputs(1, n, seed=77, step=10)
    a = new_slabs(micro[k - 1], master.clone(), m.clone(), v.clone(), with_acc=True)
    for j in range(k - 1):
        capi.cc_accumulate_local(micro[j], a.acc, n, R, j == 0)
    gpu_step(a, HP10, accum_k=k, use_acc=True)
    summed = [sum(micro[j][r].float() for j in range(k)).to(torch.bfloat16)
              for r in range(R)]
    b = new_slabs(summed, master.clone(), m.clone(), v.clone())
    gpu_step(b, HP10)
    torch.cuda.synchronize()
    for x, y in zip([a.master, a.m, a.v] + a.outs, [b.master, b.m, b.v] + b.outs):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32
                           else x.view(torch.int16),
                           y.view(torch.int32) if y.dtype == torch.float32
                           else y.view(torch.int16))


def test_rejects_host_memory_and_short_allocations():
    n = 4096
    s = new_slabs(*random_inputs(2, n, seed=1))
    host = torch.zeros(n)
    with pytest.raises(capi.CCError) as ei:
        capi.cc_fused_dp_step(s.grads, host, s.m, s.v, s.outs, n, 2, 0, **HP1)
    assert ei.value.status == capi.CC_ERR_INVALID
    # All slabs carved from one cudaMalloc allocation, master last, ending
    # exactly at the allocation's end: n elements fit, n + 8 run 32 bytes past.
    import ctypes
    torch.cuda.synchronize()
    rt = ctypes.CDLL("libcudart.so.13")
    n = 1 << 20
    pad = n + 64
    total = 16 * pad + 4 * n
    ptr = ctypes.c_void_p()
    assert rt.cudaMalloc(ctypes.byref(ptr), ctypes.c_size_t(total)) == 0
    try:
        base = ptr.value
        assert rt.cudaMemset(ctypes.c_void_p(base), 0, ctypes.c_size_t(total)) == 0
        bf = [base + 2 * pad * i for i in range(4)]            # grads[0:2], outs[0:2]
        fp = [base + 8 * pad + 4 * pad * i for i in range(2)]  # m, v
        master = base + total - 4 * n
        capi.cc_fused_dp_step(bf[:2], master, fp[0], fp[1], bf[2:], n, 2, 0,
                              stream=0, **HP1)
        assert rt.cudaDeviceSynchronize() == 0
        with pytest.raises(capi.CCError) as ei:
            capi.cc_fused_dp_step(bf[:2], master, fp[0], fp[1], bf[2:], n + 8, 2, 0,
                                  stream=0, **HP1)
        assert ei.value.status == capi.CC_ERR_INVALID
    finally:
        rt.cudaFree(ptr)
    assert "past the end" in ei.value.reason


# ---------------------------------------------------------------------------
# Full workload sizes, sampled elements, benchmark launch configuration
# ---------------------------------------------------------------------------

def sample_indices(n, boundaries, count, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    r = torch.randint(0, n, (count,), generator=g, device=DEV)
    edges = []
    for b in boundaries:
        edges += [b - 9, b - 8, b - 1, b, b + 1, b + 7, b + 8]
    edges += [0, 1, n - 1, n - 2, n - 9]
    e = torch.tensor([x for x in edges if 0 <= x < n], device=DEV, dtype=torch.long)
    return torch.unique(torch.cat([r, e]))


def uniform_cuts(n, bucket_bytes):
    per = max(8, bucket_bytes // 16 * 8)
    return list(range(0, n, per))


def check_sampled(s, hp, idx, bucket_bytes, use_acc=False, accum_k=1):
    grads, state, acc = host_copy(s, idx)
    gpu_step(s, hp, bucket_bytes, accum_k=accum_k, use_acc=use_acc)
    torch.cuda.synchronize()
    outs = oracle_step(grads, state, hp, acc=acc)
    compare_all(s, state, outs, idx=idx)


def test_full_size_bert_large_r8():
    """336M parameters, R=8, 25 MiB buckets, step 10: the benchmark's step."""
    w = wl.bert_large_r8()
    s, offsets, n_slab = planned_workload_slabs(w)
    cuts = uniform_cuts(n_slab, w.bucket_bytes) + offsets
    idx = sample_indices(n_slab, cuts, 1 << 20, seed=1)
    check_sampled(s, hp_of(w), idx, w.bucket_bytes)


def test_full_size_gpt2_slice_r4():
    """2.72e9 parameters (element indices past 2^31), R=4, loss scale 65536."""
    w = wl.gpt2_slice_r4()
    s, offsets, n_slab = planned_workload_slabs(w)
    assert n_slab > (1 << 31)
    cuts = uniform_cuts(n_slab, w.bucket_bytes)[::7] + offsets + [1 << 31, (1 << 31) + 8]
    idx = sample_indices(n_slab, cuts, 1 << 20, seed=2)
    assert (idx > (1 << 31)).sum() > 1000
    check_sampled(s, hp_of(w), idx, w.bucket_bytes)


def test_max_replicas_past_2_31_elements():
    """R = 16, the largest replica count, over 2^31 + 29 elements (about 163 GB
    of slabs): 64-bit element indexing with the most replica pointers, a
    ragged tail, 100 MiB buckets; sampled elements against the oracle."""
    R, n = 16, (1 << 31) + 29
    if torch.cuda.get_device_properties(0).total_memory < 200 * (1 << 30):
        pytest.skip("needs about 180 GB of device memory")
    torch.cuda.empty_cache()
    s = new_slabs(*random_inputs(R, n, seed=91, step=3))
    bb = 100 << 20
    cuts = uniform_cuts(n, bb)[::5] + [1 << 31, (1 << 31) + 8, (1 << 31) + 24]
    idx = sample_indices(n, cuts, 1 << 19, seed=3)
    past = torch.arange(1 << 31, n, device=DEV)          # every element past 2^31
    idx = torch.unique(torch.cat([idx, past]))
    assert int((idx >= (1 << 31)).sum()) == n - (1 << 31)
    check_sampled(s, dict(HP10, step=3), idx, bb)
    del s
    torch.cuda.empty_cache()


def test_full_size_bert_large_accumulation_k4():
    """k=4 on the 336M set at R=8: three local micro-steps, then the reducing
    step, sampled against the oracle run through the same micro-steps."""
    w = wl.bert_large_r8(accum_k=4)
    s, offsets, n_slab = planned_workload_slabs(w, micro=0, with_acc=True)
    idx = sample_indices(n_slab, uniform_cuts(n_slab, w.bucket_bytes) + offsets,
                         1 << 19, seed=3)
    ref_acc = None
    for j in range(w.accum_k - 1):
        if j > 0:
            s.grads = workload_grads(w, offsets, n_slab, micro=j)
        gj = [u16(g[idx]) for g in s.grads]
        if ref_acc is None:
            ref_acc = [np.empty(idx.numel(), np.float32) for _ in range(w.R)]
        capi.cc_accumulate_local(s.grads, s.acc, n_slab, w.R, j == 0)
        oracle.accumulate_local(gj, ref_acc, first=(j == 0))
    torch.cuda.synchronize()
    for r in range(w.R):
        assert_bits(f"acc[{r}]", f32(s.acc[r][idx]), ref_acc[r], "f32")
    s.grads = workload_grads(w, offsets, n_slab, micro=w.accum_k - 1)
    check_sampled(s, hp_of(w), idx, w.bucket_bytes, use_acc=True, accum_k=w.accum_k)


# ---------------------------------------------------------------------------
# CTA budgets (cc_fused_dp_bucket with max_ctas > 0): the wide-CTA kernel,
# and the TMA bulk-copy engine (CC_ENGINE_BULK_COPY)
# ---------------------------------------------------------------------------

ENGINES = {"wide": 0, "bulk_copy": capi.CC_ENGINE_BULK_COPY}


def bulk_step(s, hp, max_ctas, begin=0, end=None, use_acc=False, engine="wide"):
    end = s.n if end is None else end
    capi.cc_fused_dp_bucket_ex(s.grads, s.acc if use_acc else None, s.master, s.m, s.v,
                               s.outs, s.n, s.R, begin, end, max_ctas=max_ctas,
                               arith_flags=ENGINES[engine], **hp)


def check_bulk(s, hp, max_ctas, use_acc=False, label="", engine="wide"):
    grads, state, acc = host_copy(s)
    bulk_step(s, hp, max_ctas, use_acc=use_acc, engine=engine)
    torch.cuda.synchronize()
    outs = oracle_step(grads, state, hp, acc=acc if use_acc else None)
    compare_all(s, state, outs, label=label)
    assert capi.cc_device_status() == 0


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("n", [1, 7, 8, 9, 1023, 1024, 1025, 4096 + 3, 300_007])
@pytest.mark.parametrize("R", [1, 3, 8, 16])
def test_bulk_engine_ragged(R, n, engine):
    s = new_slabs(*random_inputs(R, n, seed=500 + R * 7 + n % 97, step=4))
    check_bulk(s, dict(HP10, step=4), max_ctas=5, label=f"{engine} R={R} n={n} ",
               engine=engine)


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("R", [1, 2, 8, 16])
@pytest.mark.parametrize("max_ctas", [1, 3, 152, 1000])
def test_bulk_engine_accumulators(R, max_ctas, engine):
    """With accumulators the bulk-copy engine's tile shrinks to 512 (R=8)
    or 256 (R=16)."""
    n = 100_003
    s = new_slabs(*random_inputs(R, n, seed=R + max_ctas, step=3), with_acc=True)
    g = torch.Generator(device=DEV)
    g.manual_seed(17)
    for a in s.acc:
        a.copy_(torch.randn(n, generator=g, device=DEV) * 1e-3)
    check_bulk(s, dict(HP10, step=3), max_ctas, use_acc=True, engine=engine)


@pytest.mark.parametrize("engine", list(ENGINES))
def test_bulk_engine_subrange_leaves_the_rest_untouched(engine):
    n = 50_000
    s = new_slabs(*random_inputs(4, n, seed=99, step=2))
    before = [t.clone() for t in (s.master, s.m, s.v)] + [o.clone() for o in s.outs]
    grads, state, _ = host_copy(s)
    b, e = 8 * 1000, 8 * 4000 + 5
    bulk_step(s, dict(HP10, step=2), 7, begin=b, end=e, engine=engine)
    torch.cuda.synchronize()
    sub = [x[b:e].copy() for x in state]
    outs = oracle_step([g_[b:e].copy() for g_ in grads], sub, dict(HP10, step=2))
    idx = torch.arange(b, e, device=DEV)
    compare_all(s, sub, outs, idx=idx)
    after = [s.master, s.m, s.v] + s.outs
    for x, y in zip(after, before):
        xb = x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)
        yb = y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)
        assert torch.equal(xb[:b], yb[:b]) and torch.equal(xb[e:], yb[e:])
    assert capi.cc_device_status() == 0


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("ctas", [48, 96, 152])
def test_bulk_engine_streams_every_sm(ctas, engine):
    """2^25 elements at R = 8 (32,768 bulk-copy tiles, hundreds per CTA) on
    48, 96 and all 152 SMs: the bulk-copy engine's consumer groups run far
    apart in time, and no group may read a stage before its fill has
    landed.  Every element equals the oracle and no pipeline wait runs out.
    The opt-in fast arithmetic on the same inputs gives the same bits as the
    whole-GPU kernel's."""
    R, n = 8, 1 << 25
    capi.cc_device_status(clear=True)
    inputs = random_inputs(R, n, seed=1000 + ctas, step=6)
    s = new_slabs(*[x if isinstance(x, list) else x.clone() for x in inputs])
    grads, state, _ = host_copy(s)
    hp = dict(HP10, step=6)
    bulk_step(s, hp, ctas, engine=engine)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0
    compare_all(s, state, oracle_step(grads, state, hp), label=f"{engine} {ctas} CTAs ")
    a = new_slabs(*[x if isinstance(x, list) else x.clone() for x in inputs])
    b = new_slabs(*[x if isinstance(x, list) else x.clone() for x in inputs])
    for slabs, budget in ((a, ctas), (b, 0)):
        capi.cc_fused_dp_bucket_ex(slabs.grads, None, slabs.master, slabs.m, slabs.v,
                                   slabs.outs, n, R, 0, n, max_ctas=budget,
                                   arith_flags=capi.CC_ARITH_FAST | ENGINES[engine], **hp)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0
    for x, y in zip([a.master, a.m, a.v] + a.outs, [b.master, b.m, b.v] + b.outs):
        bits = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(x.view(bits), y.view(bits))


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("offset", [0, 4])
def test_budget_slabs_aligned_to_16_or_32_bytes(engine, offset):
    """Under a CTA budget the wide form moves the fp32 state in 32-byte
    accesses when master, m and v are 32-byte aligned, and in 16-byte ones
    when they are only 16-byte aligned (offset 4 floats): same bits."""
    R, n = 8, 300_007
    grads, master, m, v = random_inputs(R, n, seed=63 + offset, step=5)

    def place(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=DEV)
        view = buf[offset:offset + t.numel()]
        assert view.data_ptr() % 32 == (16 if offset else 0)
        view.copy_(t)
        return view
    s = new_slabs(grads, place(master), place(m), place(v))
    check_bulk(s, dict(HP10, step=5), max_ctas=11, label=f"{engine} +{4 * offset} B ",
               engine=engine)


@pytest.mark.parametrize("engine", list(ENGINES))
def test_full_size_bert_large_r8_bulk_engine(engine):
    """The 336M R=8 slab in its planned buckets on a 64-SM budget."""
    w = wl.bert_large_r8()
    s, offsets, n_slab = planned_workload_slabs(w)
    _, buckets, _ = oracle.plan_buckets(w.numel(), w.bucket_bytes)
    idx = sample_indices(n_slab, [b for b, _ in buckets] + offsets, 1 << 20, seed=4)
    grads, state, _ = host_copy(s, idx)
    for b, e in buckets:
        capi.cc_fused_dp_bucket_ex(s.grads, None, s.master, s.m, s.v, s.outs, n_slab,
                                   w.R, b, e, max_ctas=64, arith_flags=ENGINES[engine],
                                   **hp_of(w))
    torch.cuda.synchronize()
    compare_all(s, state, oracle_step(grads, state, hp_of(w)), idx=idx)
    assert capi.cc_device_status() == 0


# ---------------------------------------------------------------------------
# The unfused schedule (reduce -> AdamW -> broadcast), for comparison
# ---------------------------------------------------------------------------

def unfused_step(s, hp, bucket_bytes=0):
    per = max(8, bucket_bytes // 16 * 8) if bucket_bytes else s.n
    ws = torch.empty(min(per, s.n), dtype=torch.float32, device=DEV)
    capi.cc_unfused_dp_step(s.grads, s.master, s.m, s.v, s.outs, ws, ws.numel() * 4,
                            s.n, s.R, bucket_bytes, **hp)
    return ws


@pytest.mark.parametrize("R", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("n", [1, 9, 4099, 300_007])
def test_unfused_matches_oracle(R, n):
    s = new_slabs(*random_inputs(R, n, seed=900 + R + n % 13, step=5))
    grads, state, _ = host_copy(s)
    ws = unfused_step(s, dict(HP10, step=5))
    torch.cuda.synchronize()
    compare_all(s, state, oracle_step(grads, state, dict(HP10, step=5)))
    del ws


@pytest.mark.parametrize("bucket_bytes", [16, 4096, 1 << 20])
def test_unfused_equals_fused_bit_for_bit(bucket_bytes):
    n = 3 * 1024 * 1024 + 5
    base = random_inputs(8, n, seed=21, step=10)
    a = new_slabs([g.clone() for g in base[0]], *[t.clone() for t in base[1:]])
    b = new_slabs([g.clone() for g in base[0]], *[t.clone() for t in base[1:]])
    gpu_step(a, HP10, bucket_bytes)
    unfused_step(b, HP10, bucket_bytes)
    torch.cuda.synchronize()
    for x, y in zip([a.master, a.m, a.v] + a.outs, [b.master, b.m, b.v] + b.outs):
        xv = x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)
        yv = y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)
        assert torch.equal(xv, yv)


# ---------------------------------------------------------------------------
# Replica slabs in page-locked host memory (read/written over the host link)
# ---------------------------------------------------------------------------

def test_replica_slabs_in_pinned_host_memory():
    R, n = 4, 1_000_003
    grads, master, m, v = random_inputs(R, n, seed=41, step=3)
    host_grads = [g.cpu().pin_memory() for g in grads]
    s = new_slabs(host_grads, master, m, v)
    s.outs[0] = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    s.outs[2] = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    grads_h, state, _ = host_copy(s)
    gpu_step(s, dict(HP10, step=3), bucket_bytes=1 << 20)
    torch.cuda.synchronize()
    compare_all(s, state, oracle_step(grads_h, state, dict(HP10, step=3)))
    # the unfused schedule with host-resident replicas too
    u = new_slabs(host_grads, *[t.clone() for t in random_inputs(R, n, seed=41, step=3)[1:]])
    u.outs[1] = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    grads_h, state, _ = host_copy(u)
    ws = torch.empty(n, dtype=torch.float32, device=DEV)
    capi.cc_unfused_dp_step(u.grads, u.master, u.m, u.v, u.outs, ws, 4 * n, n, R, 0,
                            **dict(HP10, step=3))
    torch.cuda.synchronize()
    compare_all(u, state, oracle_step(grads_h, state, dict(HP10, step=3)))


def test_pageable_and_short_host_ranges_are_rejected():
    R, n = 2, 1 << 20
    s = new_slabs(*random_inputs(R, n, seed=43, step=1))
    pageable = torch.zeros(n, dtype=torch.bfloat16)
    with pytest.raises(capi.CCError) as ei:
        capi.cc_fused_dp_step([pageable, s.grads[1]], s.master, s.m, s.v, s.outs, n, R, 0,
                              **HP1)
    assert ei.value.status == capi.CC_ERR_INVALID
    big = 1 << 22
    dev = new_slabs(*random_inputs(R, big, seed=44, step=1))
    short = torch.empty(n, dtype=torch.bfloat16).pin_memory()   # 2 MiB of pinned memory
    with pytest.raises(capi.CCError) as ei:
        capi.cc_fused_dp_step(dev.grads, dev.master, dev.m, dev.v, [short, dev.outs[1]],
                              big, R, 0, **HP1)
    assert ei.value.status in (capi.CC_ERR_INVALID, capi.CC_ERR_UNSUPPORTED)
    assert "past the end" in ei.value.reason or "cannot bound" in ei.value.reason


@pytest.mark.parametrize("use_acc", [False, True])
def test_fp32_slabs_aligned_to_16_but_not_32_bytes(use_acc):
    """fp32 slabs 16 bytes past a 32-byte boundary take the 128-bit path."""
    R, n = 3, 100_003
    grads, master, m, v = random_inputs(R, n, seed=61, step=4)
    def offset16(t):
        buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=DEV)
        view = buf[4:]
        assert view.data_ptr() % 32 == 16
        view.copy_(t)
        return view
    s = new_slabs(grads, offset16(master), offset16(m), offset16(v), with_acc=use_acc)
    if use_acc:
        g = torch.Generator(device=DEV)
        g.manual_seed(62)
        s.acc = [offset16(torch.randn(n, generator=g, device=DEV) * 1e-3) for _ in range(R)]
    grads_h, state, acc = host_copy(s)
    gpu_step(s, dict(HP10, step=4), bucket_bytes=64 << 10, accum_k=2 if use_acc else 1,
             use_acc=use_acc)
    torch.cuda.synchronize()
    compare_all(s, state, oracle_step(grads_h, state, dict(HP10, step=4), acc=acc))


# ---------------------------------------------------------------------------
# The ready-driven scheduler (cc_overlap_bench) steps every bucket exactly once
# per arm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("max_ctas,prio,comm_sms,budget,algo,use_acc,flags", [
    (0, 0, 0, 0, 0, False, 0), (0, 2, 0, 0, 0, False, 0), (24, 1, 0, 0, 0, False, 0),
    (0, 2, 48, 0, 0, False, 0), (8, 2, 0, 3, 0, False, 0), (0, 2, 0, 0, 1, False, 0),
    (24, 2, 0, 0, 0, False, 2), (0, 2, 0, 0, 0, True, 0), (16, 2, 0, 0, 0, True, 0),
    (16, 2, 0, 0, 0, True, 2)])
def test_overlap_bench_applies_every_bucket_once_per_arm(max_ctas, prio, comm_sms, budget,
                                                         algo, use_acc, flags):
    """With warmup 0 and one iteration the four arms step the slabs three
    times (buckets alone, overlapped, sequential; the backward-only arm does
    not step): the result must be three oracle steps, bit for bit.  Also the
    reducing step with accumulators (read, not written, by each arm), and
    budgets on the bulk-copy engine (flags 2)."""
    t = wl.bert_large_tensors(layers=4, hidden=256, ffn=1024, vocab=997, positions=64)
    numel = [x[1] for x in t]
    layer_of = [x[2] for x in t]
    offsets, buckets, n_slab = oracle.plan_buckets(numel, 96 * 1024)
    ready = oracle.bucket_ready_layers(numel, layer_of, offsets, buckets)
    assert len(buckets) >= 8 and len(set(ready)) == 4
    R = 4
    s = new_slabs(*random_inputs(R, n_slab, seed=71, step=5), with_acc=use_acc)
    if use_acc:
        gen = torch.Generator(device=DEV)
        gen.manual_seed(72)
        for a in s.acc:
            a.copy_(torch.randn(n_slab, generator=gen, device=DEV) * 1e-3)
    grads, state, acc = host_copy(s)
    hp = dict(HP10, step=5)
    M = N = K = 256
    A = torch.randn(M * K, device=DEV).to(torch.bfloat16)
    B = torch.randn(K * N, device=DEV).to(torch.bfloat16)
    C = torch.empty(M * N, dtype=torch.bfloat16, device=DEV)
    r = capi.cc_overlap_bench(grads=s.grads, master=s.master, m=s.m, v=s.v,
                              params_out=s.outs, n=n_slab, R=R, buckets=buckets,
                              ready_layers=ready, num_layers=4, gemms_per_layer=2,
                              gemm_m=M, gemm_n=N, gemm_k=K, gemm_a=A, gemm_b=B,
                              gemm_c=C, warmup=0, iters=1, max_ctas=max_ctas,
                              stream_priority=prio, comm_sms=comm_sms,
                              budget_buckets=budget, gemm_algo=algo,
                              acc=s.acc if use_acc else None, arith_flags=flags, **hp)
    assert r["num_buckets"] == len(buckets) and r["t_bwd_ms"] > 0
    assert (r["gemm_algos"] >= 1) == (algo > 0)
    if comm_sms:   # a spatial partition: green contexts on disjoint SM sets
        assert r["comm_sms"] >= comm_sms and r["compute_sms"] > 0
    torch.cuda.synchronize()
    for _ in range(3):
        outs = oracle_step(grads, state, hp, acc=acc if use_acc else None)
    compare_all(s, state, outs)
    assert capi.cc_device_status() == 0


def test_overlap_bench_rejects_bad_schedules():
    s = new_slabs(*random_inputs(2, 4096, seed=72, step=1))
    A = torch.empty(64 * 64, dtype=torch.bfloat16, device=DEV)
    base = dict(grads=s.grads, master=s.master, m=s.m, v=s.v, params_out=s.outs,
                n=4096, R=2, num_layers=2, gemms_per_layer=1, gemm_m=64, gemm_n=64,
                gemm_k=64, gemm_a=A, gemm_b=A, gemm_c=A, warmup=0, iters=1, **HP1)
    for buckets, ready, status in (([(0, 4096)], [2], capi.CC_ERR_INVALID),   # no layer 2
                                   ([(4, 4096)], [0], capi.CC_ERR_MISALIGNED),
                                   ([(0, 5000)], [0], capi.CC_ERR_INVALID)):
        with pytest.raises(capi.CCError) as ei:
            capi.cc_overlap_bench(buckets=buckets, ready_layers=ready, **base)
        assert ei.value.status == status
    for kw in (dict(gemm_algo=-1), dict(gemm_algo=10_000), dict(budget_buckets=-1)):
        with pytest.raises(capi.CCError) as ei:
            capi.cc_overlap_bench(buckets=[(0, 4096)], ready_layers=[0], **kw, **base)
        assert ei.value.status == capi.CC_ERR_INVALID


@pytest.mark.parametrize("rank,use_acc", [(-1, False), (1, False), (-1, True)])
def test_tune_bucket_bytes_measures_every_candidate(rank, use_acc):
    """The bucket-size tuner times each candidate cap's launch list with the
    overlap bench and returns the cap whose overlapped step is shortest.
    With warmup 0 and one iteration every candidate steps its buckets (or
    the rank's shards of them) three times: the slabs must equal the oracle
    stepping each element three times per candidate whose launch list covers
    it, bucket lists taken from the oracle's own planner."""
    t = wl.bert_large_tensors(layers=4, hidden=256, ffn=1024, vocab=997, positions=64)
    numel = [x[1] for x in t]
    layer_of = [x[2] for x in t]
    caps = [64 * 1024, 256 * 1024, 0]
    R = 3
    _, _, n_slab = oracle.plan_buckets(numel, 0)
    s = new_slabs(*random_inputs(R, n_slab, seed=73, step=5), with_acc=use_acc)
    if use_acc:                     # the reducing step: accumulators read by every arm
        gen = torch.Generator(device=DEV)
        gen.manual_seed(74)
        for a in s.acc:
            a.copy_(torch.randn(n_slab, generator=gen, device=DEV) * 1e-3)
    grads, state, acc = host_copy(s)
    hp = dict(HP10, step=5)
    M = N = K = 256
    A = torch.randn(M * K, device=DEV).to(torch.bfloat16)
    B = torch.randn(K * N, device=DEV).to(torch.bfloat16)
    C = torch.empty(M * N, dtype=torch.bfloat16, device=DEV)
    best, results = capi.cc_tune_bucket_bytes(
        numel=numel, layer_of=layer_of, candidates=caps, rank=rank, grads=s.grads,
        master=s.master, m=s.m, v=s.v, params_out=s.outs, n=n_slab, R=R, num_layers=4,
        gemms_per_layer=2, gemm_m=M, gemm_n=N, gemm_k=K, gemm_a=A, gemm_b=B, gemm_c=C,
        warmup=0, iters=1, acc=s.acc if use_acc else None, **hp)
    assert len(results) == len(caps)
    step_ms = [r["t_step_overlap_ms"] for r in results]
    assert best == caps[min(range(len(caps)), key=lambda i: (step_ms[i], i))]
    outs = [np.full(n_slab, 0xFFFF, dtype=np.uint16) for _ in range(R)]
    for cap, res in zip(caps, results):
        _, buckets, _ = oracle.plan_buckets(numel, cap)
        if rank >= 0:
            shards = oracle.shard_plan(buckets, R)[0]
            buckets = [row[rank] for row in shards if row[rank][1] > row[rank][0]]
        assert res["num_buckets"] == len(buckets)
        idx = np.concatenate([np.arange(lo, hi) for lo, hi in buckets])
        sub = [a[idx].copy() for a in state]
        sub_grads = [g[idx] for g in grads]
        sub_acc = [a[idx].copy() for a in acc] if use_acc else None
        for _ in range(3):
            sub_outs = oracle.fused_dp_step(sub_grads, *sub, acc=sub_acc, **hp)
        for a, b in zip(state, sub):
            a[idx] = b
        for o, b in zip(outs, sub_outs):
            o[idx] = b
    torch.cuda.synchronize()
    compare_all(s, state, outs)
    assert capi.cc_device_status() == 0


# ---------------------------------------------------------------------------
# The tensor-parallel MatMul-then-AllReduce
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("R", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("n", [1, 9, 4099, 262_147])
def test_tp_allreduce_matches_oracle(R, n):
    g = torch.Generator(device=DEV)
    g.manual_seed(R * 1000 + n % 1000)
    parts = [torch.randn(n, generator=g, device=DEV) * 10 for _ in range(R)]
    if n > 100:   # a few special values
        specials = torch.tensor([float("inf"), -float("inf"), float("nan"), 0.0, -0.0,
                                 3e38, 1e-40], device=DEV)
        parts[0][:7] = specials
    outs = [torch.full((n,), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            for _ in range(R)]
    capi.cc_tp_allreduce(parts, outs, n, R)
    torch.cuda.synchronize()
    ref = oracle.tp_allreduce([f32(p).copy() for p in parts])
    for r in range(R):
        assert_bits(f"out[{r}]", u16(outs[r]), ref[r], "bf16")


@pytest.mark.parametrize("batched", [False, True])
def test_tp_overlap_bench_outputs(batched):
    R, m, n, k, chunks = 4, 256, 128, 512, 4
    kr = k // R
    g = torch.Generator(device=DEV)
    g.manual_seed(81)
    if batched:   # one buffer per operand, R equal shards
        x = list(torch.randn(R * m * kr, generator=g, device=DEV).to(torch.bfloat16).view(R, -1))
        w = list((torch.randn(R * kr * n, generator=g, device=DEV) * 0.05)
                 .to(torch.bfloat16).view(R, -1))
        partials = list(torch.empty(R, m * n, device=DEV))
    else:
        x = [(torch.randn(m * kr, generator=g, device=DEV)).to(torch.bfloat16)
             for _ in range(R)]
        w = [(torch.randn(kr * n, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
             for _ in range(R)]
        partials = [torch.empty(m * n, device=DEV) for _ in range(R)]
    outs = [torch.empty(m * n, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    t = capi.cc_tp_overlap_bench(R=R, m=m, n=n, k=k, chunks=chunks, x=x, w=w,
                                 partials=partials, out=outs, warmup=0, iters=1,
                                 stream_priority=2)
    assert all(v > 0 for v in t.values())
    torch.cuda.synchronize()
    P = [f32(p).copy() for p in partials]
    # the AllReduce of what the GEMMs produced: bit for bit
    ref = oracle.tp_allreduce(P)
    for r in range(R):
        assert_bits(f"out[{r}]", u16(outs[r]), ref[r], "bf16")
    # the GEMMs (cuBLAS, fp32 accumulation) against a float64 matmul
    for r in range(R):
        X = x[r].float().cpu().numpy().astype(np.float64).reshape(m, kr)
        W = w[r].float().cpu().numpy().astype(np.float64).reshape(kr, n)
        exact = X @ W
        bound = kr * 2.0 ** -23 * (np.abs(X) @ np.abs(W)) + 1e-30
        assert np.all(np.abs(P[r].reshape(m, n) - exact) <= bound)


def test_tp_overlap_bench_rejects_bad_shapes():
    R = 2
    x = [torch.empty(64 * 32, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    w = [torch.empty(32 * 64, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    p = [torch.empty(64 * 64, device=DEV) for _ in range(R)]
    o = [torch.empty(64 * 64, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    for kw, status in ((dict(k=63, chunks=1), capi.CC_ERR_INVALID),
                       (dict(k=64, chunks=3), capi.CC_ERR_INVALID),
                       (dict(k=36, chunks=1), capi.CC_ERR_MISALIGNED)):
        with pytest.raises(capi.CCError) as ei:
            capi.cc_tp_overlap_bench(R=R, m=64, n=64, x=x, w=w, partials=p, out=o,
                                     warmup=0, iters=1, **kw)
        assert ei.value.status == status


# ---------------------------------------------------------------------------
# Error propagation: an injected launch failure partway through a step
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("schedule", ["fused", "unfused"])
def test_injected_launch_failure_leaves_earlier_buckets_applied(schedule):
    """Failure after 3 of 8 buckets: CC_ERR_CUDA with the reason; buckets 0-2
    were stepped, 3-7 untouched; the next call works normally."""
    R, n, bb = 2, 8 * 4096, 8192          # 4096-element buckets, 8 of them
    s = new_slabs(*random_inputs(R, n, seed=91, step=2))
    before = [f32(t).copy() for t in (s.master, s.m, s.v)]
    grads, state, _ = host_copy(s)
    hp = dict(HP10, step=2)
    ws = torch.empty(4096, dtype=torch.float32, device=DEV)

    def step():
        if schedule == "fused":
            capi.cc_fused_dp_step(s.grads, s.master, s.m, s.v, s.outs, n, R, bb, **hp)
        else:
            capi.cc_unfused_dp_step(s.grads, s.master, s.m, s.v, s.outs, ws, 4 * 4096,
                                    n, R, bb, **hp)

    capi.cc_inject_launch_failure(3)
    with pytest.raises(capi.CCError) as ei:
        step()
    assert ei.value.status == capi.CC_ERR_CUDA and "injected" in ei.value.reason
    torch.cuda.synchronize()
    outs = oracle_step(grads, state, hp)
    done, rest = 3 * 4096, slice(3 * 4096, n)
    for name, t, ref, old in zip(("master", "m", "v"), (s.master, s.m, s.v), state, before):
        got = f32(t)
        assert_bits(name, got[:done], ref[:done], "f32")
        assert_bits(name + " untouched", got[rest], old[rest], "f32")
    step()                                  # disarmed: a normal full step
    torch.cuda.synchronize()
    capi.cc_inject_launch_failure(-1)
