"""The C-ABI library on the host: it loads, exports every declared symbol,
plans buckets exactly like the oracle, and rejects bad arguments before any
launch.  No kernel runs here (no GPU needed)."""
import os
import random
import re

import pytest

import oracle
from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gradient_reduce_optimizer_gb300 import workloads as wl
from plan_fixtures import load_cases

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cc_dp.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    return capi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\bCC_API\b[^;(]*?\b(cc_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 10
    L = capi.lib()
    for name in names:
        assert hasattr(L, name), name
    # and the binding covers every one of them under the same name
    for name in names:
        assert callable(getattr(capi, name)), name


def test_header_is_plain_c_and_links(tmp_path):
    """include/cc_dp.h compiles as C99 with warnings as errors, and a C
    program that calls the ABI links against the library and runs without
    a GPU (the planner is host-only)."""
    src = tmp_path / "use_abi.c"
    src.write_text(r"""
#include <stdio.h>
#include "cc_dp.h"
int main(void) {
    size_t numel[3] = {100, 7, 300};
    size_t offsets[3], begin[4], end[4], n_padded = 0;
    int count = 0;
    int st = cc_plan_buckets(numel, 3, 512, offsets, begin, end, 4, &count, &n_padded);
    cc_overlap_cfg cfg = {0};
    (void)cfg;
    printf("%s %d %zu %zu\n", cc_status_string(st), count, n_padded, offsets[2]);
    return st == CC_OK ? 0 : 1;
}
""")
    exe = tmp_path / "use_abi"
    lib_dir = os.path.dirname(capi.LIBRARY)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER),
           str(src), "-o", str(exe), f"-L{lib_dir}", "-lcc_dp", f"-Wl,-rpath,{lib_dir}"]
    import subprocess
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    # 300 -> [0, 304), 7 -> [304, 312), 100 -> [312, 416): buckets close at >= 512 B
    assert r.stdout.split() == ["CC_OK", "2", "416", "0"]


def test_status_strings():
    assert capi.cc_status_string(0) == "CC_OK"
    for code, name in [(-1, "CC_ERR_INVALID"), (-2, "CC_ERR_ALIAS"),
                       (-3, "CC_ERR_MISALIGNED"), (-4, "CC_ERR_CUDA"),
                       (-5, "CC_ERR_UNSUPPORTED"), (-6, "CC_ERR_CAPACITY")]:
        assert capi.cc_status_string(code) == name
    assert capi.cc_status_string(-99) == "CC_ERR_UNKNOWN"


# ---------------------------------------------------------------------------
# Planner: bit-exact against the oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_planner_hand_counted(case):
    offsets, buckets, n_pad = capi.cc_plan_buckets(case["numel"],
                                                   case["bucket_bytes"])
    assert (offsets, buckets, n_pad) == (case["offsets"], case["buckets"],
                                         case["n_padded"])
    assert capi.cc_bucket_ready_layers(case["numel"], case["layer"], offsets,
                                       buckets) == case["ready"]


@pytest.mark.parametrize("tensors", ["bert", "gpt2"])
@pytest.mark.parametrize("mib", [0, 1, 4, 25, 100, 500])
def test_planner_model_lists_match_oracle(tensors, mib):
    t = wl.bert_large_tensors() if tensors == "bert" else wl.gpt2_slice_tensors()
    numel = [x[1] for x in t]
    layer_of = [x[2] for x in t]
    mine = capi.cc_plan_buckets(numel, mib * wl.MiB)
    ref = oracle.plan_buckets(numel, mib * wl.MiB)
    assert mine == ref
    assert (capi.cc_bucket_ready_layers(numel, layer_of, mine[0], mine[1]) ==
            oracle.bucket_ready_layers(numel, layer_of, ref[0], ref[1]))


@pytest.mark.parametrize("seed", range(40))
def test_planner_random_lists_match_oracle(seed):
    rnd = random.Random(1000 + seed)
    T = rnd.randint(1, 80)
    numel = [rnd.choice([0, 1, 3, 8, 15, 16, 17, 255, 4096, 99991])
             for _ in range(T)]
    if sum(numel) == 0:
        numel[-1] = 5
    layer_of = sorted(rnd.randint(0, 20) for _ in range(T))
    cap = rnd.choice([0, 1, 16, 17, 512, 8192, 1 << 20])
    mine = capi.cc_plan_buckets(numel, cap)
    ref = oracle.plan_buckets(numel, cap)
    assert mine == ref
    assert (capi.cc_bucket_ready_layers(numel, layer_of, mine[0], mine[1]) ==
            oracle.bucket_ready_layers(numel, layer_of, ref[0], ref[1]))


def test_planner_capacity_and_bad_input():
    L = capi.lib()
    import ctypes
    numel = (ctypes.c_size_t * 3)(10, 20, 30)
    offs = (ctypes.c_size_t * 3)()
    b = (ctypes.c_size_t * 1)()
    e = (ctypes.c_size_t * 1)()
    cnt = ctypes.c_int(0)
    st = L.cc_plan_buckets(numel, 3, 16, offs, b, e, 1, ctypes.byref(cnt), None)
    assert st == capi.CC_ERR_CAPACITY and cnt.value == 3
    assert L.cc_plan_buckets(numel, 0, 16, offs, b, e, 1, ctypes.byref(cnt),
                             None) == capi.CC_ERR_INVALID
    assert L.cc_plan_buckets(numel, 3, 16, offs, None, None, 2,
                             ctypes.byref(cnt), None) == capi.CC_ERR_INVALID


# ---------------------------------------------------------------------------
# Argument validation (returns before touching any device)
# ---------------------------------------------------------------------------

ADAM = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
            step=1, grad_scale=1.0)
MB = 1 << 20


def fake_slabs(R, n, base=1 << 40):
    """Aligned, non-overlapping fake addresses (never dereferenced)."""
    stride = ((4 * n + 4095) // 4096 + 1) * 4096
    addr = iter(range(base, base + stride * (3 * R + 8), stride))
    grads = [next(addr) for _ in range(R)]
    outs = [next(addr) for _ in range(R)]
    acc = [next(addr) for _ in range(R)]
    master, m, v = next(addr), next(addr), next(addr)
    return grads, acc, master, m, v, outs


def step_status(grads, master, m, v, outs, n, R, **kw):
    args = dict(ADAM)
    args.update(kw)
    accum_k = args.pop("accum_k", 1)
    try:
        capi.cc_fused_dp_step(grads, master, m, v, outs, n, R, 0,
                              accum_k=accum_k, stream=0, **args)
        return capi.CC_OK
    except capi.CCError as err:
        return err.status


@pytest.mark.parametrize("kw", [
    dict(lr=-1.0), dict(lr=float("nan")), dict(beta1=1.0), dict(beta1=-0.1),
    dict(beta2=1.0), dict(eps=-1e-8), dict(eps=float("inf")),
    dict(weight_decay=-0.1), dict(step=0), dict(grad_scale=0.0),
    dict(grad_scale=float("inf")), dict(grad_scale=1e-45), dict(accum_k=2),
    dict(accum_k=0),
])
def test_rejects_bad_hyper_parameters(kw):
    g, _, p, m, v, o = fake_slabs(2, 64)
    assert step_status(g, p, m, v, o, 64, 2, **kw) == capi.CC_ERR_INVALID


@pytest.mark.parametrize("R", [0, 17, -1])
def test_rejects_bad_replica_count(R):
    g, _, p, m, v, o = fake_slabs(16, 64)
    assert step_status(g, p, m, v, o, 64, R) == capi.CC_ERR_INVALID


def test_n_zero_is_a_no_op():
    assert step_status([0, 0], 0, 0, 0, [0, 0], 0, 2) == capi.CC_OK


def test_rejects_null_and_misaligned_and_aliased():
    g, _, p, m, v, o = fake_slabs(3, 1000)
    assert step_status(g, 0, m, v, o, 1000, 3) == capi.CC_ERR_INVALID
    assert step_status([g[0], 0, g[2]], p, m, v, o, 1000, 3) == capi.CC_ERR_INVALID
    assert step_status(g, p + 8, m, v, o, 1000, 3) == capi.CC_ERR_MISALIGNED
    assert step_status(g, p, m, v, [o[0], o[1] + 2, o[2]], 1000, 3) == \
        capi.CC_ERR_MISALIGNED
    # a parameter slab overlapping a gradient slab
    assert step_status(g, p, m, v, [o[0], g[1] + 1024, o[2]], 1000, 3) == \
        capi.CC_ERR_ALIAS
    # m overlapping master
    assert step_status(g, p, p + 16, v, o, 1000, 3) == capi.CC_ERR_ALIAS
    # two output replicas sharing memory
    assert step_status(g, p, m, v, [o[0], o[0], o[2]], 1000, 3) == capi.CC_ERR_ALIAS
    # read-only gradient slabs may alias each other
    st = step_status([g[0], g[0], g[0]], p, m, v, o, 1000, 3)
    assert st in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID)  # no device / fake ptr


def test_fake_pointers_never_reach_a_launch():
    """Valid-looking fake addresses fail at the device checks: without a GPU
    as CC_ERR_UNSUPPORTED, with one as CC_ERR_INVALID (not allocated)."""
    g, acc, p, m, v, o = fake_slabs(4, 4096)
    assert step_status(g, p, m, v, o, 4096, 4) in (capi.CC_ERR_UNSUPPORTED,
                                                    capi.CC_ERR_INVALID)


def test_bucket_and_accumulate_validation():
    g, acc, p, m, v, o = fake_slabs(2, 1000)
    with pytest.raises(capi.CCError) as ei:
        capi.cc_fused_dp_bucket(g, None, p, m, v, o, 1000, 2, 4, 100, stream=0,
                                **ADAM)
    assert ei.value.status == capi.CC_ERR_MISALIGNED
    with pytest.raises(capi.CCError) as ei:
        capi.cc_fused_dp_bucket(g, None, p, m, v, o, 1000, 2, 8, 1001, stream=0,
                                **ADAM)
    assert ei.value.status == capi.CC_ERR_INVALID
    with pytest.raises(capi.CCError) as ei:
        capi.cc_fused_dp_step_accum(g, None, p, m, v, o, 1000, 2, 0, accum_k=4,
                                    stream=0, **ADAM)
    assert ei.value.status == capi.CC_ERR_INVALID
    with pytest.raises(capi.CCError) as ei:
        capi.cc_accumulate_local(g, [acc[0], g[1]], 1000, 2, True, stream=0)
    assert ei.value.status == capi.CC_ERR_ALIAS
    with pytest.raises(capi.CCError) as ei:
        capi.cc_accumulate_local(g, [acc[0], acc[1] + 4], 1000, 2, True, stream=0)
    assert ei.value.status == capi.CC_ERR_MISALIGNED


def test_shard_validation():
    g, acc, p, m, v, o = fake_slabs(2, 1000)

    def status(begin, end, grads=g, outs=o, state=(p, m, v), accs=None, **kw):
        hp = dict(ADAM)
        hp.update(kw)
        try:
            capi.cc_fused_dp_shard(grads, accs, *state, outs, 1000, 2, begin, end, 0,
                                   stream=0, **hp)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status

    assert status(4, 100) == capi.CC_ERR_MISALIGNED
    assert status(8, 1001) == capi.CC_ERR_INVALID
    assert status(16, 8) == capi.CC_ERR_INVALID
    # an empty shard checks the hyper-parameters and touches no pointer
    assert status(64, 64, grads=None, outs=None, state=(0, 0, 0)) == capi.CC_OK
    assert status(64, 64, grads=None, outs=None, state=(0, 0, 0), lr=-1.0) == \
        capi.CC_ERR_INVALID
    assert status(8, 100, grads=[g[0], 0]) == capi.CC_ERR_INVALID
    assert status(8, 100, accs=[acc[0], None]) == capi.CC_ERR_INVALID
    # the shard's state written over a gradient slab's shard range
    assert status(8, 100, state=(g[1] + 16, m, v)) == capi.CC_ERR_ALIAS
    # master is shard-sized: m may start right after a 92-element master
    assert status(8, 100, state=(p, p + 4 * 92, v)) in (capi.CC_ERR_UNSUPPORTED,
                                                        capi.CC_ERR_INVALID)
    assert status(8, 100, state=(p, p + 4 * 88, v)) == capi.CC_ERR_ALIAS
    assert status(8, 100, state=(p + 4, m, v)) == capi.CC_ERR_MISALIGNED


def test_unfused_workspace_validation():
    g, acc, p, m, v, o = fake_slabs(2, 1000)
    ws = acc[0]                         # an unused, aligned fake range
    kw = dict(ADAM, stream=0)
    def status(workspace, nbytes, bucket_bytes=0):
        try:
            capi.cc_unfused_dp_step(g, p, m, v, o, workspace, nbytes, 1000, 2,
                                    bucket_bytes, **kw)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status
    assert status(0, 4000) == capi.CC_ERR_INVALID
    assert status(ws + 4, 4000) == capi.CC_ERR_MISALIGNED
    assert status(ws, 3999) == capi.CC_ERR_INVALID          # 4 * 1000 needed
    assert status(ws, 64, bucket_bytes=32) in (capi.CC_ERR_UNSUPPORTED,
                                              capi.CC_ERR_INVALID)  # 16 elements: enough
    assert status(p + 1024, 4000) == capi.CC_ERR_ALIAS      # inside master
    assert status(o[1], 4000) == capi.CC_ERR_ALIAS          # a parameter slab
    assert status(ws, 4000) in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID)


def test_tp_allreduce_validation():
    g, acc, p, m, v, o = fake_slabs(3, 1000)
    def status(parts, outs, R=3):
        try:
            capi.cc_tp_allreduce(parts, outs, 1000, R, stream=0)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status
    assert status(acc, o, R=0) == capi.CC_ERR_INVALID
    assert status(acc, [o[0], o[1] + 2, o[2]]) == capi.CC_ERR_MISALIGNED
    assert status(acc, [o[0], acc[1], o[2]]) == capi.CC_ERR_ALIAS    # writes over a partial
    assert status(acc, [o[0], o[0], o[2]]) == capi.CC_ERR_ALIAS      # two outputs share memory
    assert status(acc, o) in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID)


def test_inject_launch_failure_arguments():
    capi.cc_inject_launch_failure(5)
    capi.cc_inject_launch_failure(-1)
    with pytest.raises(capi.CCError) as ei:
        capi.cc_inject_launch_failure(-2)
    assert ei.value.status == capi.CC_ERR_INVALID


def test_binding_constants_match_the_header():
    """Every numeric #define of include/cc_dp.h that the binding mirrors has
    the header's value (the header is the source of truth)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    defines = {k: v for k, v in re.findall(r"#define\s+(CC_\w+)\s+(\([^\n]*\)|\d+)", text)}
    assert set(defines) >= {"CC_MAX_R", "CC_PAD_ELEMS", "CC_NOALLOC_SCRATCH_ELEMS"}
    for name, expr in defines.items():
        value = eval(expr.replace("u", ""))          # plain integer arithmetic
        assert getattr(capi, name) == value, name


def test_noalloc_size_refusals_name_their_cause():
    """The allocation-free entry point refuses, before looking at any pointer,
    a bucket larger than its fixed scratch, and says whether n or
    bucket_bytes set the bucket's size; 15 bytes past 32 MiB still floor to
    an accepted bucket."""
    cap = capi.CC_NOALLOC_SCRATCH_ELEMS
    g, acc, p, m, v, o = fake_slabs(2, cap + 1000)
    def reason(n, bucket_bytes):
        try:
            capi.cc_unfused_dp_step_noalloc(g, p, m, v, o, n, 2, bucket_bytes,
                                            stream=0, **ADAM)
            return "ok"
        except capi.CCError as err:
            return err.reason if err.status == capi.CC_ERR_INVALID else "other"
    assert "n=" in reason(cap + 8, 0) and "scratch" in reason(cap + 8, 0)
    assert "bucket_bytes=" in reason(cap + 1000, 2 * cap + 16)
    # accepted sizes go on to pointer validation (fake pointers: refused there)
    for bb in (2 * cap, 2 * cap + 15):
        r = reason(cap + 1000, bb)
        assert "scratch" not in r, r


def test_inject_bulk_stall_arguments():
    with pytest.raises(capi.CCError):
        capi.cc_inject_bulk_stall(-2, 100)
    with pytest.raises(capi.CCError):
        capi.cc_inject_bulk_stall(0, 0)
    with pytest.raises(capi.CCError):
        capi.cc_inject_bulk_stall(0, 2000000)
    capi.cc_inject_bulk_stall(-1, 0)             # disarm


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("mib", [1, 25, 500])
def test_shard_plan_matches_oracle(world, mib):
    w = wl.bert_large_r8()
    _, buckets, _ = capi.cc_plan_buckets(w.numel(), mib << 20)
    assert capi.cc_shard_plan(buckets, world) == tuple(oracle.shard_plan(buckets, world))


def test_shard_plan_random_and_ragged_match_oracle():
    rng = random.Random(17)
    for _ in range(60):
        numel = [rng.choice([1, 7, 8, 9, 64, 1000, 4099]) for _ in range(rng.randint(1, 12))]
        _, buckets, n = capi.cc_plan_buckets(numel, rng.choice([0, 16, 64, 4096]))
        if rng.random() < 0.5:              # a ragged last bucket, as a uniform cut makes
            b, e = buckets[-1]
            buckets[-1] = (b, e - rng.randint(0, 7))
        world = rng.randint(1, 9)
        assert capi.cc_shard_plan(buckets, world) == tuple(oracle.shard_plan(buckets, world))


def test_shard_plan_rejects_bad_input():
    with pytest.raises(capi.CCError) as ei:
        capi.cc_shard_plan([(0, 16)], 0)
    assert ei.value.status == capi.CC_ERR_INVALID
    with pytest.raises(capi.CCError) as ei:
        capi.cc_shard_plan([(4, 16)], 2)
    assert ei.value.status == capi.CC_ERR_MISALIGNED
    with pytest.raises(capi.CCError) as ei:
        capi.cc_shard_plan([(16, 32), (0, 8)], 2)
    assert ei.value.status == capi.CC_ERR_INVALID


def test_rank_step_validation():
    g, acc, p, m, v, o = fake_slabs(3, 1000)
    def status(**kw):
        args = dict(grad_slices=g, master=p, m=m, v=v, param_out=o[0], length=1000, R=3)
        args.update(kw)
        try:
            capi.cc_fused_dp_rank_step(args.pop("grad_slices"), args.pop("master"),
                                       args.pop("m"), args.pop("v"), args.pop("param_out"),
                                       args.pop("length"), args.pop("R"), stream=0, **ADAM)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status
    assert status(R=0) == capi.CC_ERR_INVALID
    assert status(R=17) == capi.CC_ERR_INVALID
    assert status(length=0) == capi.CC_OK                      # no-op, pointers unexamined
    assert status(param_out=o[0] + 2) == capi.CC_ERR_MISALIGNED
    assert status(param_out=g[1]) == capi.CC_ERR_ALIAS         # writes over a gradient slice
    assert status(m=p) == capi.CC_ERR_ALIAS
    assert status(grad_slices=[g[0], g[0], g[0]]) in (capi.CC_ERR_UNSUPPORTED,
                                                      capi.CC_ERR_INVALID)   # aliasing reads ok
    assert status() in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID)


def test_tune_bucket_bytes_refuses_before_measuring():
    """The bucket-size tuner plans and checks every candidate on the host
    before its first measurement: bad tensor lists, candidate counts, ranks,
    slab lengths and ready layers are refused with no device call."""
    numel = [1000, 3000, 500, 7000]
    layer_of = [0, 1, 2, 3]
    _, _, n = capi.cc_plan_buckets(numel, 0)
    R = 2
    g, acc, p, m, v, o = fake_slabs(R, n)
    kw = dict(grads=g, master=p, m=m, v=v, params_out=o, n=n, R=R, num_layers=4,
              gemms_per_layer=1, gemm_m=64, gemm_n=64, gemm_k=64, gemm_a=None, gemm_b=None,
              gemm_c=None, **ADAM)

    def status(**over):
        args = dict(kw, numel=numel, layer_of=layer_of, candidates=[4096, 16384])
        args.update(over)
        try:
            capi.cc_tune_bucket_bytes(**args)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status
    assert status(numel=[], layer_of=[]) == capi.CC_ERR_INVALID
    assert status(candidates=[]) == capi.CC_ERR_INVALID
    assert status(candidates=[4096] * (capi.CC_TUNE_MAX_CANDIDATES + 1)) == capi.CC_ERR_INVALID
    assert status(n=n + 8) == capi.CC_ERR_INVALID              # not this tensor list's slab
    assert status(rank=R) == capi.CC_ERR_INVALID
    assert status(rank=-2) == capi.CC_ERR_INVALID
    assert status(num_layers=3) == capi.CC_ERR_INVALID         # a bucket ready after layer 3
    # a one-unit slab gives rank 0 of 2 no elements
    _, _, n8 = capi.cc_plan_buckets([8], 0)
    assert status(numel=[8], layer_of=[0], n=n8, rank=0) == capi.CC_ERR_INVALID
    # well-formed: planning passes and the first measurement refuses the fake
    # (host) addresses
    assert status() in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID, capi.CC_ERR_CUDA)
    assert status(candidates=None, rank=1) in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID,
                                               capi.CC_ERR_CUDA)


def test_tp_matmul_allreduce_refuses_before_any_launch():
    """The fused tensor-parallel entry points check shapes, budgets, NULLs,
    alignment and aliasing (the workspace included) on the host before any
    device call."""
    R, m, n, k = 2, 256, 256, 256
    kr = k // R
    base = 1 << 40
    stride = 1 << 22                       # fake, aligned, disjoint device addresses
    addrs = iter(range(base, base + 64 * stride, stride))
    x = [next(addrs) for _ in range(R)]
    w = [next(addrs) for _ in range(R)]
    outs = [next(addrs) for _ in range(R)]
    ws = next(addrs)

    def ex(**over):
        args = dict(x=x, w=w, out=outs, partials=None, m=m, n=n, k=k, R=R, workspace=ws,
                    workspace_bytes=1 << 20, max_ctas=0)
        args.update(over)
        try:
            capi.cc_tp_matmul_allreduce_ex(args.pop("x"), args.pop("w"), args.pop("out"),
                                           args.pop("partials"), args.pop("m"), args.pop("n"),
                                           args.pop("k"), args.pop("R"), stream=0, **args)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status

    def query(**over):
        args = dict(m=m, n=n, k=k, R=R, max_ctas=0)
        args.update(over)
        try:
            capi.cc_tp_matmul_allreduce_workspace(**args)
            return capi.CC_OK
        except capi.CCError as err:
            return err.status

    for bad in (dict(m=m + 8), dict(n=n + 16), dict(k=k + 1), dict(k=96), dict(R=0),
                dict(R=17), dict(max_ctas=-1)):
        assert query(**bad) == capi.CC_ERR_INVALID, bad
        assert ex(**bad) == capi.CC_ERR_INVALID, bad
    assert ex(max_ctas=1) == capi.CC_ERR_INVALID                 # the kernel runs CTA pairs
    assert query(max_ctas=1) == capi.CC_ERR_INVALID
    assert ex(out=[outs[0], None]) == capi.CC_ERR_INVALID
    assert ex(workspace=ws + 8) == capi.CC_ERR_MISALIGNED
    assert ex(workspace=outs[1]) == capi.CC_ERR_ALIAS            # written twice
    assert ex(workspace=x[0] + 16 * kr) == capi.CC_ERR_ALIAS     # inside an input
    assert ex(out=[outs[0], x[1]]) == capi.CC_ERR_ALIAS
    # well-formed: the host checks pass and the device range check refuses
    # the fake addresses (no GPU here)
    assert ex() in (capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_INVALID, capi.CC_ERR_CUDA)
    assert ex(workspace=None, workspace_bytes=0) in (capi.CC_ERR_UNSUPPORTED,
                                                     capi.CC_ERR_INVALID, capi.CC_ERR_CUDA)
    assert query() in (capi.CC_OK, capi.CC_ERR_UNSUPPORTED, capi.CC_ERR_CUDA)
