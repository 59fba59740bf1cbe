"""The fused tensor-parallel MatMul + AllReduce (tcgen05 GEMM whose epilogue
sums the R ranks' partial products in rank order and stores the bf16 result
to every rank), through the C ABI.

Two pins: integer-valued operands make every partial product and every sum
exact in fp32, so the GEMM itself is checked exactly against a float64
matmul (any layout, descriptor or indexing slip changes an integer); with
real-valued operands the kernel also stores the fp32 partial products, the
outputs must equal the oracle's rank-order AllReduce of exactly those
partials bit for bit, and the partials must lie within the float64 matmul's
error bound."""
import numpy as np
import pytest
import torch

import oracle
from gradient_reduce_optimizer_gb300 import build as gbuild
from gradient_reduce_optimizer_gb300 import capi
from gpu_common import DEV, assert_bits, f32, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    capi.lib()
    capi.cc_device_status(clear=True)


def operands(R, m, n, k, seed, integer):
    kr = k // R
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    if integer:
        x = [torch.randint(-4, 5, (m, kr), generator=g, device=DEV).to(torch.bfloat16)
             for _ in range(R)]
        w = [torch.randint(-4, 5, (n, kr), generator=g, device=DEV).to(torch.bfloat16)
             for _ in range(R)]
    else:
        x = [torch.randn(m, kr, generator=g, device=DEV).to(torch.bfloat16) for _ in range(R)]
        w = [(torch.randn(n, kr, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
             for _ in range(R)]
    return x, w


# Schedules: (workspace?, CTA budget).  Without a workspace every group of
# output tiles runs whole; with one, a small last wave's groups are split
# into rank products summed by the last to finish.  A budget of 6 CTAs (3
# pairs) gives several whole waves per pair.  "split-budget" takes the
# smallest budget for which the library splits (it asks the workspace
# query); for the pair shapes with R > 1 one exists, and with it the
# groups before the split wave run whole.
SCHEDULES = {"whole": (False, 0), "split": (True, 0), "whole-3pairs": (False, 6),
             "split-budget": (True, None)}


def split_budget(m, n, k, R):
    """The smallest CTA budget at which the last wave is split (0: none)."""
    for ctas in range(4, 153, 2):
        if capi.cc_tp_matmul_allreduce_workspace(m, n, k, R, ctas) > 0:
            return ctas
    return 0


def run(x, w, m, n, k, R, with_partials=True, schedule="whole"):
    outs = [torch.full((m, n), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            for _ in range(R)]
    parts = ([torch.full((m, n), float("nan"), device=DEV) for _ in range(R)]
             if with_partials else None)
    split, max_ctas = SCHEDULES[schedule]
    if schedule == "whole":
        capi.cc_tp_matmul_allreduce(x, w, outs, parts, m, n, k, R)
    else:
        if max_ctas is None:
            max_ctas = split_budget(m, n, k, R)
            if (m // 128) % 2 == 0 and R > 1:
                assert max_ctas > 0              # these shapes can split a last wave
        ws_bytes = capi.cc_tp_matmul_allreduce_workspace(m, n, k, R, max_ctas) if split else 0
        ws = (torch.full((max(ws_bytes, 16),), 0x7F, dtype=torch.uint8, device=DEV)
              if split else None)
        capi.cc_tp_matmul_allreduce_ex(x, w, outs, parts, m, n, k, R, ws, ws_bytes, max_ctas)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0
    return outs, parts


def exact_products(x, w):
    return [x_.double().cpu().numpy() @ w_.double().cpu().numpy().T for x_, w_ in zip(x, w)]


# (R, m, n, k): one tile; several tiles and k-blocks; more tiles than SMs
# with an odd R (the two accumulators alternate across tiles); the widest R.
# Where the row tiles pair up, the pair kernel (one MMA over two SMs); else
# the single-CTA kernel.  Single 128, pair 256, pair 256, pair 192, single
# 256, single 192, pair 128 (tile widths).  The single-CTA kernel's cluster
# shapes with multicast (1x2, 2x1, 2x2) are built for sweeps
# (CC_TP_PAIR=0, CC_TP_CLUSTER_M/N).
SHAPES = [(1, 128, 128, 64), (2, 256, 256, 256), (3, 2560, 1280, 192),
          (8, 256, 384, 1024), (16, 128, 256, 1024), (2, 384, 768, 128),
          (4, 512, 640, 256)]


@pytest.mark.parametrize("schedule", list(SCHEDULES))
@pytest.mark.parametrize("R,m,n,k", SHAPES)
def test_integer_operands_are_exact(R, m, n, k, schedule):
    x, w = operands(R, m, n, k, seed=11 + R, integer=True)
    outs, parts = run(x, w, m, n, k, R, schedule=schedule)
    Y = exact_products(x, w)
    total = sum(Y)
    for r in range(R):
        np.testing.assert_array_equal(f32(parts[r]).reshape(m, n), Y[r].astype(np.float32),
                                      err_msg=f"partial {r}")
    want = torch.from_numpy(total.astype(np.float32)).to(torch.bfloat16)
    want16 = want.view(torch.int16).numpy().view(np.uint16).ravel()
    for r in range(R):
        assert_bits(f"out[{r}]", u16(outs[r]).ravel(), want16, "bf16")


@pytest.mark.parametrize("schedule", ["whole", "split-budget"])
@pytest.mark.parametrize("R,m,n,k", SHAPES)
def test_outputs_are_the_rank_order_allreduce_of_the_partials(R, m, n, k, schedule):
    x, w = operands(R, m, n, k, seed=21 + R, integer=False)
    outs, parts = run(x, w, m, n, k, R, schedule=schedule)
    P = [f32(p).ravel().copy() for p in parts]
    ref = oracle.tp_allreduce(P)
    for r in range(R):
        assert_bits(f"out[{r}]", u16(outs[r]).ravel(), ref[r], "bf16")
    kr = k // R
    for r, Yr in enumerate(exact_products(x, w)):
        X = x[r].double().cpu().numpy()
        W = w[r].double().cpu().numpy()
        bound = kr * 2.0 ** -23 * (np.abs(X) @ np.abs(W).T) + 1e-30
        err = np.abs(P[r].reshape(m, n) - Yr)
        assert np.all(err <= bound), f"partial {r}: max excess {np.max(err - bound)}"
    # neither the debug store of the partials nor the schedule changes an
    # output bit
    for other in ("whole", "split", "split-budget", "whole-3pairs"):
        outs2, _ = run(x, w, m, n, k, R, with_partials=False, schedule=other)
        for r in range(R):
            assert torch.equal(outs2[r].view(torch.int16), outs[r].view(torch.int16)), other


@pytest.mark.parametrize("schedule", ["whole", "split"])
@pytest.mark.parametrize("m", [2048, 8192, 16384])
def test_gpt2_mlp_shape_sampled(m, schedule):
    """The measured shape (R=8, n=3072, k=12288; m=8192 runs 256-column tiles
    with a split last wave of 4 groups, m=16384 one of 8 groups, m=2048
    192-column tiles): integer operands, so every output is exact; checked on
    sampled rows against float64 (the last row tiles are the split wave's)."""
    R, n, k = 8, 3072, 12288
    x, w = operands(R, m, n, k, seed=5, integer=True)
    outs, _ = run(x, w, m, n, k, R, with_partials=False, schedule=schedule)
    rows = torch.tensor([0, 1, 127, 128, m // 2 - 1, m // 2, m - 256, m - 192, m - 1],
                        device=DEV)
    total = sum(x_[rows].double() @ w_.double().T for x_, w_ in zip(x, w))
    want = total.float().to(torch.bfloat16).view(torch.int16)
    for r in range(R):
        assert torch.equal(outs[r][rows].view(torch.int16), want), f"out[{r}]"


def test_rejects_bad_shapes_and_aliases():
    R, m, n, k = 2, 128, 128, 128
    x, w = operands(R, m, n, k, seed=3, integer=True)
    outs = [torch.empty(m, n, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    for bad in ((m + 8, n, k), (m, n + 16, k), (m, n, k + 2), (m, n, 96)):
        with pytest.raises(capi.CCError) as ei:
            capi.cc_tp_matmul_allreduce(x, w, outs, None, *bad, R)
        assert ei.value.status == capi.CC_ERR_INVALID
    with pytest.raises(capi.CCError) as ei:
        capi.cc_tp_matmul_allreduce(x, w, [outs[0], outs[0]], None, m, n, k, R)
    assert ei.value.status == capi.CC_ERR_ALIAS
    with pytest.raises(capi.CCError) as ei:
        capi.cc_tp_matmul_allreduce(x, w, [outs[0], x[1]], None, m, n, k, R)
    assert ei.value.status == capi.CC_ERR_ALIAS


def test_rejects_small_workspace_and_one_cta():
    R, m, n, k = 4, 512, 640, 256
    x, w = operands(R, m, n, k, seed=4, integer=True)
    outs = [torch.empty(m, n, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    ctas = split_budget(m, n, k, R)
    need = capi.cc_tp_matmul_allreduce_workspace(m, n, k, R, ctas)
    assert ctas > 0 and need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    with pytest.raises(capi.CCError) as ei:
        capi.cc_tp_matmul_allreduce_ex(x, w, outs, None, m, n, k, R, ws, need - 16, ctas)
    assert ei.value.status == capi.CC_ERR_INVALID
    with pytest.raises(capi.CCError) as ei:
        capi.cc_tp_matmul_allreduce_ex(x, w, outs, None, m, n, k, R, None, 0, 1)
    assert ei.value.status == capi.CC_ERR_INVALID
    with pytest.raises(capi.CCError) as ei:
        capi.cc_tp_matmul_allreduce_ex(x, w, outs, None, m, n, k, R, outs[1], need, ctas)
    assert ei.value.status == capi.CC_ERR_ALIAS
    # one split-free launch later nothing is left armed
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0


def _random_cases(count=28, seed=2024):
    import random
    rnd = random.Random(seed)
    cases = []
    while len(cases) < count:
        R = rnd.choice([1, 2, 3, 4, 5, 8, 12, 16])
        m = 128 * rnd.randint(1, 24)
        n = rnd.choice([128, 192, 256, 384, 512, 576, 640, 768, 1024])
        kr = 64 * rnd.randint(1, 4)
        max_ctas = rnd.choice([0, 0, 4, 6, 10, 32])
        use_ws = rnd.random() < 0.7
        cases.append((R, m, n, kr * R, max_ctas, use_ws))
    return cases


@pytest.mark.parametrize("R,m,n,k,max_ctas,use_ws", _random_cases())
def test_random_shapes_and_schedules_are_exact(R, m, n, k, max_ctas, use_ws):
    """Seeded random shapes, CTA budgets and workspaces: whichever kernel,
    tile width and schedule (whole or split last wave) the library picks,
    integer operands give outputs equal to the bf16 rounding of the exact
    sum (|x|, |w| <= 3, so every partial and sum is exact in fp32)."""
    x, w = operands(R, m, n, k, seed=m + n + k + R, integer=True)
    outs = [torch.full((m, n), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            for _ in range(R)]
    ws_bytes = capi.cc_tp_matmul_allreduce_workspace(m, n, k, R, max_ctas) if use_ws else 0
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV) if use_ws else None
    capi.cc_tp_matmul_allreduce_ex(x, w, outs, None, m, n, k, R, ws, ws_bytes, max_ctas)
    torch.cuda.synchronize()
    assert capi.cc_device_status() == 0
    total = sum(x_.double() @ w_.double().T for x_, w_ in zip(x, w))
    want = total.float().to(torch.bfloat16).view(torch.int16)
    for r in range(R):
        assert torch.equal(outs[r].view(torch.int16), want), f"out[{r}]"
