"""Pins for the oracle: checks against things other than the oracle itself.

Each test fixes the oracle to a closed form, a library routine, exact
arithmetic, an invariant of the method, or brute force, chosen so that a
plausible slip (a dropped term, a wrong sign or index, a swapped operand, a
missing replica) fails at least one of them:

* bf16 cast: every bf16 rounding class for all 65,536 upper halves, against
  a rounding computed in float64 from frexp/rint (no bit tricks); and every
  one of the 2^32 binary32 patterns against torch's own conversion.
* step 1 closed form: with m = v = 0 and no decay, Adam's first update is
  lr * g / (|g| + eps) (bias correction exactly cancels 1 - beta).
* R = 1 against torch.optim.AdamW on CPU (fp32, foreach=False), over
  several steps, with weight decay large enough that a coupled (L2) or
  missing decay shows.
* exact integer sums: with beta1 = beta2 = 0 the new moments are the summed
  gradient and its square, exactly.
* loss scale: a power-of-two grad_scale applied to the gradients and then
  removed gives bit-identical results.
* replica identity, k-step accumulation against the single step on summed
  gradients, NaN/Inf propagation, and brute force in float64 on n <= 64.
"""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(12345)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def widen(h: np.ndarray) -> np.ndarray:
    """bf16 bits -> float64 from the fields (sign, exponent, mantissa)."""
    h = h.astype(np.int64)
    sign = np.where(h & 0x8000, -1.0, 1.0)
    e = (h >> 7) & 0xFF
    f = (h & 0x7F).astype(np.float64)
    val = np.where(e == 0, np.ldexp(f, -133),
                   np.ldexp(128.0 + f, (e - 134).astype(np.int32)))
    return sign * val


def rne_bf16_float64(x: np.ndarray) -> np.ndarray:
    """Round finite float64 values to the bf16 grid, ties to even, in float64.

    bf16 keeps 8 significant bits; its smallest step is 2**-133.  For x in
    [2**(e-1), 2**e) the step is 2**(e-8), floored at 2**-133.  np.rint
    rounds half to even; both scalings are exact.  Values past the largest
    bf16 become infinities.
    """
    out = np.empty_like(x)
    zero = x == 0
    _, e = np.frexp(x)
    q = np.maximum(e - 8, -133)
    scaled = np.ldexp(x, -q)
    out = np.ldexp(np.rint(scaled), q)
    out[zero] = x[zero]
    big = np.abs(out) >= 2.0 ** 128
    out[big] = np.copysign(np.inf, x[big])
    return out


# ---------------------------------------------------------------------------
# bf16 cast and widening
# ---------------------------------------------------------------------------

def test_bf16_widen_matches_field_decoding():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        got = oracle.bf16_widen(h).astype(np.float64)
    exp = h.astype(np.int64)
    finite = ((exp >> 7) & 0xFF) != 0xFF
    np.testing.assert_array_equal(got[finite], widen(h[finite]))
    e_ff = ~finite
    mant = (h & 0x7F) != 0
    assert np.all(np.isnan(got[e_ff & mant]))
    assert np.all(np.isinf(got[e_ff & ~mant]))


def test_bf16_round_every_rounding_class():
    """All 65,536 upper halves x lower halves that cover every RNE decision:
    below half, exactly half (ties, both parities of the kept half), above
    half, and the extremes; plus random lower halves."""
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF,
                     0xFFFF], dtype=np.uint32)
    lows = np.concatenate([lows, RNG.integers(0, 1 << 16, 24, dtype=np.uint32)])
    hi = np.arange(1 << 16, dtype=np.uint32)
    u = (hi[:, None] << 16 | lows[None, :]).ravel()
    x32 = u.view(np.float32)
    got = oracle.bf16_round(x32)
    finite = np.isfinite(x32)
    got_f = got[finite]
    exp = rne_bf16_float64(x32[finite].astype(np.float64))
    got_inf = (((got_f >> 7) & 0xFF) == 0xFF) & ((got_f & 0x7F) == 0)
    got_neg = (got_f >> 15) == 1
    fin = np.isfinite(exp)
    assert not got_inf[fin].any()
    np.testing.assert_array_equal(widen(got_f[fin]), exp[fin])
    np.testing.assert_array_equal(got_neg[fin], np.signbit(exp[fin]))
    assert got_inf[~fin].all()
    np.testing.assert_array_equal(got_neg[~fin], np.signbit(exp[~fin]))
    # signed zeros keep their sign
    z = oracle.bf16_round(np.array([0.0, -0.0], dtype=np.float32))
    assert list(z) == [0x0000, 0x8000]
    # NaN stays NaN with its sign; infinities stay infinities
    nan = x32[np.isnan(x32)]
    gn = oracle.bf16_round(nan)
    assert np.all(((gn >> 7) & 0xFF) == 0xFF) and np.all((gn & 0x7F) != 0)
    assert np.array_equal(gn >> 15, (nan.view(np.uint32) >> 31).astype(np.uint16))
    inf = np.array([np.inf, -np.inf], dtype=np.float32)
    assert list(oracle.bf16_round(inf)) == [0x7F80, 0xFF80]


def test_bf16_round_every_binary32_pattern():
    """All 2^32 binary32 bit patterns, in chunks.  Non-NaN inputs (finite
    values and infinities) against torch's CPU float->bfloat16 conversion,
    a separate implementation of round-to-nearest-even; NaN inputs stay NaN
    with their sign (torch returns one canonical NaN, so only the class is
    compared).  The float64 reference above pins every rounding class; this
    sweep leaves no input pattern unchecked."""
    chunk = 1 << 25
    base = np.arange(chunk, dtype=np.uint32)
    u = np.empty_like(base)
    for start in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(start), out=u)
        x = u.view(np.float32)
        got = oracle.bf16_round(x)
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        if ((start + chunk - 1) >> 23) & 0xFF != 0xFF:      # no NaN patterns here
            assert np.array_equal(got, ref), hex(start)
            continue
        nan = (((u >> 23) & 0xFF) == 0xFF) & ((u & 0x7FFFFF) != 0)
        keep = ~nan
        assert np.array_equal(got[keep], ref[keep]), hex(start)
        gn = got[nan]
        assert np.all(((gn >> 7) & 0xFF) == 0xFF) and np.all((gn & 0x7F) != 0), hex(start)
        assert np.array_equal(gn >> 15, (u[nan] >> 31).astype(np.uint16)), hex(start)


def test_bf16_round_agrees_with_torch_on_finite_values():
    """torch's CPU float->bfloat16 conversion rounds to nearest even too."""
    x = torch.from_numpy(RNG.standard_normal(1 << 16).astype(np.float32)) * 1e-3
    np.testing.assert_array_equal(oracle.bf16_round(x.numpy()),
                                  bf16_bits(x.to(torch.bfloat16)))


# ---------------------------------------------------------------------------
# Adam arithmetic
# ---------------------------------------------------------------------------

ADAM = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def rand_grads(R, n, sigma=1e-3):
    return [bf16_bits(torch.from_numpy(
        (RNG.standard_normal(n) * sigma).astype(np.float32)).to(torch.bfloat16))
        for _ in range(R)]


def ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(np.maximum(x, np.float32(1.2e-38))).astype(np.float64)


@pytest.mark.parametrize("R", [1, 2, 3])
@pytest.mark.parametrize("eps", [1e-8, 1e-3])
def test_step1_closed_form(R, eps):
    """m = v = 0, wd = 0, step 1: p0 - p1 = lr * g / (|g| + eps),
    m1 = (1 - b1) g, v1 = (1 - b2) g^2, with g the replica sum."""
    n = 4096
    grads = rand_grads(R, n)
    p0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.fused_dp_step(grads, master, m, v, lr=1e-3, beta1=0.9, beta2=0.999,
                         eps=eps, weight_decay=0.0, step=1, grad_scale=1.0)
    g = sum(widen(gr) for gr in grads)
    want = 1e-3 * g / (np.abs(g) + eps)
    got = p0.astype(np.float64) - master.astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= ulp32(master) + 1e-6 * 1e-3), err.max()
    b1 = float(np.float32(1) - np.float32(0.9))
    b2 = float(np.float32(1) - np.float32(0.999))
    np.testing.assert_allclose(m, b1 * g, rtol=1e-6, atol=0)
    np.testing.assert_allclose(v, b2 * g * g, rtol=1e-6, atol=1e-30)


def test_r1_matches_torch_adamw_over_steps():
    """R = 1 reduces to plain AdamW: compare with torch.optim.AdamW (CPU, fp32,
    foreach=False) for 6 steps with a strong decoupled weight decay."""
    n, steps = 8192, 6
    lr, b1, b2, eps, wd = 1e-2, 0.8, 0.95, 1e-6, 0.1
    p0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=lr, betas=(b1, b2), eps=eps,
                            weight_decay=wd, foreach=False, fused=False)
    for t in range(1, steps + 1):
        grads = rand_grads(1, n)
        out = oracle.fused_dp_step(grads, master, m, v, lr=lr, beta1=b1,
                                   beta2=b2, eps=eps, weight_decay=wd, step=t,
                                   grad_scale=1.0)
        tp.grad = torch.from_numpy(widen(grads[0]).astype(np.float32))
        opt.step()
        st = opt.state[tp]
        for name, mine, ref in (("master", master, tp.detach().numpy()),
                                ("m", m, st["exp_avg"].numpy()),
                                ("v", v, st["exp_avg_sq"].numpy())):
            scale = np.abs(ref).max()
            err = np.abs(mine.astype(np.float64) - ref).max() / scale
            assert err < 1e-5, (t, name, err)
        # the bf16 output is the rounded master
        np.testing.assert_array_equal(out[0], oracle.bf16_round(master))


def test_r3_scaled_matches_torch_adamw_on_summed_grad():
    """R = 3 with loss scale 1024: torch AdamW fed the summed, unscaled
    gradient (float64 sum, then fp32) agrees within 1e-5 relative."""
    n, R = 8192, 3
    lr, wd = 1e-3, 0.01
    grads = rand_grads(R, n)
    scaled = [bf16_bits(torch.from_numpy(widen(g).astype(np.float32) * 1024)
                        .to(torch.bfloat16)) for g in grads]
    p0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    m0 = (RNG.standard_normal(n) * 1e-4).astype(np.float32)
    v0 = ((RNG.standard_normal(n) * 1e-3) ** 2).astype(np.float32)
    master, m, v = p0.copy(), m0.copy(), v0.copy()
    oracle.fused_dp_step(scaled, master, m, v, lr=lr, beta1=0.9, beta2=0.999,
                         eps=1e-8, weight_decay=wd, step=10, grad_scale=1024.0)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=lr, betas=(0.9, 0.999), eps=1e-8,
                            weight_decay=wd, foreach=False, fused=False)
    opt.state[tp] = {"step": torch.tensor(9.0),
                     "exp_avg": torch.from_numpy(m0.copy()),
                     "exp_avg_sq": torch.from_numpy(v0.copy())}
    tp.grad = torch.from_numpy(sum(widen(g) for g in grads).astype(np.float32))
    opt.step()
    st = opt.state[tp]
    for mine, ref in ((master, tp.detach().numpy()), (m, st["exp_avg"].numpy()),
                      (v, st["exp_avg_sq"].numpy())):
        err = np.abs(mine.astype(np.float64) - ref).max() / np.abs(ref).max()
        assert err < 1e-5, err


@pytest.mark.parametrize("R", [1, 2, 3, 8, 16])
def test_integer_gradients_sum_exactly(R):
    """beta1 = beta2 = 0 makes m' the unscaled summed gradient and v' its
    square; integer gradients in [-8, 8] sum exactly in binary32."""
    n = 2048
    ints = [RNG.integers(-8, 9, n) for _ in range(R)]
    grads = [bf16_bits(torch.from_numpy(i.astype(np.float32)).to(torch.bfloat16))
             for i in ints]
    master = np.ones(n, np.float32)
    m = np.full(n, 7.0, np.float32)
    v = np.full(n, 3.0, np.float32)
    oracle.fused_dp_step(grads, master, m, v, lr=0.0, beta1=0.0, beta2=0.0,
                         eps=1e-8, weight_decay=0.0, step=1, grad_scale=1.0)
    s = np.sum(ints, axis=0)
    np.testing.assert_array_equal(m, s.astype(np.float32))
    np.testing.assert_array_equal(v, (s * s).astype(np.float32))
    np.testing.assert_array_equal(master, np.ones(n, np.float32))  # lr = 0


def test_reduction_is_left_to_right_in_binary32():
    """Three replicas where the order of addition changes the fp32 result:
    (2^24 + 1) + 1 rounds twice to 2^24, 1 + (1 + 2^24) does not."""
    big = np.float32(2.0 ** 24)
    vals = [np.array([big], np.float32), np.array([1.0], np.float32),
            np.array([1.0], np.float32)]
    grads = [bf16_bits(torch.from_numpy(x).to(torch.bfloat16)) for x in vals]
    m = np.zeros(1, np.float32)
    oracle.fused_dp_step(grads, np.zeros(1, np.float32), m,
                         np.zeros(1, np.float32), lr=0.0, beta1=0.0, beta2=0.0,
                         eps=1.0, weight_decay=0.0, step=1, grad_scale=1.0)
    assert m[0] == big  # ((2^24 + 1) + 1) with two roundings to even
    m2 = np.zeros(1, np.float32)
    oracle.fused_dp_step(grads[::-1], np.zeros(1, np.float32), m2,
                         np.zeros(1, np.float32), lr=0.0, beta1=0.0, beta2=0.0,
                         eps=1.0, weight_decay=0.0, step=1, grad_scale=1.0)
    assert m2[0] == big + 2


def test_power_of_two_loss_scale_is_exact():
    n, R = 4096, 4
    grads = rand_grads(R, n, sigma=1e-4)
    scaled = [bf16_bits(torch.from_numpy(widen(g).astype(np.float32) * 65536.0)
                        .to(torch.bfloat16)) for g in grads]
    for g, s in zip(grads, scaled):
        assert np.array_equal(widen(s), widen(g) * 65536.0)
    base = [(RNG.standard_normal(n) * 0.02).astype(np.float32),
            (RNG.standard_normal(n) * 1e-5).astype(np.float32),
            ((RNG.standard_normal(n) * 1e-4) ** 2).astype(np.float32)]
    a = [x.copy() for x in base]
    b = [x.copy() for x in base]
    kw = dict(lr=1.5e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
              step=10)
    oa = oracle.fused_dp_step(grads, *a, grad_scale=1.0, **kw)
    ob = oracle.fused_dp_step(scaled, *b, grad_scale=65536.0, **kw)
    for x, y in zip(a + oa, b + ob):
        np.testing.assert_array_equal(x, y)


def test_replicas_are_identical_and_equal_rounded_master():
    n, R = 1000, 5
    grads = rand_grads(R, n)
    master = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    out = oracle.fused_dp_step(grads, master, np.zeros(n, np.float32),
                               np.zeros(n, np.float32), weight_decay=0.01,
                               step=1, grad_scale=1.0, **ADAM)
    for r in range(1, R):
        np.testing.assert_array_equal(out[r], out[0])
    np.testing.assert_array_equal(out[0], oracle.bf16_round(master))


def test_accumulation_equals_single_step_on_summed_integer_grads():
    """k = 4: three local micro-steps then the reducing step give bit for bit
    the single step on each replica's summed gradient (exact in bf16)."""
    n, R, k = 3000, 8, 4
    micro = [[RNG.integers(-8, 9, n) for _ in range(R)] for _ in range(k)]
    as_bf16 = [[bf16_bits(torch.from_numpy(x.astype(np.float32))
                          .to(torch.bfloat16)) for x in mj] for mj in micro]
    state0 = [(RNG.standard_normal(n) * 0.02).astype(np.float32),
              (RNG.standard_normal(n) * 1e-2).astype(np.float32),
              ((RNG.standard_normal(n)) ** 2).astype(np.float32)]
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
              step=10, grad_scale=1.0)
    acc = [np.empty(n, np.float32) for _ in range(R)]
    for j in range(k - 1):
        oracle.accumulate_local(as_bf16[j], acc, first=(j == 0))
    for r in range(R):
        np.testing.assert_array_equal(
            acc[r], sum(micro[j][r] for j in range(k - 1)).astype(np.float32))
    a = [x.copy() for x in state0]
    out_a = oracle.fused_dp_step(as_bf16[k - 1], *a, acc=acc, **kw)
    summed = [bf16_bits(torch.from_numpy(
        sum(micro[j][r] for j in range(k)).astype(np.float32)).to(torch.bfloat16))
        for r in range(R)]
    b = [x.copy() for x in state0]
    out_b = oracle.fused_dp_step(summed, *b, **kw)
    for x, y in zip(a + out_a, b + out_b):
        np.testing.assert_array_equal(x, y)


def test_nan_and_inf_propagate():
    grads = [np.array([0x7F80, 0x0000, 0x7FC0], np.uint16)]  # +inf, 0, NaN
    master = np.array([1.0, 1.0, 1.0], np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    out = oracle.fused_dp_step(grads, master, m, v, weight_decay=0.0, step=1,
                               grad_scale=1.0, **ADAM)
    assert np.isnan(master[0]) and np.isinf(m[0]) and np.isinf(v[0])
    assert master[1] == 1.0 and m[1] == 0.0 and v[1] == 0.0  # zero gradient
    assert np.isnan(master[2]) and np.isnan(m[2])
    assert ((out[0][0] >> 7) & 0xFF) == 0xFF and (out[0][0] & 0x7F) != 0


def test_rejects_bad_arguments():
    g = rand_grads(1, 8)
    z = np.zeros(8, np.float32)
    with pytest.raises(ValueError):
        oracle.fused_dp_step(g, z.copy(), z.copy(), z.copy(), weight_decay=0.0,
                             step=0, grad_scale=1.0, **ADAM)
    with pytest.raises(ValueError):
        oracle.fused_dp_step(g * 17, z.copy(), z.copy(), z.copy(),
                             weight_decay=0.0, step=1, grad_scale=1.0, **ADAM)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 63, 64])
@pytest.mark.parametrize("R", [1, 2, 5, 16])
def test_brute_force_float64_tiny(n, R):
    """Every element against the definition evaluated in float64 after the
    binary32 fixed-order reduction (whose order is pinned above), within a
    forward error bound: each binary32 rounding is at most u = 2**-24
    relative, propagated through the Adam step term by term."""
    u = 2.0 ** -24
    lr, b1, b2, eps, wd, t, scale = 2e-3, 0.85, 0.99, 1e-7, 0.05, 3, 4.0
    grads = rand_grads(R, n, sigma=4e-3)
    p = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    m = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    v = ((RNG.standard_normal(n) * 1e-3) ** 2).astype(np.float32)
    P, M, V = p.copy(), m.copy(), v.copy()
    out = oracle.fused_dp_step(grads, P, M, V, lr=lr, beta1=b1, beta2=b2,
                               eps=eps, weight_decay=wd, step=t,
                               grad_scale=scale)
    f = lambda x: float(np.float32(x))  # the fp32 hyper-parameters, exactly
    B1, B2, LR, WD, EPS = f(b1), f(b2), f(lr), f(wd), f(eps)
    for i in range(n):
        s = np.float32(widen(grads[0][i:i + 1])[0])
        for r in range(1, R):
            s = np.float32(s + np.float32(widen(grads[r][i:i + 1])[0]))
        g = float(s) / scale                      # exact: scale is 2**2
        a1, a2 = B1 * float(m[i]), (1 - B1) * g   # 1 - B1 is exact (Sterbenz)
        mn = a1 + a2
        e_m = u * (abs(a1) + abs(a2) + abs(mn))
        a3, a4 = B2 * float(v[i]), (1 - B2) * g * g
        vn = a3 + a4
        e_v = u * (abs(a3) + 2 * abs(a4) + abs(vn))
        bc1, bc2 = 1 - B1 ** t, 1 - B2 ** t
        mh, vh = mn / bc1, vn / bc2
        e_mh = e_m / bc1 + 2 * u * abs(mh)
        e_vh = e_v / bc2 + 2 * u * abs(vh)
        sq = math.sqrt(vh)
        e_sq = (e_vh / (2 * sq) if sq > 0 else math.sqrt(e_vh)) + u * sq
        den = sq + EPS
        e_den = e_sq + u * den
        ratio = mh / den
        e_ratio = e_mh / den + abs(mh) * e_den / den ** 2 + u * abs(ratio)
        upd = LR * ratio
        e_upd = LR * e_ratio + u * abs(upd)
        dec = 1 - LR * WD
        pd = float(p[i]) * dec
        e_pd = abs(float(p[i])) * u * (LR * WD + 1) + u * abs(pd)
        pn = pd - upd
        e_p = e_pd + e_upd + u * abs(pn)
        for got, want, tol in ((M[i], mn, e_m), (V[i], vn, e_v), (P[i], pn, e_p)):
            assert abs(float(got) - want) <= 1.5 * tol, (i, got, want, tol)
        # the cast of the fp32 master is to the nearest bf16 (<= half a step)
        q = widen(out[0][i:i + 1])[0]
        assert abs(q - float(P[i])) <= abs(float(P[i])) * 2.0 ** -8


# ---------------------------------------------------------------------------
# The tensor-parallel AllReduce
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("R", [1, 2, 4, 16])
def test_tp_allreduce_integer_sums_exact_and_identical(R):
    """Integer partials sum exactly; small integers are exact in bf16, so the
    result is the integer sum, the same on every rank."""
    n = 5000
    ints = [RNG.integers(-15, 16, n) for _ in range(R)]
    out = oracle.tp_allreduce([i.astype(np.float32) for i in ints])
    s = np.sum(ints, axis=0)
    np.testing.assert_array_equal(widen(out[0]), s.astype(np.float64))
    for r in range(1, R):
        np.testing.assert_array_equal(out[r], out[0])


def test_tp_allreduce_rank_order():
    """Rank order is observable after the bf16 cast: (1 + 2^-24) rounds to 1
    (a tie, to even), so [1, 2^-24, -1] gives 0, while [-1, 2^-24, 1] keeps
    the 2^-24 (exact in bf16)."""
    parts = [np.array([x], np.float32) for x in (1.0, 2.0 ** -24, -1.0)]
    assert widen(oracle.tp_allreduce(parts)[0])[0] == 0.0
    assert widen(oracle.tp_allreduce(parts[::-1])[0])[0] == 2.0 ** -24


def test_tp_allreduce_matches_float64_sum_within_bound():
    """Random partials: the result is the float64 sum rounded to the bf16 grid,
    up to the fp32 summation error (R ulps of the partial sums)."""
    R, n = 8, 20000
    parts = [(RNG.standard_normal(n) * 10).astype(np.float32) for _ in range(R)]
    got = widen(oracle.tp_allreduce(parts)[0])
    exact = np.sum([p.astype(np.float64) for p in parts], axis=0)
    bound = np.abs(exact) * 2.0 ** -8 + R * 2.0 ** -24 * np.sum(
        [np.abs(p.astype(np.float64)) for p in parts], axis=0) * 2
    assert np.all(np.abs(got - exact) <= bound)
