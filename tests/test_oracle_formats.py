"""Pins of the oracle's number formats against independent formulations.

Each test checks the oracle against something other than itself: a fixture
taken from the format's specification, a different formulation of the same
rounding rule (threshold counting instead of nearest-value search), exact
rational arithmetic, or torch's own FP8/BF16 conversions.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# E2M1 rounding midpoints and the tie direction (True = the upper neighbour
# has the even index, so an exact tie rounds up).
MIDPOINTS = [(0.25, False), (0.75, True), (1.25, False), (1.75, True),
             (2.5, False), (3.5, True), (5.0, False)]
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def all_finite_bf16():
    b = np.arange(1 << 16, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return f[np.isfinite(f)]


def test_e2m1_grid_matches_spec_fixture():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_grid.txt")) if not l.startswith("#")]
    for code, val in rows:
        got = oracle.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def threshold_count(a, s):
    """Independent formulation: count thresholds mu*s passed by |x| (exact)."""
    m = np.zeros(a.shape, np.int64)
    for mu, up in MIDPOINTS:
        t = mu * s
        m += (a >= t) if up else (a > t)
    return m


@pytest.mark.parametrize("token_scale_exp", [-20, 0, 7])
def test_e2m1_rne_equals_threshold_count_exhaustive(token_scale_exp):
    """Every finite BF16 value x and every positive E4M3 block scale s_b:
    the oracle's nearest-grid search on x/s equals the threshold count."""
    x = all_finite_bf16().astype(np.float64)
    St = math.ldexp(1.0, token_scale_exp)
    for sb_code in range(1, 127):
        s = oracle.e4m3_value(sb_code) * St
        got = oracle.e2m1_rne_batch(x / s)
        want = np.minimum(threshold_count(np.abs(x), s), 7) | np.where(np.signbit(x), 8, 0)
        np.testing.assert_array_equal(got, want)


def test_e2m1_rne_exact_rationals():
    rng = np.random.default_rng(7)
    vals = [Fraction(int(n), 64) for n in rng.integers(-500, 500, 400)]
    vals += [Fraction(mu).limit_denominator() for mu, _ in MIDPOINTS]
    for v in vals:
        a = abs(v)
        d = [abs(a - Fraction(g)) for g in GRID]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        idx = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        want = idx | (8 if v < 0 else 0)
        assert oracle.e2m1_rne(float(v)) == want, v


def test_e2m1_sign_of_zero_is_kept():
    assert oracle.e2m1_rne(-0.0) == 8
    assert oracle.e2m1_rne(-0.2) == 8
    assert oracle.e2m1_rne(0.0) == 0
    assert oracle.e2m1_rne(-100.0) == 15


def test_e4m3_values_match_torch():
    codes = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    np.testing.assert_array_equal(got, want)
    assert math.isnan(oracle.e4m3_value(0x7f)) and math.isnan(oracle.e4m3_value(0xff))
    assert oracle.e4m3_value(126) == 448.0 and oracle.e4m3_value(1) == 2.0 ** -9


def test_e4m3_rne_matches_torch_in_range():
    """All finite BF16 values and all exact E4M3 midpoints in [0, 448], plus
    random float32 values; torch's cast is round-to-nearest-even in range."""
    x = all_finite_bf16().astype(np.float64)
    x = x[np.abs(x) <= 448.0]
    vals = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(3)
    rnd = rng.uniform(0, 448, 200000)
    allv = np.concatenate([x, mids, -mids, rnd.astype(np.float32).astype(np.float64)])
    got = oracle.e4m3_rne_sat_batch(allv)
    want = torch.from_numpy(allv.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, want)


def test_e4m3_saturates():
    assert oracle.e4m3_rne_sat(448.0) == 126
    assert oracle.e4m3_rne_sat(1e30) == 126
    assert oracle.e4m3_rne_sat(2.0 ** -10) == 0      # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_rne_sat(1.5 * 2.0 ** -10) == 1


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.uniform(-30, 30, 100000),
                        np.array([0.0, -0.0, 1e-40, -3e-39])])
    v32 = v.astype(np.float32)
    got = np.array([oracle.bf16_rne(float(t)) for t in v32], np.uint16)
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_token_scale_closed_form():
    """S_t = 2^k is a power of two with A in (1344 S_t, 2688 S_t], except at
    the floor k = -126; cross-checked with a frexp formula."""
    rng = np.random.default_rng(11)
    amax = np.concatenate([all_finite_bf16()[::7].astype(np.float64), [0.0, 2688.0, 1344.0]])
    amax = np.abs(amax)
    for a in amax:
        k = oracle.token_scale_exp(a)
        assert k >= -126
        S = math.ldexp(1.0, k)
        assert a <= 2688.0 * S
        if k > -126:
            assert a > 1344.0 * S
        # independent: k = ceil(log2(a / 2688)) computed with exact rationals
        if a > 0:
            q = Fraction(a) / 2688
            m, e = math.frexp(a / 2688.0)
            kk = e if Fraction(2) ** e / 2 != q else e - 1
            kk = max(kk, -126)
            assert k == kk, a
    assert oracle.token_scale_exp(0.0) == -126


def test_mx_scale_exp_brute_force():
    """Smallest e in [-127, 127] with max|x| <= 448 * 2^e, by enumeration of
    every exponent (the products 448 * 2^e are exact in float64)."""
    x = np.abs(all_finite_bf16()[::5].astype(np.float64))
    E = np.arange(-127, 128)
    ok = x[:, None] <= 448.0 * np.ldexp(1.0, E)[None, :]
    want = np.where(ok.any(axis=1), E[np.argmax(ok, axis=1)], 127)
    got = np.array([oracle.mx_scale_exp(b) for b in x])
    np.testing.assert_array_equal(got, want)
