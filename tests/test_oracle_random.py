"""Pins of the oracle's Philox4x32-10 generator and stochastic rounding."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_philox_known_answer_vectors():
    n = 0
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        got = oracle.philox4x32_10(w[0:4], w[4:6])
        assert got.tolist() == w[6:10]
        n += 1
    assert n == 3


def test_sr_byte_mapping():
    """Element idx takes byte idx%4 of word (idx/4)%4 of the Philox call with
    counter (idx/16, 0, stream, 0) and key (lo(seed), hi(seed))."""
    seed = 0x0123456789ABCDEF
    for stream in (0, 1):
        for n in (0, 1, 77, (1 << 32) + 5):
            out = oracle.philox4x32_10([n & 0xffffffff, n >> 32, stream, 0],
                                       [seed & 0xffffffff, seed >> 32])
            b = out.view(np.uint8)  # little-endian words
            got = oracle.sr_bytes(seed, stream, 16 * n, 16)
            np.testing.assert_array_equal(got, b)


def test_sr_probability_is_floor_256f_exhaustive_over_r8():
    """Over all 256 values of the random byte, the number of round-ups is
    exactly floor(256 f) with f the position of |v| between its neighbours."""
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(0, 6, 3000), np.array(GRID), rng.uniform(-6, 0, 500)])
    r = np.arange(256, dtype=np.uint8)
    for x in v:
        a = abs(x)
        i = max(j for j in range(8) if GRID[j] <= a) if a < 6 else 7
        codes = oracle.e2m1_sr_batch(np.full(256, x), r)
        mags = codes & 7
        assert set(np.unique(mags)) <= {i, min(i + 1, 7)}
        ups = int((mags == i + 1).sum()) if i < 7 else 0
        if i < 7:
            f = (a - GRID[i]) / (GRID[i + 1] - GRID[i])
            assert ups == int(np.floor(256 * f)), x
        assert np.all((codes >> 3) == (1 if np.signbit(x) else 0))


def test_sr_grid_values_never_move():
    r = np.arange(256, dtype=np.uint8)
    for g in GRID:
        for s in (1, -1):
            codes = oracle.e2m1_sr_batch(np.full(256, s * g), r)
            assert len(np.unique(codes)) == 1
            assert oracle.e2m1_value(int(codes[0])) == s * g


def test_sr_unbiased_over_philox_draws():
    """Mean decoded value over 4096 Philox draws is within 5 sigma of v + the
    known truncation bias (at most one 256th of the grid gap, downwards)."""
    vals = [0.3, 0.7, 1.1, 1.6, 2.2, 2.9, 3.3, 4.6, 5.9]
    for x in vals:
        r8 = oracle.sr_bytes(99, 0, 0, 4096)
        dec = np.array([oracle.e2m1_value(int(c)) for c in oracle.e2m1_sr_batch(np.full(4096, x), r8)])
        i = max(j for j in range(8) if GRID[j] <= x)
        gap = GRID[i + 1] - GRID[i]
        f = (x - GRID[i]) / gap
        expect = GRID[i] + gap * np.floor(256 * f) / 256
        sigma = gap * np.sqrt(f * (1 - f) / 4096) + 1e-12
        assert abs(dec.mean() - expect) < 5 * sigma + 1e-9, x
        assert abs(expect - x) <= gap / 256 + 1e-12
