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


def test_sr_u16_worked_example():
    """The 16 numbers of the first Philox call (seed 0, stream 0), derived by
    hand in the fixture from the published known-answer words."""
    want = []
    for line in open(os.path.join(GOLDEN, "sr16_worked_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        i, r = line.split()
        want.append((int(i), int(r, 16)))
    assert [i for i, _ in want] == list(range(16))
    got = oracle.sr_u16s(0, 0, 0, 16)
    assert got.tolist() == [r for _, r in want]


def _rev16(x):
    return int(format(int(x), "016b")[::-1], 2)


def test_sr_u16_mapping():
    """Element idx uses word (idx/4)%4 of the Philox call with counter
    (idx/16, hi, stream, 0) and key (lo(seed), hi(seed)): j = idx%4 takes
    b2:b0, its bit reverse, b3:b1, its bit reverse."""
    seed = 0x0123456789ABCDEF
    for stream in (0, 1, 2):
        for n in (0, 1, 77, (1 << 32) + 5):
            out = oracle.philox4x32_10([n & 0xffffffff, n >> 32, stream, 0], [seed & 0xffffffff, seed >> 32])
            want = []
            for w in out.tolist():
                b = [(w >> (8 * i)) & 0xff for i in range(4)]
                A, B = (b[2] << 8) | b[0], (b[3] << 8) | b[1]
                want += [A, _rev16(A), B, _rev16(B)]
            got = oracle.sr_u16s(seed, stream, 16 * n, 16)
            assert got.tolist() == want
            assert oracle.sr_u16(seed, stream, 16 * n + 13) == want[13]


def test_sr_u16_each_element_uniform():
    """Over all 65536 values of the two bytes an element's number is built
    from, each of the four positions takes every 16-bit value exactly once
    (the bit reverse is a bijection), so every element's number is uniform."""
    lo = np.arange(65536, dtype=np.int64)
    A = lo
    revA = np.array([_rev16(x) for x in range(65536)])
    assert np.array_equal(np.sort(A), lo) and np.array_equal(np.sort(revA), lo)


def test_sr_pair_sharing_two_bytes_independent_at_half():
    """Elements 0 and 1 of a word share the bytes b0, b2 (A and its reverse).
    At f = 1/2 their round-up events are 'top bit of A' and 'top bit of the
    reverse' = bit 15 and bit 0 of A: over all 65536 values of A they are
    independent (each pair of outcomes 16384 times)."""
    A = np.arange(65536, dtype=np.uint32)
    up0 = (A + 32768) >= 65536
    up1 = np.array([_rev16(x) for x in range(65536)]) + 32768 >= 65536
    for a in (False, True):
        for b in (False, True):
            assert int(np.count_nonzero((up0 == a) & (up1 == b))) == 16384


def test_sr_probability_is_floor_65536f_exhaustive_over_r16():
    """Over all 65536 values of the random number, the number of round-ups is
    exactly floor(65536 f) with f the position of |v| between its neighbours."""
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(0, 6, 300), np.array(GRID), rng.uniform(-6, 0, 60),
                        # on and next to a 2^-16 step of the fraction
                        np.array([0.5 + 0.5 * 12345 / 65536, 4.0 + 2.0 * 3 / 65536, 1.0 + 0.5 / 65536]),
                        np.nextafter(np.array([2.0 + 1.0 * 777 / 65536]), 10.0)])
    r = np.arange(65536, dtype=np.uint16)
    for x in v:
        a = abs(x)
        i = max(j for j in range(8) if GRID[j] <= a) if a < 6 else 7
        codes = oracle.e2m1_sr_batch(np.full(65536, x), r)
        mags = codes & 7
        assert set(np.unique(mags)) <= {i, min(i + 1, 7)}
        ups = int((mags == i + 1).sum()) if i < 7 else 0
        if i < 7:
            f = (a - GRID[i]) / (GRID[i + 1] - GRID[i])
            assert ups == int(np.floor(65536 * f)), x
            # the up decisions are exactly the largest numbers
            if ups:
                assert np.all(mags[65536 - ups:] == i + 1) and np.all(mags[:65536 - ups] == i)
        assert np.all((codes >> 3) == (1 if np.signbit(x) else 0))


def test_sr_grid_values_never_move():
    r = np.arange(65536, dtype=np.uint16)
    for g in GRID:
        for s in (1, -1):
            codes = oracle.e2m1_sr_batch(np.full(65536, s * g), r)
            assert len(np.unique(codes)) == 1
            assert oracle.e2m1_value(int(codes[0])) == s * g


def test_sr_unbiased_over_philox_draws():
    """Mean decoded value over 4096 Philox draws is within 5 sigma of v + the
    known truncation bias (at most one 65536th of the grid gap, downwards)."""
    vals = [0.3, 0.7, 1.1, 1.6, 2.2, 2.9, 3.3, 4.6, 5.9]
    for x in vals:
        r16 = oracle.sr_u16s(99, 0, 0, 4096)
        dec = np.array([oracle.e2m1_value(int(c)) for c in oracle.e2m1_sr_batch(np.full(4096, x), r16)])
        i = max(j for j in range(8) if GRID[j] <= x)
        gap = GRID[i + 1] - GRID[i]
        f = (x - GRID[i]) / gap
        expect = GRID[i] + gap * np.floor(65536 * f) / 65536
        sigma = gap * np.sqrt(f * (1 - f) / 4096) + 1e-12
        assert abs(dec.mean() - expect) < 5 * sigma + 1e-9, x
        assert abs(expect - x) <= gap / 65536 + 1e-12
