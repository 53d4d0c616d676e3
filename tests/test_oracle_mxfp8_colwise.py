"""Pins of the oracle's columnwise MXFP8 operand (reading R25).

It is the rowwise MXFP8 quantisation (R14, pinned in the format tests) of
each expert's transposed block: checked against the oracle's rowwise MXFP8
pack run on the transposes, and against a hand-worked block.
"""
import numpy as np

import oracle


def bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_equals_the_rowwise_pack_of_each_transpose():
    rng = np.random.default_rng(4)
    H, E = 96, 3
    off = np.array([0, 128, 128, 384], np.int32)      # expert 1 empty
    R_cap = 400
    x = bf16(rng.standard_normal((R_cap, H)) * np.exp(rng.standard_normal((R_cap, 1))))
    got = oracle.mxfp8_colwise(x, off, E)
    for e in range(E):
        a, n = int(off[e]), int(off[e + 1] - off[e])
        if n == 0:
            continue
        xt = np.ascontiguousarray(x[a:a + n].T)        # [H][n]: columns become tokens
        ref = oracle.mxfp8_pack(xt, np.arange(H, dtype=np.int32), 1, np.array([0, H], np.int32),
                                np.array([H], np.int32), 1, H)
        data, scl = ref[: H * n], ref[H * n:]
        assert np.array_equal(got[a * H:(a + n) * H], data), e
        assert np.array_equal(got[R_cap * H + a * H // 32: R_cap * H + (a + n) * H // 32], scl), e


def test_hand_worked_block():
    """One column of 32 rows: values 1..32 -> max 32 <= 448 * 2^-3 = 56 but
    not <= 448 * 2^-4 = 28, so e = -3 (E8M0 byte 124) and element i is the
    E4M3 rounding of the exact quotient (i + 1) * 8."""
    H, E = 32, 1
    off = np.array([0, 32], np.int32)
    x = np.zeros((32, H), np.float32)
    x[:, 5] = np.arange(1, 33)
    got = oracle.mxfp8_colwise(bf16(x), off, E)
    assert got[32 * H + 5] == 124
    col = got[5 * 32:6 * 32]
    for i in range(32):
        v = (i + 1) * 8.0                                  # 8 .. 256
        want = int(oracle.lib().or_e4m3_rne_sat(v))
        assert col[i] == want, i
    assert (got[32 * H: 32 * H + 5] == 0).all()            # all-zero columns: byte 0 (e = -127)
