"""Pins of the oracle's BF16-input columnwise-RHT quantizer with a supplied
per-expert amax (reading R24: TE PR #3755 "Optionally derive FC1 dy NVFP4
amaxes from the dGLU epilogue", PR description and test commit).

The checks tie it to things other than itself: the direct receive's
columnwise operand (already pinned) on rows whose decoded values are the BF16
input, a closed-form block, the facts the page states (the rowwise amax is
the supplied amax rounded to BF16 and equals the input's amax when that is
what is supplied; no post-RHT value above 4x that amax), and the stochastic
rounding's one-grid-step property.
"""
import numpy as np
import pytest

import oracle
import workloads

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def bf16_to_f32(u16):
    return (np.asarray(u16, np.uint32) << 16).view(np.float32)


def expert_amax(x, off, E):
    a = np.zeros(E, np.float32)
    f = np.abs(bf16_to_f32(x))
    for e in range(E):
        if off[e + 1] > off[e]:
            a[e] = f[off[e]:off[e + 1]].max()
    return a


def test_equals_the_direct_receive_on_decoded_rows():
    """Packed rows decoded to BF16 (exact) and given the direct receive's own
    rowwise amax: the columnwise operand and metadata are the direct
    receive's, byte for byte (RNE)."""
    w = workloads.make(2, T=300, H=512)
    off, cnt, dest, _ = oracle.route_plan(w.topk, w.E, w.A)
    R_cap = int(off[-1])
    rows = oracle.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, R_cap)
    dr = oracle.nvfp4_direct_receive(rows, w.H, off, w.E, sign_mask=w.sign_mask)
    x = oracle.nvfp4_unpack(rows, w.H, off, w.E)
    assert np.isfinite(bf16_to_f32(x)).all()
    got = oracle.nvfp4_colwise_rht_bf16(x, off, w.E, dr["amax_row"], sign_mask=w.sign_mask)
    for k in ("cw_codes", "cw_scales"):
        assert np.array_equal(got[k], dr[k]), k
    for k in ("amax_row", "amax_col", "scale_enc"):
        assert np.array_equal(got[k].view(np.uint32), dr[k].view(np.uint32)), k


def test_rowwise_amax_is_the_supplied_amax_rounded_to_bf16():
    rng = np.random.default_rng(1)
    H, E = 64, 3
    off = np.array([0, 128, 128, 256], np.int32)
    x = (rng.standard_normal((256, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    exact = expert_amax(x, off, E)
    # the input's own amax is a BF16 value: kept as is
    o = oracle.nvfp4_colwise_rht_bf16(x, off, E, exact)
    assert np.array_equal(o["amax_row"], exact)
    assert o["amax_row"][1] == 0 and o["scale_enc"][1] == 1.0          # the empty expert
    assert np.array_equal(o["amax_col"], (np.float32(4) * exact).astype(np.float32))
    assert o["report"]["above_4x_rowwise_amax"] == 0 and o["report"]["above_4x_block_input"] == 0
    # a supplied amax off the BF16 grid: rounded to nearest, ties to even
    sup = np.array([3.8906251, 0.0, 1.0 + 2.0 ** -8], np.float32)   # 3.890625 | 1 + 2^-8 is a tie -> 1
    o = oracle.nvfp4_colwise_rht_bf16(x, off, E, sup)
    assert o["amax_row"][0] == np.float32(3.890625)
    assert o["amax_row"][2] == np.float32(1.0)
    assert o["scale_enc"][0] == np.float32(np.float32(2688.0) / np.float32(4 * 3.890625))


def test_closed_form_block():
    """One expert of 16 rows, one column: x_r = 1 for every row.  With the
    default sign mask the transform of the constant column is
    y = 1/4 H16 sigma: its entries are (1/4) * (sum of sigma times Hadamard
    row signs), computed here with numpy from the Sylvester matrix."""
    H, E = 32, 1
    off = np.array([0, 16], np.int32)
    x = np.zeros((16, H), np.uint16)
    x[:, 0] = 0x3F80                                                # 1.0
    mask = oracle.DEFAULT_SIGN_MASK
    o = oracle.nvfp4_colwise_rht_bf16(x, off, E, np.array([1.0], np.float32), sign_mask=mask)
    sig = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    Hm = np.array([[(-1.0) ** bin(i & j).count("1") for j in range(16)] for i in range(16)])
    y = 0.25 * Hm @ sig
    # S_enc = 2688 / 4 = 672, block scale E4M3(max|y| * 672 / 6), codes E2M1(|y| * 672 / s)
    se = np.float32(672.0)
    b = np.abs(y).max()
    s_val = float(np.float32(b) * np.float32(se / np.float32(6.0)))
    s_code = int(oracle.lib().or_e4m3_rne_sat(s_val))
    s = oracle.lib().or_e4m3_value(s_code)
    assert o["cw_scales"][0] == s_code
    r = np.float32(se / np.float32(s))
    for i in range(16):
        v = float(np.float32(abs(y[i])) * r)
        m = int(oracle.lib().or_e2m1_rne(v))
        code = m | (8 if y[i] < 0 else 0)
        byte = o["cw_codes"][i // 2]
        assert (byte >> (4 * (i % 2))) & 0xF == code, i
    # the other columns are all zero: scale 0, codes +0 or -0 only
    assert (o["cw_scales"][2:] == 0).all()


def test_stochastic_rounding_stays_within_one_grid_step():
    w = workloads.make(4, T=64, H=256, E=8, k=2)
    off, cnt, dest, _ = oracle.route_plan(w.topk, w.E, w.A)
    R = int(off[-1])
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((R, w.H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    am = expert_amax(x, off, w.E)
    rne = oracle.nvfp4_colwise_rht_bf16(x, off, w.E, am)
    sr = oracle.nvfp4_colwise_rht_bf16(x, off, w.E, am, rounding=1, seed=77)
    assert np.array_equal(rne["cw_scales"], sr["cw_scales"])         # scales stay RNE
    a = np.concatenate([rne["cw_codes"] & 0xF, rne["cw_codes"] >> 4])
    b = np.concatenate([sr["cw_codes"] & 0xF, sr["cw_codes"] >> 4])
    ma, mb = a & 7, b & 7
    assert (np.abs(ma.astype(int) - mb.astype(int)) <= 1).all()
    assert (ma != mb).mean() > 0.05                                  # it does move codes
    sr2 = oracle.nvfp4_colwise_rht_bf16(x, off, w.E, am, rounding=1, seed=78)
    assert not np.array_equal(sr["cw_codes"], sr2["cw_codes"])       # keyed by the seed
