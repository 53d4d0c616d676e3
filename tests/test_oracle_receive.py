"""Pins of the oracle's direct receive (rowwise + columnwise-RHT operands).

Closed-form cases built from hand-made rows fix the transform, the
bound-derived scale and the columnwise layout; the rest are invariants the
pages state (rowwise operand = the sender's codes, rowwise amax = the BF16
amax, post-RHT amax <= 4x rowwise amax, grouped = per expert, empty experts).
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import workloads

MASK = oracle.DEFAULT_SIGN_MASK
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def sigma(mask=MASK):
    return np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])


def make_rows(codes, scale_code, St, At, H):
    """Hand-built packed rows: codes [n, H] (4-bit), one E4M3 scale code for
    every block, per-row token scale and amax."""
    n = codes.shape[0]
    S = oracle.row_bytes(H)
    rows = np.zeros((n, S), np.uint8)
    rows[:, : H // 2] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    rows[:, H // 2: H // 2 + H // 16] = scale_code
    rows[:, S - 16:S - 12] = np.full((n, 1), St, np.float32).view(np.uint8)
    rows[:, S - 12:S - 8] = np.broadcast_to(np.asarray(At, np.float32), (n,)).reshape(n, 1).copy().view(np.uint8)
    return rows


def cw_code(out, off, n, H, h, j):
    b = out["cw_codes"][off * H // 2 + h * (n // 2) + j // 2]
    return (b >> (4 * (j % 2))) & 0xF


def cw_scale(out, off, n, H, h, blk):
    return out["cw_scales"][off * H // 16 + h * (n // 16) + blk]


def test_tight_4x_case():
    """Rows whose decoded column is a * sigma_i: y_0 = 4a, other y_i = 0.
    The bound-derived scale then lands exactly on E4M3 448 and y_0 on 6."""
    H, n, m = 32, 128, 3          # magnitude index 3 -> a = 1.5
    a = GRID[m]
    codes = np.full((n, H), m, np.int64)
    sig = np.tile(sigma(), n // 16)
    codes[sig < 0] |= 8
    rows = make_rows(codes, 0x38, 1.0, a, H)      # E4M3 0x38 = 1.0
    off = np.array([0, n], np.int32)
    out = oracle.nvfp4_direct_receive(rows, H, off, 1)
    assert out["amax_row"][0] == a and out["amax_col"][0] == 4 * a
    assert out["scale_enc"][0] == np.float32(2688.0) / np.float32(4 * a)
    for h in range(H):
        for blk in range(n // 16):
            assert cw_scale(out, 0, n, H, h, blk) == 126                   # 448
            assert cw_code(out, 0, n, H, h, 16 * blk) == 7                 # +6
            for i in range(1, 16):
                assert cw_code(out, 0, n, H, h, 16 * blk + i) & 7 == 0
    assert out["report"]["above_4x_block_input"] == 0


def test_single_spike_fixes_layout_and_signs():
    """One nonzero decoded value g at (row l of block 1, column h0): every
    output of that block in column h0 has |y_i| = g/4 with sign
    sigma_l * H16[i][l]; everything else is zero."""
    H, n = 64, 128
    Hm = scipy.linalg.hadamard(16)
    for l, h0 in [(0, 0), (5, 17), (15, 63)]:
        codes = np.zeros((n, H), np.int64)
        codes[16 + l, h0] = 4                       # g = 2
        At = np.zeros(n); At[16 + l] = 2.0
        rows = make_rows(codes, 0x38, 1.0, At, H)
        out = oracle.nvfp4_direct_receive(rows, H, np.array([0, n], np.int32), 1)
        # S_enc = 2688/8 = 336, B = 0.5 -> s = 0.5*56 = 28 (exact E4M3), v = 6
        assert out["scale_enc"][0] == 336.0
        for h in range(H):
            for blk in range(n // 16):
                sc = cw_scale(out, 0, n, H, h, blk)
                for i in range(16):
                    c = cw_code(out, 0, n, H, h, 16 * blk + i)
                    if h == h0 and blk == 1:
                        assert torch.tensor([sc], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item() == 28.0
                        want_sign = sigma()[l] * Hm[i, l] < 0
                        assert c == (7 | (8 if want_sign else 0))
                    else:
                        assert c & 7 == 0 and sc == 0


def pipeline(w, rounding=0, seed=0):
    off, cnt, dest, st = oracle.route_plan(w.topk, w.E, w.A)
    Rc = oracle.rows_capacity(w.T, w.k, w.E, w.A)
    rows = oracle.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, Rc, rounding=rounding, seed=seed)
    out = oracle.nvfp4_direct_receive(rows, w.H, off, w.E, rounding=rounding, seed=seed)
    return off, cnt, dest, rows, out


def test_rowwise_is_the_senders_codes_and_metadata():
    w = workloads.make(2, T=96, H=256)
    off, cnt, dest, rows, out = pipeline(w)
    R = off[-1]
    H, S = w.H, oracle.row_bytes(w.H)
    np.testing.assert_array_equal(out["rw_codes"][:R], rows[:R, : H // 2])
    np.testing.assert_array_equal(out["rw_scales"][:R], rows[:R, H // 2: H // 2 + H // 16])
    np.testing.assert_array_equal(out["rw_row_scale"][:R], rows[:R, S - 16:S - 12].view(np.float32)[:, 0])
    x = workloads.bf16_bits_to_f32(w.tokens)
    for e in range(w.E):
        toks = [t for t in range(w.T) for j in range(w.k) if w.topk[t, j] == e]
        amax = np.abs(x[toks]).max() if toks else 0.0
        assert out["amax_row"][e] == amax                   # equals the BF16 amax
        assert out["amax_col"][e] == np.float32(4) * np.float32(amax)
        se = np.float32(2688) / np.float32(4 * amax) if amax > 0 else np.float32(1)
        assert out["scale_enc"][e] == se
        if not toks:
            assert off[e + 1] == off[e]                     # empty expert: no rows
    assert (cnt[14:] == 0).all() and out["scale_enc"][14] == 1.0


def test_grouped_equals_per_expert():
    w = workloads.make(3, T=128, H=256)
    off, cnt, dest, rows, out = pipeline(w)
    H = w.H
    for e in range(w.E):
        n = off[e + 1] - off[e]
        sub = rows[off[e]:off[e + 1]]
        one = oracle.nvfp4_direct_receive(sub, H, np.array([0, n], np.int32), 1)
        np.testing.assert_array_equal(one["cw_codes"][: n * H // 2],
                                      out["cw_codes"][off[e] * H // 2:(off[e] + n) * H // 2])
        np.testing.assert_array_equal(one["cw_scales"][: n * H // 16],
                                      out["cw_scales"][off[e] * H // 16:(off[e] + n) * H // 16])
        assert one["scale_enc"][0] == out["scale_enc"][e]


def test_columnwise_round_trip_and_bound_report():
    """Dequantise the columnwise operand, undo the RHT in float64 and compare
    with the decoded rows: a transposed layout, a wrong sign or a wrong scale
    would give an error of order 1; NVFP4 gives roughly 10%."""
    H = scipy.linalg.hadamard(16).astype(np.float64)
    w = workloads.make(1, T=256, H=256)
    off, cnt, dest, rows, out = pipeline(w)
    dec = workloads.bf16_bits_to_f32(oracle.nvfp4_unpack(rows, w.H, off, w.E)).astype(np.float64)
    e4 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    num = den = 0.0
    for e in range(w.E):
        o, n = off[e], off[e + 1] - off[e]
        cb = out["cw_codes"][o * w.H // 2:(o + n) * w.H // 2].reshape(w.H, n // 2)
        c = np.empty((w.H, n), np.int64)
        c[:, 0::2] = cb & 0xF
        c[:, 1::2] = cb >> 4
        sc = out["cw_scales"][o * w.H // 16:(o + n) * w.H // 16].reshape(w.H, n // 16)
        y = np.where(c & 8, -1.0, 1.0) * GRID[c & 7] * np.repeat(e4[sc], 16, axis=1) / out["scale_enc"][e]
        yb = y.reshape(w.H, n // 16, 16)
        d = sigma()[None, None, :] * (0.25 * np.einsum("ij,hbj->hbi", H, yb))
        ref = dec[o:o + n].T.reshape(w.H, n // 16, 16)
        num += ((d - ref) ** 2).sum()
        den += (ref ** 2).sum()
    rel = np.sqrt(num / den)
    assert 0.01 < rel < 0.2, rel
    assert out["report"]["above_4x_block_input"] == 0
    assert out["report"]["scale_saturated"] == 0


def test_sr_columnwise_stays_within_one_step():
    w = workloads.make(4, T=64, H=256, E=8, k=4)
    _, _, _, rows, sr = pipeline(w, rounding=1, seed=1234)
    off, *_ = oracle.route_plan(w.topk, w.E, w.A)
    rn = oracle.nvfp4_direct_receive(rows, w.H, off, w.E, rounding=0)
    np.testing.assert_array_equal(sr["cw_scales"], rn["cw_scales"])
    a = np.concatenate([sr["cw_codes"] & 0xF, sr["cw_codes"] >> 4])
    b = np.concatenate([rn["cw_codes"] & 0xF, rn["cw_codes"] >> 4])
    assert np.all(np.abs(GRID[a & 7] - GRID[b & 7]) <= 2.0)
    assert (a != b).mean() > 0.05        # SR does change codes
