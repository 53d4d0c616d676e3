"""Pins of the oracle's route plan, NVFP4 pack / unpack and MXFP8 pack.

The expected values come from independent formulations: a Python brute-force
route plan (sort by (expert, token)), torch's FP8 / BF16 conversions, the
threshold-count form of E2M1 rounding, closed forms of the token scale, a
hand-derived worked example, and the pack -> unpack error bound.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MIDPOINTS = [(0.25, False), (0.75, True), (1.25, False), (1.75, True),
             (2.5, False), (3.5, True), (5.0, False)]
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def bf16(x):
    return workloads.to_bf16_bits(np.asarray(x, np.float32))


def f32(b):
    return workloads.bf16_bits_to_f32(b).astype(np.float64)


def torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_e4m3_value(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


# ---------------------------------------------------------------- route plan
def brute_route(topk, E, A):
    T, k = topk.shape
    status = 0
    keep = np.full((T, k), -1)
    for t in range(T):
        seen = set()
        for j in range(k):
            e = int(topk[t, j])
            if e == -1:
                continue
            if not (0 <= e < E):
                status |= 1
                continue
            if e in seen:
                status |= 2
                continue
            seen.add(e)
            keep[t, j] = e
    pairs = sorted((int(keep[t, j]), t, j) for t in range(T) for j in range(k) if keep[t, j] >= 0)
    counts = np.array([sum(1 for p in pairs if p[0] == e) for e in range(E)])
    padded = -(-counts // A) * A
    offsets = np.concatenate([[0], np.cumsum(padded)])
    dest = np.full(T * k, -1)
    seen_e = {}
    for e, t, j in pairs:
        dest[t * k + j] = offsets[e] + seen_e.get(e, 0)
        seen_e[e] = seen_e.get(e, 0) + 1
    return offsets, counts, dest, status


@pytest.mark.parametrize("T,E,k,A", [(1, 1, 1, 128), (37, 5, 2, 128), (300, 16, 4, 256), (64, 3, 3, 128)])
def test_route_plan_brute_force(T, E, k, A):
    rng = np.random.default_rng(T * 7 + E)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    topk[rng.random((T, k)) < 0.1] = -1
    got = oracle.route_plan(topk, E, A)
    want = brute_route(topk, E, A)
    for g, w in zip(got[:3], want[:3]):
        np.testing.assert_array_equal(g, w)
    assert got[3] == want[3] == 0
    offs = got[0]
    assert np.all(offs % A == 0) and offs[-1] <= oracle.rows_capacity(T, k, E, A)
    d = got[2][got[2] >= 0]
    assert len(np.unique(d)) == len(d)


def test_route_plan_bad_and_duplicate_ids():
    topk = np.array([[0, 0], [5, 1], [-3, 2], [1, -1]], np.int32)
    got = oracle.route_plan(topk, 3, 128)
    want = brute_route(topk, 3, 128)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)
    assert got[3] == 3
    assert got[2].tolist() == [0, -1, -1, 128, -1, 256, 129, -1]


def test_route_plan_empty():
    off, cnt, dest, st = oracle.route_plan(np.zeros((0, 2), np.int32), 4, 128)
    assert off.tolist() == [0] * 5 and cnt.tolist() == [0] * 4 and st == 0


# ---------------------------------------------------------------- pack
def parse_row(row, H):
    S = oracle.row_bytes(H)
    codes = np.empty(H, np.int64)
    codes[0::2] = row[: H // 2] & 0xF
    codes[1::2] = row[: H // 2] >> 4
    scales = row[H // 2: H // 2 + H // 16]
    tr = row[S - 16:S].view(np.float32)
    tid = row[S - 8:S - 4].view(np.uint32)[0]
    return codes, scales, float(tr[0]), float(tr[1]), int(tid)


def test_pack_worked_example():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "nvfp4_pack_worked_example.txt"))
             if l.strip() and not l.startswith("#")]
    xs = {int(l[1]): [float(v) for v in l[3:]] for l in lines if l[2] == "x"}
    rows = {int(l[1]): l for l in lines if l[2] == "row"}
    for t, x in xs.items():
        row = oracle.pack_token(bf16(x), token_id=t)
        l = rows[t]
        want = bytes(int(h, 16) for h in l[3:21])
        assert bytes(row[:18]) == want, (t, row[:18].tobytes().hex())
        _, _, St, At, tid = parse_row(row, 32)
        assert St == float(l[22]) and At == float(l[24]) and tid == t


def closed_form_pack(xb):
    """Independent restatement used as a pin: torch E4M3 for the block scale,
    threshold counting for the codes."""
    x = f32(xb)
    H = x.shape[0]
    A = np.abs(x).max()
    k = -126
    if A > 0:
        m, e = math.frexp(A / 2688.0)
        k = max(e if m != 0.5 else e - 1, -126)
    S = math.ldexp(1.0, k)
    B = np.abs(x).reshape(-1, 16).max(axis=1)
    sb = torch_e4m3((B / (6.0 * S)).astype(np.float32))
    s = torch_e4m3_value(sb) * S
    a = np.abs(x).reshape(-1, 16)
    m = np.zeros(a.shape, np.int64)
    for mu, up in MIDPOINTS:
        t = mu * s[:, None]
        m += (a >= t) if up else (a > t)
    m[s == 0] = 0
    codes = m.reshape(-1) | np.where(np.signbit(x), 8, 0)
    return codes, sb, S, A


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_pack_matches_closed_form(cfg):
    w = workloads.make(cfg, T=24, H=512)
    for t in range(w.T):
        row = oracle.pack_token(w.tokens[t], token_id=t)
        codes, scales, St, At, tid = parse_row(row, w.H)
        c2, sb2, S2, A2 = closed_form_pack(w.tokens[t])
        np.testing.assert_array_equal(codes, c2)
        np.testing.assert_array_equal(scales, sb2)
        assert St == S2 and At == A2 and tid == t
        assert np.all(scales <= 126)  # no NaN, within 448


def test_pack_edge_tokens():
    H = 64
    cases = [np.zeros(H), -np.zeros(H), np.full(H, 3e38), np.full(H, 1e-38),
             np.r_[np.full(H - 1, 1e-30), 1e30], np.r_[1.0, np.full(H - 1, -0.0)]]
    for x in cases:
        xb = bf16(x)
        row = oracle.pack_token(xb)
        codes, scales, St, At, _ = parse_row(row, H)
        c2, sb2, S2, A2 = closed_form_pack(xb)
        np.testing.assert_array_equal(codes, c2)
        np.testing.assert_array_equal(scales, sb2)
        assert St == S2 and At == A2


def test_pack_unpack_error_bound_and_exactness():
    w = workloads.make(3, T=64, H=1024)
    off, cnt, dest, st = oracle.route_plan(w.topk, w.E, w.A)
    Rc = oracle.rows_capacity(w.T, w.k, w.E, w.A)
    rows = oracle.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, Rc)
    out = oracle.nvfp4_unpack(rows, w.H, off, w.E)
    x = f32(w.tokens)
    for t in range(w.T):
        for j in range(w.k):
            d = dest[t * w.k + j]
            codes, scales, St, At, tid = parse_row(rows[d], w.H)
            s = torch_e4m3_value(scales).repeat(16) * St
            # exact decode, rounded to BF16 by torch
            val = np.where(codes & 8, -1.0, 1.0) * GRID[codes & 7] * s
            want = torch.from_numpy(val).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            np.testing.assert_array_equal(out[d], want)
            # |x - x_hat| <= half the local grid gap times s, or saturation
            xh = f32(out[d])
            v = np.abs(x[t]) / np.where(s > 0, s, 1)
            gap = np.select([v < 2, v < 4], [0.5, 1.0], 2.0)
            err = np.abs(x[t] - xh)
            ok = (err <= 0.5 * gap * s * (1 + 1e-12)) | ((v > 6) & (np.abs(xh) == 6 * s)) | (s == 0)
            assert ok.all()
            assert np.max(np.abs(x[t])) == At
    # padding rows are the packing of an all-zero token with id 0xFFFFFFFF
    zero = oracle.pack_token(np.zeros(w.H, np.uint16), token_id=0xFFFFFFFF)
    for e in range(w.E):
        for r in range(off[e] + cnt[e], off[e + 1]):
            np.testing.assert_array_equal(rows[r], zero)


def test_pack_duplicates_identical_with_sr():
    w = workloads.make(4, T=40, H=256, E=8, k=4)
    off, cnt, dest, st = oracle.route_plan(w.topk, w.E, w.A)
    Rc = oracle.rows_capacity(w.T, w.k, w.E, w.A)
    rows = oracle.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, Rc, rounding=1, seed=77)
    rne = oracle.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, Rc, rounding=0)
    for t in range(w.T):
        ds = dest[t * w.k:(t + 1) * w.k]
        for d in ds[1:]:
            np.testing.assert_array_equal(rows[d], rows[ds[0]])
        c_sr, s_sr, *_ = parse_row(rows[ds[0]], w.H)
        c_rn, s_rn, *_ = parse_row(rne[ds[0]], w.H)
        np.testing.assert_array_equal(s_sr, s_rn)  # scales stay RNE
        step = np.abs(GRID[c_sr & 7] - GRID[c_rn & 7])
        assert np.all(step <= 2.0)


# ---------------------------------------------------------------- MXFP8
def test_mxfp8_pack_pins():
    w = workloads.make(5, T=48, H=512)
    off, cnt, dest, st = oracle.route_plan(w.topk, w.E, w.A)
    Rc = oracle.rows_capacity(w.T, w.k, w.E, w.A)
    buf = oracle.mxfp8_pack(w.tokens, dest, w.k, off, cnt, w.E, Rc)
    data = buf[: Rc * w.H].reshape(Rc, w.H)
    scl = buf[Rc * w.H:].reshape(Rc, w.H // 32)
    x = f32(w.tokens)
    E_ = np.arange(-127, 128)
    for t in range(w.T):
        B = np.abs(x[t]).reshape(-1, 32).max(axis=1)
        ok = B[:, None] <= 448.0 * np.ldexp(1.0, E_)[None, :]
        e = E_[np.argmax(ok, axis=1)]
        q = torch_e4m3((x[t].reshape(-1, 32) / np.ldexp(1.0, e)[:, None]).reshape(-1))
        for j in range(w.k):
            d = dest[t * w.k + j]
            np.testing.assert_array_equal(scl[d], (e + 127).astype(np.uint8))
            np.testing.assert_array_equal(data[d], q)
            assert np.all(np.abs(torch_e4m3_value(data[d])) <= 448)
    for e in range(w.E):
        for r in range(off[e] + cnt[e], off[e + 1]):
            assert not data[r].any() and not scl[r].any()
