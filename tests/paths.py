"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
(via the package's thin binding) and the oracle on the same seeded inputs, and
compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_quantization_gb300 as nq
import oracle

CANARY = 0xAB


def to_dev_bf16(tokens_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(tokens_u16).view(np.int16)).view(torch.bfloat16).cuda()


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
    if len(bad):
        i = int(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {got.size} differ; first at flat index {i}: "
                             f"got {got.reshape(-1)[i]!r} want {want.reshape(-1)[i]!r}")


class DeviceRun:
    """The hot path on the GPU for one workload, with canary-filled outputs."""

    def __init__(self, w, rowwise=True, mxfp8=False, unpack=False, R_cap=None, dispatch=False, swizzled=False,
                 amax=False):
        """amax: the pack (or dispatch) reduces the per-expert amax, and the
        direct receive takes it instead of reducing the row trailers."""
        self.w = w
        self.swizzled = swizzled
        self.expert_amax = None
        if amax:
            # canary bits where the dispatch's routing kernel must write zeros;
            # the separate pack accumulates into what the caller put there
            self.expert_amax = torch.full((w.E,), 0.0, dtype=torch.float32, device="cuda")
            if dispatch:
                self.expert_amax.view(torch.int32).fill_(0x7F7F7F7F)
        self.tok = to_dev_bf16(w.tokens)
        self.topk = torch.from_numpy(np.ascontiguousarray(w.topk)).cuda()
        self.R_cap = R_cap or nq.rows_capacity(w.T, w.k, w.E, w.A)
        S = nq.row_bytes(w.H)
        self.rows = torch.full((self.R_cap, S), CANARY, dtype=torch.uint8, device="cuda")
        if dispatch:   # route plan + pack in one call
            self.plan, _ = nq.ep_nvfp4_dispatch(self.tok, self.topk, w.E, w.A, R_cap=self.R_cap, rows=self.rows,
                                                rounding=w.rounding, seed=w.seed, expert_amax=self.expert_amax)
        else:
            self.plan = nq.ep_route_plan(self.topk, w.E, w.A, R_cap=self.R_cap)
            nq.ep_nvfp4_pack(self.tok, self.plan, rows=self.rows, rounding=w.rounding, seed=w.seed,
                             expert_amax=self.expert_amax)
        g = nq.alloc_grouped(self.R_cap, w.H, w.E, "cuda", rowwise=rowwise)
        for t in g.values():
            t.view(torch.uint8).fill_(CANARY)
        self.grouped = nq.ep_nvfp4_direct_receive(self.rows, w.H, self.plan.offsets, w.E, out=g,
                                                  rounding=w.rounding, seed=w.seed, sign_mask=w.sign_mask,
                                                  status=self.plan.status, swizzled=swizzled,
                                                  expert_amax=self.expert_amax)
        self.unpacked = None
        if unpack:
            self.unpacked = torch.full((self.R_cap, w.H), 0, dtype=torch.bfloat16, device="cuda")
            self.unpacked.view(torch.uint8).fill_(CANARY)
            nq.ep_nvfp4_unpack(self.rows, w.H, self.plan.offsets, w.E, out=self.unpacked, status=self.plan.status)
        self.mx = None
        if mxfp8:
            self.mx = torch.full((self.R_cap * w.H + self.R_cap * (w.H // 32),), CANARY, dtype=torch.uint8,
                                 device="cuda")
            nq.ep_mxfp8_pack(self.tok, self.plan, buf=self.mx)
        torch.cuda.synchronize()

    def host(self, t):
        return t.cpu().numpy()

    @property
    def status(self) -> int:
        return int(self.plan.status.item()) & 0xFFFFFFFF


class OracleRun:
    def __init__(self, w, R_cap, unpack=False, mxfp8=False, experts=None):
        self.w = w
        self.off, self.cnt, self.dest, self.status = oracle.route_plan(w.topk, w.E, w.A)
        self.rows = oracle.nvfp4_pack(w.tokens, self.dest, w.k, self.off, self.cnt, w.E, R_cap,
                                      rounding=w.rounding, seed=w.seed)
        self.dr = oracle.nvfp4_direct_receive(self.rows, w.H, self.off, w.E, rounding=w.rounding, seed=w.seed,
                                              sign_mask=w.sign_mask, experts=experts)
        self.unpacked = oracle.nvfp4_unpack(self.rows, w.H, self.off, w.E) if unpack else None
        self.mx = oracle.mxfp8_pack(w.tokens, self.dest, w.k, self.off, self.cnt, w.E, R_cap) if mxfp8 else None


def compare_runs(g: DeviceRun, o: OracleRun, check_rowwise=True):
    w = g.w
    H = w.H
    R = int(o.off[-1])
    assert_bytes_equal(g.host(g.plan.offsets), o.off, "expert_offsets")
    assert_bytes_equal(g.host(g.plan.counts), o.cnt, "expert_counts")
    assert_bytes_equal(g.host(g.plan.dest)[: w.T * w.k], o.dest, "dest")
    assert g.status == o.status, (g.status, o.status)
    rows = g.host(g.rows)
    assert_bytes_equal(rows[:R], o.rows[:R], "packed rows")
    assert (rows[R:] == CANARY).all(), "rows beyond R were written"
    gr = {k: g.host(v) for k, v in g.grouped.items()}
    odr = oracle.swizzle_grouped_scales(o.dr, H, o.off, w.E) if g.swizzled else o.dr
    for name in ("amax_row", "amax_col", "cw_scale_enc"):
        oname = "scale_enc" if name == "cw_scale_enc" else name
        assert_bytes_equal(gr[name].view(np.uint32), o.dr[oname].view(np.uint32), name)
    if g.expert_amax is not None:   # the pack's reduction is the receive's rowwise amax
        assert_bytes_equal(g.host(g.expert_amax).view(np.uint32), o.dr["amax_row"].view(np.uint32),
                           "expert_amax from the pack")
    assert_bytes_equal(gr["cw_codes"][: R * H // 2], o.dr["cw_codes"][: R * H // 2], "columnwise codes")
    assert_bytes_equal(gr["cw_scales"][: R * H // 16], odr["cw_scales"][: R * H // 16], "columnwise scales")
    assert (gr["cw_codes"][R * H // 2:] == CANARY).all()
    assert (gr["cw_scales"][R * H // 16:] == CANARY).all()
    if check_rowwise and "rw_codes" in gr:
        assert_bytes_equal(gr["rw_codes"][:R], o.dr["rw_codes"][:R], "rowwise codes")
        assert_bytes_equal(gr["rw_scales"][:R], odr["rw_scales"][:R], "rowwise scales")
        assert (gr["rw_scales"][R:] == CANARY).all()
        assert_bytes_equal(gr["rw_row_scale"][:R].view(np.uint32), o.dr["rw_row_scale"][:R].view(np.uint32),
                           "rowwise row scale")
        assert (gr["rw_codes"][R:] == CANARY).all()
    if g.unpacked is not None:
        un = g.unpacked.view(torch.int16).cpu().numpy().view(np.uint16)
        assert_bytes_equal(un[:R], o.unpacked[:R], "unpacked bf16")
        assert (un[R:].view(np.uint8) == CANARY).all()
    if g.mx is not None:
        mx = g.host(g.mx)
        Rc = g.R_cap
        data, scl = mx[: Rc * H].reshape(Rc, H), mx[Rc * H:].reshape(Rc, H // 32)
        odata, oscl = o.mx[: Rc * H].reshape(Rc, H), o.mx[Rc * H:].reshape(Rc, H // 32)
        assert_bytes_equal(data[:R], odata[:R], "mxfp8 data")
        assert_bytes_equal(scl[:R], oscl[:R], "mxfp8 scales")
        assert (data[R:] == CANARY).all() and (scl[R:] == CANARY).all()
