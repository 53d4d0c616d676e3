"""GPU parity at the full workload sizes (the dispatch-forward, imbalanced,
combine-backward and MXFP8-vs-NVFP4 batches), with the path called exactly as
the benchmark calls it.  The oracle cannot redo a whole batch in test time,
so the check is by samples it computes one by one, plus facts that hold at
any size:

* the routing plan: the whole plan, against the oracle (integer work);
* packed rows: every destination row of sampled tokens against the oracle's
  packing of that token; sampled padding rows against the oracle's padding
  row;
* per-expert metadata of every expert: A_e = max |x| over the expert's
  tokens (the definition; a numpy maximum), 4 A_e and S_enc = 2688 / (4 A_e)
  in FP32;
* direct receive: every output byte of two sampled experts (the smallest
  and a median-sized one) against the oracle run on those experts' rows;
* MXFP8 (last batch): the destination rows of sampled tokens.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantization_gb300 as nq
import oracle
import workloads
from paths import assert_bytes_equal, to_dev_bf16

pytestmark = pytest.mark.gpu

FLT_MAX = np.float32(3.4028234663852886e38)


class FullRun:
    """The benchmark's step on one full-size batch (route plan and pack in one
    dispatch call, direct receive; MXFP8 pack for the last batch), outputs
    kept on the device."""

    def __init__(self, cfg):
        w = workloads.make(cfg)
        self.w = w
        self.tok = to_dev_bf16(w.tokens)
        self.topk = torch.from_numpy(np.ascontiguousarray(w.topk)).cuda()
        # the benchmark's calls: route plan + pack in one dispatch call
        self.plan, self.rows = nq.ep_nvfp4_dispatch(self.tok, self.topk, w.E, w.A, rounding=w.rounding,
                                                    seed=w.seed)
        self.R_cap = self.plan.R_cap
        self.out = nq.ep_nvfp4_direct_receive(self.rows, w.H, self.plan.offsets, w.E, rounding=w.rounding,
                                              seed=w.seed, sign_mask=w.sign_mask, status=self.plan.status)
        self.mx = nq.ep_mxfp8_pack(self.tok, self.plan) if "mxfp8_pack" in w.ops else None
        torch.cuda.synchronize()
        self.off = self.plan.offsets.cpu().numpy()
        self.cnt = self.plan.counts.cpu().numpy()
        self.dest = self.plan.dest.cpu().numpy()[: w.T * w.k]


@pytest.fixture(scope="module", params=[2, 3, 4, 5], ids=lambda c: f"cfg{c}")
def run(request):
    r = FullRun(request.param)
    yield r
    del r
    torch.cuda.empty_cache()


def test_route_plan_whole(run):
    w = run.w
    off, cnt, dest, st = oracle.route_plan(w.topk, w.E, w.A)
    assert_bytes_equal(run.off, off, "expert_offsets")
    assert_bytes_equal(run.cnt, cnt, "expert_counts")
    assert_bytes_equal(run.dest, dest, "dest")
    assert int(run.plan.status.item()) == st == 0


def test_sampled_token_rows(run):
    w = run.w
    rng = np.random.default_rng(100 + w.T)
    sample = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 46, replace=False)]))
    for t in sample:
        want = oracle.pack_token(w.tokens[t], token_id=int(t), rounding=w.rounding, seed=w.seed, t_index=int(t))
        for j in range(w.k):
            d = int(run.dest[t * w.k + j])
            if d >= 0:
                assert_bytes_equal(run.rows[d].cpu().numpy(), want, f"row of token {t} slot {j}")


def test_sampled_padding_rows(run):
    w = run.w
    pad = np.concatenate([np.arange(run.off[e] + run.cnt[e], run.off[e + 1]) for e in range(w.E)])
    assert len(pad) > 0
    want = oracle.pack_token(np.zeros(w.H, np.uint16), token_id=0xFFFFFFFF)
    rng = np.random.default_rng(7)
    for r in rng.choice(pad, min(32, len(pad)), replace=False):
        assert_bytes_equal(run.rows[int(r)].cpu().numpy(), want, f"padding row {r}")


def test_expert_metadata_every_expert(run):
    w = run.w
    tok_amax = np.abs(workloads.bf16_bits_to_f32(w.tokens)).max(axis=1)
    a = np.zeros(w.E, np.float32)
    for e in range(w.E):
        rows_e = (w.topk == e).any(axis=1)
        if rows_e.any():
            a[e] = tok_amax[rows_e].max()
    ac = np.float32(4.0) * a
    with np.errstate(divide="ignore"):
        se = np.where(ac > 0, np.minimum(np.float32(2688.0) / ac, FLT_MAX), np.float32(1.0)).astype(np.float32)
    assert_bytes_equal(run.out["amax_row"].cpu().numpy().view(np.uint32), a.view(np.uint32), "amax_row")
    assert_bytes_equal(run.out["amax_col"].cpu().numpy().view(np.uint32), ac.view(np.uint32), "amax_col")
    assert_bytes_equal(run.out["cw_scale_enc"].cpu().numpy().view(np.uint32), se.view(np.uint32), "S_enc")


def sampled_experts(run):
    n = run.off[1:] - run.off[:-1]
    live = np.nonzero(n > 0)[0]
    by_size = live[np.argsort(n[live], kind="stable")]
    return sorted({int(by_size[0]), int(by_size[len(by_size) // 2])})


def test_direct_receive_of_sampled_experts(run):
    w = run.w
    H, S = w.H, nq.row_bytes(w.H)
    experts = sampled_experts(run)
    # the oracle's rows for those experts only (the rest stay zero and unread)
    rows = np.zeros((run.R_cap, S), np.uint8)
    src = np.full(run.R_cap, -1, np.int64)
    ok = run.dest >= 0
    src[run.dest[ok]] = np.nonzero(ok)[0] // w.k
    pad_row = oracle.pack_token(np.zeros(H, np.uint16), token_id=0xFFFFFFFF)
    for e in experts:
        for r in range(run.off[e], run.off[e + 1]):
            t = int(src[r])
            rows[r] = pad_row if t < 0 else oracle.pack_token(w.tokens[t], token_id=t, rounding=w.rounding,
                                                              seed=w.seed, t_index=t)
    o = oracle.nvfp4_direct_receive(rows, H, run.off, w.E, rounding=w.rounding, seed=w.seed,
                                    sign_mask=w.sign_mask, experts=experts)
    g = run.out
    for e in experts:
        a, b = int(run.off[e]), int(run.off[e + 1])
        for name, key in (("amax_row", "amax_row"), ("amax_col", "amax_col"), ("cw_scale_enc", "scale_enc")):
            assert_bytes_equal(g[name][e:e + 1].cpu().numpy().view(np.uint32), o[key][e:e + 1].view(np.uint32),
                               f"{name} of expert {e}")
        assert_bytes_equal(g["rw_codes"][a:b].cpu().numpy(), o["rw_codes"][a:b], f"rowwise codes of expert {e}")
        assert_bytes_equal(g["rw_scales"][a:b].cpu().numpy(), o["rw_scales"][a:b], f"rowwise scales of expert {e}")
        assert_bytes_equal(g["rw_row_scale"][a:b].cpu().numpy().view(np.uint32),
                           o["rw_row_scale"][a:b].view(np.uint32), f"row scales of expert {e}")
        assert_bytes_equal(g["cw_codes"][a * H // 2:b * H // 2].cpu().numpy(), o["cw_codes"][a * H // 2:b * H // 2],
                           f"columnwise codes of expert {e}")
        assert_bytes_equal(g["cw_scales"][a * H // 16:b * H // 16].cpu().numpy(),
                           o["cw_scales"][a * H // 16:b * H // 16], f"columnwise scales of expert {e}")
    assert o["report"]["above_4x_rowwise_amax"] == 0


def test_mxfp8_sampled_tokens(run):
    w = run.w
    if run.mx is None:
        pytest.skip("this batch has no MXFP8 pack")
    rng = np.random.default_rng(55)
    sample = np.sort(rng.choice(w.T, 40, replace=False))
    sub_dest = np.ascontiguousarray(run.dest.reshape(w.T, w.k)[sample].reshape(-1))
    want = oracle.mxfp8_pack(np.ascontiguousarray(w.tokens[sample]), sub_dest, w.k, run.off, run.cnt, w.E,
                             run.R_cap)
    Rc, H = run.R_cap, w.H
    got = run.mx.cpu().numpy()
    gd, gs = got[: Rc * H].reshape(Rc, H), got[Rc * H:].reshape(Rc, H // 32)
    wd, ws = want[: Rc * H].reshape(Rc, H), want[Rc * H:].reshape(Rc, H // 32)
    for d in sub_dest[sub_dest >= 0]:
        assert_bytes_equal(gd[d], wd[d], f"mxfp8 data row {d}")
        assert_bytes_equal(gs[d], ws[d], f"mxfp8 scale row {d}")


def test_swizzled_scales_of_sampled_experts(run):
    """The swizzled call on the full batch: for the two sampled experts, the
    columnwise scales equal the oracle's scales in the tiled layout, and the
    rowwise tiles of their rows equal the tiled rowwise scales."""
    w = run.w
    H = w.H
    if H % 128:
        pytest.skip("the tiled layout needs H % 128 == 0")
    g = nq.ep_nvfp4_direct_receive(run.rows, H, run.plan.offsets, w.E, rounding=w.rounding, seed=w.seed,
                                   sign_mask=w.sign_mask, status=run.plan.status, swizzled=True)
    lin = run.out
    torch.cuda.synchronize()
    for e in sampled_experts(run):
        a, b = int(run.off[e]), int(run.off[e + 1])
        n = b - a
        want_cw = oracle.scale_swizzle(lin["cw_scales"][a * H // 16:b * H // 16].cpu().numpy().reshape(H, n // 16))
        assert_bytes_equal(g["cw_scales"][a * H // 16:b * H // 16].cpu().numpy(), want_cw,
                           f"tiled columnwise scales of expert {e}")
        want_rw = oracle.scale_swizzle(lin["rw_scales"][a:b].cpu().numpy())
        assert_bytes_equal(g["rw_scales"].reshape(-1)[a * H // 16:b * H // 16].cpu().numpy(), want_rw,
                           f"tiled rowwise scales of expert {e}")
        assert torch.equal(g["cw_codes"][a * H // 2:b * H // 2], lin["cw_codes"][a * H // 2:b * H // 2])


def test_bf16_columnwise_paths_of_sampled_experts(run):
    """The BF16-input columnwise calls on the full batch's decoded rows (the
    unpack of the received rows, as the bench times them), checked for the
    sampled experts against the oracle run on those experts' rows alone:
    the supplied-amax RHT quantizer (given the direct receive's amaxes) and
    the columnwise MXFP8 operand."""
    w = run.w
    H = w.H
    x = nq.ep_nvfp4_unpack(run.rows, H, run.plan.offsets, w.E, status=run.plan.status)
    amax = run.out["amax_row"]
    cw = nq.ep_nvfp4_colwise_rht_bf16(x, run.plan.offsets, w.E, amax, rounding=w.rounding, seed=w.seed,
                                      sign_mask=w.sign_mask, status=run.plan.status)
    mx = nq.ep_mxfp8_colwise(x, run.plan.offsets, w.E, status=run.plan.status)
    torch.cuda.synchronize()
    assert int(run.plan.status.item()) == 0
    R_cap = run.R_cap
    am = amax.cpu().numpy()
    for e in sampled_experts(run):
        a, b = int(run.off[e]), int(run.off[e + 1])
        n = b - a
        xe = x[a:b].view(torch.int16).cpu().numpy().view(np.uint16)
        # the oracle on this expert alone: its rows at offset 0
        o = oracle.nvfp4_colwise_rht_bf16(xe, np.array([0, n], np.int32), 1, am[e:e + 1], rounding=w.rounding,
                                          seed=w.seed, sign_mask=w.sign_mask)
        # SR keys on the element's index off*H + h*n + row: the oracle's off is 0, so
        # compare codes only for RNE; scales and metadata for both
        if w.rounding == 0:
            assert_bytes_equal(cw["cw_codes"][a * H // 2:b * H // 2].cpu().numpy(), o["cw_codes"],
                               f"supplied-amax codes of expert {e}")
        assert_bytes_equal(cw["cw_scales"][a * H // 16:b * H // 16].cpu().numpy(), o["cw_scales"],
                           f"supplied-amax scales of expert {e}")
        assert cw["cw_scale_enc"][e].item() == o["scale_enc"][0]
        om = oracle.mxfp8_colwise(xe, np.array([0, n], np.int32), 1)
        got = mx.cpu().numpy()
        assert_bytes_equal(got[a * H:b * H], om[: n * H], f"columnwise MXFP8 data of expert {e}")
        assert_bytes_equal(got[R_cap * H + a * H // 32:R_cap * H + b * H // 32], om[n * H:],
                           f"columnwise MXFP8 scales of expert {e}")
