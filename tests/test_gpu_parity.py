"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, bit for bit (codes, scales, metadata, decoded BF16,
MXFP8 bytes, routing).  Sizes here are ones the oracle finishes in seconds
while still spanning several tiles and a ragged tail; the full-size configs
are in test_gpu_fullsize.py."""
import numpy as np
import pytest
import torch

import nvfp4_quantization_gb300 as nq
import oracle
import workloads
from paths import CANARY, DeviceRun, OracleRun, assert_bytes_equal, compare_runs, to_dev_bf16

pytestmark = pytest.mark.gpu


CASES = {
    "cfg1": dict(cfg=1, kw={}, unpack=True),
    "cfg2": dict(cfg=2, kw=dict(T=600, H=1024), unpack=False),
    "cfg3": dict(cfg=3, kw=dict(T=700, H=2048), unpack=True),
    "cfg4": dict(cfg=4, kw=dict(T=300, H=1024, E=64, k=8), unpack=False),
    "cfg5": dict(cfg=5, kw=dict(T=400, H=1024), unpack=False, mxfp8=True),
    "cfg1_ragged_H": dict(cfg=1, kw=dict(T=130, H=1056), unpack=True, mxfp8=True),
    "cfg4_ragged_H": dict(cfg=4, kw=dict(T=90, H=288, E=16, k=4), unpack=True, mxfp8=True),
    # more tiles than the receive has CTAs, with a strip count (6) that does not
    # divide the grid: every CTA steps to its later tiles across strip rows
    "cfg3_tile_walk": dict(cfg=3, kw=dict(T=4000, H=1312), unpack=False),
    "cfg4_tile_walk": dict(cfg=4, kw=dict(T=1200, H=1312, E=32, k=8), unpack=False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_parity_config(name):
    c = CASES[name]
    w = workloads.make(c["cfg"], **c["kw"])
    g = DeviceRun(w, unpack=c.get("unpack", False), mxfp8=c.get("mxfp8", False))
    o = OracleRun(w, g.R_cap, unpack=c.get("unpack", False), mxfp8=c.get("mxfp8", False))
    compare_runs(g, o)


@pytest.mark.parametrize("name", ["cfg1", "cfg2", "cfg4", "cfg5", "cfg4_ragged_H"])
def test_parity_dispatch(name):
    """ep_nvfp4_dispatch (route plan + pack in one call, the pack encoding
    its first tokens while the routing kernel runs) against the oracle; the
    ragged-H case takes the pack kernel without the early reads."""
    c = CASES[name]
    w = workloads.make(c["cfg"], **c["kw"])
    g = DeviceRun(w, unpack=c.get("unpack", False), mxfp8=c.get("mxfp8", False), dispatch=True)
    o = OracleRun(w, g.R_cap, unpack=c.get("unpack", False), mxfp8=c.get("mxfp8", False))
    compare_runs(g, o)


def test_parity_dispatch_sr_many_tokens_per_warp():
    """More tokens than the pack's resident warps (several tokens per warp
    after the first), stochastic rounding, through ep_nvfp4_dispatch."""
    w = workloads.make(4, T=9000, H=512, E=32, k=3)
    g = DeviceRun(w, dispatch=True)
    o = OracleRun(w, g.R_cap)
    compare_runs(g, o)


@pytest.mark.parametrize("name", ["cfg1", "cfg2", "cfg4", "cfg5"])
def test_parity_swizzled_scales(name):
    """ep_nvfp4_direct_receive_swizzled: codes, row scales and metadata as the
    linear call, both scale tensors equal to the oracle's scales put in the
    tiled layout (rowwise over rows [0, R), columnwise per expert)."""
    c = CASES[name]
    w = workloads.make(c["cfg"], **c["kw"])
    g = DeviceRun(w, swizzled=True)
    o = OracleRun(w, g.R_cap)
    compare_runs(g, o)


def test_parity_swizzled_scales_256_row_slots():
    """The tiled scale layout with expert slots aligned to 256 rows (A = 256):
    every expert's columnwise scale matrix spans whole 128-row tile pairs, and
    the rowwise matrix's tiles run across expert boundaries unchanged."""
    w = workloads.make(2, T=700, H=1024)
    w = workloads.Workload("a256", "a256", w.tokens, w.topk, E=w.E, A=256)
    for dispatch in (False, True):
        g = DeviceRun(w, swizzled=True, dispatch=dispatch, amax=dispatch)
        compare_runs(g, OracleRun(w, g.R_cap))


def test_swizzled_scales_need_h_multiple_of_128():
    w = workloads.make(1, T=64, H=1056)
    tok = to_dev_bf16(w.tokens)
    plan = nq.ep_route_plan(torch.from_numpy(w.topk).cuda(), w.E, w.A)
    rows = nq.ep_nvfp4_pack(tok, plan)
    with pytest.raises(nq.EpError) as ei:
        nq.ep_nvfp4_direct_receive(rows, w.H, plan.offsets, w.E, status=plan.status, swizzled=True)
    assert ei.value.status == -2


def test_parity_rne_and_sr_on_same_tokens():
    base = workloads.make(4, T=200, H=512, E=16, k=4)
    for rounding, seed in ((0, 0), (1, 1), (1, 0xFFFFFFFFFFFF1234)):
        base.rounding, base.seed = rounding, seed
        g = DeviceRun(base)
        o = OracleRun(base, g.R_cap)
        compare_runs(g, o)


def test_parity_without_rowwise_outputs():
    w = workloads.make(2, T=300, H=512)
    g = DeviceRun(w, rowwise=False)
    o = OracleRun(w, g.R_cap)
    compare_runs(g, o, check_rowwise=False)


def special_tokens(H=512):
    """Tokens that reach every branch of the encoder: the fast and the slow
    division paths (tiny and huge token scales, the -126 floor), zero tokens,
    negative zeros, exact ties, saturation."""
    rng = np.random.default_rng(9)
    rows = []
    for scale in (1.0, 1e-30, 1e30, 3e-37, 1e-38, 2.0 ** -110, 2.0 ** 105, 3.0e37):
        x = rng.standard_normal(H).astype(np.float32) * np.float32(scale)
        rows.append(x)
    rows.append(np.zeros(H, np.float32))
    z = np.zeros(H, np.float32)
    z[::3] = -0.0
    rows.append(z)
    ties = np.tile(np.array([6, 1, 0.5, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -5, -0.25, 4.5, 0, -0.0, 3],
                            np.float32), H // 16)
    rows.append(ties)
    rows.append(ties * np.float32(2.0 ** -100))
    one = np.zeros(H, np.float32)
    one[7] = -3.0
    rows.append(one)
    return workloads.to_bf16_bits(np.stack(rows))


def test_parity_special_tokens_and_routing_edges():
    tokens = special_tokens()
    T = tokens.shape[0]
    topk = np.array([[i % 5, (i + 2) % 5] for i in range(T)], np.int32)
    topk[1, 1] = -1           # dropped slot
    topk[2, 1] = 9            # id out of range -> status bit, dropped
    topk[3, 1] = topk[3, 0]   # repeated id -> status bit, later slot dropped
    w = workloads.Workload("special", "special", tokens, topk, E=5)
    g = DeviceRun(w, unpack=True, mxfp8=True)
    o = OracleRun(w, g.R_cap, unpack=True, mxfp8=True)
    assert o.status == 3
    compare_runs(g, o)


def test_parity_empty_and_single_token():
    for T, E in ((0, 4), (1, 1), (1, 8)):
        rng = np.random.default_rng(T + E)
        tokens = workloads.to_bf16_bits(rng.standard_normal((T, 256)).astype(np.float32))
        k = min(2, E)
        topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
            np.zeros((0, k), np.int32)
        w = workloads.Workload("edge", "edge", tokens, topk, E=E)
        g = DeviceRun(w, unpack=True, mxfp8=True)
        o = OracleRun(w, g.R_cap, unpack=True, mxfp8=True)
        compare_runs(g, o)


def test_parity_all_slots_dropped_and_one_hot_expert():
    rng = np.random.default_rng(3)
    tokens = workloads.to_bf16_bits(rng.standard_normal((700, 256)).astype(np.float32))
    topk = np.full((700, 2), -1, np.int32)
    w = workloads.Workload("dropped", "dropped", tokens, topk, E=3)
    g = DeviceRun(w)
    o = OracleRun(w, g.R_cap)
    compare_runs(g, o)
    topk = np.zeros((700, 1), np.int32) + 2   # every token to expert 2, 700 rows -> ragged 768
    w = workloads.Workload("hot", "hot", tokens, topk, E=3, A=256)
    g = DeviceRun(w, unpack=True)
    o = OracleRun(w, g.R_cap, unpack=True)
    compare_runs(g, o)


def exhaustive_encode_tokens(token_scale_exp: int, H=2048):
    """Blocks whose max fixes every positive E4M3 block scale s_b (B = 6 s_b S_t)
    filled with every BF16 magnitude in [2^-10 s, 6 s] (both signs): every
    (value, block scale) pair of the encoder's decision range appears."""
    St = 2.0 ** token_scale_exp
    e4 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    allbf = (np.arange(1 << 15, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    allbf = allbf[np.isfinite(allbf)]
    blocks = []
    for code in range(1, 127):
        s = e4[code] * St
        B = 6.0 * s
        vals = allbf[(allbf >= s * 2.0 ** -10) & (allbf <= B)]
        vals = np.concatenate([vals, -vals])
        n = len(vals)
        nb = -(-n // 15)
        pad = np.resize(vals, nb * 15).reshape(nb, 15)
        blk = np.concatenate([np.full((nb, 1), B), pad], axis=1)
        blocks.append(blk)
    blocks = np.concatenate(blocks)
    per_tok = H // 16 - 1
    ntok = -(-len(blocks) // per_tok)
    blocks = np.resize(blocks, (ntok * per_tok, 16))
    # first block of every token carries the token amax 2688 * S_t (S_t exact)
    first = np.zeros((ntok, 16))
    first[:, 0] = 2688.0 * St
    tok = np.concatenate([first[:, None, :], blocks.reshape(ntok, per_tok, 16)], axis=1).reshape(ntok, H)
    return workloads.to_bf16_bits(tok.astype(np.float32))


@pytest.mark.parametrize("kexp", [0, -20, 12, -110, 105])
def test_parity_exhaustive_encode(kexp):
    tokens = exhaustive_encode_tokens(kexp)
    T = tokens.shape[0]
    topk = (np.arange(T, dtype=np.int32) % 4).reshape(T, 1)
    for rounding in (0, 1):
        w = workloads.Workload("exh", "exh", tokens, topk, E=4, rounding=rounding, seed=17)
        g = DeviceRun(w, unpack=True)
        o = OracleRun(w, g.R_cap, unpack=True)
        compare_runs(g, o)


def test_deterministic_repeat():
    w = workloads.make(4, T=200, H=512, E=16, k=4)
    a = DeviceRun(w, mxfp8=True, unpack=True)
    b = DeviceRun(w, mxfp8=True, unpack=True)
    assert torch.equal(a.rows, b.rows)
    for k in a.grouped:
        assert torch.equal(a.grouped[k], b.grouped[k]), k
    assert torch.equal(a.mx, b.mx) and torch.equal(a.unpacked.view(torch.int16), b.unpacked.view(torch.int16))


def test_cuda_graph_capture_matches_eager():
    """Route plan + pack + direct receive captured in one CUDA graph replay to
    the same bytes as the eager calls (the library allocates nothing and never
    synchronises, so every call is capturable)."""
    w = workloads.make(2, T=500, H=1024)
    eager = DeviceRun(w)
    tok = to_dev_bf16(w.tokens)
    topk = torch.from_numpy(w.topk).cuda()
    R_cap = eager.R_cap
    plan = nq.ep_route_plan(topk, w.E, w.A, R_cap=R_cap)      # warm-up call, allocates outputs
    ws = nq.new_route_workspace(w.T, w.k, w.E, "cuda")
    rows = torch.empty((R_cap, nq.row_bytes(w.H)), dtype=torch.uint8, device="cuda")
    out = nq.alloc_grouped(R_cap, w.H, w.E, "cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            nq.ep_route_plan(topk, w.E, w.A, R_cap=R_cap, plan=plan, workspace=ws)
            nq.ep_nvfp4_pack(tok, plan, rows=rows)
            nq.ep_nvfp4_direct_receive(rows, w.H, plan.offsets, w.E, out=out, status=plan.status)
            # the same again through the one-call dispatch (a second step in the graph)
            nq.ep_nvfp4_dispatch(tok, topk, w.E, w.A, plan=plan, workspace=ws, rows=rows)
            nq.ep_nvfp4_direct_receive(rows, w.H, plan.offsets, w.E, out=out, status=plan.status)
    rows.fill_(CANARY)
    for t in out.values():
        t.view(torch.uint8).fill_(CANARY)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    R = int(plan.offsets[-1].item())
    assert torch.equal(rows[:R], eager.rows[:R])
    for k, v in out.items():
        n = {"cw_codes": R * w.H // 2, "cw_scales": R * w.H // 16}.get(k)
        ref = eager.grouped[k]
        if k.startswith("rw"):
            assert torch.equal(v[:R], ref[:R]), k
        elif n is not None:
            assert torch.equal(v[:n], ref[:n]), k
        else:
            assert torch.equal(v, ref), k


def test_pointer_off_the_input_device_is_refused():
    """Device guard: every pointer must be memory of the device that owns the
    first input.  A call whose output lives in host memory (pinned, so that
    CUDA knows it) returns EP_ERR_DEVICE and enqueues nothing: the device
    outputs it was also given keep their contents."""
    import ctypes
    from nvfp4_quantization_gb300 import _lib
    T, k, E = 64, 2, 4
    topk = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    topk[:, 1] = 1
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    dest_host = torch.full((T * k,), -7, dtype=torch.int32).pin_memory()
    ws = nq.new_route_workspace(T, k, E, "cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    R_cap = nq.rows_capacity(T, k, E, 128)
    s = _lib.lib().ep_route_plan(p(topk), T, k, E, 128, R_cap, p(off), p(cnt), p(dest_host), p(ws),
                                 ws.numel() * 4, p(st), None)
    torch.cuda.synchronize()
    assert s == -6                                    # EP_ERR_DEVICE
    assert torch.all(off == -7) and torch.all(cnt == -7) and torch.all(dest_host == -7)
    # the same call with the destination on the device runs
    dest = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    s = _lib.lib().ep_route_plan(p(topk), T, k, E, 128, R_cap, p(off), p(cnt), p(dest), p(ws), ws.numel() * 4,
                                 p(st), None)
    torch.cuda.synchronize()
    assert s == 0 and int(off[E].item()) == 2 * 128


@pytest.mark.parametrize("T,E,k", [(3000, 32, 12), (400000, 64, 2), (20000, 1024, 3), (200000, 64, 4)])
def test_route_plan_general_paths(T, E, k):
    """Routing alone on shapes that leave the register fast path: k > 8, more
    512-token chunks than resident CTAs (several chunks per CTA), and more
    chunks than the register kernel can keep resident but not than the
    general kernel can (one chunk per CTA on the general kernel)."""
    rng = np.random.default_rng(T + k)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    topk[rng.random((T, k)) < 0.02] = -1
    off, cnt, dest, st = oracle.route_plan(topk, E, 128)
    plan = nq.ep_route_plan(torch.from_numpy(topk).cuda(), E, 128)
    torch.cuda.synchronize()
    assert_bytes_equal(plan.offsets.cpu().numpy(), off, "offsets")
    assert_bytes_equal(plan.counts.cpu().numpy(), cnt, "counts")
    assert_bytes_equal(plan.dest.cpu().numpy()[: T * k], dest, "dest")
    assert int(plan.status.item()) == st == 0


@pytest.mark.parametrize("T,E,k", [(1025, 8, 3), (2048, 128, 8), (1000, 256, 5), (8192, 32, 2), (4097, 64, 1)])
def test_route_plan_small_batch_shapes(T, E, k):
    """Routing across 512-token chunk boundaries for several k (1 to 8) and
    up to 256 experts, with dropped, out-of-range and repeated ids."""
    rng = np.random.default_rng(T * 7 + k)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    topk[rng.random((T, k)) < 0.03] = -1
    bad = rng.random((T, k)) < 0.002
    topk[bad] = E + 3
    if k > 1:
        rep = rng.random(T) < 0.01
        topk[rep, 1] = topk[rep, 0]
    off, cnt, dest, st = oracle.route_plan(topk, E, 128)
    plan = nq.ep_route_plan(torch.from_numpy(topk).cuda(), E, 128)
    torch.cuda.synchronize()
    assert_bytes_equal(plan.offsets.cpu().numpy(), off, "offsets")
    assert_bytes_equal(plan.counts.cpu().numpy(), cnt, "counts")
    assert_bytes_equal(plan.dest.cpu().numpy()[: T * k], dest, "dest")
    assert int(plan.status.item()) == st


@pytest.mark.parametrize("T,E,k", [(9000, 700, 8), (16384, 256, 8), (12000, 64, 6), (16384, 752, 2),
                                   (16384, 760, 3)])
def test_route_plan_large_batches(T, E, k):
    """Batches of 8193 to 16384 tokens (more 512-token chunks than one
    thread-block cluster holds) with up to 760 experts, with dropped,
    out-of-range and repeated ids."""
    rng = np.random.default_rng(T + 13 * E + k)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    topk[rng.random((T, k)) < 0.03] = -1
    topk[rng.random((T, k)) < 0.002] = -7
    if k > 1:
        rep = rng.random(T) < 0.01
        topk[rep, k - 1] = topk[rep, 0]
    off, cnt, dest, st = oracle.route_plan(topk, E, 128)
    plan = nq.ep_route_plan(torch.from_numpy(topk).cuda(), E, 128)
    torch.cuda.synchronize()
    assert_bytes_equal(plan.offsets.cpu().numpy(), off, "offsets")
    assert_bytes_equal(plan.counts.cpu().numpy(), cnt, "counts")
    assert_bytes_equal(plan.dest.cpu().numpy()[: T * k], dest, "dest")
    assert int(plan.status.item()) == st != 0


def grouped_bf16_rows(w, R_cap):
    """Expert-grouped BF16 rows [R_cap, H] of a workload (token t at each of
    its destination rows, padding rows zero) and the exact per-expert amax."""
    off, cnt, dest, _ = oracle.route_plan(w.topk, w.E, w.A)
    x = np.zeros((R_cap, w.H), np.uint16)
    d = dest.reshape(w.T, w.k)
    for j in range(w.k):
        ok = d[:, j] >= 0
        x[d[ok, j]] = w.tokens[ok]
    f = np.abs((x.astype(np.uint32) << 16).view(np.float32))
    amax = np.zeros(w.E, np.float32)
    for e in range(w.E):
        if off[e + 1] > off[e]:
            amax[e] = f[off[e]:off[e + 1]].max()
    return x, off, amax


@pytest.mark.parametrize("name,scale", [("cfg2", 1.0), ("cfg4", 1.0), ("cfg4_ragged_H", 1.0), ("cfg1_ragged_H", 1.0),
                                        ("cfg2", 3.3)])
def test_parity_colwise_rht_bf16(name, scale):
    """ep_nvfp4_colwise_rht_bf16 (the supplied-amax path) against the oracle,
    byte for byte; the supplied amax is the input's own (as the dGLU epilogue
    gives it) or larger and off the BF16 grid; rows past R are untouched."""
    c = CASES[name]
    w = workloads.make(c["cfg"], **c["kw"])
    R_cap = nq.rows_capacity(w.T, w.k, w.E, w.A)
    x, off, amax = grouped_bf16_rows(w, R_cap)
    amax = (amax * np.float32(scale)).astype(np.float32)
    want = oracle.nvfp4_colwise_rht_bf16(x, off, w.E, amax, rounding=w.rounding, seed=w.seed, sign_mask=w.sign_mask)
    R, H = int(off[-1]), w.H
    out = {"cw_codes": torch.full((R_cap * H // 2,), CANARY, dtype=torch.uint8, device="cuda"),
           "cw_scales": torch.full((R_cap * H // 16,), CANARY, dtype=torch.uint8, device="cuda"),
           "amax_row": torch.zeros(w.E, dtype=torch.float32, device="cuda"),
           "amax_col": torch.zeros(w.E, dtype=torch.float32, device="cuda"),
           "cw_scale_enc": torch.zeros(w.E, dtype=torch.float32, device="cuda")}
    st = nq.new_status("cuda")
    nq.ep_nvfp4_colwise_rht_bf16(to_dev_bf16(x), torch.from_numpy(off).cuda(), w.E, torch.from_numpy(amax).cuda(),
                                 out=out, rounding=w.rounding, seed=w.seed, sign_mask=w.sign_mask, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g = {k: v.cpu().numpy() for k, v in out.items()}
    assert_bytes_equal(g["cw_codes"][: R * H // 2], want["cw_codes"][: R * H // 2], "columnwise codes")
    assert_bytes_equal(g["cw_scales"][: R * H // 16], want["cw_scales"][: R * H // 16], "columnwise scales")
    assert (g["cw_codes"][R * H // 2:] == CANARY).all() and (g["cw_scales"][R * H // 16:] == CANARY).all()
    for k, ok in (("amax_row", "amax_row"), ("amax_col", "amax_col"), ("cw_scale_enc", "scale_enc")):
        assert_bytes_equal(g[k].view(np.uint32), want[ok].view(np.uint32), k)
    assert want["report"]["above_4x_rowwise_amax"] == 0


def test_colwise_rht_bf16_rejects_partial_slots():
    """Expert slots that are not whole 128-row tiles: the device status says
    so and their rows are skipped (the other experts are still written)."""
    H, E = 64, 2
    off = np.array([0, 128, 200], np.int32)          # expert 1: 72 rows
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((256, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    amax = np.array([4.0, 4.0], np.float32)
    out = {"cw_codes": torch.full((256 * H // 2,), CANARY, dtype=torch.uint8, device="cuda"),
           "cw_scales": torch.full((256 * H // 16,), CANARY, dtype=torch.uint8, device="cuda"),
           "amax_row": torch.zeros(E, dtype=torch.float32, device="cuda"),
           "amax_col": torch.zeros(E, dtype=torch.float32, device="cuda"),
           "cw_scale_enc": torch.zeros(E, dtype=torch.float32, device="cuda")}
    st = nq.new_status("cuda")
    nq.ep_nvfp4_colwise_rht_bf16(to_dev_bf16(x), torch.from_numpy(off).cuda(), E, torch.from_numpy(amax).cuda(),
                                 out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & nq.EP_DEV_ERR_BAD_EXPERT
    want = oracle.nvfp4_colwise_rht_bf16(x[:128], np.array([0, 128], np.int32), 1, amax[:1])
    assert_bytes_equal(out["cw_codes"].cpu().numpy()[: 128 * H // 2], want["cw_codes"], "expert 0 codes")
    assert (out["cw_codes"].cpu().numpy()[128 * H // 2:] == CANARY).all()


@pytest.mark.parametrize("name", ["cfg5", "cfg1_ragged_H", "cfg4"])
def test_parity_mxfp8_colwise(name):
    """ep_mxfp8_colwise against the oracle, byte for byte (data and scales of
    rows [0, R)); bytes of rows past R untouched.  The ragged case has H % 64
    = 32 (a half-filled last column group)."""
    c = CASES[name]
    w = workloads.make(c["cfg"], **c["kw"])
    R_cap = nq.rows_capacity(w.T, w.k, w.E, w.A)
    x, off, _ = grouped_bf16_rows(w, R_cap)
    want = oracle.mxfp8_colwise(x, off, w.E)
    buf = torch.full((R_cap * w.H + R_cap * (w.H // 32),), CANARY, dtype=torch.uint8, device="cuda")
    st = nq.new_status("cuda")
    nq.ep_mxfp8_colwise(to_dev_bf16(x), torch.from_numpy(off).cuda(), w.E, buf=buf, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = buf.cpu().numpy()
    R, H = int(off[-1]), w.H
    assert_bytes_equal(got[: R * H], want[: R * H], "mxfp8 columnwise data")
    assert_bytes_equal(got[R_cap * H: R_cap * H + R * H // 32], want[R_cap * H: R_cap * H + R * H // 32],
                       "mxfp8 columnwise scales")
    assert (got[R * H: R_cap * H] == CANARY).all() and (got[R_cap * H + R * H // 32:] == CANARY).all()


def test_route_barrier_timeout_is_reported():
    """Failure detection without a fault: the routing plan's grid barrier is
    given an arrival count preset far beyond the grid (so no CTA can be the
    last to arrive: a flag nothing sets).  Its bounded wait gives up, the
    kernel returns with EP_DEV_ERR_TIMEOUT in the device status, and the
    context stays usable: the next plan (fresh workspace) is exact."""
    import time
    T, E, k = 3000, 32, 12          # k > 8: the cooperative kernel with the grid barrier
    rng = np.random.default_rng(21)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    tk = torch.from_numpy(topk).cuda()
    ws = nq.new_route_workspace(T, k, E, "cuda")
    ws[0] = 0x40000000
    t0 = time.perf_counter()
    plan = nq.ep_route_plan(tk, E, 128, workspace=ws)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(plan.status.item()) & nq.EP_DEV_ERR_TIMEOUT
    assert waited < 30.0
    good = nq.ep_route_plan(tk, E, 128)
    torch.cuda.synchronize()
    off, cnt, dest, st = oracle.route_plan(topk, E, 128)
    assert int(good.status.item()) == st == 0
    assert_bytes_equal(good.dest.cpu().numpy()[: T * k], dest, "dest after a timed-out plan")


def test_parity_largest_expert_count_and_slots():
    """E = 1024 experts (the largest allowed) and k = 32 slots per token:
    the general routing kernel, 1 024 mostly-padding slots, the direct
    receive's per-CTA expert tables at their full size."""
    w = workloads.make(4, T=64, H=256, E=1024, k=32)
    g = DeviceRun(w)
    o = OracleRun(w, g.R_cap)
    compare_runs(g, o)


def test_parity_wide_hidden():
    """H = 16384: the pack's multi-chunk kernel (wider than the warp kernel's
    8192) and 64 column strips in the direct receive."""
    w = workloads.make(1, T=64, H=16384)
    g = DeviceRun(w, unpack=True, mxfp8=True)
    o = OracleRun(w, g.R_cap, unpack=True, mxfp8=True)
    compare_runs(g, o)


@pytest.mark.parametrize("name,dispatch", [("cfg1", True), ("cfg2", True), ("cfg4", True), ("cfg5", False),
                                           ("cfg1_ragged_H", True), ("cfg4_ragged_H", False), ("cfg4", False)])
def test_parity_pack_reduced_amax(name, dispatch):
    """The per-expert amax max-reduced by the pack as it writes the rows
    (through ep_nvfp4_dispatch, which zeroes it in the routing kernel and
    names each slot's expert from topk_idx; or through ep_nvfp4_pack, which
    finds the expert from the row index) equals the oracle's rowwise amax bit
    for bit, and the direct receive given it (no trailer pass, the tile
    kernel writes the metadata) produces the same operands.  The ragged-H
    cases take the general pack kernel."""
    c = CASES[name]
    w = workloads.make(c["cfg"], **c["kw"])
    g = DeviceRun(w, unpack=c.get("unpack", False), dispatch=dispatch, amax=True)
    o = OracleRun(w, g.R_cap, unpack=c.get("unpack", False))
    compare_runs(g, o)


def test_parity_pack_reduced_amax_swizzled_and_edges():
    # the tiled-scale receive with the supplied amax
    w = workloads.make(2, T=600, H=1024)
    compare_runs(DeviceRun(w, swizzled=True, dispatch=True, amax=True), OracleRun(w, nq.rows_capacity(w.T, w.k, w.E, w.A)))
    # routing edges: dropped slots, out-of-range and repeated ids add nothing
    tokens = special_tokens()
    T = tokens.shape[0]
    topk = np.array([[i % 5, (i + 2) % 5] for i in range(T)], np.int32)
    topk[1, 1] = -1
    topk[2, 1] = 9
    topk[3, 1] = topk[3, 0]
    w = workloads.Workload("special", "special", tokens, topk, E=5)
    for dispatch in (False, True):
        g = DeviceRun(w, dispatch=dispatch, amax=True)
        compare_runs(g, OracleRun(w, g.R_cap))
    # no tokens / one token (capacity below one tile: the receive reduces the
    # trailers itself), empty experts (amax 0, S_enc 1)
    for T, E in ((0, 4), (1, 1), (1, 8)):
        rng = np.random.default_rng(T + E)
        tokens = workloads.to_bf16_bits(rng.standard_normal((T, 256)).astype(np.float32))
        k = min(2, E)
        topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
            np.zeros((0, k), np.int32)
        w = workloads.Workload("edge", "edge", tokens, topk, E=E)
        g = DeviceRun(w, dispatch=True, amax=True)
        compare_runs(g, OracleRun(w, g.R_cap))


def test_parity_pack_reduced_amax_largest_and_wide():
    """E = 1024, k = 32 (deepest search over the offsets in the separate
    pack) and H = 16384 (the general pack kernel)."""
    w = workloads.make(4, T=64, H=256, E=1024, k=32)
    for dispatch in (False, True):
        g = DeviceRun(w, dispatch=dispatch, amax=True)
        compare_runs(g, OracleRun(w, g.R_cap))
    w = workloads.make(1, T=64, H=16384)
    g = DeviceRun(w, dispatch=True, amax=True)
    compare_runs(g, OracleRun(w, g.R_cap))


def test_pack_amax_accumulates_into_callers_values():
    """ep_nvfp4_pack max-reduces into what the array holds: an entry above
    every token amax stays, the others end at the experts' amax."""
    w = workloads.make(2, T=300, H=512)
    tok = to_dev_bf16(w.tokens)
    plan = nq.ep_route_plan(torch.from_numpy(np.ascontiguousarray(w.topk)).cuda(), w.E, w.A)
    amax = torch.zeros(w.E, dtype=torch.float32, device="cuda")
    amax[1] = 1e30
    nq.ep_nvfp4_pack(tok, plan, expert_amax=amax)
    off, cnt, dest, _ = oracle.route_plan(w.topk, w.E, w.A)
    rows = oracle.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, plan.R_cap)
    want = oracle.nvfp4_direct_receive(rows, w.H, off, w.E)["amax_row"].copy()
    want[1] = np.float32(1e30)
    assert_bytes_equal(amax.cpu().numpy().view(np.uint32), want.view(np.uint32), "accumulated amax")
