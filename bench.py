"""Benchmark of the NVFP4 EP hot path: route plan + NVFP4 pack + direct receive.

Workload: 4096 tokens x 4096 hidden BF16 ~N(0,1) with 0.1% of entries x50;
16 experts, softmax-of-Gaussian top-2 routing with 2 experts forced empty;
alignment 128; round-to-nearest-even (the dispatch-forward configuration).
A step is one pass of the whole path over one batch: route plan (1 kernel),
NVFP4 pack with the routing gather (1 kernel), direct receive (2 kernels:
per-expert amax from the row trailers, then the tiled rowwise /
columnwise-RHT transform).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--config 1..5]

``--config`` picks another of the five synthetic workloads (the same step:
route plan + NVFP4 pack + direct receive; config 5's MXFP8 pack is not part
of it); the default is the dispatch-forward batch above.

Prints one JSON line (rank 0).  Under torchrun every rank processes its own
batch (replicas: the path shards by token batch with no exchange on one
GPU), ``value`` is the sum over ranks of tokens / the slowest rank's time.
The reference arm (``--impl reference``) times the plain CPU oracle on the
host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 pack+direct-receive tokens/s and achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
WORKLOAD_CFG = 2          # the dispatch-forward config the metric is quoted on
KERNELS_PER_STEP = 3      # route plan, pack (reducing the per-expert amax), direct receive tile transform
N_SETS = 6                # rotating buffer sets: ~560 MB touched per rotation > 129 MB L2
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--sets", type=int, default=N_SETS, help="rotating buffer sets (profiling uses 1)")
    p.add_argument("--config", type=int, default=WORKLOAD_CFG, choices=[1, 2, 3, 4, 5],
                   help="workload (default: the 4096-token dispatch-forward batch the metric is quoted on)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_workload_kwargs(rank: int) -> dict:
    """Each replica packs its own batch: rank 0 the workload's own seed, rank r
    a seed of its own (same shapes and distributions, different values)."""
    return {"seed": 2 + 1000 * rank} if rank else {}


def max_over_ranks(dist, x: float, device) -> float:
    """The largest value over all ranks (the slowest replica's time); x itself
    on one process."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region (read-only queries)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.proc = None
        self.path = None

    def start(self):
        if not self.enabled:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [t.strip() for t in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    mhz.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        finally:
            os.unlink(self.path)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(mhz)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(mhz)}


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


DR_SOURCES = ["nvfp4_quantization_gb300/csrc/receive.cu", "nvfp4_quantization_gb300/csrc/epq_device.cuh"]


def profiled_traffic(kernel: str, sources, config: int) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and on this workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d[kernel]
        if rec.get("source_sha") != source_sha(sources) or rec.get("config") != config:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def algorithmic_bytes(T, H, k, E, R, S):
    """Bytes the method must move (padding rows count: they are real rows)."""
    route = 4 * T * k * 2 + 4 * (2 * E + 1)          # ids in, dest out, offsets / counts
    pack = 2 * T * H + 4 * T * k + R * S             # tokens + dest in, rows out
    dr = R * S + R * (9 * H // 16 + 4) + R * (9 * H // 16) + 12 * E
    return route, pack, dr


class BufferSet:
    """One set of device buffers and the CUDA graphs of one step on them."""

    def __init__(self, torch, nq, w, tok_host, topk_host):
        self.tok = tok_host.cuda()
        self.topk = topk_host.cuda()
        self.plan = nq.ep_route_plan(self.topk, w.E, w.A)
        self.ws = nq.new_route_workspace(w.T, w.k, w.E, "cuda")
        self.rows = torch.empty((self.plan.R_cap, nq.row_bytes(w.H)), dtype=torch.uint8, device="cuda")
        self.out = nq.alloc_grouped(self.plan.R_cap, w.H, w.E, "cuda")
        self.amax = torch.zeros(w.E, dtype=torch.float32, device="cuda")
        self.w, self.nq = w, nq
        self.route_pack()
        self.receive()

    def route_pack(self):
        w, nq = self.w, self.nq
        # route plan + pack in one call: the pack encodes its first tokens while the routing kernel runs,
        # and reduces each expert's amax as it writes the rows
        nq.ep_nvfp4_dispatch(self.tok, self.topk, w.E, w.A, plan=self.plan, workspace=self.ws, rows=self.rows,
                             rounding=w.rounding, seed=w.seed, expert_amax=self.amax)

    def receive(self):
        w, nq = self.w, self.nq
        nq.ep_nvfp4_direct_receive(self.rows, w.H, self.plan.offsets, w.E, out=self.out, rounding=w.rounding,
                                   seed=w.seed, sign_mask=w.sign_mask, status=self.plan.status,
                                   expert_amax=self.amax)

    def capture(self, torch):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        self.gA, self.gB, self.gS = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.gA, stream=s):
                self.route_pack()
            with torch.cuda.graph(self.gB, stream=s):
                self.receive()
            with torch.cuda.graph(self.gS, stream=s):
                self.route_pack()
                self.receive()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()


def capture_rotation(torch, sets, rotations: int = 1):
    """One graph holding `rotations` rounds of one step on every buffer set,
    in rotation order."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(rotations):
                for b in sets:
                    b.route_pack()
                    b.receive()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def gpu_arm(args, rank, world, local):
    import torch

    import nvfp4_quantization_gb300 as nq
    import workloads

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier(device_ids=[local])

    w = workloads.make(args.config, **replica_workload_kwargs(rank))
    T, H, k, E = w.T, w.H, w.k, w.E
    tok_host = torch.from_numpy(w.tokens.view(np.int16)).view(torch.bfloat16)
    topk_host = torch.from_numpy(np.ascontiguousarray(w.topk))
    sets = [BufferSet(torch, nq, w, tok_host, topk_host) for _ in range(args.sets)]
    torch.cuda.synchronize()
    st = int(sets[0].plan.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st:#x} after the first pass")
    R = int(sets[0].plan.offsets[-1].item())
    S = nq.row_bytes(H)
    for b in sets:
        b.capture(torch)

    # ---- timed region: K steps, rotating buffer sets (cold L2 per step).
    # Steps go in blocks of one step per set; whole blocks run as graphs of up
    # to GRAPH_ROTATIONS blocks each (then single steps for a remainder), so
    # the device runs them back to back with a launch gap only between graphs.
    GRAPH_ROTATIONS = 50
    gR = capture_rotation(torch, sets)
    K, W = args.steps, args.warmup
    nset = len(sets)
    SAMPLE_EVERY = 10
    nblocks, rem = divmod(K, nset)
    n_big, n_small = divmod(nblocks, GRAPH_ROTATIONS)
    gBig = capture_rotation(torch, sets, GRAPH_ROTATIONS) if n_big else None
    gSmall = capture_rotation(torch, sets, n_small) if n_small else None
    for i in range(max(1, W // nset)):
        gR.replay()
    torch.cuda.synchronize()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    clocks.start()
    time.sleep(0.2)
    wall0 = time.perf_counter()
    t0.record()
    for _ in range(n_big):
        gBig.replay()
    if gSmall is not None:
        gSmall.replay()
    for j in range(rem):
        sets[j].gS.replay()
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    clk = clocks.stop()
    barrier()
    ms_total = max_over_ranks(dist, t0.elapsed_time(t1), "cuda")
    ms_step = ms_total / K
    # ---- per-call durations for the roofline, after the timed region: one
    # block in SAMPLE_EVERY again, each step replayed call by call with CUDA
    # events between the calls (which stops the calls' overlap, so these steps
    # are kept out of the step time)
    n_sampled = max(1, (nblocks + SAMPLE_EVERY - 1) // SAMPLE_EVERY)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(nset)] for _ in range(n_sampled)]
    for blk in range(n_sampled):
        for j, b in enumerate(sets):
            e = ev[blk][j]
            e[0].record()
            b.gA.replay()
            e[1].record()
            b.gB.replay()
            e[2].record()
    torch.cuda.synchronize()
    flat = [e for row in ev for e in row]
    ms_a = float(np.mean([e[0].elapsed_time(e[1]) for e in flat]))
    ms_b = float(np.mean([e[1].elapsed_time(e[2]) for e in flat]))
    st = int(sets[0].plan.status.item())
    route_b, pack_b, dr_b = algorithmic_bytes(T, H, k, E, R, S)
    set_mb = (route_b + pack_b + dr_b) / 1e6
    res = dict(set_mb=set_mb, T=T, H=H, k=k, E=E, R=R, S=S, ms_step=ms_step, ms_a=ms_a, ms_b=ms_b, wall_s=wall1 - wall0,
               clocks=clk, status=st, bytes=(route_b, pack_b, dr_b), world=world, w=w,
               n_sampled_steps=len(flat))

    # ---- end to end through the public API with host buffers
    res["e2e"] = e2e_measure(torch, nq, w, sets[:2], tok_host, topk_host, R, args.e2e_steps)
    res["e2e"]["ms"] = max_over_ranks(dist, res["e2e"]["ms"], "cuda")
    # ---- the two calls outside the step: unpack and MXFP8 pack, same batch
    res["aux"] = aux_measure(torch, nq, w, sets[0], R)
    return res


def aux_measure(torch, nq, w, b, R, reps=20):
    """CUDA-event times of ep_nvfp4_unpack (the step's rows -> BF16),
    ep_mxfp8_pack (the step's tokens) and the direct receive with both scale
    tensors in the tiled GEMM layout and, for comparison, in the linear one
    (the step's rows), each launch after a 512 MB write that flushes the L2,
    median of ``reps``."""
    H, S = w.H, nq.row_bytes(w.H)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((b.plan.R_cap, H), dtype=torch.bfloat16, device="cuda")
    mx = torch.empty(b.plan.R_cap * H + b.plan.R_cap * (H // 32), dtype=torch.uint8, device="cuda")

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    ms_u = timed(lambda: nq.ep_nvfp4_unpack(b.rows, H, b.plan.offsets, w.E, out=out, status=b.plan.status))
    ms_m = timed(lambda: nq.ep_mxfp8_pack(b.tok, b.plan, buf=mx))
    bytes_u = R * S + R * 2 * H
    bytes_m = 2 * w.T * H + 4 * w.T * w.k + R * (H + H // 32)
    res = {"unpack": {"ms": ms_u, "bytes": bytes_u}, "mxfp8_pack": {"ms": ms_m, "bytes": bytes_m}}
    # the columnwise RHT operand of the decoded rows (BF16) with the supplied
    # per-expert amax (the dGLU-epilogue path): the rows unpacked above, the
    # step's own rowwise amaxes
    cw = {"cw_codes": torch.empty(b.plan.R_cap * H // 2, dtype=torch.uint8, device="cuda"),
          "cw_scales": torch.empty(b.plan.R_cap * H // 16, dtype=torch.uint8, device="cuda"),
          "amax_row": torch.empty(w.E, dtype=torch.float32, device="cuda"),
          "amax_col": torch.empty(w.E, dtype=torch.float32, device="cuda"),
          "cw_scale_enc": torch.empty(w.E, dtype=torch.float32, device="cuda")}
    ms_c = timed(lambda: nq.ep_nvfp4_colwise_rht_bf16(out, b.plan.offsets, w.E, b.out["amax_row"], out=cw,
                                                      rounding=w.rounding, seed=w.seed, sign_mask=w.sign_mask,
                                                      status=b.plan.status))
    res["colwise_rht_bf16"] = {"ms": ms_c, "bytes": R * H * 2 + R * (9 * H // 16) + 16 * w.E}
    del cw
    # the columnwise MXFP8 operand of the same BF16 rows
    mxc = torch.empty(b.plan.R_cap * H + b.plan.R_cap * (H // 32), dtype=torch.uint8, device="cuda")
    ms_x = timed(lambda: nq.ep_mxfp8_colwise(out, b.plan.offsets, w.E, buf=mxc, status=b.plan.status))
    res["mxfp8_colwise"] = {"ms": ms_x, "bytes": R * H * 2 + R * (H + H // 32)}
    del mxc
    if H % 128 == 0:
        g = nq.alloc_grouped(b.plan.R_cap, H, w.E, "cuda")
        bytes_d = algorithmic_bytes(w.T, H, w.k, w.E, R, S)[2]
        # the receive from the rows alone (its own pass over the row trailers for
        # the per-expert amax), and with the amax the dispatch reduced, in the
        # linear and the tiled scale layouts
        for name, swz, am in (("direct_receive_rows_only", False, None), ("direct_receive_linear", False, b.amax),
                              ("direct_receive_swizzled", True, b.amax)):
            ms = timed(lambda: nq.ep_nvfp4_direct_receive(b.rows, H, b.plan.offsets, w.E, out=g, rounding=w.rounding,
                                                          seed=w.seed, sign_mask=w.sign_mask, status=b.plan.status,
                                                          swizzled=swz, expert_amax=am))
            res[name] = {"ms": ms, "bytes": bytes_d}
        del g
    del flush, out, mx
    return res


def e2e_measure(torch, nq, w, bufs, tok_host, topk_host, R, steps):
    """Each step: pinned host tokens + routing -> device, the three public
    calls (eager), grouped operands + metadata -> pinned host.  Two buffer
    sets on two streams take alternate steps, so one step's copies overlap
    the neighbouring step's kernels and copies (a serving loop's double
    buffering; four streams measured no faster: the host link is the limit);
    every step still moves its own inputs in and its outputs out."""
    H = w.H
    tok_pin = tok_host.pin_memory()
    topk_pin = topk_host.pin_memory()
    lanes = []
    for b in bufs:
        # the three per-expert metadata arrays are rows of one tensor: one copy
        srcs = [b.out["rw_codes"][:R], b.out["rw_scales"][:R], b.out["rw_row_scale"][:R],
                b.out["cw_codes"][: R * H // 2], b.out["cw_scales"][: R * H // 16], b.out["metadata"]]
        dsts = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in srcs]
        lanes.append((b, torch.cuda.Stream(), srcs, dsts))
    h2d = tok_pin.numel() * 2 + topk_pin.numel() * 4
    d2h = sum(x.numel() * x.element_size() for x in lanes[0][2])

    def step(i):
        b, st, srcs, dsts = lanes[i % len(lanes)]
        with torch.cuda.stream(st):
            b.tok.copy_(tok_pin, non_blocking=True)
            b.topk.copy_(topk_pin, non_blocking=True)
            b.route_pack()
            b.receive()
            for x, d in zip(srcs, dsts):
                d.copy_(x, non_blocking=True)

    main = torch.cuda.current_stream()
    for i in range(6):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _, st, _, _ in lanes:
        st.wait_stream(main)
    for i in range(steps):
        step(i)
    for _, st, _, _ in lanes:
        main.wait_stream(st)
    e1.record(main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ok = all(torch.equal(dsts[3][: 1 << 16].cuda(), srcs[3][: 1 << 16]) for _, _, srcs, dsts in lanes)
    return dict(ms=ms, h2d=h2d, d2h=d2h, ok=bool(ok), link=host_link_gbs(torch))


def host_link_gbs(torch, nbytes: int = 256 << 20, reps: int = 5) -> dict:
    """Plain pinned-memory copy bandwidth of this GPU's host link: each
    direction alone, and both at once (one copy each way on two streams; the
    sum of the bytes over the time), which is what an end-to-end step that
    overlaps its copies gets."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        out[name] = reps * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(main)
    s1.wait_stream(main)
    s2.wait_stream(main)
    for _ in range(reps):
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
    main.wait_stream(s1)
    main.wait_stream(s2)
    b.record(main)
    torch.cuda.synchronize()
    out["both"] = 2 * reps * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9
    return out


def oracle_pass(o, w, tokens, topk):
    """Route plan + NVFP4 pack + direct receive of one batch on the oracle."""
    off, cnt, dest, _ = o.route_plan(topk, w.E, w.A)
    R_cap = o.rows_capacity(tokens.shape[0], w.k, w.E, w.A)
    rows = o.nvfp4_pack(tokens, dest, w.k, off, cnt, w.E, R_cap, rounding=w.rounding, seed=w.seed)
    o.nvfp4_direct_receive(rows, w.H, off, w.E, rounding=w.rounding, seed=w.seed, sign_mask=w.sign_mask)


def cpu_baseline(w, budget_s: float = 15.0) -> dict:
    """The oracle, as it stands (single-threaded C), on the first n tokens of
    the batch (and their routing), n sized from a 64-token probe so that the
    timed pass takes about ``budget_s`` (the whole batch if that is shorter)."""
    import oracle as o
    o.build()
    t0 = time.perf_counter()
    oracle_pass(o, w, np.ascontiguousarray(w.tokens[:64]), np.ascontiguousarray(w.topk[:64]))
    per_tok = (time.perf_counter() - t0) / 64
    n = int(max(64, min(w.T, budget_s / max(per_tok, 1e-9))))
    tok, topk = np.ascontiguousarray(w.tokens[:n]), np.ascontiguousarray(w.topk[:n])
    t0 = time.perf_counter()
    oracle_pass(o, w, tok, topk)
    dt = time.perf_counter() - t0
    what = "the full batch" if n == w.T else f"the first {n} of {w.T} tokens"
    return {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"one pass over {what} (route plan + pack + direct receive), single-threaded C oracle, "
                      f"{dt:.2f} s"}


def reference_arm(args, rank, world):
    """--impl reference: the oracle on the host cores, each step a slice of
    the same workload sized so that warm-up + K steps take about two minutes."""
    if rank != 0:
        return None
    import oracle as o
    import workloads
    o.build()
    w = workloads.make(args.config)
    t0 = time.perf_counter()
    oracle_pass(o, w, w.tokens[:512], w.topk[:512])
    per_tok = (time.perf_counter() - t0) / 512
    K, W = args.steps, args.warmup
    n = int(max(1, min(w.T, 120.0 / max(K + W, 1) / per_tok)))

    def run(i):
        a = (i * n) % w.T
        idx = np.arange(a, a + n) % w.T
        oracle_pass(o, w, np.ascontiguousarray(w.tokens[idx]), np.ascontiguousarray(w.topk[idx]))

    for i in range(W):
        run(i)
    t0 = time.perf_counter()
    for i in range(K):
        run(W + i)
    dt = time.perf_counter() - t0
    value = n * K / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": dt * 1e3 / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.description, "tokens_per_step": n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{n} consecutive tokens of the batch (and their routing) per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    r = gpu_arm(args, rank, world, local)
    if rank != 0:
        return
    peak, peak_kind = load_peaks()
    route_b, pack_b, dr_b = r["bytes"]
    w = r["w"]
    tokens_s = world * r["T"] / (r["ms_step"] * 1e-3)
    dr_gbs = dr_b / (r["ms_b"] * 1e-3) / 1e9
    pack_gbs = (route_b + pack_b) / (r["ms_a"] * 1e-3) / 1e9
    path_gbs = (route_b + pack_b + dr_b) / (r["ms_step"] * 1e-3) / 1e9
    e2e = r["e2e"]
    line = {
        "metric": METRIC, "value": tokens_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.description, "T": r["T"], "H": r["H"], "E": r["E"], "k": r["k"], "A": w.A,
                   "R": r["R"], "rounding": "sr" if w.rounding else "rne",
                   "l2": f"{args.sets} rotating buffer sets ({r['set_mb']:.0f} MB touched per step; a set is reused "
                         f"after the others moved {(args.sets - 1) * r['set_mb']:.0f} MB through the 129 MB L2), "
                         "back-to-back CUDA-graph steps",
                   "parallelism": f"replicas x{world}"},
        "path": {"gbs": path_gbs, "frac_of_peak": path_gbs / peak, "bytes_per_step": route_b + pack_b + dr_b,
                 "route_pack_ms": r["ms_a"], "route_pack_gbs": pack_gbs, "direct_receive_ms": r["ms_b"],
                 "direct_receive_gbs": dr_gbs},
        "roofline": {"kernel": "direct_receive_kernel (ep_nvfp4_direct_receive)", "bound": "hbm",
                     "achieved": dr_gbs, "peak": peak, "unit": "GB/s", "frac": dr_gbs / peak,
                     "peak_kind": f"{peak_kind} (copy bandwidth)", "bytes_per_launch": dr_b,
                     "traffic": profiled_traffic("direct_receive", DR_SOURCES, args.config)},
        "e2e": {"value": world * r["T"] / (e2e["ms"] * 1e-3), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e["ms"],
                "api": "eager ep_nvfp4_dispatch / ep_nvfp4_direct_receive on two streams, "
                       "alternate steps (double buffering)", "checked": e2e["ok"],
                "host_link_gbs": e2e["link"],
                "link_floor_ms": max(e2e["h2d"] / (e2e["link"]["h2d"] * 1e9), e2e["d2h"] / (e2e["link"]["d2h"] * 1e9),
                                     (e2e["h2d"] + e2e["d2h"]) / (e2e["link"]["both"] * 1e9)) * 1e3,
                "floor_note": "the largest of: the step's host-to-device bytes over that direction's pinned copy "
                              "bandwidth, the same for device-to-host, and all its bytes over the bandwidth of "
                              "both directions at once"},
        "other_calls": {name: {"ms": v["ms"], "gbs": v["bytes"] / (v["ms"] * 1e-3) / 1e9,
                               "frac": v["bytes"] / (v["ms"] * 1e-3) / 1e9 / peak, "bytes": v["bytes"],
                               "note": "one call on the step's batch, L2 flushed before each launch"}
                        for name, v in r["aux"].items()},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "sampled_steps_for_kernel_times": r["n_sampled_steps"],
        "clocks": r["clocks"],
        "device_status": r["status"],
        "timed_wall_s": r["wall_s"],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
