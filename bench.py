"""Benchmark of the NVFP4 EP hot path: route plan + NVFP4 pack + direct receive.

Headline workload (the largest configuration): combine-backward gradients,
16384 tokens x 7168 hidden BF16 ~ 1e-3 N(0,1) lognormal(0,1) per token;
256 experts, top-8 uniform routing with 26 experts empty; alignment 128;
stochastic rounding (Philox seed 1234) in the pack and the columnwise
requantisation.  A step is one pass of the whole path over one batch: route
plan (1 kernel) and NVFP4 pack with the routing gather (1 kernel, which also
reduces the per-expert amax) in one ep_nvfp4_dispatch call, then the direct
receive given that amax (1 kernel: the tiled rowwise / columnwise-RHT
transform).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--config 1..5] [--no-extra-configs]

``--config`` picks another of the five synthetic workloads for the headline
(the same step).  With the default headline the line also carries, as nested
keys: ``configs`` -- the dispatch-forward (4096x4096) and imbalanced
(8192x4096) batches timed the same way, each with its own roofline block --
and ``config5`` -- the MXFP8 vs NVFP4 comparison on the StudentT(4) batch:
both packs timed, the NVFP4 step timed, and the relative RMS decode error of
each format computed from the GPU outputs.

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
WORKLOAD_CFG = 4          # the largest configuration (16384x7168, 256 experts top-8, SR)
EXTRA_CONFIGS = (2, 3)    # the other pack + direct-receive batches, nested in the same line
KERNELS_PER_STEP = 3      # route plan, pack (reducing the per-expert amax), direct receive tile transform
L2_BYTES = 129 << 20
FALLBACK_HBM_GBS = 6800.0
DEFAULT_SEEDS = {1: 0, 2: 2, 3: 3, 4: 4, 5: 5}   # each workload's own seed


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--e2e-steps", type=int, default=0, help="end-to-end steps (0: sized to about a second)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-extra-configs", action="store_true",
                   help="only the headline workload (no nested configs 2, 3 and the config-5 comparison)")
    p.add_argument("--sets", type=int, default=0, help="rotating buffer sets (0: enough to exceed the L2); rounded up to "
                   "a multiple of the streams that take alternate steps")
    p.add_argument("--config", type=int, default=WORKLOAD_CFG, choices=[1, 2, 3, 4, 5],
                   help="headline workload (default: the largest, the 16384x7168 SR combine-backward batch)")
    p.add_argument("--tokens", type=int, default=0,
                   help="a smaller batch of the same recipe (T tokens; profiling captures on scaled-down cases)")
    p.add_argument("--experts", type=int, default=0, help="expert count of the scaled-down config-4 recipe")
    return p.parse_args()


def workload_kwargs(args, rank: int) -> dict:
    """The headline workload's recipe arguments: the replica's seed, and the
    scaled-down shape when --tokens / --experts ask for one."""
    kw = replica_workload_kwargs(rank, args.config)
    if args.tokens:
        kw["T"] = args.tokens
    if args.experts and args.config == 4:
        kw["E"] = args.experts
    return kw


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_workload_kwargs(rank: int, config: int = WORKLOAD_CFG) -> dict:
    """Each replica packs its own batch: rank 0 the workload's own seed, rank r
    a seed of its own (same shapes and distributions, different values)."""
    return {"seed": DEFAULT_SEEDS[int(config)] + 1000 * rank} if rank else {}


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


def n_rotating_sets(set_bytes: int, requested: int = 0) -> int:
    """Buffer sets rotated between steps so that a set comes back only after
    the others have moved more than the L2 holds (2 at least, 6 at most)."""
    if requested > 0:
        return int(requested)
    return int(min(6, max(2, math.ceil(4 * L2_BYTES / max(set_bytes, 1)) + 1)))


class ClockSampler:
    """nvidia-smi sampling (read-only queries) of SM clocks and throttle
    reasons every 10 ms, with the sample's time stamp, so that the samples
    taken inside a timed region can be told from the rest."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True, period_ms: int = 10):
        self.gpu = gpu_index
        self.enabled = enabled
        self.period_ms = period_ms
        self.proc = None
        self.path = None
        self.rows = []

    def start(self):
        if not self.enabled:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms), "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        """Ends the sampling and keeps the samples as (unix time, sm MHz,
        max MHz, active reasons)."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        import datetime
        try:
            for line in open(self.path):
                f = [t.strip() for t in line.split(",")]
                if len(f) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    mhz, mx = float(f[2]), float(f[3])
                except ValueError:
                    continue
                reasons = {n for n, v in zip(self.REASONS, f[6:10]) if v.lower() == "active"}
                self.rows.append((ts, mhz, mx, reasons))
        finally:
            os.unlink(self.path)
        self.proc = None

    def summary(self, t0: float, t1: float, busy0: float | None = None) -> dict | None:
        """Median SM clock and the reasons seen in [t0, t1] (unix times of the
        timed region).  A region shorter than a few sampling periods may hold
        no sample; then the samples of the busy period around it ([busy0, t1]:
        the warm-up steps just before it and the region itself) are used, and
        ``window`` says so."""
        if not self.enabled:
            return None
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 1 and busy0 is not None:
            inside = [r for r in self.rows if busy0 <= r[0] <= t1 + self.period_ms * 1e-3]
            window = "warm-up steps and timed region (the timed region alone is shorter than a sample period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        reasons = sorted(set().union(*[r[3] for r in inside]))
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": float(max(r[2] for r in inside)),
                "reasons": reasons, "samples": len(inside), "window": window,
                "period_ms": self.period_ms}


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


DR_SOURCES = ["nvfp4_quantization_gb300/csrc/receive.cu", "nvfp4_quantization_gb300/csrc/epq_device.cuh"]


def profiled_traffic(kernel: str, sources, config: int) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d[kernel][str(int(config))]
        if rec.get("source_sha") != source_sha(sources):
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


def row_bytes(H: int) -> int:
    """Bytes of a packed NVFP4 row: roundup16(9H/16 + 16) (the boundary's
    ep_nvfp4_row_bytes, restated for host arithmetic)."""
    return (9 * H // 16 + 16 + 15) // 16 * 16


def rows_capacity(T: int, k: int, E: int, A: int) -> int:
    """Upper bound on the received rows of any routing, T k + E (A - 1) (the
    boundary's ep_rows_capacity, restated for host arithmetic)."""
    return T * k + E * (A - 1)


def step_layout(w, n_sets: int = 0) -> dict:
    """Buffer sets and step streams of the GPU arm's timed steps on workload
    ``w`` (host arithmetic only): the bytes one set holds, the number of
    rotating sets (a multiple of the streams) and the streams."""
    T, H, k, E = w.T, w.H, w.k, w.E
    R_cap = rows_capacity(T, k, E, w.A)
    S = row_bytes(H)
    set_bytes = 2 * T * H + 4 * T * k + R_cap * S * 2 + R_cap * (9 * H // 8 + 4)
    nset = n_rotating_sets(set_bytes, n_sets)
    ns = step_streams(set_bytes)
    nset += (-nset) % ns   # every stream keeps its own sets
    return dict(set_bytes=set_bytes, nset=nset, streams=ns, R_cap=R_cap, S=S)


def workload_config(w, R: int, world: int, n_sets: int = 0) -> dict:
    """The JSON ``config`` of a timed workload (both arms print the same):
    the batch, its received rows R and the timing method of the GPU arm."""
    lay = step_layout(w, n_sets)
    set_mb = sum(algorithmic_bytes(w.T, w.H, w.k, w.E, R, lay["S"])) / 1e6
    return {"workload": w.description, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "A": w.A, "R": R,
            "rounding": "sr" if w.rounding else "rne",
            "l2": f"{lay['nset']} rotating buffer sets ({set_mb:.0f} MB touched per step; a set is reused "
                  f"after the others moved {(lay['nset'] - 1) * set_mb:.0f} MB through the 129 MB L2), "
                  f"CUDA-graph steps, {lay['streams']} streams taking alternate steps",
            "parallelism": f"replicas x{world}"}


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
        self.gS = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.gS, stream=s):
                self.route_pack()
                self.receive()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()


def step_streams(set_bytes: int) -> int:
    """Streams that take alternate steps: four for batches whose buffer set
    holds less than 1 GB (their steps are short against the kernels' start-up
    and tail), two for larger ones (a third stream measured no faster on the
    16384-token, 256-expert batch and slower on the 64-expert one)."""
    return 4 if set_bytes < (1 << 30) else 2


def capture_rotation(torch, sets, rotations: int = 1, streams: int = 2):
    """One graph holding `rotations` rounds of one step on every buffer set,
    in rotation order, the steps dealt in turn to `streams` streams (the
    batches are independent: one stream's step runs while the other's starts
    up or drains).  Set j always runs on stream j mod `streams` (the set count
    is a multiple of it), so no set is used by two steps at once."""
    assert len(sets) % streams == 0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            lanes = [s] + [torch.cuda.Stream() for _ in range(streams - 1)]
            for x in lanes[1:]:
                x.wait_stream(s)
            for _ in range(rotations):
                for j, b in enumerate(sets):
                    with torch.cuda.stream(lanes[j % streams]):
                        b.route_pack()
                        b.receive()
            for x in lanes[1:]:
                s.wait_stream(x)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def time_steps(torch, nq, w, K, W, n_sets, barrier=None, clocks_enabled=True, gpu_index=0):
    """K steps of route plan + pack + direct receive on workload ``w``, timed
    on the device.  ``n_sets`` buffer sets are rotated between steps (cold L2
    per step); whole rotations run as CUDA graphs of up to 50 rotations (then
    single steps for a remainder), so the device runs the steps back to back
    with a launch gap only between graphs; inside a graph two streams take
    alternate steps (independent batches), so one step's start-up and tail
    overlap the other stream's step.  After the timed region each call kind
    (route plan + pack; direct receive) runs alone, back to back over the
    rotating sets in a graph of its own on one stream: its device time over
    the calls is the per-call duration of the roofline (not part of the step
    time)."""
    T, H, k, E = w.T, w.H, w.k, w.E
    tok_host = torch.from_numpy(w.tokens.view(np.int16)).view(torch.bfloat16)
    topk_host = torch.from_numpy(np.ascontiguousarray(w.topk))
    lay = step_layout(w, n_sets)
    S, nset, ns = lay["S"], lay["nset"], lay["streams"]
    assert S == nq.row_bytes(H) and lay["R_cap"] == nq.rows_capacity(T, k, E, w.A)
    sets = [BufferSet(torch, nq, w, tok_host, topk_host) for _ in range(nset)]
    torch.cuda.synchronize()
    st = int(sets[0].plan.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st:#x} after the first pass")
    R = int(sets[0].plan.offsets[-1].item())
    for b in sets:
        b.capture(torch)
    GRAPH_ROTATIONS = 50
    CALLS_TIMED = 20     # calls of each kind behind the per-call durations
    gR = capture_rotation(torch, sets, 1, ns)
    nblocks, rem = divmod(K, nset)
    n_big, n_small = divmod(nblocks, GRAPH_ROTATIONS)
    gBig = capture_rotation(torch, sets, GRAPH_ROTATIONS, ns) if n_big else None
    gSmall = capture_rotation(torch, sets, n_small, ns) if n_small else None
    clocks = ClockSampler(gpu_index, enabled=clocks_enabled)
    clocks.start()
    time.sleep(0.1)
    busy0 = time.time()
    # every graph the timed region replays runs once first (a graph's first
    # launch also uploads it), then at least W warm-up steps
    for g in (gBig, gSmall):
        if g is not None:
            g.replay()
    for j in range(rem):
        sets[j].gS.replay()
    for i in range(max(1, math.ceil(W / nset))):
        gR.replay()
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record()
    for _ in range(n_big):
        gBig.replay()
    if gSmall is not None:
        gSmall.replay()
    for j in range(rem):
        sets[j].gS.replay()
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    time.sleep(0.03)
    clocks.stop()
    clk = clocks.summary(wall0, wall1, busy0)
    ms_total = t0.elapsed_time(t1)
    # per-call durations (the roofline's): each call alone, back to back over
    # the rotating sets in one graph on one stream, device time / calls
    def calls_graph(call, rotations):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(rotations):
                    for b in sets:
                        getattr(b, call)()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return g

    call_rot = max(1, math.ceil(CALLS_TIMED / nset))
    per_call = []
    for call in ("route_pack", "receive"):
        g = calls_graph(call, call_rot)
        g.replay()   # the first launch also uploads the graph
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b_.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b_) / (call_rot * nset))
        per_call.append(float(np.median(ts)))
        del g
    ms_a, ms_b = per_call
    st = int(sets[0].plan.status.item())
    route_b, pack_b, dr_b = algorithmic_bytes(T, H, k, E, R, S)
    set_mb = (route_b + pack_b + dr_b) / 1e6
    return dict(sets=sets, tok_host=tok_host, topk_host=topk_host, nset=nset, streams=ns, set_mb=set_mb,
                n_sets_req=n_sets, T=T, H=H,
                k=k, E=E,
                R=R, S=S, ms_total=ms_total, ms_step=ms_total / K, ms_a=ms_a, ms_b=ms_b, wall_s=wall1 - wall0,
                clocks=clk, status=st, bytes=(route_b, pack_b, dr_b), w=w, n_calls_timed=call_rot * nset, K=K, W=W)


def step_report(r, peak, peak_kind, world=1, config=None, n_sets_note=True) -> dict:
    """The JSON fields of one timed workload: throughput, path and per-call
    rates, and the roofline block of the dominant kernel (the direct receive)."""
    route_b, pack_b, dr_b = r["bytes"]
    w = r["w"]
    tokens_s = world * r["T"] / (r["ms_step"] * 1e-3)
    dr_gbs = dr_b / (r["ms_b"] * 1e-3) / 1e9
    pack_gbs = (route_b + pack_b) / (r["ms_a"] * 1e-3) / 1e9
    path_gbs = (route_b + pack_b + dr_b) / (r["ms_step"] * 1e-3) / 1e9
    cfg = workload_config(w, r["R"], world, r["n_sets_req"])
    assert str(r["nset"]) + " rotating" in cfg["l2"] and f"{r['streams']} streams" in cfg["l2"]
    return {
        "value": tokens_s, "unit": UNIT, "ms_per_step": r["ms_step"], "steps": r["K"], "warmup": r["W"],
        "config": cfg,
        "path": {"gbs": path_gbs, "frac_of_peak": path_gbs / peak, "bytes_per_step": route_b + pack_b + dr_b,
                 "route_pack_ms": r["ms_a"], "route_pack_gbs": pack_gbs, "route_pack_frac": pack_gbs / peak,
                 "direct_receive_ms": r["ms_b"], "direct_receive_gbs": dr_gbs},
        "roofline": {"kernel": "direct_receive_kernel (ep_nvfp4_direct_receive)", "bound": "hbm",
                     "achieved": dr_gbs, "peak": peak, "unit": "GB/s", "frac": dr_gbs / peak,
                     "peak_kind": f"{peak_kind} (copy bandwidth)", "bytes_per_launch": dr_b,
                     "traffic": profiled_traffic("direct_receive", DR_SOURCES, config)},
        "clocks": r["clocks"],
        "device_status": r["status"],
        "calls_for_kernel_times": r["n_calls_timed"],
    }


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

    w = workloads.make(args.config, **workload_kwargs(args, rank))
    r = time_steps(torch, nq, w, args.steps, args.warmup, args.sets, barrier, not args.no_clocks, local)
    r["ms_total"] = max_over_ranks(dist, r["ms_total"], "cuda")
    r["ms_step"] = r["ms_total"] / args.steps
    r["world"] = world
    sets = r.pop("sets")
    # ---- end to end through the public API with host buffers
    e2e_steps = args.e2e_steps or int(min(200, max(20, 1000.0 / max(r["ms_step"] * 8, 1e-3))))
    r["e2e"] = e2e_measure(torch, nq, w, sets[:2], r["tok_host"], r["topk_host"], r["R"], e2e_steps)
    r["e2e"]["ms"] = max_over_ranks(dist, r["e2e"]["ms"], "cuda")
    # ---- the calls outside the step: unpack, MXFP8 pack, the BF16 columnwise
    # operands and the receive's variants, same batch
    r["aux"] = aux_measure(torch, nq, w, sets[0], r["R"])
    del sets
    torch.cuda.empty_cache()
    # ---- the other workloads (rank 0 of the replicas is enough: they are reports, not the headline)
    r["extra"] = {}
    r["config5"] = None
    if not args.no_extra_configs and args.config == WORKLOAD_CFG and not args.tokens and not args.experts:
        peak, peak_kind = load_peaks()
        for c, K in ((2, 3000), (3, 2000)):
            wc = workloads.make(c, **replica_workload_kwargs(rank, c))
            rc = time_steps(torch, nq, wc, K, max(args.warmup, 20), 0, None, not args.no_clocks, local)
            del rc["sets"]
            torch.cuda.empty_cache()
            r["extra"][str(c)] = step_report(rc, peak, peak_kind, 1, c)
        r["config5"] = config5_measure(torch, nq, workloads, rank, local, not args.no_clocks, peak, peak_kind)
        torch.cuda.empty_cache()
    return r


def config5_measure(torch, nq, workloads, rank, local, clocks_enabled, peak, peak_kind) -> dict:
    """The MXFP8 vs NVFP4 dispatch comparison on the StudentT(4) batch
    (16384 x 7168, 64 experts top-6): the NVFP4 step timed like the headline
    (RNE), both packs timed as single calls after an L2 flush, and the
    relative RMS decode error of each format, sqrt(sum (decoded - x)^2 /
    sum x^2) over every element of every token, from the GPU outputs (each
    token's first destination row; its k rows are identical)."""
    w = workloads.make(5, **replica_workload_kwargs(rank, 5))
    rc = time_steps(torch, nq, w, 200, 20, 0, None, clocks_enabled, local)
    out = step_report(rc, peak, peak_kind, 1, 5)
    b = rc["sets"][0]
    T, H, k, R_cap = w.T, w.H, w.k, b.plan.R_cap
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    mx = torch.empty(R_cap * H + R_cap * (H // 32), dtype=torch.uint8, device="cuda")

    def timed(fn, reps=10):
        for _ in range(2):
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

    ms_mx = timed(lambda: nq.ep_mxfp8_pack(b.tok, b.plan, buf=mx))
    ms_nv = timed(lambda: nq.ep_nvfp4_pack(b.tok, b.plan, rows=b.rows, rounding=w.rounding, seed=w.seed))
    bytes_mx = 2 * T * H + 4 * T * k + rc["R"] * (H + H // 32)
    bytes_nv = 2 * T * H + 4 * T * k + rc["R"] * rc["S"]
    # decode errors, token by token against the BF16 input
    first = b.plan.dest.view(T, k)[:, 0].long()
    un = nq.ep_nvfp4_unpack(b.rows, H, b.plan.offsets, w.E, status=b.plan.status)
    data = mx[: R_cap * H].view(R_cap, H)
    scl = mx[R_cap * H:].view(R_cap, H // 32)
    num_nv = num_mx = den = 0.0
    for t0 in range(0, T, 1024):
        rows_t = first[t0:t0 + 1024]
        x = b.tok[t0:t0 + 1024].double()
        d_nv = un[rows_t].double()
        e = scl[rows_t].to(torch.int32) - 127
        d_mx = data[rows_t].view(torch.float8_e4m3fn).double() * torch.pow(2.0, e.double()).repeat_interleave(32, 1)
        num_nv += float(((d_nv - x) ** 2).sum())
        num_mx += float(((d_mx - x) ** 2).sum())
        den += float((x ** 2).sum())
    torch.cuda.synchronize()
    st = int(b.plan.status.item())
    del rc["sets"], b, flush, mx, un
    out["mxfp8_pack"] = {"ms": ms_mx, "gbs": bytes_mx / (ms_mx * 1e-3) / 1e9,
                         "frac": bytes_mx / (ms_mx * 1e-3) / 1e9 / peak, "bytes": bytes_mx,
                         "note": "one call (fused gather, E8M0 per 32, E4M3), L2 flushed before each launch"}
    out["nvfp4_pack"] = {"ms": ms_nv, "gbs": bytes_nv / (ms_nv * 1e-3) / 1e9,
                         "frac": bytes_nv / (ms_nv * 1e-3) / 1e9 / peak, "bytes": bytes_nv,
                         "note": "one call on the same tokens and plan, L2 flushed before each launch"}
    out["rms_rel_err"] = {"mxfp8": math.sqrt(num_mx / den), "nvfp4": math.sqrt(num_nv / den),
                          "definition": "sqrt(sum (decoded - x)^2 / sum x^2) over all T x H elements; NVFP4 "
                                        "decoded by ep_nvfp4_unpack, MXFP8 as E4M3 element x 2^(E8M0 - 127)"}
    out["device_status"] = max(out["device_status"], st)
    return out


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
    # every output copied back by each lane's last step equals the device
    # tensor it came from, whole (nothing writes them after that step)
    ok = all(torch.equal(d.to(x.device), x) for _, _, srcs, dsts in lanes for x, d in zip(srcs, dsts))
    return dict(ms=ms, h2d=h2d, d2h=d2h, ok=bool(ok), steps=steps, link=host_link_gbs(torch))


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


def oracle_expert_pass(o, w, experts, times: dict | None = None, other_ops: bool = False) -> int:
    """The batch's route plan + pack + direct receive on the oracle,
    restricted to the experts in ``experts``: every routing slot to another
    expert is dropped, so each kept expert has exactly its rows (and padding)
    of the whole batch, the pack writes only those rows and the receive
    builds only those experts' operands.  Returns the number of routed slots
    kept; slots / k is the batch's work in tokens that the pass did.
    ``times`` (if given) receives the seconds of each call; with
    ``other_ops`` the unpack of the packed rows and the MXFP8 pack of the same
    slots follow (timed, outside the three calls of the path)."""
    topk = np.array(w.topk, copy=True)
    topk[~np.isin(topk, np.asarray(list(experts), dtype=np.int32))] = -1
    t0 = time.perf_counter()
    off, cnt, dest, _ = o.route_plan(topk, w.E, w.A)
    t1 = time.perf_counter()
    R_cap = int(off[-1])
    rows = o.nvfp4_pack(w.tokens, dest, w.k, off, cnt, w.E, max(R_cap, 1), rounding=w.rounding, seed=w.seed)
    t2 = time.perf_counter()
    o.nvfp4_direct_receive(rows, w.H, off, w.E, rounding=w.rounding, seed=w.seed, sign_mask=w.sign_mask,
                           experts=list(experts))
    t3 = time.perf_counter()
    if times is not None:
        times.update(route_plan=t1 - t0, pack=t2 - t1, direct_receive=t3 - t2)
        if other_ops:
            o.nvfp4_unpack(rows, w.H, off, w.E)
            t4 = time.perf_counter()
            o.mxfp8_pack(w.tokens, dest, w.k, off, cnt, w.E, max(R_cap, 1))
            times.update(unpack=t4 - t3, mxfp8_pack=time.perf_counter() - t4)
    return int(np.count_nonzero(topk >= 0))


def expert_loads(w) -> list[tuple[int, int]]:
    """(expert, routed slots) of every expert with at least one slot."""
    ids, counts = np.unique(w.topk[w.topk >= 0], return_counts=True)
    return [(int(e), int(c)) for e, c in zip(ids, counts)]


def expert_groups(loads, n_groups: int) -> list[list[int]]:
    """Experts split into n_groups of about equal slots (largest first, each
    to the least loaded group)."""
    groups = [[] for _ in range(n_groups)]
    tot = [0] * n_groups
    for e, c in sorted(loads, key=lambda x: -x[1]):
        g = int(np.argmin(tot))
        groups[g].append(e)
        tot[g] += c
    return [sorted(g) for g in groups if g]


def host_cpu() -> dict:
    """The host's logical CPU count and model name (lscpu, else /proc/cpuinfo)."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not name:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    name = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return {"nproc": n, "model": name or "unknown"}


_SLICE_W = None


def _oracle_group_init(cfg: int, kw: dict):
    """Pool initializer of the all-core baseline: the workload and the oracle,
    made once per process before any timed task."""
    global _SLICE_W
    import oracle as o
    import workloads
    _SLICE_W = workloads.make(cfg, **kw)
    o.lib()


def _oracle_group_worker(experts):
    """One task of the all-core baseline: the oracle's pass over one group
    of experts; returns (start, end) wall-clock seconds and the slots done."""
    import oracle as o
    t0 = time.time()
    n = oracle_expert_pass(o, _SLICE_W, experts) if experts else 0
    return t0, time.time(), n


def cpu_baseline(w, cfg: int, budget_s: float = 10.0, all_cores: bool = True, kw: dict | None = None) -> dict:
    """The oracle, as it stands (single-threaded C), timed on a bounded sample
    of the batch: the route plan, pack and direct receive restricted to the
    first m experts (each with exactly its rows and padding of the whole
    batch), m sized from a one-expert probe for about ``budget_s``; value =
    (routed slots kept / k) / seconds, i.e. tokens of the batch per second.
    Then the whole batch on all host cores: its experts split into one group
    per core (about equal slots), one process per group, started together;
    value = tokens of the batch / (last end - first start)."""
    import oracle as o
    o.build()
    loads = expert_loads(w)
    t0 = time.perf_counter()
    s1 = oracle_expert_pass(o, w, [loads[0][0]])
    per_slot = (time.perf_counter() - t0) / max(s1, 1)
    m, acc = 0, 0
    while m < len(loads) and (m == 0 or (acc + loads[m][1]) * per_slot <= budget_s):
        acc += loads[m][1]
        m += 1
    experts = [e for e, _ in loads[:m]]
    times = {}
    slots = oracle_expert_pass(o, w, experts, times, other_ops=True)
    dt = times["route_plan"] + times["pack"] + times["direct_receive"]
    hc = host_cpu()
    res = {"value": slots / w.k / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "host_cpu": hc["model"],
           "nproc": hc["nproc"],
           "sample": f"route plan + pack + direct receive of {m} of the batch's {len(loads)} routed experts "
                     f"({slots} of {int(np.count_nonzero(w.topk >= 0))} slots, each expert with its rows and "
                     f"padding of the whole batch), single-threaded C oracle, {dt:.2f} s; tokens = slots / k",
           "per_call": {"unit": UNIT, "sample": "the same slots, each call timed alone (the unpack decodes the "
                                                "packed rows, the MXFP8 pack encodes the same slots)",
                        **{op: slots / w.k / sec for op, sec in times.items()}}}
    if all_cores and hc["nproc"] > 1:
        import multiprocessing as mp
        C = hc["nproc"]
        groups = expert_groups(loads, C)
        with mp.get_context("spawn").Pool(len(groups), initializer=_oracle_group_init,
                                          initargs=(cfg, kw or {})) as pool:
            # a short task per process first, so that every process has made
            # its workload before the timed tasks start
            pool.map(_oracle_group_worker, [[]] * (2 * len(groups)), chunksize=1)
            spans = pool.map(_oracle_group_worker, groups, chunksize=1)
        wall = max(e for _, e, _ in spans) - min(s for s, _, _ in spans)
        slots_all = sum(n for _, _, n in spans)
        res["all_cores"] = {"value": slots_all / w.k / wall, "unit": UNIT, "cores": len(groups), "wall_s": wall,
                            "sample": f"the whole batch: its experts in {len(groups)} groups of about equal slots, "
                                      "one process per group (the unchanged single-threaded oracle) started "
                                      "together; tokens / (last end - first start)"}
        res["cores_all"] = len(groups)
    return res


def reference_arm(args, rank, world):
    """--impl reference: the oracle on the host cores, single-threaded; each
    step is the route plan + pack + direct receive of a group of the batch's
    experts (each with its rows and padding of the whole batch; groups taken
    in turn), the group sized so that warm-up + K steps take about two
    minutes; value = (routed slots / k) / seconds."""
    if rank != 0:
        return None
    import oracle as o
    import workloads
    o.build()
    w = workloads.make(args.config)
    loads = expert_loads(w)
    t0 = time.perf_counter()
    s1 = oracle_expert_pass(o, w, [loads[0][0]])
    per_slot = (time.perf_counter() - t0) / max(s1, 1)
    K, W = args.steps, args.warmup
    budget = 120.0 / max(K + W, 1)
    m = int(max(1, min(len(loads), budget / max(per_slot * np.mean([c for _, c in loads]), 1e-9))))
    groups = [[loads[(i * m + j) % len(loads)][0] for j in range(m)] for i in range(K + W)]
    for i in range(W):
        oracle_expert_pass(o, w, groups[i])
    slots = 0
    t0 = time.perf_counter()
    for i in range(K):
        slots += oracle_expert_pass(o, w, groups[W + i])
    dt = time.perf_counter() - t0
    value = slots / w.k / dt
    hc = host_cpu()
    R = int(o.route_plan(w.topk, w.E, w.A)[0][-1])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": dt * 1e3 / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            # the GPU arm's config of the same batch; what one step here covers is in "sample"
            "config": workload_config(w, R, world, args.sets),
            "sample": {"experts_per_step": m, "tokens_per_step": slots / w.k / max(K, 1)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "host_cpu": hc["model"],
                             "nproc": hc["nproc"],
                             "sample": f"per step the route plan + pack + direct receive of {m} of the batch's "
                                       f"{len(loads)} routed experts (each with its rows and padding of the whole "
                                       "batch; groups in turn); tokens = routed slots / k"},
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
    w = r["w"]
    rep = step_report(r, peak, peak_kind, world, args.config)
    e2e = r["e2e"]
    line = {
        "metric": METRIC, "value": rep["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": rep["config"],
        "path": rep["path"],
        "roofline": rep["roofline"],
        "e2e": {"value": world * r["T"] / (e2e["ms"] * 1e-3), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e["ms"], "steps": e2e["steps"],
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
        "calls_for_kernel_times": r["n_calls_timed"],
        "clocks": r["clocks"],
        "device_status": r["status"],
        "timed_wall_s": r["wall_s"],
    }
    if r["extra"]:
        line["configs"] = r["extra"]
    if r["config5"] is not None:
        line["config5"] = r["config5"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.config, kw=workload_kwargs(args, 0))
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
