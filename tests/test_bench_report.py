"""The GPU arm's JSON fields, composed on the host from a timing record (no
GPU): the roofline block of the direct receive (achieved = algorithmic bytes
per launch / the launch's duration, frac = achieved / peak), the path and
throughput figures, and the DRAM traffic looked up from the committed ncu
record only while it was taken on the current kernel sources."""
import json
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import workloads  # noqa: E402


def record(T=16384, H=7168, k=8, E=256, R=147200, ms_step=0.75, ms_a=0.15, ms_b=0.61):
    S = (9 * H // 16 + 16 + 15) // 16 * 16
    w = types.SimpleNamespace(description="synthetic", A=128, rounding=1, T=T, H=H, k=k, E=E)
    return dict(w=w, T=T, H=H, k=k, E=E, R=R, S=S, nset=2, streams=2, n_sets_req=0, set_mb=2600.0, ms_step=ms_step,
                ms_a=ms_a, ms_b=ms_b, K=100, W=10, clocks=None, status=0, n_calls_timed=20,
                bytes=bench.algorithmic_bytes(T, H, k, E, R, S))


def test_algorithmic_bytes_follow_their_definition():
    T, H, k, E, R = 100, 1024, 2, 4, 512
    S = (9 * H // 16 + 16 + 15) // 16 * 16
    route, pack, dr = bench.algorithmic_bytes(T, H, k, E, R, S)
    assert route == 4 * T * k * 2 + 4 * (2 * E + 1)
    assert pack == 2 * T * H + 4 * T * k + R * S
    # rows in; rowwise codes + scales + the row scale, columnwise codes + scales out; 12 B of metadata per expert
    assert dr == R * S + R * (H // 2 + H // 16 + 4) + R * (H // 2 + H // 16) + 12 * E


def test_roofline_block_is_bytes_over_the_launch_duration():
    r = record()
    rep = bench.step_report(r, 6663.2, "measured", 1, 4)
    route_b, pack_b, dr_b = r["bytes"]
    rf = rep["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] == 6663.2
    assert rf["bytes_per_launch"] == dr_b
    assert rf["achieved"] == pytest.approx(dr_b / (r["ms_b"] * 1e-3) / 1e9)
    assert rf["frac"] == pytest.approx(rf["achieved"] / 6663.2)
    p = rep["path"]
    assert p["bytes_per_step"] == route_b + pack_b + dr_b
    assert p["gbs"] == pytest.approx((route_b + pack_b + dr_b) / (r["ms_step"] * 1e-3) / 1e9)
    assert p["route_pack_gbs"] == pytest.approx((route_b + pack_b) / (r["ms_a"] * 1e-3) / 1e9)
    assert rep["value"] == pytest.approx(r["T"] / (r["ms_step"] * 1e-3))
    # N replicas: the tokens of every rank count
    assert bench.step_report(r, 6663.2, "measured", 4, 4)["value"] == pytest.approx(4 * rep["value"])


def test_traffic_comes_only_from_a_record_of_the_current_sources(tmp_path):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["direct_receive"]["4"]
    cur = bench.source_sha(bench.DR_SOURCES)
    got = bench.profiled_traffic("direct_receive", bench.DR_SOURCES, 4)
    if rec["source_sha"] == cur:
        assert got == float(rec["dram_bytes_per_launch"])
        # the record's bytes are its measured rows' bytes scaled to the full batch
        m = rec["measured"]
        assert rec["dram_bytes_per_launch"] == round((m["dram_bytes_read"] + m["dram_bytes_write"]) * 147200 /
                                                     m["rows"])
    else:
        assert got is None
    # another kernel source, or a configuration without a record: no traffic
    other = tmp_path / "other.cu"
    other.write_text("// not the receive\n")
    assert bench.profiled_traffic("direct_receive", [os.path.relpath(other, ROOT)], 4) is None
    assert bench.profiled_traffic("direct_receive", bench.DR_SOURCES, 3) is None


def test_step_streams_and_set_rounding():
    """Small batches take four streams, large ones two, and the rotating
    sets are a multiple of the stream count, so a set stays on one stream."""
    assert bench.step_streams(128 << 20) == 4 and bench.step_streams(900 << 20) == 4
    assert bench.step_streams(1 << 30) == 2 and bench.step_streams(3 << 30) == 2
    for set_bytes in (64 << 20, 128 << 20, 700 << 20, 2 << 30, 3 << 30):
        ns = bench.step_streams(set_bytes)
        n = bench.n_rotating_sets(set_bytes)
        n += (-n) % ns
        assert n % ns == 0 and n >= 2
        # step j runs on stream j mod ns; set j mod n: one stream per set
        owners = {}
        for j in range(5 * n):
            owners.setdefault(j % n, set()).add(j % ns)
        assert all(len(v) == 1 for v in owners.values())


def test_cpu_baseline_reports_each_call():
    """The oracle's CPU baseline gives the path's rate and each call's alone
    (route plan, pack, direct receive, and the unpack and MXFP8 pack of the
    same slots), with the host's CPU named; the path's rate is that of the
    three calls of the path together."""
    w = workloads.make(1)
    r = bench.cpu_baseline(w, 1, budget_s=0.5, all_cores=False)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["host_cpu"] and r["nproc"] >= 1
    pc = r["per_call"]
    for op in ("route_plan", "pack", "direct_receive", "unpack", "mxfp8_pack"):
        assert pc[op] > 0, op
    # 1 / rate adds up over the calls of the path
    inv = 1 / pc["route_plan"] + 1 / pc["pack"] + 1 / pc["direct_receive"]
    assert abs(1 / inv - r["value"]) <= 1e-6 * r["value"]
