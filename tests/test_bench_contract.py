"""The benchmark's JSON contract on the part that runs without a GPU: the
reference arm (the oracle timed on the host cores) prints one JSON line with
the keys the driver reads, on the small configuration."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert "workload" in d["config"]
    # the reference line carries the GPU arm's config of the same batch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import workloads
    w = workloads.make(1)
    R = int(oracle.route_plan(w.topk, w.E, w.A)[0][-1])
    assert d["config"] == bench.workload_config(w, R, 1)
    assert d["config"]["R"] == R and d["config"]["T"] == w.T
