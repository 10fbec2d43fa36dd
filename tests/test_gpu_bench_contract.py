"""bench.py's one-line JSON contract on the GPU (the small fp32 workload, a few steps): every required key with
sane values, and the reference arm's line beside it."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REQUIRED = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"]


def _line(args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_has_every_key():
    d = _line(["--workload", "tiny", "--steps", "3", "--warmup", "3", "--cpu-seconds", "2", "--configs", "prefill"])
    for k in REQUIRED:
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["n_gpus"] == 1 and d["steps"] == 3
    roof = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in roof, k
    assert roof["achieved"] > 0 and abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
    assert cpu["single_thread"]["cores"] == 1 and cpu["single_thread"]["value"] > 0
    # the per-pass sweep and the other configurations timed in the same process
    sw = d["sweep"][0]
    assert sw["layer_ms"] > 0 and sw["gemm1_ms"] <= sw["layer_ms"] and sw["layer_frac"] > 0
    assert list(d["configs"]) == ["prefill"]
    c = d["configs"]["prefill"]
    for k in ("value", "ms_per_step", "roofline", "clocks", "layer_frac", "routes_per_step", "gpu_launches"):
        assert k in c, k
    assert c["value"] > 0 and c["roofline"]["bound"] == "tensor" and 0 < c["roofline"]["frac"] < 1.2
    assert abs(c["value"] - c["routes_per_step"] / (c["ms_per_step"] / 1e3)) / c["value"] < 1e-3
    assert "sm_mhz" in c["clocks"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    ts = d["timing_stats"]
    assert len(ts["ms_per_step_replays"]) == 5 and ts["ms_per_step_replays"][0] == d["ms_per_step"]
    assert ts["p10"] <= ts["median"] <= ts["p90"] and ts["eager_ms_per_step"] > 0


def test_reference_arm_line():
    d = _line(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
