"""bench.py on a GPU, small: one JSON line with the contract's fields, the
bench's own parity gate bit-exact, every path and combine variant."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "64",
                        "--warmup", "8", "--graph-steps", "16", "--cpu-seconds", "0.5", *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("args", [
    ("--workload", "tiny"),
    ("--workload", "tiny", "--dispatch", "fp8", "--combine", "fp8"),
    ("--workload", "tiny", "--combine", "rank_partial"),
    ("--workload", "tiny", "--path", "regions"),
    ("--workload", "tiny", "--unfused", "--no-e2e", "--no-cpu-baseline"),
])
def test_bench_line(args):
    d = _bench(*args)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "roofline",
                "gpu_launches", "clocks", "timing"):
        assert key in d, key
    t = d["timing"]
    assert t["passes"] >= 3 and t["steps_per_pass"] == 64
    assert d["gpu_launches"] == d["launches_per_step"] * 64 * t["passes"]
    assert d["parity"] == "bit-exact"
    assert d["value"] > 0 and d["steps"] == 64 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    if "--no-e2e" not in args:
        e = d["e2e"]
        assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
        assert e["output_matches_device_run"]
    if "--no-cpu-baseline" not in args:
        c = d["cpu_baseline"]
        assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] == 1
