"""Host-side logic of the benchmark, on CPU: multi-rank timing reduction and
per-rank seeding over a 2-rank gloo group, the clocks parser, the algorithmic
byte counts, and the reference arm (the oracle) end to end."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_moe_layout_05_gb300 import workload as wl  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [3.5, 7.25][rank]
    m = bench.max_over_ranks(elapsed)
    bench.barrier()
    seed = bench.shard_seed(1, rank)
    inp = wl.make_inputs(wl.get("tiny"), seed=seed)
    q.put((rank, m, seed, int(inp.topk_ids.sum())))
    dist.destroy_process_group()


def test_two_rank_gloo_max_and_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [7.25, 7.25]         # max over ranks on both
    assert res[0][2] != res[1][2]                       # distinct seeds
    assert res[0][3] != res[1][3]                       # distinct routing


def test_max_over_ranks_without_group():
    assert bench.max_over_ranks(2.5) == 2.5


def test_clock_parser_window():
    text = ("2026/12/02 10:00:00.000, 400, 2070, 100, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "2026/12/02 10:00:01.000, 1900, 2070, 900, 0x4, Not Active, Not Active, Not Active, Active\n"
            "2026/12/02 10:00:01.100, 1950, 2070, 950, 0x4, Not Active, Not Active, Not Active, Active\n")
    import datetime
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0, 500000).timestamp()
    t1 = datetime.datetime(2026, 12, 2, 10, 0, 2).timestamp()
    c = bench.ClockSampler.parse(text, t0, t1)
    assert c == {"sm_mhz": 1925.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}


def test_algorithmic_bytes_decode():
    w = wl.get("decode_dsv3")
    b = bench.algorithmic_bytes(w, "bf16")
    # one token row read, K rows written, K slot indices read
    assert b["dispatch"] == 128 * 7168 * 2 * 9 + 128 * 8 * 4
    # K rows gathered, K weights and slots read, one row written
    assert b["combine"] == 128 * 7168 * 2 * 9 + 128 * 8 * 8
    f = bench.algorithmic_bytes(w, "fp8")
    assert f["dispatch"] == 128 * 7168 * 2 + 128 * 8 * (7168 + 4 * 56) + 128 * 8 * 4


def test_traffic_rows_keyed_by_source_hash(tmp_path):
    h = bench.kernel_source_hash("combine")
    f = tmp_path / "t.json"
    f.write_text(json.dumps({"rows": [
        {"call": "combine", "workload": "decode_dsv3", "dispatch": "bf16",
         "source_hash": h, "dram_bytes_per_launch": 123},
        {"call": "combine", "workload": "prefill_qwen3", "dispatch": "fp8",
         "source_hash": "000000000000", "dram_bytes_per_launch": 456}]}))
    assert bench.profiled_traffic("combine", "decode_dsv3", "bf16", str(f)) == 123
    assert bench.profiled_traffic("combine", "prefill_qwen3", "fp8", str(f)) is None  # stale
    assert bench.profiled_traffic("combine", "tiny", "bf16", str(f)) is None
    assert bench.profiled_traffic("combine", "decode_dsv3", "bf16", str(tmp_path / "x")) is None


def test_committed_traffic_file_parses():
    with open(bench.TRAFFIC_FILE) as f:
        rows = json.load(f)["rows"]
    for r in rows:
        assert r["call"] in bench.CALL_SOURCES
        assert r["dram_bytes_per_launch"] > 0 and len(r["source_hash"]) == 12


def test_default_workload_is_the_largest_config():
    args = bench.parse_args([])
    assert args.workload is None and wl.HEADLINE == "prefill_qwen3"
    w = wl.get(wl.HEADLINE)
    assert w.dispatch[0] == "fp8" and args.combine == "bf16"
    assert all(w.T * w.H >= v.T * v.H for v in wl.WORKLOADS.values())
    assert bench.dtype_label("fp8", "bf16").startswith("fp8-e4m3 dispatch")


def test_reference_arm_runs_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["host_cpus"] >= 1 and line["cpu_baseline"]["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["metric"] == bench.METRIC


def test_variant_options_and_launch_counts():
    """--variant picks a form the library keeps behind test hooks; each
    reports its own launches per step (host-side plan queries only)."""
    for v in ("library", "cluster", "decode_bulk", "persistent", "persistent_bulk",
              "combine_shuffle"):
        assert bench.parse_args(["--variant", v]).variant == v
    q = wl.get("prefill_qwen3")
    d = wl.get("decode_dsv3")
    assert bench.launches_per_step(q, "fp8", False) == 3          # count, rank-and-pack, combine
    assert bench.launches_per_step(q, "fp8", False, variant="persistent") == 3
    assert bench.launches_per_step(d, "bf16", False) == 2         # one fused kernel, combine
    assert bench.launches_per_step(d, "bf16", False, variant="cluster") == 2
    assert bench.launches_per_step(q, "fp8", True) == 2 + 2       # count, ranking; dispatch; combine
