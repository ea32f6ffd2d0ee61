#!/usr/bin/env python3
"""Benchmark of the single-GPU MoE layout + dispatch + combine path.

One step = moe_layout_dispatch (layout, then dispatch) -> moe_combine on one
batch of the workload.  Default: the Qwen3-235B-shaped prefill (T=16384
tokens, H=4096, E=128 experts over R=16 regions, top-8 Zipf(1.0) routing,
1 % outlier rows) with block-scaled FP8 dispatch and bf16 combine; the
stand-in experts (dequantised identity) are materialised once before timing.
Prints one JSON line: whole-job tokens/s, per-call times and HBM GB/s, the
roofline of the dominant call, an end-to-end figure through host buffers,
clocks seen during the timed region, and the CPU oracle timed on the host.
`--all` prints one such line per workload and dispatch variant.

Timing: the K steps of one pass are captured into CUDA graphs (the launch
cost of a decode-sized step is comparable to its run time); the pass is
replayed repeatedly, between a barrier and a device synchronize, until at
least --min-seconds of device time have been measured, with CUDA events on
the launching stream around every pass; ms_per_step is the median pass / K.
Every step works on one of S rotating buffer sets whose total size is at
least 3x the L2 cache, so each step starts cold in L2.  Each call of the step
is also timed alone the same way.  `--impl reference` times the CPU oracle
instead.

Multi-GPU (torchrun): every rank runs its own replica on its own tokens (no
data-path collective); the elapsed time is the maximum over ranks and the
value counts the tokens of all ranks ("weak" scaling).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
KERNELS = ("layout", "dispatch", "combine")

# workload and dispatch variants of --all (the tiny workload is a parity case)
ALL_VARIANTS = (("decode_dsv3", "bf16"), ("decode_dsv3_fp8", "fp8"),
                ("prefill_kimi_k2", "bf16"), ("prefill_kimi_k2", "fp8"),
                ("prefill_qwen3", "fp8"))


# --------------------------------------------------------------- helpers --

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200, help="steps per timed pass (K)")
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=None, help="workload name (default: prefill_qwen3)")
    p.add_argument("--dispatch", choices=("bf16", "fp8"), default=None)
    p.add_argument("--all", action="store_true",
                   help="one line per workload and dispatch variant (%s)"
                        % ", ".join(f"{n}/{d}" for n, d in ALL_VARIANTS))
    p.add_argument("--min-seconds", type=float, default=1.0,
                   help="device time over which K-step passes are repeated")
    p.add_argument("--call-seconds", type=float, default=0.4,
                   help="device time over which each call is timed alone")
    p.add_argument("--graph-steps", type=int, default=512,
                   help="steps per captured graph")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="host time spent timing the oracle baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-parity", action="store_true",
                   help="skip the bench's own oracle check of one step")
    p.add_argument("--path", choices=("packed", "regions"), default="packed",
                   help="regions: dispatch through per-rank send regions (moe_dispatch_send, "
                        "private area of --private rows, bulk sized to the worst case) and "
                        "moe_dispatch_recv back to the packed layout")
    p.add_argument("--private", type=int, default=4, help="private rows per region (--path regions)")
    p.add_argument("--unfused", action="store_true",
                   help="moe_layout + moe_dispatch as two calls instead of moe_layout_dispatch")
    p.add_argument("--variant", choices=("library", "cluster", "decode_bulk", "persistent",
                                          "persistent_bulk", "combine_shuffle"),
                   default="library",
                   help="layout+dispatch form (A/B of alternatives the library keeps behind test "
                        "hooks): cluster = decode batches counted by thread-block clusters; "
                        "decode_bulk = the decode kernel writing rows by bulk copies out of "
                        "shared memory (K = 8); persistent[_bulk] = large batches through one CTA "
                        "per SM and a shared-memory ring of bulk copies (bulk: bf16 rows stored "
                        "by bulk copies); combine_shuffle = the bf16 combine with each token's "
                        "slots and weights loaded by 8 lanes and shuffled to the warp (K = 8)")
    p.add_argument("--combine", choices=("bf16", "fp8", "rank_partial"), default="bf16",
                   help="fp8: combine reads the FP8 dispatch output directly "
                        "(moe_combine_fp8, identity experts; needs --dispatch fp8); "
                        "rank_partial: sender-side per-rank partial sums "
                        "(moe_combine_rank_partial)")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def shard_seed(base: int, rank: int) -> int:
    """Each rank draws its own tokens: weak scaling over independent batches."""
    return base + 1000003 * rank


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a host float over all ranks (identity without a group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_info() -> dict:
    """The host the CPU baseline ran on: logical CPUs and the CPU model."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip() in ("model name", "Model", "Hardware"):
                    model = val.strip()
                    break
    except OSError:
        pass
    import platform
    return {"host_cpus": os.cpu_count(), "cpu_model": model or platform.machine()}


def algorithmic_bytes(w, dispatch: str):
    """Bytes each kernel must move at minimum for one batch (one launch)."""
    T, H, K, E, R = w.T, w.H, w.K, w.E, w.R
    layout = 4 * T * K * 3 + 4 * E + 4 * (E + 1) + 4 * (R + 1)
    if dispatch == "bf16":
        disp = 2 * T * H + 2 * T * K * H + 4 * T * K
    else:
        disp = 2 * T * H + T * K * H + 4 * T * K * (H // 128) + 4 * T * K
    comb = 2 * T * K * H + 8 * T * K + 2 * T * H
    comb8 = T * K * H + 4 * T * K * (H // 128) + 8 * T * K + 2 * T * H
    row = (2 * H if dispatch == "bf16" else H + 4 * (H // 128))
    send = disp + 4 * T * K
    recv = 2 * T * K * row + 4 * (R + 1)
    return {"layout": layout, "dispatch": disp, "combine": comb, "combine_fp8": comb8,
            "dispatch_send": send, "dispatch_recv": recv,
            "combine_rank_partial": comb + 4 * T * K,
            "layout_dispatch": layout + disp - 4 * T * K}


# the sources each call's kernels are built from (their hash keys the DRAM
# traffic rows in profiles/dram_traffic.json)
CALL_SOURCES = {
    "layout": ["layout.cu", "layout_common.cuh", "layout_dispatch_prefill.cu"],
    "dispatch": ["dispatch.cu", "rowops.cuh"],
    "combine": ["combine.cu", "combine_common.cuh"],
    "combine_fp8": ["combine_fp8.cu", "combine_common.cuh"],
    "combine_rank_partial": ["combine_rank_partial.cu", "combine_common.cuh"],
    "layout_dispatch": ["layout_dispatch.cu", "layout_common.cuh", "rowops.cuh",
                        "layout.cu", "dispatch.cu", "layout_dispatch_prefill.cu"],
    "dispatch_send": ["regions.cu", "rowops.cuh"],
    "dispatch_recv": ["regions.cu"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def kernel_source_hash(kernel: str):
    srcs = CALL_SOURCES.get(kernel)
    if srcs is None:
        return None
    h = hashlib.sha256()
    for f in srcs + ["common.cuh"]:
        p = os.path.join(ROOT, "combine_moe_layout_05_gb300", "csrc", f)
        if os.path.exists(p):
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(kernel: str, workload: str, dispatch: str, path: str = TRAFFIC_FILE):
    """DRAM bytes per launch from the committed ncu capture of this call, if
    it was taken on the current source of that call; otherwise None."""
    try:
        with open(path) as f:
            rows = json.load(f)["rows"]
    except (OSError, ValueError, KeyError):
        return None
    want = kernel_source_hash(kernel)
    for r in rows:
        if (r.get("call"), r.get("workload"), r.get("dispatch"), r.get("source_hash")) == \
                (kernel, workload, dispatch, want):
            return int(r["dram_bytes_per_launch"])
    return None


def dtype_label(dispatch: str, combine: str) -> str:
    d = ("fp8-e4m3 dispatch (1x128 fp32 block scales)" if dispatch == "fp8"
         else "bf16 dispatch (bit copy)")
    c = {"bf16": "bf16 combine, fp32 accumulate",
         "fp8": "fp8-e4m3 combine input, fp32 accumulate",
         "rank_partial": "bf16 combine, fp32 per-rank partials rounded to bf16"}[combine]
    return f"{d}, {c}"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples, kept only for the span
    between mark_start() and mark_stop() (the timed region)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    KEYS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, local_index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
        ids = [v.strip() for v in vis.split(",") if v.strip()] if vis else []
        self.idx = ids[local_index] if local_index < len(ids) else str(local_index)
        self.proc, self.out, self.t0, self.t1 = None, None, None, None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", self.idx, "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    @staticmethod
    def parse(text, t0, t1):
        import datetime
        mhz, mx, reasons = [], [], set()
        for line in text.splitlines():
            r = [c.strip() for c in line.split(",")]
            if len(r) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax = float(r[1]), float(r[2])
            except ValueError:
                continue
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            mhz.append(sm)
            mx.append(smax)
            for k, v in zip(ClockSampler.KEYS, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(k)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(mhz)}

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        text = self.out.read()
        name = self.out.name
        self.out.close()
        os.unlink(name)
        return self.parse(text, self.t0, self.t1)


class Driver:
    """CUDA driver calls the benchmark needs and PyTorch does not expose in
    both supported versions: timing events recorded as graph nodes (external
    event records), pinned host buffers and asynchronous copies that can be
    captured into a graph."""

    def __init__(self):
        self.lib = ctypes.CDLL("libcuda.so.1")
        vp, u, sz = ctypes.c_void_p, ctypes.c_uint, ctypes.c_size_t
        L = self.lib
        L.cuEventCreate.argtypes = [ctypes.POINTER(vp), u]
        L.cuEventRecordWithFlags.argtypes = [vp, vp, u]
        L.cuEventDestroy_v2.argtypes = [vp]
        self.elapsed = getattr(L, "cuEventElapsedTime_v2", None) or L.cuEventElapsedTime
        self.elapsed.argtypes = [ctypes.POINTER(ctypes.c_float), vp, vp]
        L.cuMemHostAlloc.argtypes = [ctypes.POINTER(vp), sz, u]
        L.cuMemFreeHost.argtypes = [vp]
        L.cuMemcpyHtoDAsync_v2.argtypes = [ctypes.c_uint64, vp, sz, vp]
        L.cuMemcpyDtoHAsync_v2.argtypes = [vp, ctypes.c_uint64, sz, vp]
        self.events, self.host = [], []

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed (CUresult {rc})")

    def event(self):
        ev = ctypes.c_void_p()
        self._ok(self.lib.cuEventCreate(ctypes.byref(ev), 0), "cuEventCreate")
        self.events.append(ev)
        return ev

    def record(self, ev, stream_handle: int):
        self._ok(self.lib.cuEventRecordWithFlags(ev, ctypes.c_void_p(stream_handle), 1),
                 "cuEventRecordWithFlags")

    def ms(self, a, b) -> float:
        out = ctypes.c_float()
        self._ok(self.elapsed(ctypes.byref(out), a, b), "cuEventElapsedTime")
        return float(out.value)

    def pinned(self, nbytes: int):
        """Page-locked host buffer; returns (address, numpy uint8 view)."""
        import numpy as np
        p = ctypes.c_void_p()
        self._ok(self.lib.cuMemHostAlloc(ctypes.byref(p), max(nbytes, 1), 0), "cuMemHostAlloc")
        self.host.append(p)
        arr = np.ctypeslib.as_array((ctypes.c_uint8 * max(nbytes, 1)).from_address(p.value))
        return p.value, arr[:nbytes]

    def h2d(self, dst_dev: int, src_host: int, n: int, stream_handle: int):
        self._ok(self.lib.cuMemcpyHtoDAsync_v2(dst_dev, ctypes.c_void_p(src_host), n,
                                               ctypes.c_void_p(stream_handle)), "cuMemcpyHtoDAsync")

    def d2h(self, dst_host: int, src_dev: int, n: int, stream_handle: int):
        self._ok(self.lib.cuMemcpyDtoHAsync_v2(ctypes.c_void_p(dst_host), src_dev, n,
                                               ctypes.c_void_p(stream_handle)), "cuMemcpyDtoHAsync")

    def close(self):
        for ev in self.events:
            self.lib.cuEventDestroy_v2(ev)
        for p in self.host:
            self.lib.cuMemFreeHost(p)
        self.events, self.host = [], []


# ----------------------------------------------------------- our CUDA arm --

class BufferSet:
    """Inputs, layout buffers and outputs of one step, all on the device."""

    def __init__(self, w, dispatch, inp, y_host_bits, device, private_rows=None):
        import numpy as np
        import torch
        import combine_moe_layout_05_gb300 as moe
        T, H, K = w.T, w.H, w.K
        # the step's inputs sit in one contiguous buffer, so a host upload is
        # one copy: [tokens | ids | weights], each part 256-byte aligned
        self.input_layout = input_layout(w)
        self.inputs = torch.empty(self.input_layout["bytes"], dtype=torch.uint8, device=device)
        self.inputs.copy_(torch.from_numpy(pack_inputs(w, inp)))
        o = self.input_layout
        self.tokens = self.inputs[o["tokens"]:o["tokens"] + 2 * T * H].view(torch.bfloat16).view(T, H)
        self.ids = self.inputs[o["ids"]:o["ids"] + 4 * T * K].view(torch.int32).view(T, K)
        self.weights = self.inputs[o["weights"]:o["weights"] + 4 * T * K].view(torch.float32).view(T, K)
        self.layout = moe.LayoutBuffers(T, K, w.E, w.R, device=device)
        if dispatch == "bf16":
            self.packed = torch.empty((T * K, H), dtype=torch.bfloat16, device=device)
            self.scales = None
        else:
            self.packed = torch.empty((T * K, H), dtype=torch.float8_e4m3fn, device=device)
            self.scales = torch.empty((T * K, H // 128), dtype=torch.float32, device=device)
        self.y = None if y_host_bits is None else torch.from_numpy(
            y_host_bits.view(np.int16)).to(device).view(torch.bfloat16)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self.priv = self.bulk = self.priv_sc = self.bulk_sc = self.region_err = None
        if private_rows is not None:      # per-rank send regions, worst-case bulk
            P, C = private_rows, max(0, T * min(K, w.E // w.R) - private_rows)
            dt = self.packed.dtype
            self.priv = torch.zeros((w.R, P, H), dtype=dt, device=device)
            self.bulk = torch.zeros((w.R, C, H), dtype=dt, device=device)
            if dispatch == "fp8":
                self.priv_sc = torch.zeros((w.R, P, H // 128), device=device)
                self.bulk_sc = torch.zeros((w.R, C, H // 128), device=device)
            self.region_err = torch.zeros(1, dtype=torch.int32, device=device)

    def nbytes(self):
        """Bytes a step touches in this set (region buffers count only the
        rows a step fills: T*K rows, whatever their worst-case capacity)."""
        ts = [self.inputs, self.packed, self.out,
              self.layout.src_token, self.layout.dst_row]
        ts += [self.scales, self.y]
        touched = sum(t.numel() * t.element_size() for t in ts if t is not None)
        if self.priv is not None:     # the filled region rows equal the packed rows
            touched += self.packed.numel() * self.packed.element_size()
            if self.scales is not None:
                touched += self.scales.numel() * self.scales.element_size()
        return touched


def input_layout(w):
    """Byte offsets of tokens, ids and weights in one input buffer."""
    al = lambda x: (x + 255) // 256 * 256
    tok = 0
    ids = al(2 * w.T * w.H)
    wts = al(ids + 4 * w.T * w.K)
    return {"tokens": tok, "ids": ids, "weights": wts, "bytes": al(wts + 4 * w.T * w.K)}


def pack_inputs(w, inp):
    import numpy as np
    o = input_layout(w)
    buf = np.zeros(o["bytes"], np.uint8)
    for name, arr in (("tokens", inp.tokens), ("ids", inp.topk_ids), ("weights", inp.topk_weights)):
        b = np.ascontiguousarray(arr).view(np.uint8).ravel()
        buf[o[name]:o[name] + b.size] = b
    return buf


def expert_outputs(w, dispatch, inp, buf):
    """The stand-in experts' outputs for this batch (materialised once)."""
    import torch
    from combine_moe_layout_05_gb300 import experts as ex
    from combine_moe_layout_05_gb300 import workload as wl
    if w.experts == "random" or (dispatch == "fp8" and w.experts == "scale"):
        return wl.random_rows(w.T * w.K, w.H, inp.expert_rows_seed)
    if dispatch == "fp8":
        y = ex.dequant_rows(buf.packed, buf.scales)
    elif w.experts == "scale":
        y = ex.scale_rows(buf.packed, buf.layout.expert_offsets, torch.from_numpy(inp.expert_scale))
    else:
        y = buf.packed.clone()
    return y.view(torch.int16).cpu().numpy().view("uint16")


def variant_layout_dispatch(moe, variant, fp8):
    """moe_layout_dispatch in an alternative form, through the library's test
    hooks (not part of its public header); returns fn(buffer_set)."""
    lib = moe.load()
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    if variant in ("cluster", "decode_bulk"):
        f = lib.moe_testing_layout_dispatch_decode
        f.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, i32, P]
    else:
        f = lib.moe_testing_layout_pack
        f.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                      ctypes.c_uint64, i32, i32, P]
    f.restype = i32

    def run(b):
        import torch
        L = b.layout
        T, H = b.tokens.shape
        args = [b.ids.data_ptr(), b.tokens.data_ptr(), T, H, L.K, L.E, L.R, int(fp8),
                L.expert_counts.data_ptr(), L.expert_offsets.data_ptr(), L.rank_offsets.data_ptr(),
                L.src_token.data_ptr(), L.dst_row.data_ptr(), L.dev_error.data_ptr(),
                b.packed.data_ptr(), b.scales.data_ptr() if fp8 else None]
        s = torch.cuda.current_stream().cuda_stream
        if variant in ("cluster", "decode_bulk"):
            st = f(*args, 1 if variant == "cluster" else 2, s)
        else:
            st = f(*args, L.workspace.data_ptr(), 0, -1, int(variant == "persistent_bulk"), s)
        if st != 0:
            raise RuntimeError(f"{variant} layout+dispatch refused these sizes (status {st})")
    return run


def step_ops(moe, dispatch, unfused=False, combine="bf16", path="packed", variant="library"):
    """The calls of one step, as (name, fn(buffer_set)) in launch order."""
    fp8 = dispatch == "fp8"
    if path == "regions":
        ops = [("layout", lambda b: b.layout.run(b.ids)),
               ("dispatch_send", lambda b: moe.moe_dispatch_send(
                   b.tokens, b.ids, b.layout.dst_row, b.layout.rank_offsets, b.layout.E,
                   b.layout.R, b.priv, b.bulk, b.priv_sc, b.bulk_sc, fp8=fp8,
                   dev_error=b.region_err)),
               ("dispatch_recv", lambda b: moe.moe_dispatch_recv(
                   b.priv, b.bulk, b.layout.rank_offsets, b.layout.T, b.layout.K, b.packed,
                   b.priv_sc, b.bulk_sc, b.scales, fp8=fp8))]
    elif unfused:
        ops = [("layout", lambda b: b.layout.run(b.ids)),
               ("dispatch", lambda b: moe.moe_dispatch(b.tokens, b.layout.dst_row,
                                                       b.packed, b.scales, fp8=fp8))]
    elif variant not in ("library", "combine_shuffle"):
        ops = [("layout_dispatch", variant_layout_dispatch(moe, variant, fp8))]
    else:
        ops = [("layout_dispatch", lambda b: b.layout.run_dispatch(
            b.ids, b.tokens, b.packed, b.scales, fp8=fp8))]
    if combine == "fp8":
        ops.append(("combine_fp8", lambda b: moe.moe_combine_fp8(
            b.packed, b.scales, b.weights, b.layout.dst_row, b.out)))
    elif combine == "rank_partial":
        ops.append(("combine_rank_partial", lambda b: moe.moe_combine_rank_partial(
            b.y, b.weights, b.ids, b.layout.dst_row, b.layout.E, b.layout.R, b.out)))
    elif variant == "combine_shuffle":
        ops.append(("combine", variant_combine_shuffle(moe)))
    else:
        ops.append(("combine", lambda b: moe.moe_combine(b.y, b.weights, b.layout.dst_row, b.out)))
    return ops


def variant_combine_shuffle(moe):
    """moe_combine in the form kept behind the library's test hook (slots and
    weights loaded by 8 lanes and shuffled to the warp); returns fn(buffer_set)."""
    f = moe.load().moe_testing_combine_shfl
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, P, i32, i32, i32, P, P]
    f.restype = i32

    def run(b):
        import torch
        T, K = b.weights.shape
        st = f(b.y.data_ptr(), b.weights.data_ptr(), b.layout.dst_row.data_ptr(), T, b.out.shape[1],
               K, b.out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise RuntimeError(f"combine_shuffle refused these sizes (status {st})")
    return run


def run_step(moe, buf, dispatch, unfused=False, combine="bf16", path="packed", variant="library"):
    for _, fn in step_ops(moe, dispatch, unfused, combine, path, variant):
        fn(buf)


def capture(torch, steps_fn, n_steps):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        steps_fn(n_steps, s.cuda_stream)
    return g


def check_parity(w, dispatch, inp, buf, combine="bf16"):
    """The bench's own gate: one step of set 0 against the oracle."""
    import numpy as np
    import torch
    import oracle
    ref = oracle.layout(inp.topk_ids, w.E, w.R)
    ok = np.array_equal(buf.layout.dst_row.cpu().numpy(), ref.dst_row)
    ok &= np.array_equal(buf.layout.expert_offsets.cpu().numpy(), ref.expert_offsets)
    if dispatch == "bf16":
        exp = oracle.dispatch_bf16(inp.tokens, ref.dst_row)
        ok &= np.array_equal(buf.packed.view(torch.int16).cpu().numpy().view(np.uint16), exp)
    else:
        ec, es = oracle.dispatch_fp8(inp.tokens, ref.dst_row)
        ok &= np.array_equal(buf.packed.view(torch.uint8).cpu().numpy(), ec)
        ok &= np.array_equal(buf.scales.cpu().numpy().view(np.uint32), es.view(np.uint32))
    if combine == "fp8":
        exp_out = oracle.combine_fp8(ec, es, inp.topk_weights, ref.dst_row)
    elif combine == "rank_partial":
        y = buf.y.view(torch.int16).cpu().numpy().view(np.uint16)
        exp_out = oracle.combine_rank_partial(y, inp.topk_weights, inp.topk_ids, ref.dst_row,
                                              w.E, w.R)
    else:
        y = buf.y.view(torch.int16).cpu().numpy().view(np.uint16)
        exp_out = oracle.combine(y, inp.topk_weights, ref.dst_row)
    ok &= np.array_equal(buf.out.view(torch.int16).cpu().numpy().view(np.uint16), exp_out)
    return "bit-exact" if ok else "MISMATCH"


def time_oracle(w, dispatch, inp, y_bits, seconds: float, max_tokens=None, combine="bf16"):
    """Oracle steps (layout + dispatch + combine) on the host until `seconds`
    have passed; returns (tokens/s, tokens per step, steps)."""
    import oracle
    T = w.T if max_tokens is None else max(1, min(w.T, max_tokens))
    ids, x, wts = inp.topk_ids[:T], inp.tokens[:T], inp.topk_weights[:T]
    n, t0 = 0, time.perf_counter()
    while True:
        ref = oracle.layout(ids, w.E, w.R)
        if dispatch == "bf16":
            oracle.dispatch_bf16(x, ref.dst_row)
        else:
            codes, scales = oracle.dispatch_fp8(x, ref.dst_row)
        if combine == "fp8":
            oracle.combine_fp8(codes, scales, wts, ref.dst_row)
        elif combine == "rank_partial":
            oracle.combine_rank_partial(y_bits[: T * w.K], wts, inp.topk_ids[:T], ref.dst_row,
                                        w.E, w.R)
        else:
            oracle.combine(y_bits[: T * w.K], wts, ref.dst_row)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return T * n / el, T, n


class StepGraphs:
    """n_steps consecutive calls of fn(set j mod n_sets), captured into CUDA
    graphs of G steps plus one graph of the remainder; replay() enqueues all
    n_steps on the current stream."""

    def __init__(self, torch, body, n_steps, G):
        self.torch = torch
        self.g = capture(torch, body, G) if n_steps >= G else None
        self.reps = n_steps // G
        rem = n_steps % G
        self.gr = capture(torch, body, rem) if rem else None

    def replay(self):
        for _ in range(self.reps):
            self.g.replay()
        if self.gr is not None:
            self.gr.replay()


def timed_passes(torch, replay, min_seconds, min_passes=3, max_passes=100000):
    """Replays one pass (replay()) until at least min_seconds of device time
    are covered, with a CUDA event on the current stream between passes.
    Returns the list of pass times in ms.  The caller synchronises and
    brackets the call with barriers."""
    s = torch.cuda.current_stream()
    probe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    probe[0].record(s)
    replay()
    probe[1].record(s)
    probe[1].synchronize()
    first = max(probe[0].elapsed_time(probe[1]), 1e-3)
    n = int(min(max_passes, max(min_passes, math.ceil(1e3 * min_seconds / first))))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    ev[0].record(s)
    for i in range(n):
        replay()
        ev[i + 1].record(s)
    ev[n].synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]


def measure_ours(args, w, dispatch, combine, rank, world, local, device, first_line=True):
    """One bench line for workload w (dict), measured on this rank."""
    import numpy as np
    import torch
    import combine_moe_layout_05_gb300 as moe

    inp = wl_inputs(w, rank)
    if combine == "fp8" and dispatch != "fp8":
        raise SystemExit("--combine fp8 needs FP8 dispatch (--dispatch fp8)")
    ops = step_ops(moe, dispatch, args.unfused, combine, args.path, args.variant)
    priv_rows = args.private if args.path == "regions" else None

    # rotating buffer sets: total >= 3x L2, so every step starts cold in L2
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    first = BufferSet(w, dispatch, inp, None, device, priv_rows)
    for _, fn in ops[:-1]:
        fn(first)
    torch.cuda.synchronize()
    y_bits = expert_outputs(w, dispatch, inp, first) if combine != "fp8" else None
    per_set = first.nbytes() + (0 if y_bits is None else y_bits.nbytes)
    n_sets = max(2, math.ceil(3 * l2 / per_set))
    del first
    sets = [BufferSet(w, dispatch, inp, y_bits, device, priv_rows) for _ in range(n_sets)]
    for b in sets:                       # eager pass: attributes, parity data
        run_step(moe, b, dispatch, args.unfused, combine, args.path, args.variant)
    torch.cuda.synchronize()

    K = args.steps
    G = max(n_sets, (min(args.graph_steps, max(K, 1)) // n_sets) * n_sets)
    step = lambda b: run_step(moe, b, dispatch, args.unfused, combine, args.path, args.variant)
    graphs = StepGraphs(torch, lambda m, sh: [step(sets[j % n_sets]) for j in range(m)], K, G)
    for _ in range(max(1, math.ceil(args.warmup / max(K, 1)))):
        graphs.replay()
    torch.cuda.synchronize()
    parity = None
    if rank == 0 and not args.no_parity:
        parity = check_parity(w, dispatch, inp, sets[(K - 1) % n_sets if K else 0], combine)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(device)
    torch.cuda.synchronize()
    sampler.mark_start()
    passes = timed_passes(torch, graphs.replay, args.min_seconds)
    torch.cuda.synchronize()
    sampler.mark_stop()
    barrier(device)
    time.sleep(0.15)
    clocks = sampler.stop()
    pass_ms = max_over_ranks(statistics.median(passes), device)
    del graphs

    # each call of the step alone: K launches over the same rotating sets
    ab = algorithmic_bytes(w, dispatch)
    peak, peak_src = read_peaks()
    kernels = {}
    for name, fn in ops:
        cg = StepGraphs(torch, lambda m, sh, fn=fn: [fn(sets[j % n_sets]) for j in range(m)], K, G)
        cg.replay()
        torch.cuda.synchronize()
        cp = timed_passes(torch, cg.replay, args.call_seconds)
        us = 1e3 * max_over_ranks(statistics.median(cp), device) / K
        kernels[name] = {"us": round(us, 3), "gbs": round(ab[name] / (us * 1e-6) / 1e9, 1),
                         "bytes": ab[name], "passes": len(cp)}
        del cg
    dom = max(kernels, key=lambda k: kernels[k]["us"])
    achieved = kernels[dom]["gbs"]

    e2e = None
    if not args.no_e2e:
        drv = Driver()
        try:
            e2e = run_e2e(args, w, dispatch, combine, inp, sets, n_sets, G, device, torch, moe, drv)
        finally:
            drv.close()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        tps, tsamp, nst = time_oracle(w, dispatch, inp, y_bits, args.cpu_seconds, combine=combine)
        cpu = {"value": round(tps, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
               **host_info(),
               "sample": f"{nst} oracle steps (layout + {dispatch} dispatch + {combine} combine) "
                         f"of the full {w.name} batch (T={tsamp}), single thread, "
                         f"{args.cpu_seconds:.0f} s budget"}

    value = world * w.T * K / (pass_ms * 1e-3)
    lps = launches_per_step(w, dispatch, args.unfused, args.path, args.variant)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(pass_ms / K, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(dispatch, combine),
        "data": "synthetic",
        "timing": {"passes": len(passes), "steps_per_pass": K,
                   "pass_ms_median": round(statistics.median(passes), 4),
                   "pass_ms_min": round(min(passes), 4), "pass_ms_max": round(max(passes), 4),
                   "device_seconds": round(sum(passes) / 1e3, 3),
                   "method": "K-step pass replayed until >= %.1f s of device time; CUDA "
                             "events on the launching stream between passes; median pass "
                             "(max over ranks) / K" % args.min_seconds},
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "R": w.R,
                   "K": w.K, "dispatch": dispatch,
                   "combine": {"fp8": "e4m3 + block scales in (identity experts), f32 accumulate",
                               "rank_partial": "bf16 in, per-rank f32 partials rounded to bf16, "
                                               "f32 sum over ranks",
                               "bf16": "bf16 in, f32 accumulate"}[combine],
                   "experts": w.experts, "routing": w.routing,
                   "calls": [n for n, _ in ops], "path": args.path, "variant": args.variant,
                   "l2": f"{n_sets} rotating buffer sets, {n_sets * per_set / 1e6:.0f} MB "
                         f"> 3x L2 ({l2 / 1e6:.0f} MB); every step cold in L2",
                   "launch": f"CUDA graphs of {G} steps, programmatic dependent launch",
                   "kernel_timing": "each call alone: K launches in CUDA graphs over the "
                                    "same rotating sets, passes repeated, median pass",
                   "parallelism": f"replicas x{world}"},
        "kernels": kernels,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": peak_src,
                     "traffic": (profiled_traffic(dom, w.name, dispatch)
                                 if args.variant == "library" else None)},
        "e2e": e2e, "gpu_launches": lps * K * len(passes), "launches_per_step": lps,
        "clocks": clocks, "cpu_baseline": cpu, "parity": parity,
    }
    del sets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def wl_inputs(w, rank):
    from combine_moe_layout_05_gb300 import workload as wl
    return wl.make_inputs(w, seed=shard_seed(w.seed, rank))


def run_ours(args):
    import torch
    import combine_moe_layout_05_gb300 as moe
    from combine_moe_layout_05_gb300 import build as moe_build
    from combine_moe_layout_05_gb300 import workload as wl

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0:
        moe_build.build()
    barrier(device)
    moe_build.build()
    moe.load()

    if args.all:
        variants = list(ALL_VARIANTS)
    else:
        name = args.workload or wl.HEADLINE
        w = wl.get(name)
        variants = [(name, args.dispatch or w.dispatch[0])]
    for name, dispatch in variants:
        line = measure_ours(args, wl.get(name), dispatch, args.combine, rank, world, local, device)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def launches_per_step(w, dispatch, unfused, path="packed", variant="library") -> int:
    """Kernels this library launches per step (mirrors the C ABI's plans)."""
    import combine_moe_layout_05_gb300 as moe
    if variant in ("cluster", "decode_bulk"):
        return 2
    if variant.startswith("persistent"):
        return 3
    layout_kernels = moe.moe_layout_kernels(w.T, w.K, w.E)
    if path == "regions":
        return layout_kernels + 3
    if unfused:
        return layout_kernels + 2
    return moe.moe_layout_dispatch_kernels(w.T, w.H, w.K, w.E, dispatch == "fp8") + 1


def run_e2e(args, w, dispatch, combine, inp, sets, n_sets, G, device, torch, moe, drv):
    """The same steps through host buffers, as a serving loop runs them: each
    step copies its tokens, ids and weights (one contiguous buffer) from
    page-locked host memory, runs the calls, and copies its output back to
    page-locked host memory, all inside the timed region.  Copies and compute
    sit on three streams (host-to-device, compute, device-to-host) so step
    j+1's upload and step j-1's download overlap step j's kernels; events
    order each buffer set's reuse (an upload waits for the compute that last
    read the set, a compute waits for the download that last read its
    output).  Passes of K steps are repeated like the device-resident run."""
    import numpy as np
    packed_in = pack_inputs(w, inp)
    h2d = packed_in.nbytes
    d2h = w.T * w.H * 2
    host = []
    for _ in range(n_sets):
        addr, view = drv.pinned(h2d)
        view[:] = packed_in
        host.append({"inputs": addr, "out": drv.pinned(d2h)[0]})
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def body(n, sh):
        comp = torch.cuda.current_stream()
        up.wait_stream(comp)                  # fork the side streams into the capture
        down.wait_stream(comp)
        comp_done, down_done = {}, {}
        for j in range(n):
            b, h = sets[j % n_sets], host[j % n_sets]
            with torch.cuda.stream(up):
                if j - n_sets in comp_done:   # the set's previous compute has read it
                    up.wait_event(comp_done[j - n_sets])
                drv.h2d(b.inputs.data_ptr(), h["inputs"], h2d, up.cuda_stream)
                up_done = torch.cuda.Event()
                up_done.record(up)
            comp.wait_event(up_done)
            if j - n_sets in down_done:       # the set's previous output was read
                comp.wait_event(down_done[j - n_sets])
            run_step(moe, b, dispatch, args.unfused, combine, args.path, args.variant)
            comp_done[j] = torch.cuda.Event()
            comp_done[j].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[j])
                drv.d2h(h["out"], b.out.data_ptr(), d2h, down.cuda_stream)
                down_done[j] = torch.cuda.Event()
                down_done[j].record(down)
        comp.wait_stream(up)                  # join
        comp.wait_stream(down)

    K = args.steps
    torch.cuda.synchronize()
    graphs = StepGraphs(torch, body, K, G)
    graphs.replay()
    torch.cuda.synchronize()
    barrier(device)
    torch.cuda.synchronize()
    passes = timed_passes(torch, graphs.replay, args.min_seconds / 2)
    torch.cuda.synchronize()
    barrier(device)
    ms = max_over_ranks(statistics.median(passes), device)
    _, world, _ = dist_env()
    # the copies brought back the same result the device-resident steps made
    out0 = np.ctypeslib.as_array((ctypes.c_uint8 * d2h).from_address(host[0]["out"]))
    same = np.array_equal(out0, sets[0].out.view(torch.uint8).cpu().numpy().ravel())
    del graphs
    return {"value": round(world * w.T * K / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / K, 6), "passes": len(passes),
            "output_matches_device_run": bool(same),
            "pipeline": "H2D, compute and D2H on three streams, overlapping across steps"}


# ------------------------------------------------------- reference (oracle) --

def host_expert_outputs(w, dispatch, inp, dst_row, expert_offsets):
    """The stand-in experts' outputs computed on the host (reference arm)."""
    import numpy as np
    import torch
    import oracle
    from combine_moe_layout_05_gb300 import experts as ex
    from combine_moe_layout_05_gb300 import workload as wl
    if w.experts == "random" or (dispatch == "fp8" and w.experts == "scale"):
        return wl.random_rows(w.T * w.K, w.H, inp.expert_rows_seed)
    if dispatch == "fp8":
        codes, scales = oracle.dispatch_fp8(inp.tokens, dst_row)
        y = ex.dequant_rows(torch.from_numpy(codes).view(torch.float8_e4m3fn),
                            torch.from_numpy(scales))
    else:
        packed = torch.from_numpy(oracle.dispatch_bf16(inp.tokens, dst_row).view(np.int16))
        packed = packed.view(torch.bfloat16)
        if w.experts == "scale":
            y = ex.scale_rows(packed, torch.from_numpy(expert_offsets),
                              torch.from_numpy(inp.expert_scale))
        else:
            y = packed
    return y.view(torch.int16).numpy().view(np.uint16)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from combine_moe_layout_05_gb300 import workload as wl
    oracle.build()
    w = wl.get(args.workload or wl.HEADLINE)
    dispatch = args.dispatch or w.dispatch[0]
    inp = wl.make_inputs(w)
    ref = oracle.layout(inp.topk_ids, w.E, w.R)
    y_bits = None if args.combine == "fp8" else host_expert_outputs(
        w, dispatch, inp, ref.dst_row, ref.expert_offsets)
    # size each step so the whole run stays within about 90 s of host time
    t0 = time.perf_counter()
    time_oracle(w, dispatch, inp, y_bits, 0.0, combine=args.combine)
    full = time.perf_counter() - t0
    budget = 90.0 / max(1, args.steps + args.warmup)
    T_s = max(1, min(w.T, int(w.T * budget / max(full, 1e-9))))
    for _ in range(args.warmup):
        time_oracle(w, dispatch, inp, y_bits, 0.0, max_tokens=T_s, combine=args.combine)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(w, dispatch, inp, y_bits, 0.0, max_tokens=T_s, combine=args.combine)
    el = time.perf_counter() - t0
    value = T_s * args.steps / el
    sample = (f"each step: oracle layout + {dispatch} dispatch + {args.combine} combine on "
              f"the first {T_s} of the {w.T} tokens of {w.name}, single thread")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(dispatch, args.combine),
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "R": w.R, "K": w.K,
                   "dispatch": dispatch, "sample_tokens_per_step": T_s},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": 1,
                         "kind": "oracle", "sample": sample, **host_info()},
        "e2e": {"value": round(value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
