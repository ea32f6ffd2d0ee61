"""moe_layout_static: the layout entry point that allocates nothing.

Callers such as a plugin inside an inference engine that owns all device
memory, or a serving loop that must not enter the device allocator while it
runs, cannot allocate the workspace that large batches need; this entry
point keeps that scratch in a fixed array inside the library.  The GPU test calls it through the C ABI
twice in a row (the second call reuses the array the first one left behind)
and checks every output against moe_layout with a caller-allocated
workspace.  This file is collected last on purpose, so a run that stops at the
first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import build as moe_build
from combine_moe_layout_05_gb300 import workload as wl

P, i32 = ctypes.c_void_p, ctypes.c_int32
SCRATCH_BYTES = 96 << 10
MOE_OK, MOE_ERR_WORKSPACE = 0, 4


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    handle = moe.load()
    handle.moe_layout_static.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P]
    handle.moe_layout_static.restype = ctypes.c_int
    return handle


def test_rejects_batches_beyond_the_scratch(lib):
    # host-side check, nothing is launched: one expert, 40 M entries
    T, K, E = 40_000_000, 1, 1
    assert moe.moe_layout_workspace_bytes(T, K, E) > SCRATCH_BYTES
    st = lib.moe_layout_static(P(0x10000), T, K, E, 1, P(0x10000), P(0x10000),
                               P(0x10000), P(0x10000), P(0x10000), None, None)
    assert st == MOE_ERR_WORKSPACE


def _outputs(T, K, E, R):
    i = dict(dtype=torch.int32, device="cuda")
    return [torch.full((E,), -7, **i), torch.full((E + 1,), -7, **i),
            torch.full((R + 1,), -7, **i), torch.full((max(T * K, 1),), -7, **i),
            torch.full((T, K), -7, **i), torch.full((1,), -7, **i)]


def _static(lib, ids, E, R):
    T, K = ids.shape
    outs = _outputs(T, K, E, R)
    st = lib.moe_layout_static(P(ids.data_ptr()), T, K, E, R,
                               *[P(t.data_ptr()) for t in outs],
                               P(torch.cuda.current_stream().cuda_stream))
    assert st == MOE_OK, moe.moe_status_string(st)
    return outs


def _with_workspace(ids, E, R):
    T, K = ids.shape
    outs = _outputs(T, K, E, R)
    ws = moe.moe_layout_workspace_bytes(T, K, E)
    work = torch.empty(max(ws, 1), dtype=torch.uint8, device="cuda")
    moe.moe_layout(ids, E, R, *outs[:5], dev_error=outs[5], workspace=work if ws else None)
    return outs


@pytest.mark.gpu
def test_static_scratch_matches_workspace_layout_twice(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # large batches: the multi-launch layout on the scratch array, one call
    # after another, each reusing what the previous one left there
    rng = np.random.default_rng(5)
    big = [(32768, 8, 128, 16), (20000, 8, 384, 48)]
    for T, K, E, R in big:
        assert 0 < moe.moe_layout_workspace_bytes(T, K, E) <= SCRATCH_BYTES
        ids = torch.from_numpy(wl.routing_uniform(T, E, K, rng)).cuda()
        got = _static(lib, ids, E, R)
        exp = _with_workspace(ids, E, R)
        torch.cuda.synchronize()
        for g, e in zip(got, exp):       # integer outputs: exact
            assert torch.equal(g, e)
    # the prefill workloads
    for w in (wl.get("prefill_kimi_k2"), wl.get("prefill_qwen3")):
        assert 0 < moe.moe_layout_workspace_bytes(w.T, w.K, w.E) <= SCRATCH_BYTES
        ids = torch.from_numpy(wl.make_inputs(w).topk_ids).cuda()
        got = _static(lib, ids, w.E, w.R)
        exp = _with_workspace(ids, w.E, w.R)
        torch.cuda.synchronize()
        for g, e in zip(got, exp):
            assert torch.equal(g, e)
    # a batch small enough to need no scratch goes through the same call
    w = wl.get("decode_dsv3")
    ids = torch.from_numpy(wl.make_inputs(w).topk_ids).cuda()
    got, exp = _static(lib, ids, w.E, w.R), _with_workspace(ids, w.E, w.R)
    torch.cuda.synchronize()
    for g, e in zip(got, exp):
        assert torch.equal(g, e)
