"""GPU parity of moe_dispatch_send / moe_dispatch_recv (per-rank send regions
with a private area) against the oracle's dispatch_send / dispatch_recv, bit
for bit: region contents, overflow flag, and send + recv == dispatch."""
import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import workload as wl

from gpu_util import bf16_dev, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_layout_05_gb300 import build
    build.build()
    moe.load()


def _u8(t):
    return t.view(torch.uint8).cpu().numpy()


def run_regions(oracle, inp, E, R, P, C, fp8):
    T, K = inp.topk_ids.shape
    H = inp.tokens.shape[1]
    ref = oracle.layout(inp.topk_ids, E, R)
    dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    priv = torch.zeros((R, P, H), dtype=dt, device="cuda")
    bulk = torch.zeros((R, C, H), dtype=dt, device="cuda")
    nb = H // 128
    ps = torch.zeros((R, P, nb), device="cuda") if fp8 else None
    bs = torch.zeros((R, C, nb), device="cuda") if fp8 else None
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ids_d, dst_d, ro_d = i32_dev(inp.topk_ids), i32_dev(ref.dst_row), i32_dev(ref.rank_offsets)
    moe.moe_dispatch_send(bf16_dev(inp.tokens), ids_d, dst_d, ro_d, E, R, priv, bulk, ps, bs,
                          fp8=fp8, dev_error=err)
    packed = torch.zeros((T * K, H), dtype=dt, device="cuda")
    sc = torch.zeros((T * K, nb), device="cuda") if fp8 else None
    moe.moe_dispatch_recv(priv, bulk, ro_d, T, K, packed, ps, bs, sc, fp8=fp8)
    torch.cuda.synchronize()
    if fp8:
        exp_rows, exp_sc = oracle.dispatch_fp8(inp.tokens, ref.dst_row)
    else:
        exp_rows, exp_sc = oracle.dispatch_bf16(inp.tokens, ref.dst_row), None
    epriv, eps, ebulk, ebs, eerr = oracle.dispatch_send(exp_rows, exp_sc, ref.rank_offsets, P, C)
    assert int(err.item()) == eerr
    assert np.array_equal(_u8(priv).reshape(epriv.shape), epriv)
    assert np.array_equal(_u8(bulk).reshape(ebulk.shape), ebulk)
    if fp8:
        assert np.array_equal(ps.cpu().numpy().view(np.uint32), eps.view(np.uint32))
        assert np.array_equal(bs.cpu().numpy().view(np.uint32), ebs.view(np.uint32))
    back, back_sc = oracle.dispatch_recv(epriv, eps, ebulk, ebs, ref.rank_offsets, T * K)
    assert np.array_equal(_u8(packed).reshape(back.shape), back)
    if fp8:
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), back_sc.view(np.uint32))
    return eerr


@pytest.mark.parametrize("name,fp8", [("decode_dsv3", False), ("decode_dsv3_fp8", True),
                                      ("prefill_kimi_k2", False), ("prefill_kimi_k2", True)])
@pytest.mark.parametrize("P", [0, 4])
def test_regions_full_size(oracle, name, fp8, P):
    w = wl.get(name)
    inp = wl.make_inputs(w)
    # bulk areas sized to the fullest rank exactly (the worst case
    # T * min(K, E/R) rows per region would also fit, at far more memory)
    ref = oracle.layout(inp.topk_ids, w.E, w.R)
    C = max(0, int(np.diff(ref.rank_offsets).max()) - P)
    assert C <= w.T * min(w.K, w.E // w.R)
    assert run_regions(oracle, inp, w.E, w.R, P, C, fp8) == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_regions_overflow_and_all_private(oracle, fp8):
    w = wl.get("tiny")
    inp = wl.make_inputs(w)
    assert run_regions(oracle, inp, w.E, w.R, 2, 5, fp8) == 4       # bulk too small
    assert run_regions(oracle, inp, w.E, w.R, 1000, 0, fp8) == 0    # everything private


@pytest.mark.parametrize("T,H,K,E,R,P,fp8", [
    (9, 8, 2, 4, 1, 0, False),          # one 16-byte vector per row, one region
    (17, 24, 5, 10, 5, 0, False),       # 3 vectors per row
    (37, 1032, 3, 12, 4, 2, False),     # 129 vectors: a partial last group of 4 per thread
    (50, 384, 8, 64, 64, 1, True),      # R = E, FP8
    (300, 7168, 8, 256, 32, 3, True),
])
def test_regions_shapes(oracle, T, H, K, E, R, P, fp8):
    import types
    rng = np.random.default_rng(T + H)
    ids = wl.routing_uniform(T, E, K, rng)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    inp = types.SimpleNamespace(topk_ids=ids, tokens=x)
    ref = oracle.layout(ids, E, R)
    C = max(0, int(np.diff(ref.rank_offsets).max()) - P)
    assert run_regions(oracle, inp, E, R, P, C, fp8) == 0
