"""GPU parity of the decode forms of moe_layout_dispatch against the oracle,
bit for bit: the single-kernel form the library uses (every block counts all
ids itself), through the public call and through a test hook, and the
cluster form (the blocks of one token's row split the id count and add their
partial sums through distributed shared memory) and the single-kernel form
writing its rows by bulk copies out of shared memory, which measured slower
and are reachable only through the hook."""
import ctypes

import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import workload as wl

from gpu_util import bf16_dev, bf16_host, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_layout_05_gb300 import build
    build.build()
    moe.load()


def _hook():
    f = moe.load().moe_testing_layout_dispatch_decode
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, i32, P]
    f.restype = i32
    return f


def _run(T, H, K, E, R, fp8, x, ids, variant):
    buf = moe.LayoutBuffers(T, K, E, R)
    for t in (buf.expert_counts, buf.expert_offsets, buf.rank_offsets, buf.src_token,
              buf.dst_row, buf.dev_error):
        t.fill_(-7)
    if fp8:
        packed = torch.empty((T * K, H), dtype=torch.float8_e4m3fn, device="cuda")
        packed.view(torch.uint8).fill_(0x7F)
        scales = torch.full((T * K, H // 128), float("nan"), device="cuda")
    else:
        packed = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
        packed.view(torch.int16).fill_(-1)
        scales = None
    ids_d, x_d = i32_dev(ids), bf16_dev(x)
    if variant is None:
        buf.run_dispatch(ids_d, x_d, packed, scales, fp8=bool(fp8))
    else:
        st = _hook()(ids_d.data_ptr(), x_d.data_ptr(), T, H, K, E, R, fp8,
                     buf.expert_counts.data_ptr(), buf.expert_offsets.data_ptr(),
                     buf.rank_offsets.data_ptr(), buf.src_token.data_ptr(), buf.dst_row.data_ptr(),
                     buf.dev_error.data_ptr(), packed.data_ptr(),
                     scales.data_ptr() if fp8 else None, variant,
                     torch.cuda.current_stream().cuda_stream)
        assert st == 0, st
    torch.cuda.synchronize()
    return buf, packed, scales


def _check(oracle, buf, packed, scales, ref, x, E, fp8):
    assert int(buf.dev_error.item()) == ref.error
    assert np.array_equal(buf.expert_counts.cpu().numpy(), ref.expert_counts)
    assert np.array_equal(buf.expert_offsets.cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(buf.rank_offsets.cpu().numpy(), ref.rank_offsets)
    assert np.array_equal(buf.dst_row.cpu().numpy(), ref.dst_row)
    n = int(ref.expert_offsets[E])
    assert np.array_equal(buf.src_token.cpu().numpy()[:n], ref.src_token[:n])
    if fp8:
        ec, es = oracle.dispatch_fp8(x, ref.dst_row)
        assert np.array_equal(packed.view(torch.uint8).cpu().numpy()[:n], ec[:n])
        assert np.array_equal(scales.cpu().numpy().view(np.uint32)[:n], es.view(np.uint32)[:n])
    else:
        assert np.array_equal(bf16_host(packed)[:n], oracle.dispatch_bf16(x, ref.dst_row)[:n])


DECODE_SHAPES = [  # T, H, K, E, R, fp8: clusters of 7 x 128, 7 x 64, 2 .. 8 blocks
    (128, 7168, 8, 256, 32, 0),    # DeepSeek-V3 decode
    (256, 7168, 8, 256, 32, 1),    # FP8 decode
    (128, 7168, 8, 256, 32, 1),
    (100, 1024, 6, 64, 8, 0),
    (37, 4096, 8, 128, 16, 1),
    (64, 1024, 3, 16, 4, 0),       # runtime K
    (10, 2048, 1, 8, 2, 1),        # K = 1
    (1, 7168, 2, 3, 1, 0),         # one token, E + 1 = 4 T
    (200, 8192, 7, 384, 48, 0),    # 8 blocks per cluster
]


@pytest.mark.parametrize("variant", [None, 1, 0, 2])
@pytest.mark.parametrize("T,H,K,E,R,fp8", DECODE_SHAPES)
def test_decode_forms_match_oracle(oracle, T, H, K, E, R, fp8, variant):
    if variant == 2 and K != 8:
        pytest.skip("the bulk-store form takes K = 8 only")
    rng = np.random.default_rng(T * 13 + H + K)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)
                        * np.exp2(rng.integers(-8, 8, (T, 1))).astype(np.float32))
    ids = wl.routing_uniform(T, E, K, rng)
    ref = oracle.layout(ids, E, R)
    buf, packed, scales = _run(T, H, K, E, R, fp8, x, ids, variant)
    _check(oracle, buf, packed, scales, ref, x, E, fp8)


@pytest.mark.parametrize("fp8", [0, 1])
def test_cluster_form_bad_ids(oracle, fp8):
    T, H, K, E, R = 50, 2048, 4, 16, 4
    rng = np.random.default_rng(7)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids = wl.routing_uniform(T, E, K, rng)
    ids[0, 0] = E + 3
    ids[9, 3] = ids[9, 1]
    ids[T - 1, K - 1] = -1
    ids[T // 2, 0] = E
    ref = oracle.layout(ids, E, R)
    assert ref.error == 3
    buf, packed, scales = _run(T, H, K, E, R, fp8, x, ids, 1)
    _check(oracle, buf, packed, scales, ref, x, E, fp8)


def test_more_experts_than_four_per_token(oracle):
    """E + 1 > 4 T, a shape the cluster form does not cover."""
    T, H, K, E, R = 120, 7168, 8, 480, 16
    rng = np.random.default_rng(3)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids = wl.routing_uniform(T, E, K, rng)
    ref = oracle.layout(ids, E, R)
    buf, packed, scales = _run(T, H, K, E, R, 0, x, ids, None)
    _check(oracle, buf, packed, scales, ref, x, E, 0)
