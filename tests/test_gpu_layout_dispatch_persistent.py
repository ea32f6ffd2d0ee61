"""GPU parity of the persistent form of the large-batch layout + dispatch (one
CTA per SM, token rows staged in a shared-memory ring by bulk copies; kept
for comparison and reachable only through a test hook) against the oracle,
bit for bit, in its 16-byte-store and bulk-store forms, and its bounded
waits: a CTA made to wait on a barrier that nothing signals reports
MOE_DEV_ERR_TIMEOUT and finishes."""
import ctypes
import time

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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _hook():
    f = moe.load().moe_testing_layout_pack
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                  ctypes.c_uint64, i32, i32, P]
    f.restype = i32
    return f


def _inputs(T, H, K, E, seed):
    rng = np.random.default_rng(seed)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)
                        * np.exp2(rng.integers(-6, 6, (T, 1))).astype(np.float32))
    return x, wl.routing_zipf(T, E, K, 1.1, rng)


def _run(T, H, K, E, R, fp8, x, ids, bulk=0, stall_cta=-1, wait_ns=0):
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
    st = _hook()(ids_d.data_ptr(), x_d.data_ptr(), T, H, K, E, R, fp8,
                 buf.expert_counts.data_ptr(), buf.expert_offsets.data_ptr(),
                 buf.rank_offsets.data_ptr(), buf.src_token.data_ptr(), buf.dst_row.data_ptr(),
                 buf.dev_error.data_ptr(), packed.data_ptr(), scales.data_ptr() if fp8 else None,
                 buf.workspace.data_ptr(), wait_ns, stall_cta, bulk,
                 torch.cuda.current_stream().cuda_stream)
    assert st == 0, st
    torch.cuda.synchronize()
    return buf, packed, scales


def _check(oracle, buf, ref, x, packed, scales, E, fp8, rows=None, err=None):
    assert int(buf.dev_error.item()) == (ref.error if err is None else err)
    assert np.array_equal(buf.expert_counts.cpu().numpy(), ref.expert_counts)
    assert np.array_equal(buf.expert_offsets.cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(buf.rank_offsets.cpu().numpy(), ref.rank_offsets)
    assert np.array_equal(buf.dst_row.cpu().numpy(), ref.dst_row)
    n = int(ref.expert_offsets[E])
    assert np.array_equal(buf.src_token.cpu().numpy()[:n], ref.src_token[:n])
    sel = slice(0, n) if rows is None else rows
    if fp8:
        ec, es = oracle.dispatch_fp8(x, ref.dst_row)
        assert np.array_equal(packed.view(torch.uint8).cpu().numpy()[sel], ec[sel])
        assert np.array_equal(scales.cpu().numpy().view(np.uint32)[sel], es.view(np.uint32)[sel])
    else:
        assert np.array_equal(bf16_host(packed)[sel], oracle.dispatch_bf16(x, ref.dst_row)[sel])


SHAPES = [  # T, H, K, E, R, fp8, bulk
    (4096, 7168, 8, 384, 48, 0, 0),   # Kimi-K2 prefill shape
    (4096, 7168, 8, 384, 48, 0, 1),
    (4096, 7168, 8, 384, 48, 1, 0),
    (16384, 4096, 8, 128, 16, 1, 0),  # Qwen3 prefill shape
    (3001, 136, 5, 40, 8, 0, 1),      # runtime K, rows not a multiple of 128 bytes
    (9001, 8, 1, 16, 4, 0, 0),        # K = 1, 16-byte rows
    (300, 128, 32, 64, 4, 1, 0),      # K = 32
    (50000, 64, 8, 128, 16, 0, 1),    # several ranking pieces per CTA
    (40000, 128, 6, 96, 12, 1, 0),
]


@pytest.mark.parametrize("T,H,K,E,R,fp8,bulk", SHAPES)
def test_persistent_form_matches_oracle(oracle, T, H, K, E, R, fp8, bulk):
    x, ids = _inputs(T, H, K, E, seed=T + 31 * K + E)
    ids[1, 0] = -1
    ref = oracle.layout(ids, E, R)
    buf, packed, scales = _run(T, H, K, E, R, fp8, x, ids, bulk=bulk)
    _check(oracle, buf, ref, x, packed, scales, E, fp8)


def test_persistent_shapes_cover_ragged_ranges_and_pieces():
    sms = _sms()
    assert any(T % sms for T, *_ in SHAPES)
    assert any(T * K // sms > 2048 for T, H, K, *_ in SHAPES)


@pytest.mark.parametrize("fp8,bulk", [(0, 0), (0, 1), (1, 0)])
def test_persistent_bounded_wait(oracle, fp8, bulk):
    """CTA 3 waits for its first row on a barrier that nothing signals, with a
    2 ms bound: the call completes, the error word is exactly the timeout bit,
    the layout is complete and every row owned by another CTA is packed."""
    T, H, K, E, R = 4000, 256, 8, 64, 8
    x, ids = _inputs(T, H, K, E, seed=11)
    ref = oracle.layout(ids, E, R)
    t0 = time.time()
    buf, packed, scales = _run(T, H, K, E, R, fp8, x, ids, bulk=bulk, stall_cta=3,
                               wait_ns=2_000_000)
    assert time.time() - t0 < 30
    sms = _sms()
    per, extra = T // sms, T % sms
    a = 3 * per + min(3, extra)
    b = a + per + (1 if 3 < extra else 0)
    others = np.unique(np.concatenate([ref.dst_row[:a].ravel(), ref.dst_row[b:].ravel()]))
    _check(oracle, buf, ref, x, packed, scales, E, fp8, rows=others,
           err=moe.MOE_DEV_ERR_TIMEOUT)
