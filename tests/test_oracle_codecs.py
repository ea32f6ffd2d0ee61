"""Pins for the oracle's bf16 and e4m3 codecs.

The codecs are checked against PyTorch's own conversions (an independent
library implementation of the same formats) exhaustively where the domain is
small, on constructed round-to-nearest-even ties, and against hand-derived
codes from the format definitions (tests/golden/e4m3_hand.txt).
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x_f32, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_e4m3_satfinite(x_f32: np.ndarray) -> np.ndarray:
    # satfinite: clamp to the largest finite magnitude, then round to nearest
    # even (PyTorch's conversion maps values >= 480 to NaN instead).
    t = torch.from_numpy(np.ascontiguousarray(x_f32, np.float32))
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_bf16_decode_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_encode_random_and_ties(oracle):
    rng = np.random.default_rng(123)
    rand = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    hi = np.arange(65536, dtype=np.uint32) << 16
    ties = hi | 0x8000                         # exact midpoints between neighbours
    near = np.concatenate([ties - 1, ties + 1, hi, hi | 0x7FFF, hi | 0x8001])
    specials = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000,
                         0x7F7FFFFF, 0x7F7F8000, 0x00000001, 0x807FFFFF],
                        np.uint32)
    allbits = np.concatenate([rand, ties, near, specials]).view(np.float32)
    finite = allbits[~np.isnan(allbits)]
    got = oracle.f32_to_bf16_array(finite)
    assert np.array_equal(got, torch_bf16_bits(finite))
    # NaN stays NaN
    nans = allbits[np.isnan(allbits)][:1000]
    g = oracle.f32_to_bf16_array(nans)
    assert np.all((g & 0x7F80) == 0x7F80) and np.all((g & 0x7F) != 0)


def test_e4m3_decode_exhaustive(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_to_f32(int(c)) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _e4m3_values():
    codes = np.arange(128, dtype=np.uint8)
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    return v[:127]                              # 0 .. 448, ascending


def test_e4m3_encode_vs_library(oracle):
    rng = np.random.default_rng(7)
    v = _e4m3_values().astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2                 # exact ties (representable in fp32)
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(0))
    mag = np.exp2(rng.uniform(-14, 10, size=400_000)).astype(np.float32)
    sgn = np.where(rng.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    big = np.array([448, 449, 463.99, 464, 464.01, 479, 480, 1e6, 3.4e38,
                    np.inf], np.float32)
    tiny = np.array([0.0, 2**-10, 2**-11, 3 * 2**-11, 1e-30, 1e-45], np.float32)
    x = np.concatenate([mids32, up, dn, v.astype(np.float32), mag * sgn,
                        big, tiny])
    x = np.concatenate([x, -x])
    got = oracle.f32_to_e4m3_array(x)
    assert np.array_equal(got, torch_e4m3_satfinite(x))


def test_e4m3_encode_is_nearest_even_by_search(oracle):
    """Brute force: nearest of the 127 non-negative finite values, ties to the
    even code, saturating; independent of both implementations' bit tricks."""
    rng = np.random.default_rng(11)
    v = _e4m3_values().astype(np.float64)
    x = np.concatenate([np.exp2(rng.uniform(-12, 9.5, 20000)),
                        (v[:-1] + v[1:]) / 2]).astype(np.float32)
    a = np.minimum(x.astype(np.float64), 448.0)
    d = np.abs(a[:, None] - v[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    codes = np.arange(127)
    pick = np.where(cand, codes[None, :], 1 << 20)
    even = np.where(cand & (codes[None, :] % 2 == 0), codes[None, :], 1 << 20)
    exp = np.where(cand.sum(axis=1) > 1, even.min(axis=1), pick.min(axis=1))
    got = oracle.f32_to_e4m3_array(x)
    assert np.array_equal(got, exp.astype(np.uint8))


def test_e4m3_hand_golden(oracle):
    """Codes derived by hand from the e4m3 definition (fixture cites it)."""
    path = os.path.join(GOLDEN, "e4m3_hand.txt")
    n = 0
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        val, code = line.split()
        x = float.fromhex(val) if val.startswith(("0x", "-0x")) else float(val)
        assert oracle.f32_to_e4m3(x) == int(code, 16), (val, code)
        n += 1
    assert n >= 15
