"""The fp16 facts the fused decode kernel's pairwise counting relies on,
checked with numpy's IEEE binary16 (no GPU): an expert id x in [0, 1024] is
the fp16 value 1024 + x with bit pattern 0x6400 + x, exact and ordered like
the ids, and 2048 (an invalid id) compares above all of them; a count c of at
most 32 stays exact in fp16 sums and comes back as (c + 1024) - 0x6400."""
import numpy as np


def test_ids_encode_exactly_and_in_order():
    x = np.arange(0, 1025, dtype=np.int64)
    h = (1024 + x).astype(np.float16)
    assert np.array_equal(h.astype(np.int64), 1024 + x)              # exact
    assert np.array_equal(h.view(np.uint16).astype(np.int64), 0x6400 + x)
    assert np.all(np.diff(h) > 0)                                       # ordered
    invalid = np.float16(2048.0)
    assert invalid.view(np.uint16) == 0x6400 + 1024
    assert np.all(h[:-1] < invalid)                     # every valid id (x < 1024) is below


def test_counts_stay_exact_and_decode():
    one = np.float16(1.0)
    acc = np.float16(0.0)
    for c in range(1, 33):                              # one fp16 add per counted entry
        acc = np.float16(acc + one)
        assert float(acc) == c
        bits = int(np.float16(acc + np.float16(1024.0)).view(np.uint16))
        assert bits - 0x6400 == c
    # two packed lanes decode independently: the subtraction never borrows
    lo, hi = 7, 32
    word = (0x6400 + lo) | ((0x6400 + hi) << 16)
    v = word - 0x64006400
    assert v & 0xFFFF == lo and v >> 16 == hi
