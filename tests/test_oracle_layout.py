"""Pins for the oracle's layout (counts, offsets, stable slot map).

Checked against: the invariants the method fixes (counts sum to T*K, offsets
are their prefix sums, every (token, k) entry lands in exactly one row of its
expert's range), numpy's stable argsort (a library routine for the same stable
order), brute force over every routing of tiny shapes, and a hand-derived
example (tests/golden/layout_hand.txt).
"""
import itertools
import os

import numpy as np
import pytest

from combine_moe_layout_05_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_layout_invariants(lay, ids, E, R):
    T, K = ids.shape
    n = T * K
    c, off, ro = lay.expert_counts, lay.expert_offsets, lay.rank_offsets
    assert c.sum() == n
    assert off[0] == 0 and off[E] == n
    assert np.array_equal(np.diff(off), c)
    assert np.array_equal(ro, off[np.arange(R + 1) * (E // R)])
    d = lay.dst_row.ravel()
    assert np.array_equal(np.sort(d), np.arange(n))          # a permutation
    e = ids.ravel()
    assert np.all(d >= off[e]) and np.all(d < off[e + 1])     # right bucket
    t = np.arange(n) // K
    assert np.array_equal(lay.src_token[d], t)
    # inside a bucket, rows follow token order
    s = lay.src_token
    for ee in range(E):
        seg = s[off[ee]:off[ee + 1]]
        assert np.all(np.diff(seg) >= 0)


def check_against_stable_argsort(lay, ids):
    T, K = ids.shape
    order = np.argsort(ids.ravel(), kind="stable")
    assert np.array_equal(lay.src_token, (order // K).astype(np.int32))
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(lay.dst_row.ravel(), inv.astype(np.int32))
    assert np.array_equal(lay.expert_counts,
                          np.bincount(ids.ravel(), minlength=lay.expert_counts.size))


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_layout_workloads(oracle, name):
    w = wl.get(name)
    inp = wl.make_inputs(w)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    assert lay.error == 0
    check_layout_invariants(lay, inp.topk_ids, w.E, w.R)
    check_against_stable_argsort(lay, inp.topk_ids)


def brute_force_slots(ids, E):
    """Slot of every entry straight from the definition: the number of entries
    of smaller experts plus the number of earlier entries of the same expert."""
    flat = [int(v) for v in ids.ravel()]
    out = []
    for i, e in enumerate(flat):
        smaller = sum(1 for v in flat if v < e)
        earlier = sum(1 for v in flat[:i] if v == e)
        out.append(smaller + earlier)
    return out


def test_layout_brute_force_all_tiny_routings(oracle):
    cases = 0
    for T in range(0, 4):
        for K in (1, 2):
            for E in range(K, 5):
                for R in [r for r in range(1, E + 1) if E % r == 0]:
                    for flat in itertools.product(range(E), repeat=T * K):
                        ids = np.array(flat, np.int32).reshape(T, K)
                        lay = oracle.layout(ids, E, R)
                        dup = any(len(set(row)) < K for row in ids.tolist())
                        assert lay.error == (2 if dup else 0)
                        assert lay.dst_row.ravel().tolist() == brute_force_slots(ids, E)
                        counts = [sum(1 for v in flat if v == e) for e in range(E)]
                        assert lay.expert_counts.tolist() == counts
                        assert lay.expert_offsets.tolist() == [sum(counts[:e]) for e in range(E + 1)]
                        assert lay.rank_offsets.tolist() == [sum(counts[:r * (E // R)]) for r in range(R + 1)]
                        cases += 1
    assert cases > 5000


def test_layout_hand_golden(oracle):
    vals = {}
    for line in open(os.path.join(GOLDEN, "layout_hand.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            key, rest = line.split(":", 1)
            vals[key.strip()] = [int(v) for v in rest.split()]
    T, K, E, R = vals["shape"]
    ids = np.array(vals["topk_ids"], np.int32).reshape(T, K)
    lay = oracle.layout(ids, E, R)
    assert lay.error == 0
    assert lay.expert_counts.tolist() == vals["expert_counts"]
    assert lay.expert_offsets.tolist() == vals["expert_offsets"]
    assert lay.rank_offsets.tolist() == vals["rank_offsets"]
    assert lay.dst_row.ravel().tolist() == vals["dst_row"]
    assert lay.src_token.tolist() == vals["src_token"]


def test_layout_out_of_range_ids(oracle):
    ids = np.array([[0, 5], [-1, 2], [3, 3]], np.int32)   # E = 4
    lay = oracle.layout(ids, 4, 2)
    assert lay.error == 1 | 2
    assert lay.dst_row.ravel().tolist() == [0, -1, -1, 1, 2, 3]
    assert lay.expert_counts.tolist() == [1, 0, 1, 2]
    assert lay.expert_offsets.tolist() == [0, 1, 1, 2, 4]
    assert lay.src_token[:4].tolist() == [0, 1, 2, 2]
    assert lay.src_token[4:].tolist() == [-1, -1]            # untouched rows


def test_layout_empty_batch(oracle):
    lay = oracle.layout(np.zeros((0, 4), np.int32), 16, 4)
    assert lay.error == 0
    assert not lay.expert_counts.any() and not lay.expert_offsets.any()
    assert not lay.rank_offsets.any()


def test_layout_forced_empty_experts(oracle):
    """Zipf routing with most experts never picked still gives a valid map."""
    rng = np.random.default_rng(5)
    ids = rng.permutation(np.arange(3))[None, :].repeat(50, 0).astype(np.int32)
    lay = oracle.layout(ids, 64, 8)
    assert lay.expert_counts[3:].sum() == 0
    check_layout_invariants(lay, ids, 64, 8)
    check_against_stable_argsort(lay, ids)
