"""Seeded synthetic MoE routing workloads.

This module draws inputs only: hidden rows, top-k expert ids and routing
weights.  It holds none of the layout / dispatch / combine arithmetic, and both
the CUDA path and the CPU oracle consume exactly the arrays it returns.

The shapes follow the settings the method is evaluated on (Perplexity,
"Enabling trillion-parameter models on AWS EFA", section "Evaluation":
DeepSeek-V3 / Kimi-K2 with hidden size 7168, decode batch 128, prefill batch
4096, block-scaled FP8 dispatch, bf16 combine), plus a tiny case for brute
force and a large Qwen3-shaped prefill with outlier rows.  No router trace or
dataset is used; routing is drawn from the distributions below.

Recipe (all draws from numpy's PCG64, one independent child stream per array
from ``SeedSequence(seed)``):
  * hidden rows: N(0,1) in fp32, rounded to bf16 (round to nearest even);
    with outliers, a seeded 1 % of rows is multiplied by 100 in fp32 and
    rounded to bf16 again;
  * uniform routing: each token takes the first K entries of a uniformly
    random permutation of the E experts (K distinct ids);
  * Zipf(s) routing: experts are placed in a seeded random order; the expert
    at position i (1-based) has weight i^-s; each token draws K distinct
    experts one after another in proportion to those weights, redrawing
    duplicates.  This is sampled exactly with Gumbel-top-K keys
    (log weight + Gumbel noise, the K largest in descending order);
  * routing weights: softmax, in fp64, of K N(0,1) logits, stored as fp32;
  * per-expert scalars for the scaling stand-in experts: U(0.5, 1.5) fp32;
  * random expert outputs: N(0,1) rounded to bf16.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # hidden size
    E: int            # experts
    R: int            # destination ranks (regions), E % R == 0
    K: int            # experts per token
    routing: str      # "uniform" | "zipf"
    zipf_s: float
    experts: str      # "identity" | "scale" | "random" | "dequant"
    dispatch: tuple   # subset of ("bf16", "fp8")
    outlier_frac: float
    seed: int


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 64, 256, 8, 2, 2, "uniform", 0.0, "identity",
                 ("bf16", "fp8"), 0.0, 0),
        Workload("decode_dsv3", 128, 7168, 256, 32, 8, "uniform", 0.0, "scale",
                 ("bf16",), 0.0, 1),
        Workload("decode_dsv3_fp8", 256, 7168, 256, 32, 8, "uniform", 0.0,
                 "random", ("fp8",), 0.0, 2),
        Workload("prefill_kimi_k2", 4096, 7168, 384, 48, 8, "zipf", 1.2,
                 "scale", ("bf16", "fp8"), 0.0, 3),
        Workload("prefill_qwen3", 16384, 4096, 128, 16, 8, "zipf", 1.0,
                 "dequant", ("fp8",), 0.01, 4),
    ]
}

# The workload the benchmark's headline line is measured on: the largest
# configuration (FP8 dispatch, bf16 combine).
HEADLINE = "prefill_qwen3"


def get(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(n)]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, PyTorch's conversion) as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def hidden(T: int, H: int, rng, outlier_frac: float = 0.0, rng_rows=None):
    x = to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    if outlier_frac > 0.0 and T > 0:
        n = max(1, int(round(outlier_frac * T)))
        rows = np.sort(rng_rows.choice(T, size=n, replace=False))
        x[rows] = to_bf16_bits(bf16_bits_to_f32(x[rows]) * np.float32(100.0))
    return x


def routing_uniform(T: int, E: int, K: int, rng) -> np.ndarray:
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int32)


def routing_zipf(T: int, E: int, K: int, s: float, rng) -> np.ndarray:
    perm = rng.permutation(E)
    logw = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    u = rng.random((T, E))
    u = np.clip(u, np.finfo(np.float64).tiny, 1.0)
    keys = logw[None, :] - np.log(-np.log(u))
    pos = np.argsort(-keys, axis=1, kind="stable")[:, :K]
    return perm[pos].astype(np.int32)


def routing_weights(T: int, K: int, rng) -> np.ndarray:
    z = rng.standard_normal((T, K))
    z = z - z.max(axis=1, keepdims=True) if T else z
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True) if T else 1.0
    return p.astype(np.float32)


@dataclasses.dataclass
class Inputs:
    tokens: np.ndarray         # [T, H] uint16 (bf16 bits)
    topk_ids: np.ndarray       # [T, K] int32
    topk_weights: np.ndarray   # [T, K] float32
    expert_scale: np.ndarray   # [E] float32, used by the "scale" stand-in
    expert_rows_seed: int      # seed for "random" expert outputs


def make_inputs(w: Workload, seed: int | None = None, T: int | None = None) -> Inputs:
    """Draw one batch of a workload.  ``T`` overrides the token count (tests)."""
    seed = w.seed if seed is None else seed
    T = w.T if T is None else T
    r_x, r_rows, r_ids, r_w, r_s, r_y = _streams(seed, 6)
    tokens = hidden(T, w.H, r_x, w.outlier_frac, r_rows)
    if w.routing == "uniform":
        ids = routing_uniform(T, w.E, w.K, r_ids)
    elif w.routing == "zipf":
        ids = routing_zipf(T, w.E, w.K, w.zipf_s, r_ids)
    else:
        raise ValueError(w.routing)
    weights = routing_weights(T, w.K, r_w)
    scale = r_s.uniform(0.5, 1.5, size=w.E).astype(np.float32)
    return Inputs(tokens, np.ascontiguousarray(ids), weights, scale,
                  int(r_y.integers(0, 2**31 - 1)))


def random_rows(n: int, H: int, seed: int) -> np.ndarray:
    """N(0,1) bf16 rows, the "random" expert outputs."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return to_bf16_bits(rng.standard_normal((n, H), dtype=np.float32))
