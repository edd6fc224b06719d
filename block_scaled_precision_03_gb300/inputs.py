"""Seeded synthetic inputs for the block-scaled linear layer.

This module only draws random numbers and rounds them to BF16 bit
patterns; it holds none of the quantization or GEMM arithmetic, so both
the CUDA path and the CPU oracle may take their inputs from it.

The workloads follow the shapes the pages and the benchmark statement
use (no dataset is read anywhere):

* tiny MXFP8 linear: A, B 256 x 256 ~ N(0, 1)
* Llama-3-8B MLP up-projection forward: X 8192 x 4096 ~ N(0, 1) with an
  independent 0.1 % of entries scaled x50 (outliers), W 14336 x 4096 ~
  N(0, 0.02^2)
* its backward: dY 8192 x 14336, random sign, magnitude 2^U(-20, 4)
* NVFP4 forward: X 8192 x 4096 ~ N(0,1), W 4096 x 4096 ~ N(0, 0.02^2),
  X' 8192 x 14336 ~ N(0,1), W' 4096 x 14336 ~ N(0, 0.02^2)
* MoE grouped path (DeepSeek-V3-like expert layer of the MoE FP4 page,
  section 4): 64 experts, 32768 token-expert rows, per-expert counts
  multinomial(32768, p_k ~ k^-1.1), hidden 7168, N = 2048; activations
  ~ N(0, 1), expert weights ~ N(0, 0.02^2).

Large draws are split into fixed 2^24-element chunks, each with its own
child seed of ``numpy.random.SeedSequence(seed)``, so the values do not
depend on how many threads generate them.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 24


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round FP32 values to BF16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _chunked(n: int, seed: int, fill) -> np.ndarray:
    """Draw n float32 values chunk by chunk (deterministic chunk seeds) and
    return them rounded to BF16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, (n + CHUNK - 1) // CHUNK)
    seeds = np.random.SeedSequence(seed).spawn(nchunks)

    def work(i):
        lo, hi = i * CHUNK, min(n, (i + 1) * CHUNK)
        buf = np.empty(hi - lo, dtype=np.float32)
        fill(np.random.default_rng(seeds[i]), buf)
        out[lo:hi] = f32_to_bf16_bits(buf)

    threads = min(nchunks, os.cpu_count() or 1, 16)
    if threads <= 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal_bf16(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) draws rounded to BF16 bit patterns."""
    n = int(np.prod(shape))

    def fill(rng, dst):
        rng.standard_normal(out=dst, dtype=np.float32)
        if std != 1.0:
            dst *= np.float32(std)

    return _chunked(n, seed, fill).reshape(shape)


def outlier_activations_bf16(shape, seed: int, rate: float = 0.001, factor: float = 50.0):
    """N(0,1) with an independent Bernoulli(rate) mask of entries scaled by factor."""
    n = int(np.prod(shape))

    def fill(rng, dst):
        rng.standard_normal(out=dst, dtype=np.float32)
        mask = rng.random(dst.size, dtype=np.float32) < rate
        dst[mask] *= np.float32(factor)

    return _chunked(n, seed, fill).reshape(shape)


def loguniform_grad_bf16(shape, seed: int, lo_exp: float = -20.0, hi_exp: float = 4.0):
    """Random sign times 2^U(lo_exp, hi_exp)."""
    n = int(np.prod(shape))

    def fill(rng, dst):
        e = rng.uniform(lo_exp, hi_exp, dst.size).astype(np.float32)
        sign = np.where(rng.random(dst.size, dtype=np.float32) < 0.5, -1.0, 1.0).astype(np.float32)
        dst[:] = sign * np.exp2(e)

    return _chunked(n, seed, fill).reshape(shape)


def zipf_group_counts(total_rows: int, groups: int, s: float, seed: int) -> np.ndarray:
    """Per-expert row counts ~ multinomial(total_rows, p_k ~ k^-s), k = 1..groups."""
    k = np.arange(1, groups + 1, dtype=np.float64)
    p = k ** (-s)
    p /= p.sum()
    return np.random.default_rng(seed).multinomial(total_rows, p).astype(np.int64)


def group_offsets(counts: np.ndarray) -> np.ndarray:
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    off[1:] = np.cumsum(counts)
    return off


# ----------------------------------------------------------------- configs
def tiny_linear(seed_a: int = 0, seed_b: int = 1, m: int = 256, n: int = 256, k: int = 256):
    return {"A": normal_bf16((m, k), seed_a), "B": normal_bf16((n, k), seed_b)}


def llama_up_proj(m: int = 8192, n: int = 14336, k: int = 4096, seed: int = 0):
    return {"X": outlier_activations_bf16((m, k), seed),
            "W": normal_bf16((n, k), seed + 1, std=0.02)}


def llama_up_proj_backward(m: int = 8192, n: int = 14336, k: int = 4096, seed: int = 0):
    d = llama_up_proj(m, n, k, seed)
    d["dY"] = loguniform_grad_bf16((m, n), seed + 2)
    return d


def nvfp4_forward(m: int = 8192, n: int = 4096, k: int = 4096, k2: int = 14336, seed: int = 0):
    return {"X": normal_bf16((m, k), seed), "W": normal_bf16((n, k), seed + 1, std=0.02),
            "X2": normal_bf16((m, k2), seed + 2), "W2": normal_bf16((n, k2), seed + 3, std=0.02)}


def moe_grouped(rows: int = 32768, experts: int = 64, k: int = 7168, n: int = 2048,
                zipf_s: float = 1.1, seed: int = 0):
    counts = zipf_group_counts(rows, experts, zipf_s, seed)
    return {"counts": counts, "offsets": group_offsets(counts),
            "A": normal_bf16((rows, k), seed + 1),
            "W": normal_bf16((experts, n, k), seed + 2, std=0.02)}
