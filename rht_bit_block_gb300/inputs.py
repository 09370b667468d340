"""Seeded synthetic inputs for the UFP4 quantizer and GEMM (numpy only).

This module holds no arithmetic of the method: it draws random numbers with
numpy's PCG64, rounds them to bf16 (round-to-nearest-even on the fp32 bit
pattern) and returns the bf16 bit patterns as uint16 arrays.  Both the CUDA
path's tests and the oracle read the same arrays, so input generation is never
a parity question.

Workload shapes follow the pages' model families (UFP4 summary, sections 核心贡献
and 实验: Dense 1.5B, MoE 7.9B and MoE 124B pretraining; 2D-block tutorial: 0.1 %
outliers); the distributions are stated per function.
"""
from __future__ import annotations

import numpy as np

SIGN_SEED = 0x5EED0001
SR_SEED = 1234


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs: the
    largest finite pattern plus the rounding increment stays below 2^32, so
    32-bit arithmetic does not wrap)."""
    a = np.asarray(a, dtype=np.float32)
    flat = np.ascontiguousarray(a).reshape(-1)
    out = np.empty(flat.size, dtype=np.uint16)
    step = 1 << 20  # in slices that stay in cache (whole-array temporaries are much slower)
    for i in range(0, flat.size, step):
        u = flat[i:i + step].view(np.uint32).copy()
        u += (u >> 16) & 1
        u += 0x7FFF
        u >>= 16
        out[i:i + step] = u
    return out.reshape(a.shape)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rows: int, cols: int, seed: int, std: float = 1.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return f32_to_bf16_bits(rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(std))


def with_element_outliers(x_bf16: np.ndarray, frac: float, factor: float, seed: int) -> np.ndarray:
    """Multiply round(frac * size) distinct, seeded positions by `factor`."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = int(round(frac * x_bf16.size))
    pos = rng.choice(x_bf16.size, size=k, replace=False)
    # only the chosen entries change (bf16 -> fp32 -> bf16 is the identity elsewhere)
    out = np.array(x_bf16, dtype=np.uint16, copy=True)
    flat = out.reshape(-1)
    flat[pos] = f32_to_bf16_bits(bf16_bits_to_f32(flat[pos]) * np.float32(factor))
    return out


def with_column_outliers(x_bf16: np.ndarray, frac: float, factor: float, seed: int) -> np.ndarray:
    """Multiply round(frac * cols) seeded channels (columns) by `factor`."""
    x = bf16_bits_to_f32(x_bf16).copy()
    rng = np.random.Generator(np.random.PCG64(seed))
    k = max(1, int(round(frac * x.shape[1])))
    cols = rng.choice(x.shape[1], size=k, replace=False)
    x[:, cols] *= np.float32(factor)
    return f32_to_bf16_bits(x)


def student_t_bf16(rows: int, cols: int, seed: int, nu: float = 3.0, scale: float = 1e-3) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return f32_to_bf16_bits((rng.standard_t(nu, size=(rows, cols)) * scale).astype(np.float32))


# ------------------------------------------------------------ named workloads
def tiny_check(rows: int = 256, cols: int = 1024) -> np.ndarray:
    """Tiny quantizer check: N(0,1) with 0.1 % element outliers x50."""
    return with_element_outliers(normal_bf16(rows, cols, 101), 1e-3, 50.0, 102)


def dense_fprop(m: int = 8192, n: int = 5632, k: int = 2048):
    """Dense-1.5B-like FPROP operands: X tokens x hidden, N(0,1) with 0.1 % of
    the channels (columns) x30; W N(0, 0.02^2)."""
    x = with_column_outliers(normal_bf16(m, k, 201), 1e-3, 30.0, 202)
    w = normal_bf16(n, k, 203, std=0.02)
    return x, w


def dy_sr(m: int = 8192, n: int = 2048):
    """dY for the stochastic-rounding path: 1e-3 * Student-t(3); W N(0, 0.02^2)."""
    dy = student_t_bf16(m, n, 301)
    w = normal_bf16(n, n, 302, std=0.02)
    return dy, w


def moe_routing(tokens: int = 16384, experts: int = 8, top_k: int = 2, seed: int = 401):
    """Seeded top-k routing over N(0,1) logits (softmax is monotone, so the
    top-k of the softmax is the top-k of the logits; ties go to the lower
    expert id).  Returns the per-expert token lists in ascending token order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((tokens, experts), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    return [np.sort(np.nonzero((order == e).any(axis=1))[0]) for e in range(experts)]


def moe_step(tokens: int = 16384, experts: int = 8, hidden: int = 2048, ffn: int = 1408):
    """MoE-7.9B-like expert FFN step: routed token lists, X (tokens x hidden),
    W_e (experts x ffn x hidden), dY_e per expert (1e-3 * Student-t(3))."""
    lists = moe_routing(tokens, experts)
    x = normal_bf16(tokens, hidden, 402)
    w = normal_bf16(experts * ffn, hidden, 403, std=0.02).reshape(experts, ffn, hidden)
    total = sum(len(l) for l in lists)
    dy = student_t_bf16(total, ffn, 404)
    return lists, x, w, dy


def large_sweep(m: int = 16384, k: int = 7168, n: int = 7168):
    """MoE-124B-like large shapes: N(0,1) with 0.1 % element outliers x50."""
    x = with_element_outliers(normal_bf16(m, k, 501), 1e-3, 50.0, 502)
    w = with_element_outliers(normal_bf16(n, k, 503), 1e-3, 50.0, 504)
    return x, w
