"""CPU oracle for the allreduce fused with RMSNorm.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

The "NCCL Roadmap Nov 2026 - Jan 2027 の解説" post (section "GENK と Flow")
mentions a Device API example that folds a Transformer RMSNorm into one kernel
with the reduce-scatter and all-gather (receive, sum, send out). It gives no
formula; the reading used here is the standard RMSNorm of each row of the
reduced activations:

    s[t, :] = fold over ranks, ascending, of x_r[t, :]   (fp32 adds, as allreduce)
    y[t, j] = s[t, j] / sqrt(mean_k(s[t, k]^2) + eps) * gamma[j]

with s kept in fp32 before any rounding (the point of fusing), the
normalisation evaluated in fp64, and y rounded once to the output type
(fp64 -> fp32 round to nearest, then to bf16 round to nearest even).
"""
from __future__ import annotations

import numpy as np


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def rank_sum_f32(xs, dtype: str) -> np.ndarray:
    """Ascending-rank fp32 fold of the rank buffers (bf16 widened exactly)."""
    vals = [bf16_to_f32(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32) for x in xs]
    acc = vals[0].copy()
    for v in vals[1:]:
        acc = (acc + v).astype(np.float32)
    return acc


def allreduce_rmsnorm(xs, gamma, rows: int, hidden: int, eps: float, dtype: str):
    """Returns (y in the output type, y in fp64 before rounding)."""
    s = rank_sum_f32(xs, dtype).astype(np.float64).reshape(rows, hidden)
    g = (bf16_to_f32(gamma) if dtype == "bf16" else np.asarray(gamma, np.float32)).astype(np.float64)
    ms = np.mean(s * s, axis=1, keepdims=True)
    y = s / np.sqrt(ms + eps) * g[None, :]
    y32 = y.astype(np.float32).ravel()
    return (f32_to_bf16(y32) if dtype == "bf16" else y32), y.ravel()
