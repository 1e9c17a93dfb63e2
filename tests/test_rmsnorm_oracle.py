"""Pins for the allreduce + RMSNorm oracle (oracle/rmsnorm.py):
torch's own fp64 rms_norm on the same reduced rows, closed forms (constant
rows, scale invariance), the rank fold equals the allreduce oracle's fp32
result, and the bf16 rounding matches the allreduce oracle's rounding."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from oracle import rmsnorm as rn


@pytest.mark.parametrize("dtype,kind", [("f32", "uniform_f32"), ("bf16", "normal_bf16")])
def test_matches_torch_rms_norm_in_fp64(dtype, kind):
    p, rows, hidden, eps = 4, 16, 512, 1e-6
    xs = datagen.rank_buffers(kind, 4, p, rows * hidden)
    gamma = datagen.rank_buffers(kind, 8, 1, hidden)[0]
    y, y64 = rn.allreduce_rmsnorm(xs, gamma, rows, hidden, eps, dtype)
    s = torch.from_numpy(rn.rank_sum_f32(xs, dtype).astype(np.float64).reshape(rows, hidden))
    g = torch.from_numpy((rn.bf16_to_f32(gamma) if dtype == "bf16" else gamma).astype(np.float64))
    ref = torch.nn.functional.rms_norm(s, (hidden,), weight=g, eps=eps).numpy().ravel()
    assert np.allclose(y64, ref, rtol=1e-12, atol=0)


def test_rank_fold_is_the_allreduce():
    xs = datagen.rank_buffers("uniform_f32", 2, 8, 10_000)
    assert np.array_equal(rn.rank_sum_f32(xs, "f32"), oracle.allreduce(xs, "f32", "sum")[0])
    xb = datagen.rank_buffers("normal_bf16", 2, 8, 10_000)
    assert np.array_equal(rn.f32_to_bf16(rn.rank_sum_f32(xb, "bf16")),
                          oracle.allreduce(xb, "bf16", "sum")[0])


def test_constant_rows_normalise_to_gamma():
    rows, hidden = 3, 64
    xs = [np.full(rows * hidden, v, np.float32) for v in (1.5, -0.25, 0.75)]  # s = 2.0
    gamma = np.linspace(-1, 1, hidden).astype(np.float32)
    _, y64 = rn.allreduce_rmsnorm(xs, gamma, rows, hidden, 0.0, "f32")
    assert np.allclose(y64.reshape(rows, hidden), gamma[None, :], rtol=0, atol=1e-15)


def test_scale_invariance_without_eps():
    rows, hidden = 4, 128
    xs = datagen.rank_buffers("uniform_f32", 3, 2, rows * hidden)
    gamma = np.ones(hidden, np.float32)
    _, a = rn.allreduce_rmsnorm(xs, gamma, rows, hidden, 0.0, "f32")
    _, b = rn.allreduce_rmsnorm([x * np.float32(4.0) for x in xs], gamma, rows, hidden, 0.0, "f32")
    assert np.allclose(a, b, rtol=1e-13)
    # each normalised row has unit root mean square
    assert np.allclose(np.sqrt(np.mean(a.reshape(rows, hidden) ** 2, axis=1)), 1.0, rtol=1e-12)
