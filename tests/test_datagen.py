"""Pins for the seeded input generator (SplitMix64 streams).

The generator is pinned to the published SplitMix64 outputs, restated here in
pure Python (independent code), and its value recipes are checked by range,
lattice and moment properties.
"""
import math

import numpy as np
import pytest

import datagen

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def py_mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def py_draw(s0, d):
    return py_mix((s0 + (d + 1) * GAMMA) & M64)


def py_state(seed, rank):
    return py_mix((seed + GAMMA) & M64) ^ (((rank + 1) * 0xD1B54A32D192ED03) & M64)


def test_splitmix64_published_vectors(golden_dir):
    rows = [ln.split() for ln in (golden_dir / "splitmix64_seed1234567.txt").read_text().splitlines()
            if ln and not ln.startswith("#")]
    assert len(rows) == 5
    state0 = int(rows[0][0])
    got = datagen.raw(state0, 0, 5)
    for (s, i, v) in rows:
        assert int(s) == state0
        assert int(got[int(i)]) == int(v)
        assert py_draw(state0, int(i)) == int(v)


def test_counter_based_ranges_agree():
    s0 = datagen.stream_state(7, 3)
    full = datagen.raw(s0, 0, 300)
    part = datagen.raw(s0, 100, 50)
    assert np.array_equal(full[100:150], part)


@pytest.mark.parametrize("seed,rank", [(0, 0), (0, 1), (2, 7), (3, 5), (12345, 63)])
def test_stream_state_formula(seed, rank):
    assert datagen.stream_state(seed, rank) == py_state(seed, rank)


@pytest.mark.parametrize("seed,rank", [(0, 0), (1, 3), (2, 7)])
def test_uniform_matches_restatement(seed, rank):
    n = 2000
    x = datagen.uniform_f32(seed, rank, n)
    s0 = py_state(seed, rank)
    exp = np.array([(2 * (py_draw(s0, i) >> 40) - (1 << 24)) / 16777216.0 for i in range(n)],
                   dtype=np.float64)
    assert np.array_equal(x.astype(np.float64), exp)


def test_uniform_range_lattice_moments():
    x = datagen.uniform_f32(2, 4, 1 << 20).astype(np.float64)
    assert x.min() >= -1.0 and x.max() < 1.0
    # every value is a multiple of 2^-23
    assert np.all(np.floor(x * 2 ** 23) == x * 2 ** 23)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0 / 3.0) < 5e-3


def test_int32_matches_restatement_and_range():
    n = 3000
    x = datagen.int32(2, 1, n, -1000, 1000)
    s0 = py_state(2, 1)
    exp = [-1000 + py_draw(s0, i) % 2001 for i in range(n)]
    assert x.tolist() == exp
    big = datagen.int32(2, 5, 1 << 20)
    assert big.min() == -1000 and big.max() == 1000


def test_normal_bf16_recipe_and_moments():
    n = 400
    s0 = py_state(1, 2)
    xb = datagen.normal_bf16(1, 2, n)
    xf = datagen.normal_f32(1, 2, n)
    for i in range(n):
        u1 = ((py_draw(s0, 2 * i) >> 11) + 1) * 2.0 ** -53
        u2 = (py_draw(s0, 2 * i + 1) >> 11) * 2.0 ** -53
        z = math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
        assert float(xf[i]) == float(np.float32(z))
    # bf16 bits = round-to-nearest-even of the f32 value (independent rounding:
    # pick the nearer of the two bf16 neighbours, the even one on a tie)
    bits = xf.view(np.uint32).astype(np.int64)
    for i in range(n):
        lo = (bits[i] >> 16) & 0xFFFF
        rem = bits[i] & 0xFFFF
        if rem > 0x8000 or (rem == 0x8000 and (lo & 1)):
            exp = lo + 1
        else:
            exp = lo
        assert int(xb[i]) == exp
    big = datagen.normal_f32(3, 0, 1 << 20, 0.0, 0.02).astype(np.float64)
    assert abs(big.mean()) < 2e-4
    assert abs(big.std() - 0.02) < 2e-4


def test_thread_count_does_not_change_bits():
    a = datagen.normal_bf16(4, 3, 300_000, nthreads=1)
    b = datagen.normal_bf16(4, 3, 300_000, nthreads=7)
    assert np.array_equal(a, b)
    c = datagen.uniform_f32(0, 1, 300_001, nthreads=1)
    d = datagen.uniform_f32(0, 1, 300_001, nthreads=5)
    assert np.array_equal(c, d)


def test_streams_differ_across_ranks_and_seeds():
    a = datagen.uniform_f32(0, 0, 64)
    b = datagen.uniform_f32(0, 1, 64)
    c = datagen.uniform_f32(1, 0, 64)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
