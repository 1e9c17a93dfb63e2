"""Pins for the CPU oracle (``oracle/``), checked against things other than itself.

What pins what:
  * brute force on tiny inputs against an independent restatement written
    here (Python loops, numpy float32 scalars, exact-rational bf16 rounding);
  * closed forms: integer-valued inputs sum exactly in any order; P copies of
    one buffer of small integers sum to exactly P times it;
  * a crafted case where per-step bf16 rounding differs from one final
    rounding, and the bf16 round-half-to-even ties;
  * order-free invariants for int32 sum (wrapping), min and max;
  * a negative control: reversing the rank order changes fp32 sums;
  * cross-collective invariants: every allreduce output identical,
    reduce-scatter then all-gather equals allreduce, P = 1 is a copy,
    in-place equals out-of-place, threaded equals single-threaded.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import datagen
import oracle

rng = np.random.default_rng(20261202)

PS = [1, 2, 3, 5, 8]
COUNTS = [0, 1, 2, 3, 7, 8, 15, 16, 17, 33, 64, 67]


# ---------------------------------------------------------------- restatement
def f32_bits(x):
    return np.array([x], dtype=np.float32).view(np.uint32)[0]


def bf16_widen_ref(h):
    """bf16 bit pattern -> exact Python float (sign, exponent, 7-bit fraction)."""
    h = int(h)
    s = -1.0 if h & 0x8000 else 1.0
    e = (h >> 7) & 0xFF
    f = h & 0x7F
    if e == 0:
        return s * f * 2.0 ** -133
    return s * (1.0 + f / 128.0) * 2.0 ** (e - 127)


def bf16_round_ref(v: float) -> int:
    """Exact-rational round-to-nearest-even of a finite float to bf16 bits."""
    neg = v < 0 or (v == 0 and np.signbit(v))
    a = Fraction(abs(v))
    if a == 0:
        return 0x8000 if neg else 0
    e = 0
    while a >= 2 ** (e + 1):
        e += 1
    while a < 2 ** e:
        e -= 1
    q = Fraction(2) ** max(e - 7, -133)       # 8 significant bits, subnormal floor
    k = a // q
    rem = a / q - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    val = float(k * q)
    bits = int(f32_bits(np.float32(val)))
    assert bits & 0xFFFF == 0
    out = bits >> 16
    return out | 0x8000 if neg else out


def fold_ref(op, vals):
    acc = vals[0]
    for x in vals[1:]:
        if op == "sum":
            acc = acc + x
        elif op == "min":
            acc = x if x < acc else acc
        else:
            acc = x if x > acc else acc
    return acc


def reduce_ref(dtype, op, column):
    """Reduce one element across ranks, the plain way."""
    if dtype == "f32":
        return np.float32(fold_ref(op, [np.float32(v) for v in column]))
    if dtype == "bf16":
        acc = fold_ref(op, [np.float32(bf16_widen_ref(v)) for v in column])
        return np.uint16(bf16_round_ref(float(acc)))
    # int32: Python integers, wrapped to two's complement at the end (sum) or
    # compared exactly (min / max)
    if op == "sum":
        s = sum(int(v) for v in column)
        return np.int32(((s + 2 ** 31) % 2 ** 32) - 2 ** 31)
    return np.int32(fold_ref(op, [int(v) for v in column]))


def make_inputs(dtype, p, n):
    if dtype == "f32":
        xs = [rng.uniform(-1, 1, n).astype(np.float32) for _ in range(p)]
        # sprinkle exact ties and signed zeros to exercise min / max tie rules
        for x in xs:
            if n >= 4:
                x[0] = 0.0
                x[1] = -0.0
                x[2] = 0.5
        return xs
    if dtype == "bf16":
        xs = []
        for _ in range(p):
            f = rng.normal(0, 3, n).astype(np.float32)
            b = (f.view(np.uint32) >> 16).astype(np.uint16)
            if n >= 4:
                b[0] = 0x0000
                b[1] = 0x8000
                b[2] = 0x3F00
            xs.append(b)
        return xs
    xs = [rng.integers(-2 ** 31, 2 ** 31, n, dtype=np.int64).astype(np.int32) for _ in range(p)]
    for x in xs:
        if n >= 2:
            x[0] = 2 ** 31 - 1
            x[1] = 7
    return xs


def same_bits(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "min", "max"])
@pytest.mark.parametrize("p", PS)
def test_allreduce_brute_force(dtype, op, p):
    for n in COUNTS:
        xs = make_inputs(dtype, p, n)
        outs = oracle.allreduce(xs, dtype, op)
        exp = np.array([reduce_ref(dtype, op, [x[i] for x in xs]) for i in range(n)],
                       dtype=outs[0].dtype)
        for r in range(p):
            assert same_bits(outs[r], exp), (dtype, op, p, n, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("p", [1, 2, 3, 8])
def test_reduce_scatter_brute_force(dtype, op, p):
    for rc in [0, 1, 3, 8, 17]:
        xs = make_inputs(dtype, p, p * rc)
        outs = oracle.reduce_scatter(xs, dtype, op)
        for s in range(p):
            exp = np.array([reduce_ref(dtype, op, [x[s * rc + j] for x in xs])
                            for j in range(rc)], dtype=outs[s].dtype)
            assert same_bits(outs[s], exp), (dtype, op, p, rc, s)


@pytest.mark.parametrize("dtype", [np.float32, np.uint16, np.int32])
@pytest.mark.parametrize("p", [1, 2, 3, 8])
def test_allgather_brute_force(dtype, p):
    for sc in [0, 1, 5, 16, 33]:
        xs = [rng.integers(0, 60000, sc).astype(dtype) for _ in range(p)]
        outs = oracle.allgather(xs)
        for r in range(p):
            exp = np.array([xs[k][j] for k in range(p) for j in range(sc)], dtype=dtype)
            assert same_bits(outs[r], exp)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("p", [2, 4, 8, 64])
def test_f32_integer_valued_sum_is_exact(p):
    n = 4099
    xs = [rng.integers(-1000, 1001, n).astype(np.float32) for _ in range(p)]
    out = oracle.allreduce(xs, "f32", "sum")[0]
    exact = np.sum(np.stack(xs).astype(np.int64), axis=0)
    assert np.array_equal(out.astype(np.int64), exact)


@pytest.mark.parametrize("p", [2, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_p_copies_sum_to_p_times(p, dtype):
    n = 5000
    small = rng.integers(-30, 31, n)
    if dtype == "f32":
        x = small.astype(np.float32)
        out = oracle.allreduce([x.copy() for _ in range(p)], "f32", "sum")[0]
        assert np.array_equal(out, (p * small).astype(np.float32))
    else:
        x = (small.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        out = oracle.allreduce([x.copy() for _ in range(p)], "bf16", "sum")[0]
        got = (out.astype(np.uint32) << 16).view(np.float32)
        # |p * small| <= 240 < 256: exactly representable with 8 significant bits
        assert np.array_equal(got, (p * small).astype(np.float32))


def test_bf16_rounds_once_not_per_step():
    one = 0x3F80            # 1.0
    e8 = 0x3B80             # 2^-8
    xs = [np.array([one], np.uint16), np.array([e8], np.uint16), np.array([e8], np.uint16)]
    out = oracle.allreduce(xs, "bf16", "sum")[0]
    # fp32 accumulation: 1 + 2^-8 + 2^-8 = 1 + 2^-7 exactly -> 0x3F81.
    # Per-step bf16 rounding would tie 1 + 2^-8 back to 1.0 twice -> 0x3F80.
    assert int(out[0]) == 0x3F81


def test_bf16_round_half_to_even():
    one = 0x3F80
    e8 = 0x3B80             # 2^-8: 1 + 2^-8 is a tie between 1 and 1 + 2^-7
    e8x3 = 0x3C40           # 3 * 2^-8: 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6
    out = oracle.allreduce([np.array([one, one], np.uint16),
                            np.array([e8, e8x3], np.uint16)], "bf16", "sum")[0]
    assert int(out[0]) == 0x3F80
    assert int(out[1]) == 0x3F82


def test_bf16_identity_on_every_finite_pattern():
    pats = np.arange(65536, dtype=np.uint32)
    finite = ((pats >> 7) & 0xFF) != 0xFF
    x = pats[finite].astype(np.uint16)
    out = oracle.allreduce([x], "bf16", "sum")[0]
    assert np.array_equal(out, x)


def test_bf16_rounding_matches_rational_rounding():
    n = 20000
    a = (rng.normal(0, 1, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    b = (rng.normal(0, 1e-2, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out = oracle.allreduce([a, b], "bf16", "sum")[0]
    af = (a.astype(np.uint32) << 16).view(np.float32)
    bf = (b.astype(np.uint32) << 16).view(np.float32)
    s = (af + bf).astype(np.float32)
    for i in range(0, n, 7):
        assert int(out[i]) == bf16_round_ref(float(s[i])), i


# ---------------------------------------------------------------- invariants
def test_int32_sum_wraps_and_is_order_free():
    p, n = 8, 3000
    xs = [rng.integers(-2 ** 31, 2 ** 31, n, dtype=np.int64).astype(np.int32) for _ in range(p)]
    exp = ((np.sum(np.stack(xs).astype(np.int64), axis=0) + 2 ** 31) % 2 ** 32) - 2 ** 31
    base = oracle.allreduce(xs, "i32", "sum")[0]
    assert np.array_equal(base.astype(np.int64), exp)
    for perm in list(itertools.permutations(range(p)))[:: 5000]:
        out = oracle.allreduce([xs[i] for i in perm], "i32", "sum")[0]
        assert np.array_equal(out, base)
    wrap = oracle.allreduce([np.array([2 ** 31 - 1], np.int32), np.array([1], np.int32)],
                            "i32", "sum")[0]
    assert int(wrap[0]) == -2 ** 31


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_min_max_equal_library_extrema_any_order(dtype):
    p, n = 8, 2000
    xs = (datagen.rank_buffers("uniform_f32", 2, p, n) if dtype == "f32"
          else datagen.rank_buffers("int32", 2, p, n))
    st = np.stack(xs)
    mn = oracle.allreduce(xs, dtype, "min")[0]
    mx = oracle.allreduce(xs, dtype, "max")[0]
    assert np.array_equal(mn, st.min(axis=0))
    assert np.array_equal(mx, st.max(axis=0))
    rev = xs[::-1]
    assert np.array_equal(oracle.allreduce(rev, dtype, "min")[0], mn)
    assert np.array_equal(oracle.allreduce(rev, dtype, "max")[0], mx)


def test_signed_zero_tie_keeps_earlier_rank():
    pz = np.array([0.0], np.float32)
    nz = np.array([-0.0], np.float32)
    assert not np.signbit(oracle.allreduce([pz, nz], "f32", "min")[0][0])
    assert np.signbit(oracle.allreduce([nz, pz], "f32", "min")[0][0])
    assert not np.signbit(oracle.allreduce([pz, nz], "f32", "max")[0][0])
    assert np.signbit(oracle.allreduce([nz, pz], "f32", "max")[0][0])


def test_negative_control_rank_order_matters_for_f32_sum():
    p, n = 8, 4096
    xs = datagen.rank_buffers("uniform_f32", 2, p, n)
    out = oracle.allreduce(xs, "f32", "sum")[0]
    asc = xs[0].copy()
    for x in xs[1:]:
        asc = (asc + x).astype(np.float32)
    rev = xs[-1].copy()
    for x in xs[-2::-1]:
        rev = (rev + x).astype(np.float32)
    assert np.array_equal(out, asc)
    assert np.count_nonzero(out != rev) > n // 20


@pytest.mark.parametrize("dtype,kind", [("f32", "uniform_f32"), ("bf16", "normal_bf16"),
                                        ("i32", "int32")])
def test_all_allreduce_outputs_identical(dtype, kind):
    xs = datagen.rank_buffers(kind, 5, 6, 777)
    outs = oracle.allreduce(xs, dtype, "sum")
    for o in outs[1:]:
        assert same_bits(o, outs[0])


@pytest.mark.parametrize("dtype,kind", [("f32", "uniform_f32"), ("bf16", "normal_bf16"),
                                        ("i32", "int32")])
@pytest.mark.parametrize("p", [1, 2, 4, 8])
def test_reduce_scatter_then_allgather_equals_allreduce(dtype, kind, p):
    rc = 1001
    xs = datagen.rank_buffers(kind, 1, p, p * rc)
    ar = oracle.allreduce(xs, dtype, "sum")
    rs = oracle.reduce_scatter(xs, dtype, "sum")
    ag = oracle.allgather(rs)
    for r in range(p):
        assert same_bits(ag[r], ar[r])


@pytest.mark.parametrize("dtype,kind", [("f32", "uniform_f32"), ("bf16", "normal_bf16"),
                                        ("i32", "int32")])
def test_p1_is_a_copy(dtype, kind):
    x = datagen.rank_buffers(kind, 3, 1, 1234)
    assert same_bits(oracle.allreduce(x, dtype, "sum")[0], x[0])
    assert same_bits(oracle.reduce_scatter(x, dtype, "sum")[0], x[0])
    assert same_bits(oracle.allgather(x)[0], x[0])


def test_in_place_equals_out_of_place():
    p, n = 4, 1000
    xs = datagen.rank_buffers("uniform_f32", 9, p, n)
    ref = oracle.allreduce(xs, "f32", "sum")
    buf = [x.copy() for x in xs]
    ptrs = [b.ctypes.data for b in buf]
    oracle.allreduce_ptrs("f32", "sum", p, n, ptrs, ptrs)
    for r in range(p):
        assert same_bits(buf[r], ref[r])
    # reduce-scatter in place: recv[r] = send[r] + r * rc elements
    rc = 250
    rs_ref = oracle.reduce_scatter(xs, "f32", "sum")
    buf = [x.copy() for x in xs]
    oracle.reduce_scatter_ptrs("f32", "sum", p, rc, [b.ctypes.data for b in buf],
                               [b.ctypes.data + r * rc * 4 for r, b in enumerate(buf)])
    for r in range(p):
        assert same_bits(buf[r][r * rc:(r + 1) * rc], rs_ref[r])
    # all-gather in place: send[r] = recv[r] + r * sc elements
    sc = 250
    parts = [x[:sc].copy() for x in xs]
    ag_ref = oracle.allgather(parts)
    recv = [np.zeros(p * sc, np.float32) for _ in range(p)]
    for r in range(p):
        recv[r][r * sc:(r + 1) * sc] = parts[r]
    oracle.allgather_ptrs(4, p, sc, [b.ctypes.data + r * sc * 4 for r, b in enumerate(recv)],
                          [b.ctypes.data for b in recv])
    for r in range(p):
        assert same_bits(recv[r], ag_ref[r])


@pytest.mark.parametrize("dtype,kind", [("f32", "uniform_f32"), ("bf16", "normal_bf16")])
def test_threaded_variant_same_bits(dtype, kind):
    p, n = 8, 200_003
    xs = datagen.rank_buffers(kind, 0, p, n)
    a = oracle.allreduce(xs, dtype, "sum", nthreads=1)
    b = oracle.allreduce(xs, dtype, "sum", nthreads=6)
    for r in range(p):
        assert same_bits(a[r], b[r])
    rs1 = oracle.reduce_scatter([x[: (n // p) * p] for x in xs], dtype, "sum", nthreads=1)
    rs2 = oracle.reduce_scatter([x[: (n // p) * p] for x in xs], dtype, "sum", nthreads=5)
    for r in range(p):
        assert same_bits(rs1[r], rs2[r])
    ag1 = oracle.allgather(rs1, nthreads=1)
    ag2 = oracle.allgather(rs1, nthreads=3)
    for r in range(p):
        assert same_bits(ag1[r], ag2[r])


def test_rejects_bad_arguments():
    x = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle.allreduce_ptrs(7, "sum", 1, 4, [x.ctypes.data], [x.ctypes.data])
    with pytest.raises(ValueError):
        oracle.allreduce_ptrs("f32", 9, 1, 4, [x.ctypes.data], [x.ctypes.data])
    with pytest.raises(ValueError):
        oracle.allreduce_ptrs("f32", "sum", 0, 4, [], [])
    with pytest.raises(ValueError):
        oracle.allreduce_ptrs("f32", "sum", 1, 4, [0], [x.ctypes.data])
