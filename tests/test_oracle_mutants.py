"""The oracle's pins catch plausible mistakes.

Each case below plants one mistake in a copy of ``oracle/oracle.c`` (a
dropped term, a wrong order, sign, index or rounding), builds that copy on the
CPU, points the oracle module at it and runs the pin checks of
``test_oracle.py``. Every planted mistake must fail at least one pin.
"""
import subprocess
from pathlib import Path

import pytest

import oracle
import test_oracle as pins

SRC = Path(oracle.__file__).resolve().parent / "oracle.c"

MUTANTS = {
    "drop_last_rank_f32": (
        "for (int r = 1; r < nranks; ++r) acc = or_fold_f32(op, acc, ((const float*)send[r])[si]);",
        "for (int r = 1; r < nranks - 1; ++r) acc = or_fold_f32(op, acc, ((const float*)send[r])[si]);"),
    "descending_rank_order_f32": (
        "float acc = ((const float*)send[0])[si];\n"
        "    for (int r = 1; r < nranks; ++r) acc = or_fold_f32(op, acc, ((const float*)send[r])[si]);",
        "float acc = ((const float*)send[nranks - 1])[si];\n"
        "    for (int r = nranks - 2; r >= 0; --r) acc = or_fold_f32(op, acc, ((const float*)send[r])[si]);"),
    "bf16_truncates": ("u = u + 0x7FFFu + keep_lsb;", "u = u;"),
    "bf16_round_half_up": ("u = u + 0x7FFFu + keep_lsb;", "u = u + 0x8000u;"),
    "bf16_rounds_every_step": (
        "acc = or_fold_f32(op, acc, or_bf16_widen(((const uint16_t*)send[r])[si]));",
        "acc = or_bf16_widen(or_bf16_round(or_fold_f32(op, acc, or_bf16_widen(((const uint16_t*)send[r])[si]))));"),
    "bf16_widen_shift": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    "min_computes_max": ("case OR_MIN: return (x < acc) ? x : acc;\n    default: return (x > acc) ? x : acc;\n  }\n}\n\nstatic int32_t",
                         "case OR_MIN: return (x > acc) ? x : acc;\n    default: return (x > acc) ? x : acc;\n  }\n}\n\nstatic int32_t"),
    "min_tie_takes_later_rank": ("case OR_MIN: return (x < acc) ? x : acc;\n    default: return (x > acc) ? x : acc;\n  }\n}\n\nstatic int32_t",
                                 "case OR_MIN: return (x <= acc) ? x : acc;\n    default: return (x > acc) ? x : acc;\n  }\n}\n\nstatic int32_t"),
    "i32_sum_wrong_sign": ("(uint32_t)acc + (uint32_t)x", "(uint32_t)acc - (uint32_t)x"),
    "rs_index_transposed": ("(uint64_t)s * recvcount + j, recv[s], j",
                            "(uint64_t)j * nranks + s, recv[s], j"),
    "rs_wrong_destination": ("(uint64_t)s * recvcount + j, recv[s], j",
                             "(uint64_t)s * recvcount + j, recv[nranks - 1 - s], j"),
    "ag_block_index_transposed": ("((uint64_t)k * sendcount + j) * (uint64_t)elem_size",
                                  "((uint64_t)r * sendcount + j) * (uint64_t)elem_size"),
    "ar_writes_rank0_only": ("for (int r = 0; r < nranks; ++r) memcpy(",
                             "for (int r = 0; r < 1; ++r) memcpy("),
    "threaded_ranges_leave_gaps": (
        "jobs[t].end = proto.n * (uint64_t)(t + 1) / (uint64_t)nthreads;",
        "jobs[t].end = proto.n * (uint64_t)(t + 1) / (uint64_t)nthreads - (t + 1 < nthreads ? 1 : 0);"),
}


def _checks():
    c = []
    for dt in ("f32", "bf16", "i32"):
        for op in ("sum", "min", "max"):
            c.append(lambda dt=dt, op=op: pins.test_allreduce_brute_force(dt, op, 3))
            c.append(lambda dt=dt, op=op: pins.test_allreduce_brute_force(dt, op, 8))
        c.append(lambda dt=dt: pins.test_reduce_scatter_brute_force(dt, "sum", 3))
    c += [
        lambda: pins.test_allgather_brute_force(pins.np.float32, 3),
        lambda: pins.test_f32_integer_valued_sum_is_exact(8),
        lambda: pins.test_p_copies_sum_to_p_times(8, "bf16"),
        pins.test_bf16_rounds_once_not_per_step,
        pins.test_bf16_round_half_to_even,
        pins.test_bf16_identity_on_every_finite_pattern,
        pins.test_bf16_rounding_matches_rational_rounding,
        pins.test_int32_sum_wraps_and_is_order_free,
        lambda: pins.test_min_max_equal_library_extrema_any_order("f32"),
        pins.test_signed_zero_tie_keeps_earlier_rank,
        pins.test_negative_control_rank_order_matters_for_f32_sum,
        lambda: pins.test_reduce_scatter_then_allgather_equals_allreduce("f32", "uniform_f32", 4),
        pins.test_in_place_equals_out_of_place,
        lambda: pins.test_threaded_variant_same_bits("f32", "uniform_f32"),
    ]
    return c


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    text = SRC.read_text()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "oracle_mut.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-fno-fast-math", "-ffp-contract=off", "-o", str(lib), str(src)])
    failed = 0
    oracle.use_library(lib)
    try:
        for check in _checks():
            try:
                check()
            except (AssertionError, ValueError):
                failed += 1
    finally:
        oracle.use_library(None)
    assert failed >= 1, f"planted mistake {name} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = tmp_path / "liboracle_copy.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-fno-fast-math", "-ffp-contract=off", "-o", str(lib), str(SRC)])
    oracle.use_library(lib)
    try:
        for check in _checks():
            check()
    finally:
        oracle.use_library(None)
