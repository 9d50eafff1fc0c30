"""Planted mistakes in the oracle (on the CPU): each mutant of oracle.c is a
plausible error -- a dropped term, a wrong seed, order, sign, index or
rounding rule, a swapped operand -- compiled on its own, and run through a
battery of the pins.  At least one pin must reject every mutant, and the
unmodified oracle must pass all of them."""
import os
import shutil

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text to replace in oracle.c, replacement)
MUTANTS = [
    ("seed_with_zero",
     "  float acc = load_elem((const uint8_t*)x[0] + i * es, dtype);\n  for (int r = 1; r < W; r++)",
     "  float acc = 0.0f;\n  for (int r = 0; r < W; r++)"),
    ("drop_last_rank", "  for (int r = 1; r < W; r++) acc = acc + load_elem((const uint8_t*)x[r] + i * es, dtype);",
     "  for (int r = 1; r < W - 1; r++) acc = acc + load_elem((const uint8_t*)x[r] + i * es, dtype);"),
    ("reverse_rank_order",
     "  float acc = load_elem((const uint8_t*)x[0] + i * es, dtype);\n  for (int r = 1; r < W; r++) acc = acc + load_elem((const uint8_t*)x[r] + i * es, dtype);",
     "  float acc = load_elem((const uint8_t*)x[W - 1] + i * es, dtype);\n  for (int r = W - 2; r >= 0; r--) acc = acc + load_elem((const uint8_t*)x[r] + i * es, dtype);"),
    ("truncate_instead_of_rne", "    if (rem > half || (rem == half && (kept & 1ull))) kept += 1;", "    (void)half;"),
    ("ties_away_from_zero", "    if (rem > half || (rem == half && (kept & 1ull))) kept += 1;", "    if (rem >= half) kept += 1;"),
    ("flush_subnormals", "  return sbit | (uint32_t)kept;                             /* subnormal               */",
     "  return sbit;"),
    ("sum_of_squares_not_mean", "    const double rms = 1.0 / sqrt(ss / (double)N + (double)eps);",
     "    const double rms = 1.0 / sqrt(ss + (double)eps);"),
    ("eps_outside_sqrt", "    const double rms = 1.0 / sqrt(ss / (double)N + (double)eps);",
     "    const double rms = 1.0 / sqrt(ss / (double)N) + (double)eps;"),
    ("weight_from_residual",
     "      const double w = (double)load_elem((const uint8_t*)weight + j * es, dtype);",
     "      const double w = (double)load_elem((const uint8_t*)residual + j * es, dtype);"),
    ("h_from_rounded_sum",
     "      const float h = acc + load_elem((const uint8_t*)residual + i * es, dtype);\n      if (ar)",
     "      const float h = orc_bf16_to_f32(orc_f32_to_bf16(acc)) + load_elem((const uint8_t*)residual + i * es, dtype);\n      if (ar)"),
    ("ll128_flag_first_word", "    st64(line + 120, flag);", "    memmove(line + 8, line, 112);\n    st64(line, flag);"),
    ("ll128_checks_word_14", "      const uint64_t flag = ld64((const uint8_t*)wires[r] + 128 * k + 8 * 15);",
     "      const uint64_t flag = ld64((const uint8_t*)wires[r] + 128 * k + 8 * 14);"),
    ("ll_data_and_flag_swapped", "    st32(line + 0, (uint32_t)d);          /* data1 */\n    st32(line + 4, flag);                 /* flag1 */",
     "    st32(line + 4, (uint32_t)d);          /* data1 */\n    st32(line + 0, flag);                 /* flag1 */"),
    ("ll_ignores_flag2", "      if (flag1 != expected_flag || flag2 != expected_flag) {", "      if (flag1 != expected_flag) {"),
    ("stale_line_not_zeroed", "      if (!line_ok) { memset(out, 0, (size_t)es); continue; }\n      const int64_t wire_off",
     "      const int64_t wire_off"),
    ("two_shot_no_rotation", "      const int r = (int)((owner + k) % W);", "      const int r = k;"),
    ("two_shot_no_remainder_owner", "    if (owner > W - 1) owner = W - 1;  /* the last rank takes the remainder */",
     "    if (owner > W - 1) owner = 0;"),
    ("lamport_no_scrub", "    if (v == 0x8000u) v = 0;  /* scrub -0.0 */", "    (void)0;"),
    ("lamport_reads_next_region", "  const uint8_t* region = base + (int64_t)(round % 3) * region_bytes;",
     "  const uint8_t* region = base + (int64_t)((round + 1) % 3) * region_bytes;"),
    ("lamport_refills_next_region", "  orc_lamport_fill(base + (int64_t)((round + 2) % 3) * region_bytes, region_bytes / 4);",
     "  orc_lamport_fill(base + (int64_t)((round + 1) % 3) * region_bytes, region_bytes / 4);"),
    ("lamport_stale_row_not_zeroed", "      memset((uint8_t*)residual_out + 2 * m * N, 0, (size_t)(2 * N));", ""),
    ("lamport_checks_first_word_only", "      for (int64_t j = 0; j < N; j += 2) {", "      for (int64_t j = 0; j < 2; j += 2) {"),
]


def battery(orc):
    """(name, callable) pins that are cheap enough to run once per mutant."""
    return [
        ("negative_zero_seed", lambda: pins.test_reduce_negative_zero_seed(orc)),
        ("identical_ranks", lambda: pins.test_reduce_identical_ranks_is_W_times_x(orc, "bf16", 3)),
        ("rank_order", lambda: pins.test_reduce_is_sequential_fp32_adds_in_rank_order(orc, "fp32")),
        ("subnormals", lambda: pins.test_reduce_keeps_subnormals(orc)),
        ("f32_to_bf16", lambda: pins.test_f32_to_bf16_every_rounding_class(orc)),
        ("f64_to_f16", lambda: pins.test_f64_narrowing(orc, "fp16")),
        ("textbook_rmsnorm", lambda: pins.test_fused_zero_x_is_textbook_rmsnorm(orc, "bf16")),
        ("constant_row", lambda: pins.test_fused_constant_row_normalises_to_sign_times_weight(orc, 0.375)),
        ("single_column", lambda: pins.test_fused_single_column(orc)),
        ("unrounded_sum", lambda: pins.test_fused_residual_uses_unrounded_sum(orc)),
        ("buffer_table", lambda: pins.test_protocol_buffer_table(orc)),
        ("ll128_golden", lambda: pins.test_ll128_golden_lines(orc)),
        ("ll_golden", lambda: pins.test_ll_golden_line(orc)),
        ("single_stale_ll128", lambda: pins.test_each_single_stale_line_detected_alone(orc, "ll128")),
        ("single_stale_ll", lambda: pins.test_each_single_stale_line_detected_alone(orc, "ll")),
        ("ll_flag2", lambda: pins.test_ll_second_flag_alone_is_checked(orc)),
        ("two_shot_rotation", lambda: pins.test_two_shot_is_rotated_one_shot_per_shard(orc, 5, 23)),
        ("lamport_push_brute_force", lambda: pins.test_lamport_push_never_writes_the_sentinel(orc)),
        ("lamport_round", lambda: pins.test_lamport_round_equals_fused_op_on_scrubbed_inputs(orc)),
        ("lamport_missing_word", lambda: pins.test_lamport_missing_word_makes_its_row_stale(orc, (1, 2, 128))),
    ]


def run_battery(orc):
    failed = []
    for name, fn in battery(orc):
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unmodified_oracle_passes_the_battery():
    assert run_battery(oracle.default()) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_each_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / f"oracle_{name}.c"
    mutant.write_text(src.replace(old, new))
    shutil.copy(os.path.join(os.path.dirname(SRC), "oracle.h"), tmp_path / "oracle.h")
    lib = oracle.build(force=True, src=str(mutant), out=str(tmp_path / f"lib_{name}.so"))
    caught = run_battery(oracle.Oracle(lib))
    assert caught, f"no pin rejects the mutant {name}"
