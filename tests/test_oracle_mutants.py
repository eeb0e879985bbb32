"""Plant plausible mistakes in copies of the CPU oracle and check that the pins
catch every one of them (no GPU). The oracle source itself is not changed: each
mutant is a patched copy built in a temporary directory."""
import importlib.util
import os
import shutil

import numpy as np
import pytest

import oracle as oracle_pkg
from oracle_pins import (check_bf16_rounding, check_bruteforce, check_combine_all,
                         check_hand_example, check_hand_example_aligned,
                         check_hand_example_rank3, check_invariants, check_view_against_reference,
                         check_e4m3_rounding, check_lowlatency_hand, check_lowlatency_cast_exact,
                         check_lowlatency_against_exact_layout)

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "epd_oracle.c")

MUTANTS = {
    "inclusive_scan": ("expert_start_loc[e] = (int32_t)run;\n        run += tokens_per_expert[e];",
                       "run += tokens_per_expert[e];\n        expert_start_loc[e] = (int32_t)run;"),
    "interleaved_ranks": ("return (int)(e / (E / R));", "return (int)(e % R);"),
    "interleaved_nodes": ("return r / (R / N);", "return r % N;"),
    "pairs_not_tokens": ("in_rank = 1;", "in_rank += 1;"),
    "dropped_fill_increment": ("fill_count[e] += 1;", "", 0),
    "dropped_fill_increment_view": ("fill_count[e] += 1;", "", 1),
    "m_indices_wrong_operand": ("m_indices[s] = (int32_t)e;", "m_indices[s] = (int32_t)t;"),
    "unfilled_rows_not_cleared": ("for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;", "",
                                  0),
    "first_row_not_cleared": ("for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;",
                              "for (int64_t s = 1; s < capacity; ++s) m_indices[s] = -1;", 0),
    "unfilled_rows_not_cleared_view": (
        "for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;", "", 1),
    "alignment_rounds_down": ("run += (c + alignment - 1) / alignment * alignment;",
                              "run += c / alignment * alignment;"),
    "view_global_ids": ("m_indices[s] = (int32_t)(e - e_begin);", "m_indices[s] = (int32_t)e;"),
    "view_base_not_subtracted": ("int64_t s = (int64_t)expert_start_loc[e] - base + fill_count[e];",
                                 "int64_t s = (int64_t)expert_start_loc[e] + fill_count[e];"),
    "scale_col_major_swapped": ("if (scale_col_major) out_scale[(int64_t)c * scale_ld + s] = v;",
                                "if (scale_col_major) out_scale[s * scale_ld + c] = v;"),
    "view_range_off_by_one": ("if (e < e_begin || e >= e_end) {", "if (e < e_begin || e > e_end) {"),
    "e4m3_truncates": ("double r = nearbyint(a / spacing) * spacing;",
                       "double r = floor(a / spacing) * spacing;"),
    "e4m3_no_saturation": ("if (r > 448.0) r = 448.0;         /* saturate */", ""),
    "cast_scale_not_divided": ("float scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
                               "float scale = amax > 0.0f ? amax : 1.0f;"),
    "cast_amax_signed": ("float v = fabsf((float)oracle_double_from_bf16(x[(int64_t)t * H + h]));",
                         "float v = (float)oracle_double_from_bf16(x[(int64_t)t * H + h]);"),
    "rectangle_overflow_kept": ("if (r >= rows_per_expert) {", "if (r > rows_per_expert) {"),
    "rectangle_scale_row_major": (
        "out_scale[((e - e_begin) * (int64_t)C + c) * rows_per_expert + r] = scale;",
        "out_scale[((e - e_begin) * rows_per_expert + r) * (int64_t)C + c] = scale;"),
    "alignment_ignored": ("run += (c + alignment - 1) / alignment * alignment;", "run += c;"),
    "weight_wrong_index": ("acc += (double)topk_weights[(int64_t)t * k + j] *",
                           "acc += (double)topk_weights[(int64_t)t * k] *"),
    "combine_wrong_sign": ("acc += (double)topk_weights", "acc -= (double)topk_weights"),
    "combine_skips_slot0": ("if (s < 0) continue;", "if (s <= 0) continue;"),
    "rounding_truncates": ("double rounded = nearbyint(scaled);", "double rounded = floor(scaled);"),
    "rounding_ties_away": ("double rounded = nearbyint(scaled);", "double rounded = round(scaled);"),
    "per_node_unset": ("if (e >= 0 && node_of_rank(rank_of_expert(e, E, R), R, N) == n) in_node = 1;",
                       "if (e > 0 && node_of_rank(rank_of_expert(e, E, R), R, N) == n) in_node = 1;"),
}


def _mutate(src, before, after, which):
    """Replace occurrence `which` (0-based) of `before`; `which` None needs it unique."""
    n = src.count(before)
    if which is None:
        assert n == 1, f"mutation site not unique ({n})"
        return src.replace(before, after)
    assert n > which, f"mutation site {which} missing ({n})"
    i = -1
    for _ in range(which + 1):
        i = src.index(before, i + 1)
    return src[:i] + after + src[i + len(before):]


def _load_mutant(tmp_path, name):
    spec = MUTANTS[name]
    before, after = spec[0], spec[1]
    which = spec[2] if len(spec) > 2 else None
    src = open(SRC).read()
    d = tmp_path / name
    (d / "_build").mkdir(parents=True)
    (d / "epd_oracle.c").write_text(_mutate(src, before, after, which))
    shutil.copy(oracle_pkg.__file__, d / "__init__.py")
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}", d / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _run_pins(orc):
    check_hand_example(orc)
    check_hand_example_aligned(orc)
    check_bruteforce(orc, 2, 2, 4, 2, 1, limit=2000, alignment=4)
    check_hand_example_rank3(orc)
    check_e4m3_rounding(orc, n=2000)
    check_lowlatency_hand(orc)
    check_lowlatency_cast_exact(orc)
    t = np.array([[3, 7], [3, 1], [0, 15], [7, 6], [7, 3]], np.int64)
    check_lowlatency_against_exact_layout(orc, t, 16, 2, 0, 16, seed=5)
    for flat in [(0, 3, 1, 2, -1, 3), (3, 3, 2, 1, 0, 0), (1, 2, 2, 3, 3, -1)]:
        t = np.array(flat, np.int64).reshape(3, 2)
        check_view_against_reference(orc, t, 4, 1, 4, 1, True)
        check_view_against_reference(orc, t, 4, 2, 3, 1, False)
    check_bruteforce(orc, 3, 2, 4, 2, 1, limit=3000)
    check_bruteforce(orc, 2, 2, 4, 4, 2, limit=3000)
    rng = np.random.default_rng(0)
    topk = rng.integers(-1, 32, size=(50, 6)).astype(np.int64)
    check_invariants(orc, topk, 32, 8, 2)
    check_combine_all(orc)
    check_bf16_rounding(orc, n=4000)


def test_unmutated_copy_passes(tmp_path):
    d = tmp_path / "clean"
    (d / "_build").mkdir(parents=True)
    shutil.copy(SRC, d / "epd_oracle.c")
    shutil.copy(oracle_pkg.__file__, d / "__init__.py")
    spec = importlib.util.spec_from_file_location("oracle_clean_copy", d / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    _run_pins(mod)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    mod = _load_mutant(tmp_path, name)
    with pytest.raises((AssertionError, mod.OracleError)):
        _run_pins(mod)
