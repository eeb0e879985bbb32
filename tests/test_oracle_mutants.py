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
                         check_hand_example, check_hand_example_aligned, check_invariants)

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "epd_oracle.c")

MUTANTS = {
    "inclusive_scan": ("expert_start_loc[e] = (int32_t)run;\n        run += tokens_per_expert[e];",
                       "run += tokens_per_expert[e];\n        expert_start_loc[e] = (int32_t)run;"),
    "interleaved_ranks": ("return (int)(e / (E / R));", "return (int)(e % R);"),
    "interleaved_nodes": ("return r / (R / N);", "return r % N;"),
    "pairs_not_tokens": ("in_rank = 1;", "in_rank += 1;"),
    "dropped_fill_increment": ("fill_count[e] += 1;", ""),
    "m_indices_wrong_operand": ("m_indices[s] = (int32_t)e;", "m_indices[s] = (int32_t)t;"),
    "unfilled_rows_not_cleared": ("for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;", ""),
    "first_row_not_cleared": ("for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;",
                              "for (int64_t s = 1; s < capacity; ++s) m_indices[s] = -1;"),
    "alignment_rounds_down": ("run += (c + alignment - 1) / alignment * alignment;",
                              "run += c / alignment * alignment;"),
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


def _load_mutant(tmp_path, name):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not unique"
    d = tmp_path / name
    (d / "_build").mkdir(parents=True)
    (d / "epd_oracle.c").write_text(src.replace(before, after))
    shutil.copy(oracle_pkg.__file__, d / "__init__.py")
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}", d / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _run_pins(orc):
    check_hand_example(orc)
    check_hand_example_aligned(orc)
    check_bruteforce(orc, 2, 2, 4, 2, 1, limit=2000, alignment=4)
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
