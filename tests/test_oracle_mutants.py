"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of oracle.c (on the CPU), builds it, and requires that at
least one pin from test_oracle.py fails against the mutant."""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "wrong_sign": ("acc[i] += p;", "acc[i] -= p;"),
    "dropped_x_factor": ("double p = a * xj;", "double p = a;"),
    "transposed_index": ("A->row_idx[dst] = i;", "A->row_idx[dst] = j;"),
    "zero_x_active": ("if (x_val && !(x_val[e] != 0.0f)) continue;      /* inactive entry */", ""),
    "visited_ignored": ("if (semiring == 1 && visited && visited[i]) continue;\n        y_idx[t] = (int32_t)i;\n        if (semiring == 0) {\n            if (y_val) y_val[t] = acc[i];",
                        "y_idx[t] = (int32_t)i;\n        if (semiring == 0) {\n            if (y_val) y_val[t] = acc[i];"),
    "bfs_level_off_by_one": ("levels[i] = levels[u] + 1;", "levels[i] = levels[u] + 2;"),
    "th0_not_strict": ("if (z < th0) cls = 0;", "if (z <= th0) cls = 0;"),
    "th1_not_strict": ("else if (z > th1) cls = 1;", "else if (z >= th1) cls = 1;"),
    "force_classes_swapped": ("if (skew_r / skew_c > th2) cls = 3;", "if (skew_r / skew_c > th2) cls = 2;"),
    "csc2csr_wrong": ("blk_csc2csr[q] = p;", "blk_csc2csr[q] = q;"),
    "abs_sum_signed": ("sab[i] += fabs(p);", "sab[i] += p;"),
    "threshold_inclusive": ("if (!(a <= (double)tau)) idx_out[k++]", "if (a >= (double)tau) idx_out[k++]"),
    "spmv_row_index_for_column": ("double p = (double)vals[k] * (double)x[j];", "double p = (double)vals[k] * (double)x[i];"),
    "spmv_abs_signed": ("            sab += fabs(p);\n        }\n        y[i] = acc;", "            sab += p;\n        }\n        y[i] = acc;"),
}

PIN_FUNCS = [
    lambda: [pins.test_push_matches_dense_brute_force(s, sr) for s in range(4) for sr in (0, 1)],
    lambda: [pins.test_integer_values_are_exact(s) for s in range(2)],
    pins.test_unit_vector_returns_column,
    pins.test_activity_rules,
    pins.test_bfs_grid_is_manhattan_distance,
    lambda: [pins.test_block_views_match_figure5(bs) for bs in (4, 16)],
    pins.test_format_classes_by_density,
    pins.test_format_classes_by_skew,
    pins.test_activation_mask_rule,
    lambda: [pins.test_decode_layer_matches_dense_brute_force(s) for s in range(3)],
    lambda: [pins.test_spmv_csr_matches_dense_brute_force(s) for s in range(3)],
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-w", "-o", str(lib),
                           str(mutated), "-lm"])
    caught = 0
    with oracle.use_library(str(lib)):
        for f in PIN_FUNCS:
            try:
                f()
            except (AssertionError, RuntimeError):
                caught += 1
    assert caught > 0, f"mutant {name} survived every pin"
