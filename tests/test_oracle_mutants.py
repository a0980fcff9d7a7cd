"""Planted mistakes: every plausible slip in the oracle must fail a pin.

Each case copies oracle.c, plants one mistake (a dropped term, a wrong sign,
index or operand), builds it in a temporary directory and runs the oracle pin
suites against that build in a child process.  The suites must fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "carried_sum_sign": ("sum += row_sum;", "sum -= row_sum;"),
    "initial_dropped": ("double sum = initial;", "double sum = 0.0;"),
    "tile_row_index": ("int64_t source_row = row + t;", "int64_t source_row = t;"),
    "split_advance": ("while (remaining >= tile_size) {\n        row += tile_size;",
                      "while (remaining >= tile_size) {\n        row += tile_size - 1;"),
    "tile_advance": ("        }\n        row += tile_size;", "        }\n        row += tile_size - 1;"),
    "tail_start": ("tail += row_across_lanes(values + r * lanes, lanes);",
                   "tail += row_across_lanes(values + (r - row) * lanes, lanes);"),
    "tail_last_row_dropped": ("for (int64_t r = row; r < row + remaining; ++r)",
                              "for (int64_t r = row; r + 1 < row + remaining; ++r)"),
    "lane_index": ("s += (double)row[lane];", "s += (double)row[0];"),
    "column_sum_index": ("sum += (double)values[row * lanes + lane];",
                         "sum += (double)values[row * lanes];"),
    "no_sign_extension": ("out[j] = byte >= 128 ? byte - 256 : byte;", "out[j] = byte;"),
    "big_endian_unpack": ("(word >> (8 * j))", "(word >> (8 * (3 - j)))"),
    "dot_operand_reversed": ("(int64_t)x[b * k + kk]", "(int64_t)x[b * k + (k - 1 - kk)]"),
    "dot_vector_scale": ("(double)scale_x[b]", "(double)scale_x[0]"),
    "ceil_division": ("(element_count + workgroup_size - 1)", "(element_count + workgroup_size)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation site for {name} not unique in oracle.c"
    src = tmp_path / "oracle.c"
    src.write_text(text.replace(before, after))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(lib), str(src)])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_rowsum.py"),
                        os.path.join(ROOT, "tests", "test_oracle_dot.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
