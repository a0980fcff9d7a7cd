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
    "f16_exponent_bias": ("ldexpf((float)(m + 1024), e - 25)", "ldexpf((float)(m + 1024), e - 24)"),
    "f16_subnormal_hidden_bit": ("v = ldexpf((float)m, -24);", "v = ldexpf((float)(m + 1024), -24);"),
    "packed_unfused_step": ("sum = fmaf(scaled, a[j], sum);", "sum = sum + scaled * a[j];"),
    "packed_stream_map": ("l % streams) * 4", "(l + 1) % streams) * 4"),
    "packed_scale_lane": ("oracle_f16_to_f32(scales[at])", "oracle_f16_to_f32(scales[at - l])"),
    "packed_last_record_dropped": ("for (int64_t r = 0; r < count; ++r) {\n                const int64_t at",
                                   "for (int64_t r = 0; r + 1 < count; ++r) {\n                const int64_t at"),
    "packed_initial_dropped": ("float sum = initial ? initial[p * lanes + l] : 0.0f;", "float sum = 0.0f;"),
    "packed_element_order": ("sum = fmaf(scaled, a[j], sum);",
                             "sum = fmaf((float)ints[3 - j] * scale, a[3 - j], sum);"),
    "lane_sum_row_order": ("sum = sum + seg[(row * lanes + lane) * width + j];",
                           "sum = sum + seg[((count - 1 - row) * lanes + lane) * width + j];"),
    "lane_sum_element_order": ("sum = sum + seg[(row * lanes + lane) * width + j];",
                               "sum = sum + seg[(row * lanes + lane) * width + (width - 1 - j)];"),
    "lane_sum_lane_index": ("sum = sum + seg[(row * lanes + lane) * width + j];",
                            "sum = sum + seg[(row * lanes + 0) * width + j];"),
    "lane_sum_last_row_dropped": ("for (int64_t row = 0; row < count; ++row)\n                for (int64_t j = 0;",
                                  "for (int64_t row = 0; row + 1 < count; ++row)\n                for (int64_t j = 0;"),
    "guarded_reads_past_count": ("                if (row < count) {\n                    float component_sum",
                                 "                if (row < end) {\n                    float component_sum"),
    "guarded_column_bound": ("for (int64_t column = 0; column < columns; ++column)",
                             "for (int64_t column = 0; column <= columns && column < 4; ++column)"),
    "guarded_active_bound": ("lane < active_lanes ? seg", "lane <= active_lanes ? seg"),
    "guarded_row_order": ("? seg[(row * lanes + lane) * 4 + column]", "? seg[((count - 1 - row) * lanes + lane) * 4 + column]"),
    "routed_missing_not_skipped": ("            if (id < 0)\n                continue;   // a missing route",
                                   "            if (id < -1000)\n                continue;   // a missing route"),
    "routed_fused_step": ("                const float weighted = w * row[h];\n                out[t * width + h] = out[t * width + h] + weighted;",
                          "                out[t * width + h] = fmaf(w, row[h], out[t * width + h]);"),
    "routed_route_order": ("const int32_t id = ids[t * routes + r];", "const int32_t id = ids[t * routes + (routes - 1 - r)];"),
    "routed_weight_index": ("const float w = weights[t * routes + r];", "const float w = weights[t * routes];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation site for {name} not unique in oracle.c"
    src = tmp_path / "oracle.c"
    src.write_text(text.replace(before, after))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-o", str(lib), str(src), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_rowsum.py"),
                        os.path.join(ROOT, "tests", "test_oracle_dot.py"),
                        os.path.join(ROOT, "tests", "test_oracle_packed_dot.py"),
                        os.path.join(ROOT, "tests", "test_oracle_lane_sums.py"),
                        os.path.join(ROOT, "tests", "test_oracle_routed.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
