"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/lora_oracle.c (a dropped
term, a wrong sign, index, offset or operand, an unstable sort, a missed
special case), builds it with the oracle's own flags, and runs the pin
modules (tests/test_oracle_meta.py, tests/test_oracle_shrink_expand.py) in a
child process bound to that build: at least one pin must fail.  The
unaltered source, built the same way, must pass them all.  Every planted
mistake keeps its reads and writes inside the buffers it is given.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lora_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_meta.py"),
        os.path.join(ROOT, "tests", "test_oracle_shrink_expand.py")]

# (name, text in lora_oracle.c, replacement)
MUTANTS = [
    # bf16 widening
    ("widen_shift", "uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    # metadata
    ("meta_unstable_sort", "sorted_idx[bin_start[b] + seen[b]] = (int32_t)t;",
     "sorted_idx[bin_start[b] + (bin_count[b] - 1 - seen[b])] = (int32_t)t;"),
    ("meta_cumsum_shifted", "start_loc[k + 1] = (int32_t)acc;", "start_loc[k] = (int32_t)acc;"),
    ("meta_empty_not_no_lora", "if (bin_count[0] == T) {", "if (bin_count[0] == T && T > 0) {"),
    ("meta_active_id_off_by_one", "active_ids[n_active] = k - 1;", "active_ids[n_active] = k;"),
    ("meta_minus_one_not_listed", "if (bin_count[k] > 0) {", "if (k > 0 && bin_count[k] > 0) {"),
    ("meta_invalid_not_counted", "++invalid;", ";"),
    ("meta_copy_sanitised", "mapping_copy[t] = map[t];",
     "mapping_copy[t] = valid_id(map[t], num_loras) ? map[t] : -1;"),
    # shrink
    ("shrink_scale_dropped", "v += scale * dot;", "v += dot;"),
    ("shrink_overwrites", "double v = (double)buf_in[o];", "double v = 0.0;"),
    ("shrink_first_slice_only", "const uint16_t *arow = A[s] + ((int64_t)id * r + i) * H;",
     "const uint16_t *arow = A[0] + ((int64_t)id * r + i) * H;"),
    ("shrink_rank_rows_reversed", "const uint16_t *arow = A[s] + ((int64_t)id * r + i) * H;",
     "const uint16_t *arow = A[s] + ((int64_t)id * r + (r - 1 - i)) * H;"),
    ("shrink_row_stride_ignored", "const uint16_t *xrow = x + t * x_ld;",
     "const uint16_t *xrow = x + t * H;"),
    # expand
    ("expand_b_transposed", "v += (double)xrow[k] * bf16_to_f64(brow[k]);",
     "v += (double)xrow[k] * bf16_to_f64(B[s][(int64_t)id * n * r + (int64_t)k * n + j]);"),
    ("expand_x_first_slice", "const float *xrow = xin + ((int64_t)s * T + t) * r;",
     "const float *xrow = xin + ((int64_t)0 * T + t) * r;"),
    ("expand_offset_start_ignored", "int64_t off = offset_start;", "int64_t off = 0;"),
    ("expand_slices_not_advanced", "off += n;", "off += 0;"),
    ("expand_add_inputs_inverted", "y_out[o] = (add_inputs ? y_out[o] : 0.0) + v;",
     "y_out[o] = (add_inputs ? 0.0 : y_out[o]) + v;"),
    ("expand_bias_column_fixed", "v += bf16_to_f64(bias[s][(int64_t)id * n + j]);",
     "v += bf16_to_f64(bias[s][(int64_t)id * n]);"),
]


def _build(tmp_path, name, text):
    src = tmp_path / (name + ".c")
    src.write_text(text)
    sys.path.insert(0, ROOT)
    import oracle
    return oracle.compile_source(str(src), str(tmp_path / ("lib" + name + ".so")))


def _run_pins(lib):
    env = dict(os.environ, ORACLE_MUTANT_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-m", "not gpu",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_unaltered_copy_passes_every_pin(tmp_path):
    r = _run_pins(_build(tmp_path, "unaltered", open(SRC).read()))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


def test_mutants_are_distinct_and_apply_once():
    text = open(SRC).read()
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)
    for name, old, new in MUTANTS:
        assert text.count(old) == 1, name
        assert old != new, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1
    r = _run_pins(_build(tmp_path, name, text.replace(old, new)))
    # pytest exits 1 when a test failed; 2-5 would be a harness problem
    assert r.returncode == 1, (name, r.returncode, r.stdout[-2000:], r.stderr[-2000:])
    assert " failed" in r.stdout, (name, r.stdout[-2000:])
