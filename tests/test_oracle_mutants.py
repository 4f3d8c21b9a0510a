"""The oracle's pins have teeth: plant a plausible mistake in a copy of the oracle source,
rebuild it on the CPU, and check that at least one pin in test_oracle.py fails."""
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
import test_oracle as pins

SRC = obuild.SRC

# (name, original text, planted mistake)
MUTANTS = [
    ("threshold strictly greater", ">= threshold) hit = 1", "> threshold) hit = 1"),
    ("absmax includes outlier columns",
     "if (outlier && outlier[j]) continue;\n      float v = fabsf(",
     ";\n      float v = fabsf("),
    ("dequantize by 127 not 127^2", "/ (127.0 * 127.0)", "/ 127.0"),
    ("outlier product dropped", "y += f;", "y += 0.0 * f;"),
    ("weight row stride transposed", "jb->CB + o * jb->in", "jb->CB + o"),
    ("zeropoint sign of Z", "float t = p - z;", "float t = p + z;"),
    ("truncation instead of rounding", "return clamp_code(rintf(p));", "return clamp_code(truncf(p));"),
    ("scale 128 instead of 127", "? 127.0f / absmax", "? 128.0f / absmax"),
    ("outlier weight not dequantized", "* SCB[o]) / 127.0f", "* 1.0f) / 127.0f"),
    ("bias subtracted", "y += (double)h2f(jb->bias[o]);", "y -= (double)h2f(jb->bias[o]);"),
    ("ReLU dropped", "if (relu && !(v > 0.0)) v = 0.0;", "if (relu && 0) v = 0.0;"),
    ("ReLU mirrors negatives", "if (relu && !(v > 0.0)) v = 0.0;",
     "if (relu && !(v > 0.0)) v = -v;"),
    ("intermediate rounded twice", "_Float16 t = (_Float16)v;", "_Float16 t = (_Float16)(float)v;"),
    ("zeropoint correction dropped",
     "double az = (double)a + (double)jb->rowZ[r] * (double)jb->cbin[o];",
     "double az = (double)a;"),
    ("zeropoint correction over outlier columns too", "if (!mask[j]) cbin[o] += CB[o * in + j];",
     "cbin[o] += CB[o * in + j];"),
    ("zeropoint scale inverted", "/ (127.0 * (double)jb->rowS[r])",
     "* (double)jb->rowS[r] / 127.0"),
    ("block absmax over the whole row",
     "for (int64_t j = j0; j < j1; ++j) {\n        float v = fabsf(h2f(X[i * cols + j]));",
     "for (int64_t j = 0; j < cols; ++j) {\n        float v = fabsf(h2f(X[i * cols + j]));"),
    ("block one column short", "(j0 + block < cols) ? j0 + block : cols",
     "(j0 + block - 1 < cols) ? j0 + block - 1 : cols"),
    ("block absmax stored transposed", "absmax[i * nblocks + k] = a;", "absmax[k * rows + i] = a;"),
    ("ragged last block dropped", "const int64_t nblocks = (cols + block - 1) / block;",
     "const int64_t nblocks = cols / block;"),
    ("zeropoint range over outlier columns",
     "if (outlier && outlier[j]) continue;\n    float v = h2f(x[j]);",
     ";\n    float v = h2f(x[j]);"),
]

PIN_TESTS = [
    pins.test_absmax_worked_example_from_page,
    pins.test_outlier_columns_threshold_edge_and_bruteforce,
    pins.test_weight_quantization_roundtrip_bound_and_range,
    pins.test_weight_quantization_integer_rows_are_exact,
    pins.test_integer_case_reduces_to_exact_integer_matmul,
    lambda: pins.test_general_case_within_quantization_error_bound("tiny"),
    pins.test_acc_equals_library_integer_matmul_and_codes_in_range,
    pins.test_zeropoint_uses_full_range_on_one_sided_rows,
    pins.test_zeropoint_zero_maps_exactly_and_constant_row,
    lambda: pins.test_integer_ffn_block_reduces_to_exact_integer_chain(True),
    pins.test_ffn_without_activation_is_two_chained_matmuls,
    pins.test_activation_rounding_is_one_step_from_fp64,
    lambda: pins.test_zeropoint_matmul_on_one_sided_grid_rows_is_exact(True),
    pins.test_zeropoint_matmul_constant_and_all_outlier_rows,
    pins.test_zeropoint_matmul_within_quantization_error_bound,
    lambda: pins.test_blockwise_power_of_two_blocks_are_exact(64, 3 * 64 + 20),
    pins.test_blockwise_page_example_as_one_block,
    pins.test_blockwise_with_one_block_per_row_is_the_row_quantizer,
    lambda: pins.test_blockwise_half_step_bound_range_and_independence(64),
]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor not unique: {orig!r}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(orig, bad))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *obuild.CFLAGS, str(mut), "-o", str(so), "-lm"], check=True,
                   capture_output=True)
    saved = oracle._lib
    oracle._lib = oracle.load(str(so))
    failed = []
    try:
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                failed.append(getattr(t, "__name__", "general bound"))
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake: {name}"
