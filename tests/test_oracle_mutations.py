"""The oracle's pins are sensitive: each plausible slip planted in a copy of the
oracle's C source (on the CPU, in a temporary directory) makes at least one pin
fail.  The oracle in the repository is never modified."""

import os
import shutil

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.test_oracle import (run_activation_pins, run_attention_pins, run_epilogue_pins,
                               run_int_pins, run_paged_pins)

SRC = os.path.join(os.path.dirname(oracle.__file__), "sbgemm_ref.c")

# (name, text in the source, replacement)
MUTATIONS = [
    ("drop_last_k_term", "for (int64_t k = 0; k < K; ++k) {\n        const double a",
     "for (int64_t k = 0; k < K - 1; ++k) {\n        const double a"),
    ("wrong_sign", "acc[n] += p;", "acc[n] -= p;"),
    ("transposed_A", "m * j->rsA + k * j->csA", "m * j->csA + k * j->rsA"),
    ("transposed_B_index", "brow[n * j->csB]", "brow[n * j->rsB]"),
    ("alpha_scales_c0", "r += c0;\n            t += fabs(c0);",
     "r += j->alpha * c0;\n            t += fabs(c0);"),
    ("ignore_B_batch_stride", "j->B + b * j->bsB + k * j->rsB", "j->B + k * j->rsB"),
    ("c0_row_col_swapped", "m * j->rsC + n * j->csC", "m * j->csC + n * j->rsC"),
    ("bound_without_abs", "mag[n] += fabs(p);", "mag[n] += p;"),
    ("output_rows_batch_major_swapped", "double* out = j->ref + (b * j->M + m) * N;",
     "double* out = j->ref + (m * j->batch + b) * N;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmut.so")
    oracle.build(force=True, src=str(mutated), out=so)
    lib = oracle.load(so)
    assert run_int_pins(lib=lib) > 0, f"planted mistake {name} went unnoticed"


def test_unmutated_copy_passes(tmp_path):
    shutil.copy(SRC, tmp_path / "same.c")
    so = str(tmp_path / "libsame.so")
    oracle.build(force=True, src=str(tmp_path / "same.c"), out=so)
    lib = oracle.load(so)
    assert run_int_pins(lib=lib) == 0
    assert run_activation_pins(lib=lib) == 0 and run_epilogue_pins(lib=lib) == 0
    assert run_attention_pins(lib=lib) == 0
    assert run_paged_pins(lib=lib) == 0


# Slips in the fused epilogue's activations and added operand.
EPILOGUE_MUTATIONS = [
    ("relu_leaky", "case 1: *out = z > 0.0 ? z : 0.0;", "case 1: *out = z > 0.0 ? z : 0.01 * z;"),
    ("sigmoid_sign", "case 2: *out = 1.0 / (1.0 + exp(-z));", "case 2: *out = 1.0 / (1.0 + exp(z));"),
    ("silu_without_z", "case 3: *out = z / (1.0 + exp(-z));", "case 3: *out = 1.0 / (1.0 + exp(-z));"),
    ("gelu_tanh_coefficient", "(z + 0.044715 * z", "(z + 0.04715 * z"),
    ("gelu_tanh_square_not_cube", "z * z * z", "z * z"),
    ("gelu_erf_without_sqrt2", "erf(z / sqrt(2.0))", "erf(z)"),
    ("gelu_erf_without_half", "case 5: *out = 0.5 * z *", "case 5: *out = z *"),
    ("addend_rows_cols_swapped", "D[b * bsD + m * rsD + n * csD]", "D[b * bsD + m * csD + n * rsD]"),
    ("addend_bound_without_abs", "if (bound) bound[p] += fabs(d);", "if (bound) bound[p] += d;"),
]


@pytest.mark.parametrize("name,old,new", EPILOGUE_MUTATIONS, ids=[m[0] for m in EPILOGUE_MUTATIONS])
def test_planted_epilogue_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmut.so")
    oracle.build(force=True, src=str(mutated), out=so)
    lib = oracle.load(so)
    assert run_activation_pins(lib=lib) + run_epilogue_pins(lib=lib) > 0, \
        f"planted mistake {name} went unnoticed"


# Slips in the attention oracle.
ATTENTION_MUTATIONS = [
    ("causal_off_by_one", "const int64_t kept = causal ? (m % q_len) + N - q_len + 1 : N;",
     "const int64_t kept = causal ? (m % q_len) + N - q_len : N;"),
    ("key_index_uses_row", "(double)K[b * bsK + n * rsK + d * csK];", "(double)K[b * bsK + m * rsK + d * csK];"),
    ("exponent_sign", "s[n] = exp(s[n] - mx);", "s[n] = exp(mx - s[n]);"),
    ("not_normalised", "O[(b * M + m) * Dv + e] = o / l;", "O[(b * M + m) * Dv + e] = o;"),
    ("alpha_dropped", "s[n] = (double)alpha * acc;", "s[n] = acc;"),
    ("weight_without_abs", "w += s[n] * fabs(v);", "w += s[n] * v;"),
    ("value_index_transposed", "(double)V[b * bsV + n * rsV + e * csV];", "(double)V[b * bsV + e * rsV + n * csV];"),
]


@pytest.mark.parametrize("name,old,new", ATTENTION_MUTATIONS, ids=[m[0] for m in ATTENTION_MUTATIONS])
def test_planted_attention_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmut.so")
    oracle.build(force=True, src=str(mutated), out=so)
    lib = oracle.load(so)
    assert run_attention_pins(lib=lib) > 0, f"planted mistake {name} went unnoticed"


# Slips in the paged-cache reader.
PAGED_MUTATIONS = [
    ("block_index_modulo", "const int64_t block_pos = pos / block_size;",
     "const int64_t block_pos = pos % block_size;"),
    ("offset_divides", "const int64_t offset = pos % block_size;", "const int64_t offset = pos / block_size;"),
    ("head_stride_dropped", "* n_kv_heads + head) * head_dim", "+ head) * head_dim"),
    ("table_row_ignored", "block_table[seq * max_blocks + block_pos]", "block_table[block_pos]"),
    ("block_stride_dropped", "((block * block_size + offset)", "((block + offset)"),
    ("last_position_dropped", "for (int64_t pos = 0; pos < len; ++pos) {",
     "for (int64_t pos = 0; pos + 1 < len; ++pos) {"),
]


@pytest.mark.parametrize("name,old,new", PAGED_MUTATIONS, ids=[m[0] for m in PAGED_MUTATIONS])
def test_planted_paged_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmut.so")
    oracle.build(force=True, src=str(mutated), out=so)
    lib = oracle.load(so)
    assert run_paged_pins(lib=lib) > 0, f"planted mistake {name} went unnoticed"
