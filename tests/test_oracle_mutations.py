"""Each plausible mistake planted in a copy of the oracle (on the CPU) must be
caught by at least one pin.  The committed oracle.c is never modified: every
mutant is compiled from a rewritten copy into a temporary directory."""
import os

import pytest

from oracle import Oracle
from oracle import build as obuild
from oracle_pins import ALL_PINS

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("drop_onehot", "double onehot = (i == y) ? 1.0 : 0.0;", "double onehot = 0.0;"),
    ("onehot_wrong_column", "double onehot = (i == y) ? 1.0 : 0.0;",
     "double onehot = (i == (y + 1) % V) ? 1.0 : 0.0;"),
    ("divide_by_n_plus_1", "const double kf = j->reduction == ORACLE_MEAN ? s / (double)j->n : s;",
     "const double kf = j->reduction == ORACLE_MEAN ? s / (double)(j->n + 1) : s;"),
    ("sum_divides_by_n", "const double kf = j->reduction == ORACLE_MEAN ? s / (double)j->n : s;",
     "const double kf = j->reduction != ORACLE_NONE ? s / (double)j->n : s;"),
    ("grad_scale_ignored", "            if (j->grad_scale)\n",
     "            if (0)\n"),
    ("none_scale_wrong_row", "s = j->reduction == ORACLE_NONE ? j->grad_scale[r] : j->grad_scale[0];",
     "s = j->reduction == ORACLE_NONE ? j->grad_scale[k] : j->grad_scale[0];"),
    ("half_exponent_bias", "v = ldexp((double)(frac + 1024), exp - 25);",
     "v = ldexp((double)(frac + 1024), exp - 24);"),
    ("half_subnormal_scale", "v = ldexp((double)frac, -24);",
     "v = ldexp((double)frac, -25);"),
    ("loss_sign", "*loss = m + log(Z) - load_elem(x, dtype, y);",
     "*loss = m - log(Z) - load_elem(x, dtype, y);"),
    ("loss_drops_max", "*loss = m + log(Z) - load_elem(x, dtype, y);",
     "*loss = log(Z) - load_elem(x, dtype, y);"),
    ("loss_wrong_target", "*loss = m + log(Z) - load_elem(x, dtype, y);",
     "*loss = m + log(Z) - load_elem(x, dtype, (y + 1) % V);"),
    ("no_max_subtraction", "    /* pass 2: the normaliser */\n    csum_t z",
     "    m = 0.0;\n    /* pass 2: the normaliser */\n    csum_t z"),
    ("gradient_not_normalised", "double p = exp(load_elem(x, dtype, i) - m) / Z;",
     "double p = exp(load_elem(x, dtype, i) - m);"),
    ("ignored_rows_not_skipped", "    if (y == ignore_index) {\n        if (grad)",
     "    if (y == ignore_index && 0) {\n        if (grad)"),
    ("count_includes_ignored", "        if (y == ignore_index)\n            continue;\n        ++n;",
     "        ++n;\n        if (y == ignore_index)\n            continue;"),
    ("mean_over_all_rows", "return csum_value(&s) / (double)n;",
     "return csum_value(&s) / (double)M;"),
    ("softmax_not_normalised", "y[i] = exp(load_elem(x, dtype, i) - m) / Z;",
     "y[i] = exp(load_elem(x, dtype, i) - m);"),
    ("softmax_bwd_swapped", "dx[i] = load_elem(y, dtype, i) * (load_elem(dy, dtype, i) - S);",
     "dx[i] = load_elem(dy, dtype, i) * (load_elem(y, dtype, i) - S);"),
    ("softmax_bwd_drops_sum", "dx[i] = load_elem(y, dtype, i) * (load_elem(dy, dtype, i) - S);",
     "dx[i] = load_elem(y, dtype, i) * load_elem(dy, dtype, i);"),
    ("softmax_bwd_sum_of_dy", "csum_add(&s, load_elem(y, dtype, i) * load_elem(dy, dtype, i));",
     "csum_add(&s, load_elem(dy, dtype, i));"),
    ("bf16_wrong_shift", "uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;",
     "uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 15;"),
    ("row_stride_ignored", "(size_t)r * (size_t)j->a_stride * es;",
     "(size_t)r * (size_t)j->ncols * es;"),
    ("bsr_block_transposed", "return blockid * block * block + rxm * block + rxn;",
     "return blockid * block * block + rxn * block + rxm;"),
    ("bsr_entry_stride_2", "return lut[offset + 4 * rbn];", "return lut[offset + 2 * rbn];"),
    ("bsr_scale_ignored", "(load_elem(dy, dtype, z * dy_zstride + e) - S) *\n"
     "                                                 scale;",
     "(load_elem(dy, dtype, z * dy_zstride + e) - S);"),
    ("bsr_sum_skips_last_block",
     "csum_t s = {0.0, 0.0};\n                for (int64_t rbn = 0; rbn < size; ++rbn) {",
     "csum_t s = {0.0, 0.0};\n                for (int64_t rbn = 0; rbn < size - 1; ++rbn) {"),
    ("bsr_dy_batch_stride_of_y", "load_elem(dy, dtype, z * dy_zstride + e));",
     "load_elem(dy, dtype, z * y_zstride + e));"),
    ("bsr_last_row_of_block_skipped", "for (int64_t rxm = 0; rxm < block; ++rxm) {",
     "for (int64_t rxm = 0; rxm < block - 1; ++rxm) {"),
    ("bsr_sizemax_not_checked", "int ok = size >= 0 && size <= sizemax;", "int ok = size >= 0;"),
    ("bsr_sum_of_y", "csum_add(&s, load_elem(y, dtype, z * y_zstride + e) *\n"
     "                                         load_elem(dy, dtype, z * dy_zstride + e));",
     "csum_add(&s, load_elem(y, dtype, z * y_zstride + e));"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    with open(obuild.SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = obuild.compile_source(str(mutant_src), str(tmp_path / "liboracle_mutant.so"))
    o = Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
