"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies the oracle source, makes one plausible mistake in it
(a dropped weight, a wrong column offset, an unstable tie order, a wrong
exponent bias, ...), compiles the copy into a temporary directory and runs
the pin suite against it.  At least one pin has to fail, otherwise the pins
would not be pinning that part of the oracle.  The committed oracle is never
modified.
"""

import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tbe_oracle.c")

MUTANTS = {
    "fwd_drops_weight": ("double w = weighted ? (double)per_sample_weights[i] : 1.0;", "double w = 1.0;"),
    "bwd_drops_weight": ("double w = weighted ? (double)per_sample_weights[pos] : 1.0;", "double w = 1.0;"),
    "bwd_wrong_column": ("grad_out + b * sumD + D_offsets[t];", "grad_out + b * sumD;"),
    "bwd_wrong_sample": ("int64_t b = g % B;", "int64_t b = g / B;"),
    "fwd_drops_last_lookup": (
        "for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) {\n      int64_t id = indices[i];\n"
        "      if (id < 0 || id >= rows) { /* reported, contributes nothing */",
        "for (int64_t i = offsets[g]; i + 1 < offsets[g + 1]; ++i) {\n      int64_t id = indices[i];\n"
        "      if (id < 0 || id >= rows) { /* reported, contributes nothing */"),
    "fwd_sign": ("s[c] += term; /* a repeated id is simply added again */", "s[c] -= term;"),
    "unstable_ties": ("if (a->pos != b->pos) return a->pos < b->pos ? -1 : 1;",
                      "if (a->pos != b->pos) return a->pos > b->pos ? -1 : 1;"),
    "key_without_table_base": ("p[i].key = ok ? table_row_base[t] + id : total_rows;",
                               "p[i].key = ok ? id : total_rows;"),
    "run_start_off_by_one": ("run_starts[U] = (int32_t)j;", "run_starts[U] = (int32_t)(j + (j > 0));"),
    "unique_count_inclusive": ("while (c < U && unique_rows[c] < table_row_base[t]) ++c;",
                               "while (c < U && unique_rows[c] <= table_row_base[t]) ++c;"),
    "f32_rounds_toward_zero": ("((float*)out)[i] = (float)in[i]; /* C conversion: nearest-even */",
                               "((float*)out)[i] = nextafterf((float)in[i], 0.0f) == (float)in[i] ? (float)in[i] : "
                               "(fabs((double)(float)in[i]) > fabs(in[i]) ? nextafterf((float)in[i], 0.0f) : "
                               "(float)in[i]);"),
    "f16_truncates": ("double q = rint(ldexp(a, 11 - e)); /* in [1024, 2048] */",
                      "double q = floor(ldexp(a, 11 - e));"),
    "bf16_rounds_up": ("double q = rint(ldexp(a, 8 - e)); /* in [128, 256] */",
                       "double q = ceil(ldexp(a, 8 - e));"),
    "f16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "bf16_bias": ("v = ldexp((double)(m | 0x80), e - 134);", "v = ldexp((double)(m | 0x80), e - 133);"),
    "histogram_transposed": ("counts[(int64_t)b * rows_t + id] += 1;", "counts[(int64_t)id * B + b] += 1;"),
    "bwd_unsorted_position": ("int32_t pos = sorted_pos[j];", "int32_t pos = (int32_t)j;"),
    "offsets_not_checked": ("if (offsets[g + 1] < offsets[g]) return ORC_BAD_OFFSETS;", ";"),
    "adagrad_sum_not_mean": ("double m = (double)momentum[row] + sq / (double)D;",
                             "double m = (double)momentum[row] + sq;"),
    "adagrad_momentum_reset": ("double m = (double)momentum[row] + sq / (double)D;",
                               "double m = sq / (double)D;"),
    "adagrad_momentum_by_id": ("double m = (double)momentum[row] + sq / (double)D;",
                               "double m = (double)momentum[id] + sq / (double)D;"),
    "adagrad_eps_inside_sqrt": ("step = lr / (sqrt(m) + eps);", "step = lr / sqrt(m + eps);"),
    "adagrad_rms_of_update": ("step = lr / (sqrt(m) + eps);", "step = lr / (m + eps);"),
    "update_sign": ("table_elem(weights, weights_offsets[t], weights_dtype[t], D, id, c) - step * g[c];",
                    "table_elem(weights, weights_offsets[t], weights_dtype[t], D, id, c) + step * g[c];"),
    "mean_divides_by_len_plus_one": ("values[(int64_t)b * sumD + c] /= (double)len;",
                                     "values[(int64_t)b * sumD + c] /= (double)(len + 1);"),
    "mean_scales_first_column_only": ("for (int32_t c = D_offsets[t]; c < D_offsets[t + 1]; ++c) values",
                                      "for (int32_t c = D_offsets[t]; c < D_offsets[t] + 1; ++c) values"),
    "update_reads_first_row": ("table_elem(weights, weights_offsets[t], weights_dtype[t], D, id, c) - step * g[c];",
                               "table_elem(weights, weights_offsets[t], weights_dtype[t], D, 0, c) - step * g[c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.build(str(mutated), so)
    lib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin caught mutant {name}"
