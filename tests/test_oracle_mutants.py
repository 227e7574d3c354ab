"""The pins have teeth: plant one plausible mistake at a time in a copy of the
oracle's C source (on the CPU, in a temporary directory), compile it, and check
that at least one pin of tests/test_oracle_pins.py rejects it."""
from __future__ import annotations

import os

import pytest

import oracle
from test_oracle_pins import PINS as GEMV_PINS
from test_oracle_pins_collectives import PINS as COLLECTIVE_PINS

PINS = GEMV_PINS + COLLECTIVE_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTANTS = [
    ("drop_last_rank", "for (int i = 0; i < g->R; ++i) y +=", "for (int i = 0; i < g->R - 1; ++i) y +="),
    ("overwrite_not_accumulate", "y += rank_partial(g, g->order[i], b, n);", "y = rank_partial(g, g->order[i], b, n);"),
    ("drop_last_k", "for (int k = 0; k < g->Kr; ++k)", "for (int k = 0; k < g->Kr - 1; ++k)"),
    ("w_row_uses_b", "g->W + ((size_t)r * g->N + n) * g->Kr", "g->W + ((size_t)r * g->N + b) * g->Kr"),
    ("x_always_rank0", "g->x + ((size_t)r * g->B + b) * g->Kr", "g->x + ((size_t)0 * g->B + b) * g->Kr"),
    ("negated_product", "p += val[w[k]] * val[xv[k]];", "p -= val[w[k]] * val[xv[k]];"),
    ("ties_away", "(rem == half && (keep & 1))", "(rem == half)"),
    ("truncate", "if (rem > half || (rem == half && (keep & 1))) keep += 1;", "(void)half;"),
    ("decode_exponent_off", "ldexp((double)(128 + m), e - 134)", "ldexp((double)(128 + m), e - 133)"),
    ("subnormal_scale", "ldexp((double)m, -133)", "ldexp((double)m, -134)"),
    ("ar_skip_rank0", "for (int j = 0; j < a->R; ++j) s +=", "for (int j = 1; j < a->R; ++j) s +="),
    ("ar_one_replica", "for (int r = 0; r < a->R; ++r) a->out", "for (int r = 0; r < 1; ++r) a->out"),
    ("gemv_one_replica", "for (int s = 0; s < g->R; ++s)\n                    g->y_out", "for (int s = 0; s < 1; ++s)\n                    g->y_out"),
    ("order_ignored", "y += rank_partial(g, g->order[i], b, n);", "y += rank_partial(g, i, b, n);"),
    ("rs_wrong_block", "const size_t i = (size_t)s * c + j;", "const size_t i = (size_t)j * R + s;"),
    ("rs_skip_last_rank", "for (int r = 0; r < R; ++r) acc += val[in[(size_t)r * n + i]];",
     "for (int r = 0; r < R - 1; ++r) acc += val[in[(size_t)r * n + i]];"),
    ("gemv_rs_rows_by_rank", "y_ref[(size_t)(s * Bs + i) * N + n]", "y_ref[(size_t)(i * R + s) * N + n]"),
    ("rmsnorm_no_bias", "if (bias) z[h] += val[bias[h]];", "(void)bias;"),
    ("rmsnorm_eps_outside", "1.0 / sqrt(ss / (double)H + eps)", "1.0 / (sqrt(ss / (double)H) + eps)"),
    ("rmsnorm_sum_not_mean", "1.0 / sqrt(ss / (double)H + eps)", "1.0 / sqrt(ss + eps)"),
    ("rmsnorm_no_gamma", "(gamma ? val[gamma[h]] : 1.0)", "1.0"),
    ("rmsnorm_bias_after_norm_sum", "ss += z[h] * z[h];", "ss += (z[h] - (bias ? val[bias[h]] : 0.0)) * (z[h] - (bias ? val[bias[h]] : 0.0));"),
    ("tile_root_ignored", "out[(size_t)roots[i] * out_slot + out_off", "out[(size_t)0 * out_slot + out_off"),
    ("tile_ld_swapped", "(size_t)a * ld_in + (size_t)c]];", "(size_t)a * ld_out + (size_t)c]];"),
    ("tile_transposed", "in_off[i] + (size_t)a * ld_in + (size_t)c]", "in_off[i] + (size_t)c * ld_in + (size_t)a]"),
    ("tile_repeat_root_allowed", "used[roots[i]]) return -1;", "0) return -1;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in oracle.c"
    mut = tmp_path / "oracle_mutant.c"
    mut.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mut), out=str(tmp_path / "liboracle_mutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, pytest.fail.Exception) as e:  # noqa: PERF203
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant {name} passed every pin"
