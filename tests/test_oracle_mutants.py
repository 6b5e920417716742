"""Plants plausible mistakes in copies of the oracle source and checks that some pin fails.

Each mutant is one textual change to oracle/dflash_oracle.c: a reversed tie-break, a
dropped term, a transposed operand, a wrong index, a double rounding, and so on. The
copy is compiled into a temporary library and loaded. Every pin of tests/oracle_pins.py
runs against it, and at least one must fail. This shows that the pins would catch that
kind of error in the real oracle. The real oracle source is never modified.
"""

import os
import tempfile

import pytest

import oracle
import oracle_pins
from oracle.build import SOURCE, compile_oracle

# (name, original text, mutated text). Each original must occur exactly once.
MUTANTS = [
    ("tie_break_reversed",
     "/* -0 == +0 here */\n    return (a->id < b->id) ? -1 : (a->id > b->id ? 1 : 0);",
     "/* -0 == +0 here */\n    return (a->id > b->id) ? -1 : (a->id < b->id ? 1 : 0);"),
    ("value_order_reversed",
     "if (ca == 1 && a->v != b->v) return a->v > b->v ? -1 : 1;",
     "if (ca == 1 && a->v != b->v) return a->v < b->v ? -1 : 1;"),
    ("lmhead_value_order_reversed",
     "if (a->v != b->v) return a->v > b->v ? -1 : 1;",
     "if (a->v != b->v) return a->v < b->v ? -1 : 1;"),
    ("signed_zero_distinct",
     "if (ca == 1 && a->v != b->v) return a->v > b->v ? -1 : 1;",
     "if (ca == 1 && (a->v != b->v || signbit(a->v) != signbit(b->v)))"
     " return (a->v > b->v || (a->v == b->v && !signbit(a->v))) ? -1 : 1;"),
    ("nan_classes_swapped",
     "if (isnan(v)) return signbit(v) ? 0 : 2;",
     "if (isnan(v)) return signbit(v) ? 2 : 0;"),
    ("unary_from_position_not_id",
     "processed_logit(e[k].v, c->softcap, c->scale);",
     "processed_logit(row[k], c->softcap, c->scale);"),
    ("processor_scale_before_cap",
     "if (softcap > 0.0) v = softcap * tanh(v / softcap);\n    return (float)(v * scale);",
     "v *= scale;\n    if (softcap > 0.0) v = softcap * tanh(v / softcap);\n    return (float)v;"),
    ("processor_cap_ignored",
     "if (softcap > 0.0) v = softcap * tanh(v / softcap);",
     "(void)softcap;"),
    ("processor_not_applied",
     "c->unary[r * c->K + k] = processed_logit(e[k].v, c->softcap, c->scale);",
     "c->unary[r * c->K + k] = e[k].v;"),
    ("lmhead_transposed",
     "const uint16_t* w = c->lm_head + v * c->H;   /* LM head row v: [V, H] */",
     "const uint16_t* w = c->lm_head + v;"),
    ("lmhead_tie_break_reversed",
     "return (a->id < b->id) ? -1 : (a->id > b->id ? 1 : 0);\n}\n\nstatic void lmhead_row",
     "return (a->id > b->id) ? -1 : (a->id < b->id ? 1 : 0);\n}\n\nstatic void lmhead_row"),
    ("projection_weight_transposed",
     "s += bf16_to_double(wj[i]) * bf16_to_double(x[i]);",
     "s += bf16_to_double(c->w[i * c->rank + j]) * bf16_to_double(x[i]); (void)wj;"),
    ("projection_rounds_twice",
     "c->h_out[r * c->rank + j] = oracle_bf16_round(s);",
     "c->h_out[r * c->rank + j] = oracle_bf16_round((double)(float)s);"),
    ("bf16_ties_away",
     "double q = nearbyint(x / ulp);",
     "double q = round(x / ulp);"),
    ("bf16_truncates",
     "double q = nearbyint(x / ulp);",
     "double q = trunc(x / ulp);"),
    ("bf16_no_subnormal_floor",
     "if (E < -126) E = -126;",
     ";"),
    ("edges_drop_unary",
     "double s = (double)c->unary[row * K + cc];",
     "double s = 0.0;"),
    ("edges_unary_of_predecessor",
     "double s = (double)c->unary[row * K + cc];",
     "double s = (double)c->unary[row * K + q];"),
    ("edges_predecessor_same_step",
     "c->cand[(row - 1) * K + q]",
     "c->cand[row * K + q]"),
    ("edges_anchor_ignored",
     "(p == 0) ? c->anchors[r] :",
     "(p == 0) ? c->cand[row * K + q] :"),
    ("edges_codebooks_swapped",
     "const uint16_t* a = c->pred_cb + pid * c->rank;",
     "const uint16_t* a = c->succ_cb + pid * c->rank;"),
    ("edges_output_transposed",
     "float* out = &c->edges[(row * K + q) * K + cc];",
     "float* out = &c->edges[(row * K + cc) * K + q];"),
    ("edges_h_of_previous_step",
     "const uint16_t* hp = c->h + row * c->rank;",
     "const uint16_t* hp = c->h + (p == 0 ? row : row - 1) * c->rank;"),
    ("edges_sign_flipped",
     "s += bf16_to_double(a[j]) * bf16_to_double(hp[j]) * bf16_to_double(b[j]);",
     "s -= bf16_to_double(a[j]) * bf16_to_double(hp[j]) * bf16_to_double(b[j]);"),
    ("edges_subnormal_codebook_flushed",
     "s += bf16_to_double(a[j]) * bf16_to_double(hp[j]) * bf16_to_double(b[j]);",
     "s += (fabs(bf16_to_double(a[j])) < 0x1p-126 ? 0.0 : bf16_to_double(a[j])) * "
     "bf16_to_double(hp[j]) * bf16_to_double(b[j]);"),
    ("edges_h_dropped",
     "s += bf16_to_double(a[j]) * bf16_to_double(hp[j]) * bf16_to_double(b[j]);",
     "s += bf16_to_double(a[j]) * bf16_to_double(b[j]);"),
    ("best_path_ties_to_higher_predecessor",
     "if (s > best) {",
     "if (s >= best) {"),
    ("best_path_final_tie_to_higher",
     "if (v[j] > v[cur]) cur = j;",
     "if (v[j] >= v[cur]) cur = j;"),
    ("best_path_first_step_diagonal_row",
     "for (int j = 0; j < K; ++j) v[j] = E[j];",
     "for (int j = 0; j < K; ++j) v[j] = E[j * K + j];"),
    ("best_path_predecessor_not_kept",
     "keep[p * K + j] = (unsigned char)bq;",
     "keep[p * K + j] = (unsigned char)0;"),
    ("best_path_transposed_scores",
     "const float s = v[q] + Ep[q * K + j];",
     "const float s = v[q] + Ep[j * K + q];"),
    ("best_path_tokens_from_previous_step",
     "c->tokens[r * S + p] = c->cand[(r * S + p) * K + cur];",
     "c->tokens[r * S + p] = c->cand[(r * S + (p > 0 ? p - 1 : p)) * K + cur];"),
]


@pytest.fixture(scope="module")
def source_text():
    with open(SOURCE) as f:
        return f.read()


def test_mutant_texts_occur_once(source_text):
    for name, old, _ in MUTANTS:
        assert source_text.count(old) == 1, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(source_text, name, old, new):
    mutated = source_text.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, f"mutant_{name}.c")
        with open(src, "w") as f:
            f.write(mutated)
        lib = compile_oracle(src, os.path.join(d, f"libmutant_{name}.so"))
        orc = oracle.Oracle(lib)
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"no pin detects the mutant {name}"
