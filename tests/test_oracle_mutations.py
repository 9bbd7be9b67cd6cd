"""Plant plausible mistakes in copies of the oracle and check that the pins catch each one.

Every mutant is a text edit of ``oracle/moe_oracle.c`` (a dropped term, a wrong sign or
index, a transposed operand, a changed tie-break ...), compiled with gcc into a temporary
library; all pins of ``oracle_pins`` then run against it and at least one must fail.
The real oracle source is never modified.  Every edit keeps all memory accesses in bounds.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

# (name, [(old, new), ...]) -- every ``old`` must occur in the source.
MUTANTS = [
    ("silu_sign", [("exp(-g[i])", "exp(g[i])")]),
    ("silu_on_up", [("p[i] = g[i] / (1.0 + exp(-g[i])) * u[i];",
                     "p[i] = u[i] / (1.0 + exp(-u[i])) * g[i];")]),
    ("gate_reads_up", [("accumulate_row(w, w->w_gate, w->j_gate, w->cb_gate, e, hh, x, g);",
                        "accumulate_row(w, w->w_up, w->j_up, w->cb_up, e, hh, x, g);")]),
    ("residual_dropped", [("o[n] = residual ? bf16_bits_to_double(residual[(size_t)m * H + n]) : 0.0;",
                           "o[n] = 0.0;")]),
    ("down_columns_reversed", [("y[n] += p[i] * bf16_bits_to_double(drow[n]);",
                                "y[n] += p[i] * bf16_bits_to_double(drow[H - 1 - n]);")]),
    ("affinity_of_slot0", [("o[n] += a[r] * yall[r * H + n];",
                            "o[n] += a[(size_t)m * k] * yall[r * H + n];")]),
    ("combine_slots_reversed", [("const size_t r = (size_t)m * k + j;\n            const int e = topk_ids[r];",
                                 "const size_t r = (size_t)m * k + (k - 1 - j);\n            const int e = topk_ids[(size_t)m * k + j];")]),
    ("tie_to_higher_id", [("if (best < 0 || v > bestv)", "if (best < 0 || v >= bestv)")]),
    ("select_in_fp64", [("float bestv = 0.0f;", "double bestv = 0.0;"),
                        ("float v = to_f32(l[e]);", "double v = l[e];")]),
    ("renorm_unshifted", [("a[j] = exp(l[ids[j]] - l0) / denom;", "a[j] = exp(l[ids[j]]) / denom;")]),
    ("full_softmax_unnormalised", [("a[j] = exp(l[ids[j]] - lmax) / denom;",
                                    "a[j] = exp(l[ids[j]] - lmax);")]),
    ("gap_sign", [("gap[m] = l[ids[k - 1]] - l[next];", "gap[m] = l[next] - l[ids[k - 1]];")]),
    ("bias_dropped", [("row[e] += (double)bias[e];", "row[e] += 0.0;")]),
    ("router_transposed", [("row[e] += x * bf16_bits_to_double(wrow[e]);",
                            "row[e] += x * bf16_bits_to_double(w_router[(size_t)e * H + hh]);")]),
    ("bf16_widening", [("((uint32_t)bits) << 16", "((uint32_t)bits) << 15")]),
    ("vq_element_index", [("const int q = hh / d, t = hh % d;",
                           "const int q = hh / d, t = (hh + 1) % d;")]),
    ("vq_block_index", [("const uint8_t *jrow = J + ((size_t)e * (H / d) + q) * I;",
                         "const uint8_t *jrow = J + ((size_t)e * (H / d) + (H / d - 1 - q)) * I;")]),
    ("sentinel_value", [("const int32_t sentinel = (int32_t)R;", "const int32_t sentinel = -1;")]),
    ("over_padding", [("int64_t blocks = (n + b - 1) / b;", "int64_t blocks = n / b + 1;")]),
    ("routes_descending", [("for (int64_t r = 0; r < R; ++r) {\n            if (topk_ids[r] == e)",
                            "for (int64_t r = R - 1; r >= 0; --r) {\n            if (topk_ids[r] == e)")]),
    ("tail_blocks_zero", [("expert_block_ids[q] = -1;", "expert_block_ids[q] = 0;")]),
    ("low_rank_dropped", [("                add_low_rank(w, h + (size_t)m * H, e, zg, zu, g, u);",
                           "                (void)zg;")]),
    ("low_rank_basis_permuted", [("zg[rho] += x * bf16_bits_to_double(w->d_gate[(size_t)hh * R + rho]);",
                                    "zg[rho] += x * bf16_bits_to_double(w->d_gate[(size_t)(hh % R) * R + (rho * 7 + hh) % R]);")]),
    ("low_rank_gate_basis_for_up", [("zu[rho] += x * bf16_bits_to_double(w->d_up[(size_t)hh * R + rho]);",
                                     "zu[rho] += x * bf16_bits_to_double(w->d_gate[(size_t)hh * R + rho]);")]),
    ("low_rank_wrong_expert", [("const uint16_t *cg = w->c_gate + ((size_t)e * R + rho) * I;",
                                "const uint16_t *cg = w->c_gate + ((size_t)((e + 1) % w->E) * R + rho) * I;")]),
]


def _build_mutant(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, "mutation %s does not apply: %r" % (name, old)
        src = src.replace(old, new)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("lib%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    str(c), "-o", str(so), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, edits):
    so = _build_mutant(tmp_path, name, edits)
    caught = []
    with oracle.using_library(so):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, RuntimeError) as exc:
                caught.append((pin.__name__, type(exc).__name__))
    assert caught, "no pin caught the planted mistake %r" % name


def test_pins_pass_on_real_oracle():
    for pin in oracle_pins.ALL_PINS:
        pin()
