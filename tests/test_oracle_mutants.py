"""Planted mistakes in the oracle fail its pins.

Each mutant copies ``oracle/oracle.c``, changes one thing a careless author
might get wrong (a flipped comparison, a transposed operand, a wrong row
index, a dropped clamp, an fp32 accumulator, ...), builds it with gcc and runs
the pin suite against it in a child process.  The test passes when some pin
rejects the mutant (a crash counts as rejected).  All of this runs on the CPU.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, original text, replacement, expected number of occurrences)
MUTANTS = [
    ("argmax_tie_highest", "if (row[v] > best) {", "if (row[v] >= best) {", 1),
    ("accept_le", "(double)u_acc[i] * (double)qi[x] < (double)pi[x]",
     "(double)u_acc[i] * (double)qi[x] <= (double)pi[x]", 1),
    ("accept_p_q_swapped", "(double)u_acc[i] * (double)qi[x] < (double)pi[x]",
     "(double)u_acc[i] * (double)pi[x] < (double)qi[x]", 1),
    ("accept_fp32_product", "(double)u_acc[i] * (double)qi[x] < (double)pi[x]",
     "(double)(u_acc[i] * qi[x]) < (double)pi[x]", 1),
    ("residual_sign", "double d = (double)p[v] - (double)q[v];\n            r[v] = d",
     "double d = (double)q[v] - (double)p[v];\n            r[v] = d", 1),
    ("residual_no_clamp", "r[v] = d > 0.0 ? d : 0.0;", "r[v] = d;", 1),
    ("bonus_row_k_minus_1", "residual_row(p + (int64_t)K * p_stride, NULL, V, r);",
     "residual_row(p + (int64_t)(K - 1) * p_stride, NULL, V, r);", 1),
    ("icdf_ge", "if (C > T)", "if (C >= T)", 1),
    ("icdf_reversed_uniform", "double T = u * R;", "double T = (1.0 - u) * R;", 1),
    ("icdf_fp32_sums", "double R = 0.0;\n    for (int64_t v = 0; v < V; ++v)\n        R += r[v];",
     "float R = 0.0f;\n    for (int64_t v = 0; v < V; ++v)\n        R += (float)r[v];", 1),
    ("greedy_n_plus_1", "*n_out = i;\n            *next_out = (int32_t)a;",
     "*n_out = i + 1;\n            *next_out = (int32_t)a;", 1),
    ("greedy_emits_draft", "*n_out = i;\n            *next_out = (int32_t)a;",
     "*n_out = i;\n            *next_out = t[i];", 1),
    ("greedy_bonus_row_k_minus_1",
     "*next_out = (int32_t)orc_argmax_lowest(p + (int64_t)K * p_stride, V);",
     "*next_out = (int32_t)orc_argmax_lowest(p + (int64_t)(K - 1) * p_stride, V);", 1),
    ("sample_n_plus_1", "*n_out = i;\n            *next_out = (int32_t)j;",
     "*n_out = i + 1;\n            *next_out = (int32_t)j;", 1),
    ("resample_wrong_row", "residual_row(pi, qi, V, r);",
     "residual_row(pi + p_stride, qi, V, r);", 1),
    ("no_zero_mass_fallback", "if (j < 0) {\n                residual_row(pi, NULL, V, r);",
     "if (0) {\n                residual_row(pi, NULL, V, r);", 1),
    ("token_range_off_by_one", "(int64_t)t[i] >= V", "(int64_t)t[i] > V", 1),
    ("round_modes_swapped", "if (m == 0) {", "if (m == 1 && 0) {", 1),
    ("commit_next_misplaced", "row[len + n] = next[b];", "row[len + n - 1] = next[b];", 1),
    ("alpha_max_not_min", "a += x < y ? x : y;", "a += x > y ? x : y;", 1),
    ("alpha_unnormalised_q", "const double y = (double)qr[v] / Q;", "const double y = (double)qr[v];", 1),
    ("alpha_expected_off_by_one", "reach *= a;    /* P(n > i) = prod_{j <= i} alpha_j */\n            mean += reach;",
     "mean += reach;\n            reach *= a;", 1),
    ("logits_no_temperature", "out[v] = exp(((double)z[v] - m) / tau);",
     "out[v] = exp(((double)z[v] - m));", 1),
    ("logits_no_max_shift", "out[v] = exp(((double)z[v] - m) / tau);",
     "out[v] = exp((double)z[v] / tau);", 1),
    ("logits_draft_unwarped", "orc_softmax(zq + (int64_t)i * zq_stride, V, tau, qr);",
     "orc_softmax(zq + (int64_t)i * zq_stride, V, 1.0, qr);", 1),
    ("logits_bonus_row_k_minus_1", "orc_softmax(zp + (int64_t)K * zp_stride, V, tau, pr);",
     "orc_softmax(zp + (int64_t)(K - 1) * zp_stride, V, tau, pr);", 1),
    ("threads_drop_tail", "j->b1 = (int)((int64_t)B * (k + 1) / nthreads);",
     "j->b1 = (int)((int64_t)B * (k + 1) / nthreads) - (k == nthreads - 1 && k > 0);", 1),
]

RUNNER = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {here!r}]
    import oracle, oracle_pins
    orc = oracle.Oracle({lib!r})
    for pin in oracle_pins.PINS:
        try:
            pin(orc)
        except Exception as e:
            print("REJECTED_BY", pin.__name__, type(e).__name__)
            sys.exit(3)
    print("SURVIVED")
""")


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_rejected(tmp_path, name, old, new, count):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == count, f"mutation site for {name} not found exactly {count}x"
    mutated = src.replace(old, new)
    cpath = tmp_path / "oracle_mut.c"
    cpath.write_text(mutated)
    lib = str(tmp_path / "liboracle_mut.so")
    oracle.compile_source(str(cpath), lib)
    code = RUNNER.format(root=ROOT, here=HERE, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600)
    assert "SURVIVED" not in r.stdout, f"mutant {name} passed every pin:\n{r.stdout}{r.stderr}"
    assert r.returncode != 0
