"""The oracle's pins must catch plausible mistakes.  Each case plants one mistake in a copy of
the oracle's C source (on the CPU), builds it, and runs the pin suite against it: the suite has
to fail.  The mistakes are the kinds a reader could make when writing the layer out: a dropped
term, a wrong sign, a wrong index or a transposed operand, a wrong tie rule or sort order."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pmoe_oracle.c")

MUTANTS = {
    "tie_prefers_higher_id": ("logits[e] > logits[best]", "logits[e] >= logits[best]"),
    "softmax_sign": ("denom += exp((double)logits[e] - mx)", "denom += exp(mx - (double)logits[e])"),
    "no_renormalize": ("for (int j = 0; j < k; ++j) w[j] /= s;", ";"),
    "drop_up_projection": ("double a = g / (1.0 + exp(-g)) * u;", "double a = g / (1.0 + exp(-g));"),
    "silu_sign": ("double a = g / (1.0 + exp(-g)) * u;", "double a = g / (1.0 + exp(g)) * u;"),
    "gate_reads_up_page": ("g += orc_bf16_to_f64(w1[c]) * xd[c];", "g += orc_bf16_to_f64(w3[c]) * xd[c];"),
    "down_transposed": ("acc += orc_bf16_to_f64(w2[n]) * h[n];",
                        "acc += orc_bf16_to_f64(W2[(int64_t)n * d + m]) * h[n];"),
    "drop_combine_weight": ("for (int m = 0; m < d; ++m) acc[m] += w[j] * y[m];",
                            "for (int m = 0; m < d; ++m) acc[m] += y[m];"),
    "drop_shared_expert": ("        orc_expert_ffn(d, L->S * f, L->W1s, L->W3s, L->W2s, x, round_h, y);\n"
                           "        for (int m = 0; m < d; ++m) acc[m] += y[m];",
                           "        orc_expert_ffn(d, L->S * f, L->W1s, L->W3s, L->W2s, x, round_h, y);"),
    "align_unstable": ("for (int64_t i = 0; i < NP; ++i) {\n            int owner",
                       "for (int64_t i = NP - 1; i >= 0; --i) {\n            int owner"),
    "align_wrong_pad": ("sorted_ids[pos++] = (int32_t)NP;", "sorted_ids[pos++] = (int32_t)(NP - 1);"),
    "bf16_truncates": ("double r = rint(x / q) * q;", "double r = trunc(x / q) * q;"),
    "h_not_rounded": ("h[n] = round_h ? orc_bf16_to_f64(orc_f64_to_bf16(a)) : a;", "h[n] = a;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: %s" % name
    mutated = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                           str(so), str(c), "-lm"])
    env = dict(os.environ, PMOE_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode != 0, "pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
