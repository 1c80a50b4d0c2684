"""Plant mistakes in copies of the oracle (on the CPU) and check that the pins
catch every one of them.  A pin suite that passes a broken oracle pins
nothing.  (Swapping "first minimum wins" for "last minimum wins" in the grid
search is not listed: two candidates' MSEs never tie exactly on finite data,
so that mutant computes the same codes.)"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "smoe_oracle.c")

# (name, exact source text, replacement)
MUTANTS = [
    ("encode adds -L", "    q = q + L;\n", "    q = q - L;\n"),
    ("encode truncates", "    float r = rintf(q);\n", "    float r = floorf(q);\n"),
    ("decode divides by 2L", "    float lv = ((float)c - L) / L;\n",
     "    float lv = ((float)c - L) / (2.0f * L);\n"),
    ("pack MSB-first", "<< ((i % per) * bits));",
     "<< (8 - bits - (i % per) * bits));"),
    ("ties to higher index", "if (best < 0 || key[e] > key[best])",
     "if (best < 0 || key[e] >= key[best])"),
    ("bias enters weights", "            double pj = p[ids[t * k + j]];\n",
     "            double pj = p[ids[t * k + j]] * (bias ? 1.0 + bias[ids[t * k + j]] : 1.0);\n"),
    ("router transposed", "(double)bf16_bits_to_f32(wr_bf16[(int64_t)e * d + i])",
     "(double)bf16_bits_to_f32(wr_bf16[(int64_t)i * E + e])"),
    ("MSE not squared", "            acc += e * e;\n", "            acc += fabs(e);\n"),
    ("no SiLU", "double hv = (double)g / (1.0 + exp(-(double)g)) * (double)u;",
     "double hv = (double)g * (double)u;"),
    ("no renorm", "weights[t * k + j] = (float)((norm ? pj / sel : pj) * (double)routed_scaling_factor);",
     "weights[t * k + j] = (float)(pj * (double)routed_scaling_factor);"),
    ("sigmoid router scores by softmax", "        if (router_sigmoid) {\n",
     "        if (0) {\n"),
    ("scaling factor ignored", "* (double)routed_scaling_factor);", ");"),
    ("mask ignored by the softmax", "p[e] = routable(mask, e) ? exp((double)l[e] - m) : 0.0;",
     "p[e] = exp((double)l[e] - m);"),
    ("mask ignored by the selection", "if (taken[e] || !routable(mask, e))", "if (taken[e])"),
    ("grid off by one", "double v = (double)j * step + start;",
     "double v = (double)(j + 1) * step + start;"),
    ("shared gate ignored", "                sw = 1.0 / (1.0 + exp(-z));\n",
     "                sw = 1.0;\n"),
    ("expert depth ignored", "oracle_expert_ffn(b, d, f, expert_bits ? expert_bits[e] : bits, xt, o, NULL)",
     "oracle_expert_ffn(b, d, f, bits, xt, o, NULL)"),
    ("f16 truncates", "double m = rint((ldexp(a, -E) - 1.0) * 1024.0);",
     "double m = floor((ldexp(a, -E) - 1.0) * 1024.0);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for '{name}' not found"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-pthread", "-o", str(so), str(mut), "-lm"])
    env = dict(os.environ, SMOE_ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_quant.py"),
                        os.path.join(ROOT, "tests", "test_oracle_route_forward.py"),
                        os.path.join(ROOT, "tests", "test_oracle_router_variants.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins passed a mutant oracle ({name})"
