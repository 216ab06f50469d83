"""The pins must be strong enough to catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/oracle_attn.c (on the CPU), builds
it, and runs the pin suite against it: the suite must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_attn.c")

MUTANTS = {
    "causal_off_by_one": ("int64_t n = L - rows_of(p, b) + i + 1;", "int64_t n = L - rows_of(p, b) + i;"),
    "causal_reversed": ("int64_t n = L - rows_of(p, b) + i + 1;", "int64_t n = L - i;"),
    "slot_index": ("* p->P + t % p->P) * p->D;", "* p->P + (t + 1) % p->P) * p->D;"),
    "pool_transposed": ("(((int64_t)page * p->Hkv + g) * p->P", "(((int64_t)g * p->num_pages + page) * p->P"),
    "page_index": ("p->table[(int64_t)b * p->max_pages + t / p->P]", "p->table[(int64_t)b * p->max_pages + t % p->max_pages]"),
    "dot_operand": ("(double)qrow[d] * (double)krow[d]", "(double)qrow[d] * (double)krow[0]"),
    "scale_dropped": ("double s = p->scale * acc;", "double s = acc;"),
    "window_off_by_one": ("int64_t lo = pos - p->window + 1;", "int64_t lo = pos - p->window;"),
    "softcap_inside_scale": ("s = p->softcap * tanh(s / p->softcap);", "s = p->softcap * tanh(s);"),
    "sink_sign": ("if (sinks) l += exp((double)sinks[h] - M);", "if (sinks) l += exp(M - (double)sinks[h]);"),
    "fold_sink_dropped": ("l = l * cs + exp(sk - m_new);", "l = l * cs;"),
    "ragged_position": ("int64_t n = L - rows_of(p, b) + i + 1;", "int64_t n = L - p->q_len + i + 1;"),
    "append_slot": ("const int64_t dst = (((int64_t)page * Hkv + g) * P + t % P) * D;",
                    "const int64_t dst = (((int64_t)page * Hkv + g) * P + j % P) * D;"),
    "exp_sign": ("double w = exp(s[t] - M);", "double w = exp(M - s[t]);"),
    "normalise_dropped": ("for (int d = 0; d < D; ++d) o[d] /= l;", ""),
    "gqa_interleaved": ("int g = h / G;\n        if (q_lens", "int g = h % p.Hkv;\n        if (q_lens"),
    "fold_rescale_dropped": ("l *= c;", ""),
    "fold_rescale_sign": ("double c = exp(m - m_new);", "double c = exp(m_new - m);"),
    "merge_weight_dropped": ("L += w * l[s];", "L += l[s];"),
    "lse_shift_dropped": ("if (lse) lse[j] = M + log(l);", "if (lse) lse[j] = log(l);"),
    "row_head_index": ("*h = (int)((r / p->q_len) % p->Hq);", "*h = (int)(r % p->Hq);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    orig, mutated = MUTANTS[name]
    src = open(SRC).read()
    assert orig in src, f"mutation site for {name} not found"
    bad_src = tmp_path / "oracle_attn.c"
    bad_src.write_text(src.replace(orig, mutated, 1))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           str(bad_src), "-o", str(lib), "-lm"])
    env = dict(os.environ, ATLAS_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"mutant {name} passed every pin:\n{res.stdout[-2000:]}"
