"""Each plausible mistake planted in a copy of the oracle fails a pin.

The copies are built on the host from text edits of oracle.c and loaded in
a child pytest run of tests/test_oracle_pins.py; the run must fail.
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "tie_to_higher_index": ("return (x->j > y->j) - (x->j < y->j);",
                            "return (x->j < y->j) - (x->j > y->j);"),
    "score_sign_flipped": ("c[j].score = acc;", "c[j].score = -acc;"),
    "last_candidate_dropped": ("for (int64_t j = 0; j < l; ++j) {", "for (int64_t j = 0; j + 1 < l; ++j) {"),
    "kv_head_interleaved": ("    int64_t kvh = b * Hkv + h / g;\n    const int64_t qoff",
                            "    int64_t kvh = b * Hkv + h % Hkv;\n    const int64_t qoff"),
    "summary_over_S": ("acc / (double)(t1 - t0)", "acc / (double)S"),
    "own_token_dropped": ("for (int64_t tau = l * S; tau <= t; ++tau)", "for (int64_t tau = l * S; tau < t; ++tau)"),
    "scale_dropped": ("x[u] = scale * acc;", "x[u] = acc;"),
    "max_not_subtracted_in_lse": ("lse[o] = mx + log(denom);", "lse[o] = log(denom);"),
    "group_sum_first_head_only": ("for (int64_t hh = grp * g; hh < grp * g + g; ++hh) {",
                                  "for (int64_t hh = grp * g; hh < grp * g + 1; ++hh) {"),
    "quantize_ties_away_from_zero": ("float t = rintf(x / s);", "float t = roundf(x / s);"),
    "quantize_scale_over_128": ("const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    "quantize4_ties_away_from_zero": ("float t4 = rintf(x / s4);", "float t4 = roundf(x / s4);"),
    "quantize4_scale_over_8": ("const float s4 = amax4 / 7.0f;", "const float s4 = amax4 / 8.0f;"),
    "values_from_keys": ("load_f64(dtype, V, (kvh * L_cap + tok[u]) * d + c)",
                         "load_f64(dtype, K, (kvh * L_cap + tok[u]) * d + c)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "oracle_mut.c")
        so = os.path.join(td, "liboracle_mut.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"],
                       check=True)
        env = dict(os.environ, ORACLE_SO=so)
        res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q",
                              os.path.join(HERE, "test_oracle_pins.py")],
                             cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert res.returncode != 0, "mutant %s passed every pin:\n%s" % (name, res.stdout[-2000:])
