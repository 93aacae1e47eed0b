"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (on the host,
in a temporary directory), builds it, and reruns the pin suite against it with
``PKV_ORACLE_LIB`` pointing at the broken build.  Every mutant must make at
least one pin fail.
"""

import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "gqa_head_map": ("int g = h / group;", "int g = h % num_kv_heads;"),
    "causal_off_by_one": ("int ntok = pos + 1;", "int ntok = pos;"),
    "prefill_ignores_prior": ("row_pos[first + j] = L - n + j;", "row_pos[first + j] = j + (n == 1 ? L - 1 : 0);"),
    "wrong_row_in_block": ("t % block_size) * head_dim;\n            double acc",
                           "(t + 1) % block_size) * head_dim;\n            double acc"),
    "scale_dropped": ("x[t] = scale * acc;", "x[t] = acc;"),
    "max_not_subtracted": ("double w = exp(x[t] - m);", "double w = exp(x[t]);"),
    "no_normalisation": ("o[j] /= den;", "o[j] /= (den > 0 ? 1.0 : 1.0);"),
    "values_from_keys": ("o[j] += w * (widen(v_cache,", "o[j] += w * (widen(k_cache,"),
    "append_wrong_head": ("size_t src = ((size_t)i * num_kv_heads + g) * row;",
                          "size_t src = ((size_t)i * num_kv_heads + (num_kv_heads - 1 - g)) * row;"),
    "copy_only_keys": ("memmove((char *)v_cache + dst * blk", "if (0) memmove((char *)v_cache + dst * blk"),
    "bf16_wrong_half": ("bits = ((uint32_t)h) << 16;", "bits = ((uint32_t)h) << 15;"),
    "e4m3_ties_to_odd": ("(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    "e4m3_max_code_missing": ("for (int c = 0; c < 127; c++)", "for (int c = 0; c < 126; c++)"),
    "e4m3_subnormal_exponent": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3_bias_off_by_one": ("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    "fp8_append_scale_ignored": ("oracle_e4m3_encode(xk / k_scale[g]);", "oracle_e4m3_encode(xk);"),
    "fp8_value_scale_dropped": ("* (widen(v_cache, vbase + j, kv_dtype) * vs);",
                                "* (widen(v_cache, vbase + j, kv_dtype) * 1.0);"),
}


def _run(name, tmp):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"mutant {name}: anchor not found"
    mutated = src.replace(before, after, 1)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    open(c, "w").write(mutated)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", so, c, "-lm"])
    env = dict(os.environ, PKV_ORACLE_LIB=so, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(4) as ex:
            codes = dict(zip(MUTANTS, ex.map(lambda n: _run(n, tmp), MUTANTS)))
    survived = [n for n, rc in codes.items() if rc == 0]
    assert not survived, f"mutants not caught by any pin: {survived}"
