"""The oracle's pins must catch plausible mistakes (CPU only).

Each case plants one mistake in a private copy of oracle.c (a dropped term, a
wrong sign or index, a reversed tie rule, an off-by-one), builds it into a
temporary library and runs the oracle pin tests against it in a subprocess.
Every planted mistake must make at least one pin fail.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MISTAKES = {
    "causal mask drops the diagonal": ("int64_t n = t - s0 + 1;", "int64_t n = t - s0 + (t == s0);"),
    "wrong GQA head mapping": ("int kvh = h / G;\n    int64_t b = seq_of_token",
                               "int kvh = h % Hkv;\n    int64_t b = seq_of_token"),
    "softmax scale dropped": ("double s = scale * dot;", "double s = dot;"),
    "LSE sign": ("if (lse) *lse = m + log(l);", "if (lse) *lse = m - log(l);"),
    "value operand transposed": (
        "for (int64_t j = 0; j < n; ++j) acc += score_buf[j] * bf16_bits_to_f64(vals[j][d]);",
        "for (int64_t j = 0; j < n; ++j) acc += score_buf[j] * bf16_bits_to_f64(vals[d % n][j % D]);"),
    "parent index ignored": ("int src = parent ? parent[b] : b;", "int src = b;"),
    "new row appended one slot late": ("} else if (s == L_prev && append) {",
                                       "} else if (s == L_prev + 1 && append) {"),
    "suffix read from the wrong KV head": (
        "keys[Lp + s] = ks_out + (((int64_t)b * Smax + s) * Hkv + kvh) * D;",
        "keys[Lp + s] = ks_out + (((int64_t)b * Smax + s) * Hkv + 0) * D;"),
    "log-prob sign": ("float lp = x - lse[b];", "float lp = x + lse[b];"),
    "cumulative score dropped": ("float sc = cum[b] + lp;", "float sc = lp;"),
    "token tie rule reversed": ("if (a->v != c->v) return a->v < c->v ? -1 : 1;",
                                "if (a->v != c->v) return a->v > c->v ? -1 : 1;"),
    "parent tie rule reversed": ("if (a->b != c->b) return a->b < c->b ? -1 : 1;",
                                 "if (a->b != c->b) return a->b > c->b ? -1 : 1;"),
    "log-normaliser without the sum": ("lse_out[b] = (float)(m + log(s));", "lse_out[b] = (float)(m);"),
    "logit tie rule reversed": ("if (a->x > c->x) return -1;", "if (a->x < c->x) return -1;"),
    "logit tie key dropped": ("if (a->x > c->x) return -1;\n    if (a->x < c->x) return 1;\n", ""),
}

PIN_FILES = ["test_oracle_prefill.py", "test_oracle_decode.py", "test_oracle_select.py"]


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MISTAKES[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for '{name}' not found exactly once"
    c_path = tmp_path / "oracle_mut.c"
    lib = tmp_path / "liboracle_mut.so"
    c_path.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    str(c_path), "-o", str(lib), "-lm"], check=True)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider"]
                       + [os.path.join(HERE, f) for f in PIN_FILES],
                       env=dict(os.environ, SLM_ORACLE_LIB=str(lib)), cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin:\n{r.stdout[-2000:]}"
