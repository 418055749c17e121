"""The pins must be strong enough to catch a plausible slip in the oracle.

Each case plants one mistake in a temporary copy of ``oracle/oracle.c`` (on the CPU),
builds it, and runs the pin suite against it with ``ORACLE_SO``; the suite must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "attention residual dropped":
        ("for (int i = 0; i < dim; i++) m->x[i] = m->x[i] + m->tmp[i];\n        orc_rmsnorm(m->xn, m->x, L->ffn_norm",
         "for (int i = 0; i < dim; i++) m->x[i] = m->tmp[i];\n        orc_rmsnorm(m->xn, m->x, L->ffn_norm"),
    "rope sign flipped": ("u[i] = a * c - b * s;", "u[i] = a * c + b * s;"),
    "rope adjacent pairs": ("float b = u[i + half];", "float b = u[i ^ 1];"),
    "rope frequency exponent": ("-2.0 * (double)i / (double)head_dim", "-1.0 * (double)i / (double)head_dim"),
    "gqa head mapping modulo": ("int g = h / group;\n            orc_attend(m->o", "int g = h % KV;\n            orc_attend(m->o"),
    "matvec transposed": ("acc = acc + row[j] * x[j];", "acc = acc + w[(size_t)j * n_out + i] * x[j];"),
    "rmsnorm mean over n-1": ("float ms = ss / (float)n;", "float ms = ss / (float)(n - 1);"),
    "rmsnorm missing gain": ("out[i] = (x[i] * r) * g[i];", "out[i] = x[i] * r;"),
    "attention scale sqrt missing": ("float scale = 1.0f / sqrtf((float)head_dim);", "float scale = 1.0f / (float)head_dim;"),
    "attention excludes current position":
        ("pos + 1, hd, m->scores);", "(pos > 0 ? pos : 1), hd, m->scores);"),
    "silu uses the wrong sign": ("h[i] = (a[i] / (1.0f + expf(-a[i]))) * b[i];", "h[i] = (a[i] / (1.0f + expf(a[i]))) * b[i];"),
    "swiglu gate and up swapped":
        ("orc_silu_mul(m->h, m->a, m->b, c->hidden);", "orc_silu_mul(m->h, m->b, m->a, c->hidden);"),
    "argmax last index on tie": ("if (x[i] > x[best]) best = i;", "if (x[i] >= x[best]) best = i;"),
    "bf16 round truncates": ("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0u;"),
    "kv written one slot late": ("float *kd = m->kc + kv_index(m, l, seq, g, pos);",
                                 "float *kd = m->kc + kv_index(m, l, seq, g, pos + 1 < c->max_seq ? pos + 1 : pos);"),
    "final norm skipped": ("orc_matvec(logits, m->emb, m->xn, dim, c->vocab);", "orc_matvec(logits, m->emb, m->x, dim, c->vocab);"),
}


# block-quantised int8 weights: caught by tests/test_oracle_q8.py
Q8_MUTANTS = {
    "q8 halves to even": ("float v = s > 0.0f ? roundf(w[i] / s) : 0.0f;", "float v = s > 0.0f ? rintf(w[i] / s) : 0.0f;"),
    "q8 scale over 128": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "q8 blocks of 16": ("b1 = b0 + ORC_Q8_BLOCK < n ? b0 + ORC_Q8_BLOCK : n;", "b1 = b0 + 16 < n ? b0 + 16 : n;"),
    "q8 embedding left unquantised": ("int rc = q8_dequantize_rows((float *)m->emb, (size_t)c->vocab, (int)dim);",
                                      "int rc = ORC_OK;"),
    "q8 w2 blocks along the output axis": ("rc = q8_dequantize_rows((float *)L->w2, dim, (int)hid);",
                                           "rc = q8_dequantize_rows((float *)L->w2, hid, (int)dim);"),
}
PIN_FILE = {name: "test_oracle_pins.py" for name in MUTANTS}
PIN_FILE.update({name: "test_oracle_q8.py" for name in Q8_MUTANTS})
MUTANTS.update(Q8_MUTANTS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique for {name!r}"
    mut = tmp_path / "oracle.c"
    mut.write_text(src.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    so = tmp_path / "liboracle.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                    "-o", str(so), str(mut), "-lm"], check=True)
    env = dict(os.environ, ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", PIN_FILE[name])],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
