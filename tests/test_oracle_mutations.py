"""Plant mistakes in a copy of the oracle (on the CPU) and check that the pins catch
each one: a pin that no plausible slip can fail pins nothing."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lora_oracle.c")

MUTATIONS = {
    "dropped_scale": ("acc += h[j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);\n            y[t * d_out + n] += s * acc;",
                      "acc += h[j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);\n            y[t * d_out + n] += acc;"),
    "expand_scale": ("(double)hin[t * ldh + j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);\n            y[t * d_out + n] += s * acc;",
                     "(double)hin[t * ldh + j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);\n            y[t * d_out + n] += acc;"),
    "transposed_A": ("/* shrink: x . A_i (d_in -> r) */\n            double acc = 0.0;\n            for (int64_t k = 0; k < d_in; ++k)\n                acc += oracle_bf16_to_double(x[t * ldx + k]) * pool_elem(&p, desc[i].a_page0, j * d_in + k, &oob);",
                     "/* shrink: x . A_i (d_in -> r) */\n            double acc = 0.0;\n            for (int64_t k = 0; k < d_in; ++k)\n                acc += oracle_bf16_to_double(x[t * ldx + k]) * pool_elem(&p, desc[i].a_page0, k * r + j, &oob);"),
    "transposed_B": ("acc += h[j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);",
                     "acc += h[j] * pool_elem(&p, desc[i].b_page0, n * r + j, &oob);"),
    "wrong_sign": ("acc += h[j] * pool_elem", "acc -= h[j] * pool_elem"),
    "page_offset": ("return oracle_bf16_to_double(p->pool[page * p->page_elems + e % p->page_elems]);",
                    "return oracle_bf16_to_double(p->pool[page * p->page_elems + (e + 1) % p->page_elems]);"),
    "page_slot": ("int64_t slot = page0 + e / p->page_elems;\n    if (slot < 0 || slot >= p->n_page_list) { *bad = 1; return 0.0; }",
                  "int64_t slot = page0 + (e / p->page_elems) / 2;\n    if (slot < 0 || slot >= p->n_page_list) { *bad = 1; return 0.0; }"),
    "unstable_group": ("for (int32_t t = 0; t < T; ++t)              /* ascending token index */",
                       "for (int32_t t = T - 1; t >= 0; --t)        /* descending */"),
    "ties_away": ("double r = nearbyint(v / q) * q;", "double r = round(v / q) * q;"),
    "sizing_bytes": ("return (d_in * rank + rank * d_out) * bytes_per_param;",
                     "return (d_in * rank + rank * d_out) * 2;"),
    "y0_dropped": ("y[t * d_out + n] = oracle_bf16_to_double(y0[t * ldy0 + n]);\n        int32_t i = ids[t];\n        if (i == -1) continue;\n        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }\n        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);\n        if (bad || desc[i].rank > 256)",
                   "y[t * d_out + n] = (ids[t] >= 0) ? 0.0 : oracle_bf16_to_double(y0[t * ldy0 + n]);\n        int32_t i = ids[t];\n        if (i == -1) continue;\n        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }\n        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);\n        if (bad || desc[i].rank > 256)"),
    "grad_dA_scale": ("+= s * u[j] * oracle_bf16_to_double(x[t * ldx + k]);",
                      "+= u[j] * oracle_bf16_to_double(x[t * ldx + k]);"),
    "grad_dB_transposed": ("grad[pool_pos(&p, desc[i].b_page0, j * d_out + n)]",
                           "grad[pool_pos(&p, desc[i].b_page0, n * r + j)]"),
    "grad_u_from_A": ("acc += oracle_bf16_to_double(g[t * ldg + n]) * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);",
                      "acc += oracle_bf16_to_double(g[t * ldg + n]) * pool_elem(&p, desc[i].b_page0, n * r + j, &oob);"),
    "grad_dx_dropped_scale": ("dx[t * d_in + k] = s * acc;", "dx[t * d_in + k] = acc;"),
    "base_weight_column": ("* oracle_bf16_to_double(w0[n * ldw + k]);", "* oracle_bf16_to_double(w0[n * ldw + (k + 1) % d_in]);"),
    "base_dropped_under_adapter": ("y[t * d_out + n] += s * term;", "y[t * d_out + n] = s * term;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found once: " + name
    mutated = tmp_path / "lora_oracle.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liblora_oracle_mut.so"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(lib), str(mutated), "-lm"])
    env = dict(os.environ, LORA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, "pins did not catch mutation %s:\n%s" % (name, r.stdout[-2000:])
