"""Plant plausible mistakes in a copy of the oracle and check that the pins catch
each one.  The original oracle source is never modified: each mutant is a
patched copy compiled into a temporary directory and run in a child process
(a broken index can crash it, which also counts as caught)."""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

# (name, text in pkv_oracle.c, replacement) -- each replaced once
MUTATIONS = [
    ("gqa_modulo_mapping", "const int hkv = hq / group;", "const int hkv = hq % a->n_kv_heads;"),
    ("q_row_uses_kv_head", "((int64_t)b * a->n_q_heads + hq) * D",
     "((int64_t)b * a->n_q_heads + hkv) * D"),
    ("k_slot_off_by_one", "a->k_pool + (((int64_t)page * a->n_kv_heads + hkv) * P + (t % P)) * D",
     "a->k_pool + (((int64_t)page * a->n_kv_heads + hkv) * P + ((t + 1) % P)) * D"),
    ("v_pool_transposed", "a->v_pool + (((int64_t)page * a->n_kv_heads + hkv) * P + (t % P)) * D",
     "a->v_pool + (((int64_t)hkv * a->num_pages + page) * P + (t % P)) * D"),
    ("page_index_mod", "const int32_t page = a->table[(int64_t)b * a->table_stride + t / P];\n"
                       "        if (page < 0",
     "const int32_t page = a->table[(int64_t)b * a->table_stride + t % P];\n"
     "        if (page < 0"),
    ("scale_dropped", "s[t] = a->scale * dot;", "s[t] = dot;"),
    ("exp_sign_flipped", "const double w = exp(s[t] - M);", "const double w = exp(M - s[t]);"),
    ("no_max_shift", "double M = s[0];", "double M = 0.0;"),
    ("no_normalisation", "out_row[d] /= den;", "out_row[d] /= 1.0;"),
    ("last_token_dropped", "for (int t = 0; t < L; ++t) {\n            const int32_t page",
     "for (int t = 0; t + 1 < L; ++t) {\n            const int32_t page"),
    ("exponent_bias_off", "const int bias = (1 << (ebits - 1)) - 1;",
     "const int bias = (1 << (ebits - 1));"),
    ("subnormal_scale", "mag = ldexp((double)m, 1 - bias - mbits);",
     "mag = ldexp((double)m, -bias - mbits);"),
    ("append_slot_off_by_one", "* page_size + p % page_size) * head_dim;",
     "* page_size + (p + 1) % page_size) * head_dim;"),
    ("append_ignores_padding", "if (p < 0) continue;\n        const int32_t page = table",
     "if (p < -1) continue;\n        const int32_t page = table"),
    ("gather_slot_wrong", "* page_size + t % page_size) * head_dim;",
     "* page_size + t % (page_size - 1)) * head_dim;"),
    ("rope_wrong_partner", "const double x1 = pkv_oracle_decode_bits(x[row + half + i], dtype);",
     "const double x1 = pkv_oracle_decode_bits(x[row + (half + i + 1) % head_dim], dtype);"),
    ("rope_sine_sign", "const double y0 = x0 * c - x1 * sn;", "const double y0 = x0 * c + x1 * sn;"),
    ("rope_frequency_exponent", "pow(theta, -2.0 * i / head_dim)", "pow(theta, -1.0 * i / head_dim)"),
    ("encode_ties_away", "double r = nearbyint(ldexp(a, mbits - e));",
     "double r = round(ldexp(a, mbits - e));"),
    ("encode_no_carry", "if (r == ldexp(1.0, mbits + 1)) {", "if (r == ldexp(1.0, mbits + 2)) {"),
    ("encode_subnormal_spacing", "nearbyint(ldexp(a, mbits - emin))",
     "nearbyint(ldexp(a, mbits - emin + 1))"),
    ("multi_query_causal_off_by_one", "const int n_att = lens[b] - n_queries + j + 1;",
     "const int n_att = lens[b] - n_queries + j;"),
    ("multi_query_sees_all_tokens", "const int n_att = lens[b] - n_queries + j + 1;",
     "const int n_att = lens[b];"),
    ("multi_query_early_row_sees_all", "n_att > 0 ? n_att : 0, out + r * head_dim",
     "n_att, out + r * head_dim"),
    ("norm_sum_not_mean", "const double inv_rms = 1.0 / sqrt(ss / head_dim + eps);",
     "const double inv_rms = 1.0 / sqrt(ss + eps);"),
    ("norm_weight_of_partner", "pkv_oracle_decode_bits(w[d], dtype);",
     "pkv_oracle_decode_bits(w[(d + head_dim / 2) % head_dim], dtype);"),
    ("norm_eps_dropped_twice", "const double inv_rms = 1.0 / sqrt(ss / head_dim + eps);",
     "const double inv_rms = 1.0 / sqrt(ss / head_dim + 2.0 * eps + 1e-3);"),
]

RUNNER = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, oracle_pins
    orc = oracle.Oracle({lib!r})
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except Exception as e:
            failed.append(check.__name__)
            break  # one failing pin is enough to catch a mutant
    print("FAILED:", ",".join(failed))
    sys.exit(1 if failed else 0)
""")


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / "mut.c"
    c.write_text(mutated)
    lib = tmp_path / "libmut.so"
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(c), "-o", str(lib),
                        "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=str(lib))
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert p.returncode != 0, f"mutation {name} survived every pin:\n{p.stdout}\n{p.stderr}"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness on an unmodified copy passes every pin."""
    c = tmp_path / "same.c"
    shutil.copy(SRC, c)
    lib = tmp_path / "libsame.so"
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(c), "-o", str(lib),
                        "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=str(lib))
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
