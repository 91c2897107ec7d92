"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
in ``test_oracle_pins.py`` and ``test_oracle_bwd_pins.py`` catch every one of
them.

Each mutant is ``oracle/ora.c`` with one textual change, compiled into a
temporary library and loaded by a child pytest run through ``RA_ORACLE_LIB``.
The child run must fail; the unmodified source must pass.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ora.c")

MUTANTS = {
    "dropped_scale": [("return J->scale * acc;", "return acc;")],
    "gqa_modulo_mapping": [("int g = h / (J->H / J->Hkv);", "int g = h % J->Hkv;")],
    "causal_excludes_diagonal": [("int n_allowed = J->causal ? s + 1 : J->S;",
                                  "int n_allowed = J->causal ? (s > 0 ? s : 1) : J->S;"),
                                 ("t1 = s + 1; /* keys", "t1 = (s > 0 ? s : 1); /* keys")],
    "lse_log2": [("J->lse[r] = M + log(L);", "J->lse[r] = M + log2(L);"),
                 ("J->lse[r] = m + log(l);", "J->lse[r] = m + log2(l);")],
    "fold_weight_sign": [("exp(m - mn);", "exp(mn - m);")],
    "fold_drops_old_accumulator": [("o[d] = o[d] * a + oc[d] * c;", "o[d] = oc[d] * c;")],
    "key_row_uses_query_index": [("(((int64_t)b * J->S + t) * J->Hkv + g) * J->D;\n    double acc",
                                  "(((int64_t)b * J->S + s) * J->Hkv + g) * J->D;\n    double acc")],
    "value_row_off_by_one": [("return J->v + (((int64_t)b * J->S + t)",
                              "return J->v + (((int64_t)b * J->S + (t + 1) % J->S)")],
    "merge_weight_uses_max": [("double w = exp(lp - L);", "double w = exp(lp - M);")],
    "block_ignores_key_offset": [("if (causal && k_pos0 + t > q_pos0 + s) {",
                                  "if (causal && t > q_pos0 + s) {")],
    "block_empty_row_not_zeroed": [("                if (!any) {\n                    *l = -INFINITY;",
                                    "                if (!any) {\n                    o[0] = 1.0;\n                    *l = -INFINITY;")],
    "ring_skips_last_chunk": [("for (int step = 0; step < J->P; ++step)",
                               "for (int step = 0; step < J->P - (J->P > 1); ++step)")],
    # backward pass
    "bwd_drops_delta": [("const double ds = x[t] * (dp[t] - delta);",
                         "const double ds = x[t] * dp[t];")],
    "bwd_dk_unscaled": [("dk[kv + d] += J->scale * ds * widen_bf16(qr[d]);",
                         "dk[kv + d] += ds * widen_bf16(qr[d]);")],
    "bwd_dv_uses_ds": [("dv[kv + d] += x[t] * widen_bf16(dor[d]);",
                        "dv[kv + d] += ds * widen_bf16(dor[d]);")],
    "bwd_dp_uses_query": [("acc += widen_bf16(dor[d]) * widen_bf16(vr[d]);",
                           "acc += widen_bf16(dor[d]) * widen_bf16(qr[d]);")],
    "bwd_dq_uses_value_rows": [("const uint16_t *kr = J->k + kv;", "const uint16_t *kr = J->v + kv;")],
    "bwd_group_mapping": [("const int D = J->D, g = h / (J->H / J->Hkv);",
                           "const int D = J->D, g = h % J->Hkv;")],
    "bwd_causal_excludes_diagonal": [("    const int n_allowed = J->causal ? s + 1 : J->S;",
                                      "    const int n_allowed = J->causal ? (s > 0 ? s : 1) : J->S;")],
    "bwd_delta_unweighted": [("delta += x[t] * acc;", "delta += acc;")],
    "bwd_given_output_row_misread": [("delta += widen_bf16(dor[d]) * widen_bf16(outr[d]);",
                                      "delta += widen_bf16(dor[d]) * widen_bf16(outr[0]);")],
}


def _child(env_lib):
    env = dict(os.environ)
    if env_lib:
        env["RA_ORACLE_LIB"] = env_lib
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                           os.path.join(ROOT, "tests", "test_oracle_bwd_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _build(src_text, out_dir, name):
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", so, c, "-lm", "-lpthread"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    so = _build(src, str(tmp_path), name)
    r = _child(so)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


def test_unmutated_source_passes(tmp_path):
    so = _build(open(SRC).read(), str(tmp_path), "clean")
    r = _child(so)
    assert r.returncode == 0, r.stdout[-3000:]
