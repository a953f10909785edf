"""The oracle's pins must be able to fail.

Each case plants one plausible mistake in a private copy of oracle.c (on the
CPU, in a temporary directory), rebuilds it, and runs the pin tests against the
mutated copy: every mutation must make at least one pin fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "rope_interleaved_pairs": ("double x0 = v[i], x1 = v[i + half];\n        v[i] = x0 * c - x1 * s;\n"
                               "        v[i + half] = x1 * c + x0 * s;",
                               "double x0 = v[2*i], x1 = v[2*i+1];\n        v[2*i] = x0 * c - x1 * s;\n"
                               "        v[2*i+1] = x1 * c + x0 * s;"),
    "rope_sign": ("v[i] = x0 * c - x1 * s;", "v[i] = x0 * c + x1 * s;"),
    "rope_frequency": ("-(2.0 * (double)i) / (double)hd", "-((double)i) / (double)hd"),
    "gqa_head_map": ("int g = h / group;", "int g = h % kvh;"),
    "causal_off_by_one": ("vcache + base, pos + 1, hd", "vcache + base, pos, hd"),
    "rms_eps_outside_sqrt": ("1.0 / sqrt(ss / (double)n + eps)", "1.0 / (sqrt(ss / (double)n) + eps)"),
    "rms_sum_not_mean": ("1.0 / sqrt(ss / (double)n + eps)", "1.0 / sqrt(ss + eps)"),
    "attention_unscaled": ("s[t] = acc * scale;", "s[t] = acc;"),
    "silu_sign": ("return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    "kv_rounding": ("kcache[base + d] = oracle_round_bf16(k[(int64_t)g * hd + d]);",
                    "kcache[base + d] = (uint16_t)(oracle_round_bf16(k[(int64_t)g * hd + d]) ^ 1);"),
    "residual_dropped": ("for (int i = 0; i < H; ++i) x[i] += o[i];\n        /* segment C",
                         "for (int i = 0; i < H; ++i) x[i] = o[i];\n        /* segment C"),
    "gate_up_swapped": ("u[j] = oracle_silu(gate[j]) * up[j];", "u[j] = oracle_silu(up[j]) * gate[j];"),
    "topp_own_mass_included": ("const int kept = above < top_p * z;", "const int kept = above + grp < top_p * z;"),
    "topp_untempered": ("x[v] = y * inv_temp;", "x[v] = y;"),
    "q8_truncating_codes": ("if (sg > 0.0f) c = rintf((float)bf2d(W[idx]) / sg);",
                            "if (sg > 0.0f) c = truncf((float)bf2d(W[idx]) / sg);"),
    "q8_scale_255": ("const float sg = amax / 127.0f;", "const float sg = amax / 255.0f;"),
    "q8_down_row_scaled": ("oracle_gemv_q8(m->q8->q[k][l], m->q8->s[k][l], k == 6, rows, cols, x, y);",
                           "oracle_gemv_q8(m->q8->q[k][l], m->q8->s[k][l], 0, rows, cols, x, y);"),
    "q4_scale_8": ("const float s4 = amax / 7.0f;", "const float s4 = amax / 8.0f;"),
    "q4_signed_max": ("amax = fabsf(w) > amax ? fabsf(w) : amax;", "amax = w > amax ? w : amax;"),
    "q4_truncating_codes": ("rintf((float)bf2d(W[at]) / s4)", "truncf((float)bf2d(W[at]) / s4)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    a, b = MUTATIONS[name]
    assert src.count(a) == 1, f"mutation anchor for {name} no longer matches oracle.c"
    ign = shutil.ignore_patterns("_build", "__pycache__")
    for d in ("oracle", "synth", "tests"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d, ignore=ign)
    (tmp_path / "oracle" / "oracle.c").write_text(src.replace(a, b))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} was not caught:\n{r.stdout[-2000:]}"
