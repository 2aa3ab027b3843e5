"""The pins catch planted mistakes (CPU only).

Each case copies the oracle's C source, plants one plausible mistake in it (a
single textual edit), builds the copy with the oracle's own gcc flags and runs
the pin suite against it in a fresh process; at least one pin must fail.  A
control case builds the unchanged source the same way and must pass, so a
broken harness cannot pass for a caught mistake.  The copies live in a
temporary directory; the oracle itself is not touched.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_finalize_oracle.c")

# (name, text in the source, replacement, occurrences replaced)
MUTATIONS = [
    ("eps outside the square root", "1.0 / sqrt(sum_sq / (double)hidden + eps)",
     "1.0 / (sqrt(sum_sq / (double)hidden) + eps)", 1),
    ("negative indices valid", "if (i < 0 || i >= rows)", "if (i >= rows)", 1),
    ("index == rows valid", "if (i < 0 || i >= rows)", "if (i < 0 || i > rows)", 1),
    ("gain dropped after the norm", "y = v[h] * r * (double)g;", "y = v[h] * r;", 1),
    ("gain center dropped", "bf16_bits_to_float(norm_weight[h]) + gain_center",
     "bf16_bits_to_float(norm_weight[h])", 2),
    ("mean over hidden + 1", "sum_sq / (double)hidden", "sum_sq / (double)(hidden + 1)", 1),
    ("index map transposed", "int64_t i = idx[t * top_k + k];",
     "int64_t i = idx[k * num_tokens + t];", 1),
    ("weight of the wrong slot", "w = ((const float *)weights)[t * top_k + k];",
     "w = ((const float *)weights)[t * top_k];", 1),
    ("packed word's high half taken", "[t * top_k + k] & 0xFFFFu)", "[t * top_k + k] >> 16)", 1),
    ("Beam round before the scale dropped",
     "float scaled = bf16_bits_to_float(rounded) * routed_scale;",
     "float scaled = acc[h] * routed_scale;", 1),
    ("Beam round after the scale dropped",
     "v[h] = bf16_bits_to_double(oracle_bf16_from_double((double)scaled));",
     "v[h] = (double)scaled;", 1),
    ("post_weight ignored", "double gamma = post_weight ? bf16_bits_to_double(post_weight[h]) : 1.0;",
     "double gamma = 1.0;", 1),
    ("residual scales swapped", "fmaf(scale_residual, r, scale_x * x)",
     "fmaf(scale_x, r, scale_residual * x)", 1),
    ("residual dropped", "float sum = fmaf(scale_residual, r, scale_x * x);",
     "float sum = scale_x * x;", 1),
    ("hidden not rounded before the next norm", "v[h] = bf16_bits_to_double(b);",
     "v[h] = (double)sum;", 1),
    ("next_weight ignored", "double gamma = next_weight ? bf16_bits_to_double(next_weight[h]) : 1.0;",
     "double gamma = 1.0;", 1),
    ("post_eps used by the next norm", "inverse_rms(v, hidden, (double)next_eps)",
     "inverse_rms(v, hidden, (double)post_eps)", 1),
    ("ties rounded away from zero", "rint(x / spacing)", "round(x / spacing)", 1),
    ("sign lost", "return (uint16_t)(u >> 16);", "return (uint16_t)((u >> 16) & 0x7FFFu);", 1),
    ("slots summed in descending order", "for (int32_t k = 0; k < top_k; ++k) {",
     "for (int32_t k = top_k - 1; k >= 0; --k) {", 1),
    ("gain applied on the wrong side of the norm",
     "v[h] = weight_before_norm ? (double)acc[h] * (double)g : (double)acc[h];",
     "v[h] = !weight_before_norm ? (double)acc[h] * (double)g : (double)acc[h];", 1),
    ("FP32 reduction replaced by a plain multiply-add",
     "acc[h] = fmaf(w, bf16_bits_to_float(x[h]), acc[h]);",
     "acc[h] = acc[h] + w * bf16_bits_to_float(x[h]);", 1),
    ("gain center added in float64", "float g = bf16_bits_to_float(norm_weight[h]) + gain_center;",
     "double g = (double)bf16_bits_to_float(norm_weight[h]) + (double)gain_center;", 2),
    ("Beam scale product in float64",
     "float scaled = bf16_bits_to_float(rounded) * routed_scale; /* FP32 product */",
     "double scaled = (double)bf16_bits_to_float(rounded) * (double)routed_scale;", 1),
    ("residual sum in float64", "float sum = fmaf(scale_residual, r, scale_x * x);",
     "double sum = (double)scale_residual * r + (double)scale_x * x;", 1),
    ("routed_scale applied before the first round",
     "uint16_t rounded = oracle_bf16_from_double((double)acc[h]);",
     "uint16_t rounded = oracle_bf16_from_double((double)(acc[h] * routed_scale));\n"
     "            routed_scale = 1.0f;", 1),
    ("unweighted post norm skipped", "if (!has_post_norm) {",
     "if (!has_post_norm || !post_weight) {", 1),
    ("eps divided by hidden", "sum_sq / (double)hidden + eps)", "sum_sq / (double)hidden + eps / hidden)", 1),
]


def _build(source: str, tmp_path, name: str) -> str:
    import oracle
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(source)
    subprocess.run(["gcc", *oracle.GCC_FLAGS, str(c), "-o", str(so), "-lm"], check=True)
    return str(so)


def _pins_pass(so: str) -> bool:
    env = dict(os.environ, MF_ORACLE_SO=so)
    p = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_golden.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return p.returncode == 0


def test_unchanged_source_passes_the_pins(tmp_path):
    assert _pins_pass(_build(open(SRC).read(), tmp_path, "unchanged"))


@pytest.mark.parametrize("name,old,new,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new, count):
    src = open(SRC).read()
    assert src.count(old) == count, f"the text to mutate occurs {src.count(old)} times"
    mutated = src.replace(old, new)
    assert mutated != src
    assert not _pins_pass(_build(mutated, tmp_path, "mutant")), f"no pin caught: {name}"
