"""Planted mistakes in the oracle, on the CPU: each variant below is oracle.c
with one plausible error written in (a swapped table entry, a wrong sign,
rounding direction or tie rule, a dropped term, a transposed operand, an index
one block off), compiled on its own and run against the pins of
test_oracle_pins.py.  A variant that passes every pin would be a mistake the
pins cannot see; each one must fail at least one of them.

The variants are built into a scratch folder under oracle/ and loaded through
ORACLE_LIB by a separate pytest process, so the oracle in use is never changed.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("e2m1_table_1.5_2_swapped",
     "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 2.0, 1.5, 3.0, 4.0, 6.0}"),
    ("e2m1_sign_dropped",
     "  double v = mag[code & 7];\n  return (code & 8) ? -v : v;", "  double v = mag[code & 7];\n  return v;"),
    ("ue8m0_bias_128", "return ldexp(1.0, s - 127);", "return ldexp(1.0, s - 128);"),
    ("e4m3_exponent_bias_off_by_one",
     "v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);"),
    ("e4m3_ties_to_odd_code",
     "  for (int c = 0; c <= 0x7E; ++c) {\n    double d = fabs(orc_e4m3_value(c) - a);\n"
     "    if (d < bestd || (d == bestd && (c % 2) == 0)) {",
     "  for (int c = 0; c <= 0x7E; ++c) {\n    double d = fabs(orc_e4m3_value(c) - a);\n"
     "    if (d < bestd || (d == bestd && (c % 2) == 1)) {"),
    ("fp8_block_scale_to_256_not_448",
     "while (e < 127 && amax > ldexp(448.0, e)) ++e;", "while (e < 127 && amax > ldexp(256.0, e)) ++e;"),
    ("bf16_round_truncates",
     "r = ldexp(rint(ldexp(a, 8 - E)), E - 8);", "r = ldexp(floor(ldexp(a, 8 - E)), E - 8);"),
    ("e2m1_encode_ties_to_odd_code",
     "  for (int c = 0; c <= 7; ++c) {\n    double d = fabs(orc_e2m1_value(c) - a);\n"
     "    if (d < bestd || (d == bestd && (c % 2) == 0)) {",
     "  for (int c = 0; c <= 7; ++c) {\n    double d = fabs(orc_e2m1_value(c) - a);\n"
     "    if (d < bestd || (d == bestd && (c % 2) == 1)) {"),
    ("fp4_block_scale_to_4_not_6",
     "while (e < 127 && amax > ldexp(6.0, e)) ++e;", "while (e < 127 && amax > ldexp(4.0, e)) ++e;"),
    ("fp4_activation_high_nibble_first",
     "(uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));", "(uint8_t)(c[2 * i + 1] | (c[2 * i] << 4));"),
    ("router_bias_dropped", "      if (b) acc += (double)b[e];", "      (void)b;"),
    ("router_logits_accumulated_in_fp32",
     "      double acc = 0.0;\n      for (int h = 0; h < H; ++h)\n        acc += orc_bf16_value",
     "      float acc = 0.0f;\n      for (int h = 0; h < H; ++h)\n        acc += (float)orc_bf16_value"),
    ("topk_ties_to_higher_index",
     "return (a->index < b->index) ? -1 : (a->index > b->index);",
     "return (a->index > b->index) ? -1 : (a->index < b->index);"),
    ("softmax_over_all_experts",
     "for (int j = 0; j < k; ++j) den += exp(a[j].key - m);",
     "for (int j = 0; j < E; ++j) den += exp(a[j].key - m);"),
    ("sigmoid_weights_include_the_bias",
     "w[(size_t)t * k + j] = (double)sc[a[j].index] / den * scale;",
     "w[(size_t)t * k + j] = ((double)sc[a[j].index] + (bias ? bias[a[j].index] : 0.0)) / den * scale;"),
    ("sigmoid_exp_sign_flipped",
     "float orc_sigmoid_f32(float l) { return 1.0f / (1.0f + orc_exp_f32(-l)); }",
     "float orc_sigmoid_f32(float l) { return 1.0f / (1.0f + orc_exp_f32(l)); }"),
    ("segments_slots_reversed_within_an_expert",
     "    for (int s = 0; s < S; ++s)\n      if (idx[s] == e) perm[p++] = s;",
     "    for (int s = S - 1; s >= 0; --s)\n      if (idx[s] == e) perm[p++] = s;"),
    ("weight_nibbles_swapped",
     "int code = (c % 2 == 0) ? (byte & 15) : (byte >> 4);", "int code = (c % 2 == 0) ? (byte >> 4) : (byte & 15);"),
    ("weight_scale_of_the_next_column_block",
     "orc_ue8m0_table[m->scales[(size_t)r * (K / 32) + c / 32]]",
     "orc_ue8m0_table[m->scales[(size_t)r * (K / 32) + (c / 32 + 1) % (K / 32)]]"),
    ("fp8_weight_block_scale_of_the_next_column_block",
     "orc_ue8m0_table[m->scales[(size_t)(r / 32) * (K / 32) + c / 32]]",
     "orc_ue8m0_table[m->scales[(size_t)(r / 32) * (K / 32) + (c / 32 + 1) % (K / 32)]]"),
    ("x_block_scale_dropped",
     "xh[c] = orc_act_value(act4, xq[c]) * orc_ue8m0_value(xs[c / 32]);", "xh[c] = orc_act_value(act4, xq[c]);"),
    ("silu_on_the_up_projection", "h[i] = g / (1.0 + exp(-g)) * u;", "h[i] = u / (1.0 + exp(-u)) * g;"),
    ("h_not_quantised_before_down",
     "hh[i] = orc_act_value(act4, hq[i]) * orc_ue8m0_value(hs[i / 32]);", "hh[i] = h[i];"),
    ("shared_experts_dropped", "for (int s = 0; s < n_shared; ++s) {", "for (int s = 0; s < 0; ++s) {"),
    ("routing_weight_not_applied",
     "acc[r] += w[(size_t)t * k + j] * o[r];", "acc[r] += o[r];"),
    ("residual_added_before_y_is_rounded",
     "yb = orc_bf16_round(orc_bf16_value(residual[p]) + orc_bf16_value(yb));",
     "yb = orc_bf16_round(orc_bf16_value(residual[p]) + acc[r]);"),
    ("rmsnorm_mean_over_h_minus_1",
     "double inv = 1.0 / sqrt(ss / H + eps);", "double inv = 1.0 / sqrt(ss / (H - 1) + eps);"),
]


def _run_pins(name: str, old: str, new: str, scratch: str) -> tuple[int, str]:
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the planted text must occur exactly once in oracle.c"
    d = os.path.join(scratch, name)
    os.makedirs(d)
    with open(os.path.join(d, "oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(d, "liboracle.so")
    oracle.compile_library(os.path.join(d, "oracle.c"), lib)
    env = dict(os.environ, ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-1000:]


@pytest.fixture(scope="module")
def outcomes():
    scratch = tempfile.mkdtemp(prefix="_mutants_", dir=os.path.join(ROOT, "oracle"))
    try:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            futs = {m[0]: ex.submit(_run_pins, *m, scratch) for m in MUTANTS}
            yield {n: f.result() for n, f in futs.items()}
    finally:
        shutil.rmtree(scratch, ignore_errors=True)


def test_unchanged_oracle_passes_the_pins(tmp_path_factory):
    # the harness itself: oracle.c copied and built the same way passes
    scratch = tempfile.mkdtemp(prefix="_mutants_", dir=os.path.join(ROOT, "oracle"))
    try:
        rc, out = _run_pins("unchanged", "static double orc_ue8m0_table[256];",
                            "static double orc_ue8m0_table[256];", scratch)
    finally:
        shutil.rmtree(scratch, ignore_errors=True)
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(outcomes, name):
    rc, out = outcomes[name]
    # pytest exits 1 when a test failed; anything else (a crash, a collection
    # error) would not show that a pin caught the mistake
    assert rc == 1 and " failed" in out, f"{name} passed every pin or did not run cleanly:\n{out}"
