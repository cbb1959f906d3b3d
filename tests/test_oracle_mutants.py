"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the pins catch them.

Each mutant is a one-token edit of ``oracle/x3conv_oracle.c`` compiled into a temporary
library; the pin functions of ``test_oracle_pins`` are then run against it, and at least one must
fail. This shows that the pins constrain every part of the oracle they are meant to constrain.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "x3conv_oracle.c")

MUTANTS = {
    "flipped_kernel_rows": ("const int ih = stride * oh + kh - 1;", "const int ih = stride * oh + 1 - kh;"),
    "pad_offset_cols": ("const int iw = stride * ow + kw - 1;", "const int iw = stride * ow + kw;"),
    "weight_kh_kw_swapped": ("* 3 + kh) * 3 + kw] *\n                                       x[",
                             "* 3 + kw) * 3 + kh] *\n                                       x["),
    "bias_dropped_2d": ("float acc = b ? b[co] : 0.0f;\n                    for (int ci",
                        "float acc = 0.0f;\n                    for (int ci"),
    "temporal_order_reversed": ("const int f = t + kt;", "const int f = t + 2 - kt;"),
    "carry_frames_swapped": ("* 2 + f) * plane;", "* 2 + (1 - f)) * plane;"),
    "relu_missing": ("return v < 0.0f ? 0.0f : v;", "return v;"),
    "clamp_lower_bound": ("fmaxf(-1.0f, v)", "fmaxf(0.0f, v)"),
    "f16_ties_away": ("if (rem > 0x1000u || (rem == 0x1000u && (keep & 1u))) keep += 1u;",
                      "if (rem >= 0x1000u) keep += 1u;"),
    "bf16_truncates": ("if (rem > 0x8000u || (rem == 0x8000u && (keep & 1u))) keep += 1u;", ""),
    "unpatchify_dy_dx_swapped": ("c * 4 + dy * 2 + dx", "c * 4 + dx * 2 + dy"),
    "stride_ignored_rows": ("const int ih = stride * oh + kh - 1;", "const int ih = oh + kh - 1;"),
    "two_pass_g_not_rounded": ("if (round_g) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));", ""),
    "two_pass_tap_transposed": ("(i * 3 + j) * 12 + c];", "(j * 3 + i) * 12 + c];"),
    "two_pass_bias_dropped": ("float acc = b ? b[c] : 0.0f;", "float acc = 0.0f;"),
}


def _pins():
    """(name, callable(oracle_module)) for every pin, with fixed parameters."""
    pins = [
        ("f16_encode", P.test_f16_encode_matches_numpy),
        ("bf16_encode", P.test_bf16_encode_matches_torch),
        ("torch2d_s1", lambda m: P.test_conv2d_vs_torch_f64(m, 1)),
        ("torch2d_s2", lambda m: P.test_conv2d_vs_torch_f64(m, 2)),
        ("torch3d", P.test_conv3d_vs_torch_f64_causal),
        ("brute3d", lambda m: P.test_conv3d_vs_brute_force(m, (1, 2, 3, 2, 3, 4), True)),
        ("int_exact", lambda m: P.test_conv2d_integer_exact_vs_int64(m, "int")),
        ("identity", P.test_identity_and_delta_kernels),
        ("unpatchify", P.test_unpatchify_is_a_bijection),
        ("act_rounding", P.test_act_commutes_with_rounding),
        ("head_split", P.test_head_split_identity),
        ("head_exact", P.test_head_two_pass_exact_when_g_is_representable),
        ("head_rounds_g", P.test_head_two_pass_rounds_g_before_the_spatial_sum),
    ]
    for case in P._golden_cases():
        pins.append((case["name"], lambda m, c=case: P.test_hand_worked_values(m, c)))
    return pins


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_oracle_mutants_are_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    cpath = tmp_path / "mutant.c"
    cpath.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-o", str(so),
                    str(cpath), "-lm"], check=True)
    saved = oracle._lib
    oracle._lib = oracle.configure(ctypes.CDLL(str(so)))
    caught = []
    try:
        for pin_name, fn in _pins():
            try:
                fn(oracle)
            except AssertionError:
                caught.append(pin_name)
    finally:
        oracle._lib = saved
    assert caught, f"no pin caught the planted mistake {name}"
