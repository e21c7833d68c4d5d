"""Mutation check for the oracle's pins (CPU only).

Each case plants one plausible mistake in a temporary copy of the oracle's C
source, builds it, and re-runs the pins of tests/test_oracle.py against it. At
least one pin must fail for every mistake; otherwise the pins would not pin.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "wq_oracle.c")

MUTATIONS = {
    "nibble_order_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "unpack_unsigned": ("nib >= 8 ? nib - 16 : nib", "nib"),
    "group_index_off_by_one": ("(g > 0) ? k / g : 0", "(g > 0) ? (k + 1) / g : 0"),
    "channel_index_dropped": ("(Ns == 1) ? 0 : n", "0"),
    "offset_scaled": ("if (O) wk += so_at(O, Gs, Ns, g, k, n);",
                      "if (O) wk += so_at(O, Gs, Ns, g, k, n) * so_at(S, Gs, Ns, g, k, n);"),
    "bias_dropped": ("(bias ? bias[n] : 0.0)", "0.0"),
    "residual_dropped": ("double yv = v + residual[m * N + n];", "double yv = v;"),
    "mean_over_wrong_dim": ("ss / (double)N + eps", "ss / (double)(N + 1) + eps"),
    "eps_outside_sqrt": ("sqrt(ss / (double)N + eps)", "(sqrt(ss / (double)N) + eps)"),
    "gamma_reversed": ("yv / rms * gamma[n]", "yv / rms * gamma[N - 1 - n]"),
    "x_reversed_k": ("double xk = x1[m * K + k];", "double xk = x1[m * K + (K - 1 - k)];"),
    "weight_row_shifted": ("double wk = (double)q[k * N + n]", "double wk = (double)q[((k + 1) % K) * N + n]"),
    "tiled_t_and_jl_swapped": ("int64_t h = kk / 32, t = (kk % 32) / 8, jl = (kk % 8) / 4, e = kk % 4;",
                               "int64_t h = kk / 32, jl = (kk % 32) / 16, t = (kk % 16) / 4, e = kk % 4;"),
    "tiled_upper_nibble_pairs": ("int64_t p = (e < 2 ? 0 : 2) + upper + 4 * (e % 2);",
                                 "int64_t p = (e < 2 ? 0 : 4) + upper + 2 * (e % 2);"),
    "fp4_tie_to_odd": ("(dc == db && (c % 2 == 0))", "(dc == db && (c % 2 == 1))"),
    "fp4_max_magnitude_8": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 8.0}"),
    "mx_slice_of_32_off": ("k < K && k < 32 * (j + 1)", "k < K && k < 32 * (j + 1) + 1"),
    "mx_scale2_transposed": ("(int)s2[j * N + n] - 127", "(int)s2[n * J + j] - 127"),
    "dq_round_half_away": ("float rr = rintf(r);", "float rr = roundf(r);"),
    "dq_scale_off_by_one": ("volatile float s = amax / (float)qmax;", "volatile float s = amax / (float)(qmax + 1);"),
    "dq_smooth_ignored": ("if (smooth) v = v * smooth[k];", "(void)smooth;"),
    "dq_max_not_abs": ("float a = fabsf(v);", "float a = v;"),
    "tiled_word_major_in_tile": ("* 512 + lane * 16 + j * 4 + p / 2;", "* 512 + j * 128 + lane * 4 + p / 2;"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames, values = params[0].args[0], params[0].args[1]
            argnames = [a.strip() for a in argnames.split(",")]
            for v in values:
                v = v if isinstance(v, (tuple, list)) else (v,)
                out.append((f"{name}{v}", fn, dict(zip(argnames, v))))
        else:
            out.append((name, fn, {}))
    return out


@pytest.mark.parametrize("mut", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(mut, tmp_path):
    old, new = MUTATIONS[mut]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {mut} not found exactly once"
    csrc = tmp_path / "mut.c"
    csrc.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", "-std=c11", "-o", str(so),
                           str(csrc), "-lm"])
    failed = []
    with oracle.use_library(str(so)):
        for name, fn, kw in _pin_functions():
            try:
                fn(**kw)
            except Exception:  # noqa: BLE001 - any failure counts as caught
                failed.append(name)
    assert failed, f"no pin failed for planted mistake '{mut}'"
