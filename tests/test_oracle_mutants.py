"""Planted mistakes: each test compiles a copy of the oracle's C source with one
plausible error written into it (on the CPU, in a temporary directory) and
checks that at least one of the oracle pins rejects that copy.  This shows the
pins constrain every term of the definition, not only the oracle as written.
"""
import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "A_positive": ("double A = -exp(A_log_c[n]);", "double A = exp(A_log_c[n]);"),
    "dA_without_dt": ("double dA = exp(dt * A);", "double dA = exp(A);"),
    "dB_without_dt": ("double dB = dt * Bt[n];", "double dB = Bt[n];"),
    "input_before_silu": ("h[n] = dA * h[n] + dB * u;", "h[n] = dA * h[n] + dB * pre;"),
    "readout_with_D_slip": ("yss += Ct[n] * h[n];", "yss += Dc * h[n];"),
    "readout_of_previous_state": (
        "h[n] = dA * h[n] + dB * u;\n        yss += Ct[n] * h[n];",
        "yss += Ct[n] * h[n];\n        h[n] = dA * h[n] + dB * u;"),
    "skip_dropped": ("yss += Dc * u;", ""),
    "gate_without_silu": ("return yss * silu(z);", "return yss * z;"),
    "conv_taps_reversed": ("pre += w_c[k] * s[k];\n    pre += w_c[K - 1] * x;",
                           "pre += w_c[K - 1 - k] * s[k];\n    pre += w_c[0] * x;"),
    "conv_state_shift_wrong_end": ("if (K > 1) s[K - 2] = x;", "if (K > 1) s[0] = x;"),
    "softplus_threshold_wrong": ("v > 20.0 ? v :", "v > 2.0 ? v :"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "chunk_carry_without_decay": ("P[n] * H[(size_t)j * N + n] + h[n]",
                                  "H[(size_t)j * N + n] + h[n]"),
    "final_h_not_written": ("final_h[((size_t)b * D + c) * N + n] = h[n];",
                            "final_h[((size_t)b * D + c) * N + n] = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"lib_{name}.so"))
    failed = []
    try:
        pins.LIB["lib"] = oracle._load(path)
        for pin in pins.PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
                break
    finally:
        pins.LIB["lib"] = None
    assert failed, f"no pin rejects the mutant {name}"
