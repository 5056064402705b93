"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake (a dropped term, a wrong sign or index, a transposed operand, a
wrong constant or rounding rule) in a temporary copy of ``oracle/sp_oracle.cpp``, builds it, and
runs the codec and invariant pin suites against that build in a child process: at least one pin
must fail. The committed oracle is never modified.
"""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

from oracle import build as oracle_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "drop_last_partial": ("for (int r = 0; r < a.tp; ++r)", "for (int r = 0; r < a.tp - 1; ++r)"),
    "transposed_partials": ("a.partials[(r * a.T_pad + t) * H + j]", "a.partials[(t * a.tp + r) * H + j]"),
    "drop_bias": ("h[j] = s + b + res + add;", "h[j] = s + res + add + 0 * b;"),
    "drop_residual": ("h[j] = s + b + res + add;", "h[j] = s + b + add + 0 * res;"),
    "bias_sign": ("h[j] = s + b + res + add;", "h[j] = s - b + res + add;"),
    "drop_addend": ("h[j] = s + b + res + add;", "h[j] = s + b + res + 0 * add;"),
    "addend_row_index": ("a.addend[t * H + j]", "a.addend[j]"),
    "partial_scale_ignored": ("s += ps * bf16_value(", "s += bf16_value("),
    "partial_scale_on_everything": ("h[j] = s + b + res + add;",
                                    "h[j] = s + ps * (b + res + add);"),
    "residual_row_index": ("a.residual[t * H + j]", "a.residual[j]"),
    "eps_outside_sqrt": ("1.0 / std::sqrt(mean_sq + static_cast<double>(a.eps))",
                         "1.0 / (std::sqrt(mean_sq) + static_cast<double>(a.eps))"),
    "sum_not_mean": ("sum_sq / static_cast<double>(H)", "sum_sq / static_cast<double>(H + 0 * H + 1)"),
    "drop_weight": ("y[j] = h[j] * inv_rms * bf16_value(a.weight[j]);", "y[j] = h[j] * inv_rms;"),
    "static_scale_multiplies": ("as_fp32(y[j] / scale)", "as_fp32(y[j] * scale)"),
    "per_token_qmax": ("amax / 448.0", "amax / 240.0"),
    "nvfp4_nibble_order": ("lo | (hi << 4)", "hi | (lo << 4)"),
    "nvfp4_scale_no_div6": ("gs * amax / 6.0", "gs * amax / 4.0"),
    "padding_off_by_one": ("if (t >= a.T_valid) {", "if (t > a.T_valid) {"),
    "round_half_away": ("std::nearbyint(a / quantum)", "std::round(a / quantum)"),
    "no_subnormals": ("std::max(e2 - 1, emin)", "(e2 - 1)"),
    "e4m3_max_480": ("{4, 3, 7, 448.0, true}", "{4, 3, 7, 480.0, true}"),
    "bf16_saturates": ("std::ldexp(255.0, 120), false}", "std::ldexp(255.0, 120), true}"),
    "fc2_contiguous_batch_ids": ("ids[j * P + k] = j + k * D;", "ids[j * P + k] = j * P + k;"),
    "fc2_member_order": ("out + i * row_out + m * row_in", "out + i * row_out + (D - 1 - m) * row_in"),
    "swizzle_row_terms_swapped": ("(r % 32) * 16 + (r / 32) * 4 + c", "(r / 32) * 16 + (r % 32) * 4 + c"),
    "residual_out_unrounded_sum": ("a.residual_out[t * H + j] = bf16_code(h[j]);",
                                   "a.residual_out[t * H + j] = bf16_code(h[j] - bf16_value(a.weight[j]) + 1.0);"),
}


def _run_mutant(name: str, old: str, new: str, workdir: str) -> tuple[str, int, str]:
    with open(oracle_build.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, f"{name}: pattern not found"
    src = src.replace(old, new)
    cpp = os.path.join(workdir, f"{name}.cpp")
    lib = os.path.join(workdir, f"lib_{name}.so")
    with open(cpp, "w") as f:
        f.write(src)
    oracle_build.build(cpp, lib, extra_flags=["-w"])
    env = dict(os.environ, SP_ORACLE_LIBRARY=lib)
    proc = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         "tests/test_oracle_codecs.py", "tests/test_oracle_invariants.py",
         "tests/test_oracle_fc2.py"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, proc.returncode, proc.stdout[-400:]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            results = list(ex.map(lambda kv: _run_mutant(kv[0], *kv[1], tmp), MUTANTS.items()))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"mutants not caught by any pin: {survivors}"
    assert all(rc == 1 for _, rc, _ in results), [(n, rc, o) for n, rc, o in results if rc != 1]


def test_unmutated_copy_passes():
    with tempfile.TemporaryDirectory() as tmp:
        name, rc, out = _run_mutant("identity", "namespace {", "namespace {", tmp)
    assert rc == 0, out
