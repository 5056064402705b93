"""Write ``nvfp4_global_scale.json``: the static NVFP4 global scale of the NVFP4 workload.

The pages fix no value for NVFP4's fp32 global scale (vLLM SP/AsyncTP/quant notes §四 only say
the blocks carry their own scales and never cross a rank). The usual static calibration maps the
largest magnitude to the top of E4M3 block scale x E2M1 code, 448 * 6 = 2688:

    gs = 2688 / max |y|

with y taken from the fp64 oracle on a 256-row draw of the workload (its own seed), rounded to
three significant digits. Only the oracle and the seeded input generator are used.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from sequence_reduce_add_gb300 import synth  # noqa: E402

ROWS = 256


def calibrate() -> float:
    w = synth.workload("tp8_T16384_H5120_nvfp4")
    w["mode"] = "none"  # draw the same tensors; only y is needed
    inp = synth.make_inputs(w, T_pad=ROWS, T_valid=ROWS, seed=synth.BASE_SEED + 5)
    res = oracle.fused_reduce_norm(
        synth.bf16_bits(inp["partials"]), synth.bf16_bits(inp["residual"]),
        synth.bf16_bits(inp["weight"]), synth.bf16_bits(inp["bias"]), inp["eps"], "none", None,
        ROWS, want_y=True, threads=os.cpu_count() or 1)
    assert res["status"] == 0
    amax = float(np.abs(res["y"]).max())
    return float(f"{2688.0 / amax:.3g}"), amax


if __name__ == "__main__":
    gs, amax = calibrate()
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "nvfp4_global_scale.json")
    with open(out, "w") as f:
        json.dump({"global_scale": gs, "amax_y": amax, "rows": ROWS,
                   "written_by": "tests/golden/calibrate_nvfp4_global_scale.py"}, f, indent=2)
        f.write("\n")
    print(out, gs, amax)
