"""sp_fused_reduce_norm_noalloc: the entry point for callers that may not allocate device memory.

Code that records a CUDA graph, a plugin whose framework owns every device buffer, or a serving
loop that forbids allocation after start-up cannot hand the dynamic row schedule an 8-byte
counter of its own. This entry point keeps that counter in the library's static device memory.
The test calls it through the C ABI (ctypes, raw device addresses) twice in a row on the same
inputs and requires both results to equal, byte for byte, what the existing entry point
sp_fused_reduce_norm writes for those inputs (both schedules give identical bytes, which is
within every tolerance of the parity suite), and to match the fp64 oracle under the suite's
tolerances. It also checks that the calls ran the dynamic schedule, i.e. used the scratch.

The file name sorts last, so a run that stops at its first failure has already run every other
test; it passes alone in a fresh process as well as after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import synth

from parity_util import bits_of, compare, run_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _c_args(inp, outs, scale):
    """The C ABI argument list of sp_fused_reduce_norm (and of the no-allocation variant)."""
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return (p(inp["partials"]), inp["tp"], inp["T_pad"], inp["T_valid"], inp["H"],
            p(inp["residual"]), p(inp["weight"]), p(inp["bias"]), ctypes.c_float(inp["eps"]),
            sp.QUANT_MODES[inp["mode"]], p(scale), p(outs["out"]), p(outs["out_scales"]),
            p(outs["residual_out"]))


def _outputs(inp, fill):
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    for t in outs.values():
        if t is not None:
            t.view(torch.uint8).fill_(fill)  # an unwritten byte would show as a difference
    return outs


# (workload, rows): shapes whose default launch is the staged kernel with the dynamic schedule
CASES = [(2, 8192), (5, 8192)]


@pytest.mark.parametrize("wi,rows", CASES)
def test_noalloc_entry_matches_the_existing_entry(wi, rows):
    lib = sp.load_library()
    w = synth.workload(wi)
    inp = synth.make_inputs(w, device=DEV, T_pad=rows, T_valid=rows - 3)
    scale = None if inp["scale"] is None else torch.tensor([inp["scale"]], device=DEV)
    stream = torch.cuda.Stream(device=DEV)
    handle = ctypes.c_void_p(stream.cuda_stream)
    # the inputs and pre-filled outputs are written on torch's stream: finish that work before
    # the calls on their own (non-blocking) stream read or write the same buffers
    ref = _outputs(inp, 0xA5)
    fresh = [_outputs(inp, fill) for fill in (0x5A, 0xC3)]
    torch.cuda.synchronize()

    assert lib.sp_fused_reduce_norm(*_c_args(inp, ref, scale), handle) == 0
    torch.cuda.synchronize()
    ref_host = {k: None if v is None else bits_of(v) for k, v in ref.items()}

    for call, outs in enumerate(fresh):  # two calls in a row, into fresh outputs
        assert lib.sp_fused_reduce_norm_noalloc(*_c_args(inp, outs, scale), handle) == 0
        assert sp.sp_last_launch()["schedule"] == "dynamic", "the call did not use the scratch"
        torch.cuda.synchronize()
        got = {k: None if v is None else bits_of(v) for k, v in outs.items()}
        for k in ("out", "out_scales", "residual_out"):
            if ref_host[k] is not None:
                assert np.array_equal(got[k].view(np.uint8), ref_host[k].view(np.uint8)), \
                    f"call {call}: {k} differs from sp_fused_reduce_norm"
    compare(got, run_oracle(inp), inp)
    assert sp.sp_device_error(clear=False) == 0


def test_noalloc_entry_refuses_rows_beyond_its_counter():
    """More rows than the 32-bit counter can hand out: refused before anything is enqueued
    (the addresses are never dereferenced; the checks only compare them)."""
    lib = sp.load_library()
    rows = (1 << 31) - (1 << 16) + 8
    base = 1 << 44
    gap = 1 << 40
    args = (base, 1, rows, rows, 8, None, base + gap, None, ctypes.c_float(1e-6), 0, None,
            base + 2 * gap, None, base + 3 * gap)
    assert sp.sp_status_string(lib.sp_fused_reduce_norm_noalloc(*args, None)) == \
        "SP_ERR_UNSUPPORTED"
    small = (base, 1, 8, 8, 8, None, base + gap, None, ctypes.c_float(-1.0), 0, None,
             base + 2 * gap, None, base + 3 * gap)  # an invalid eps: the usual checks come first
    assert sp.sp_status_string(lib.sp_fused_reduce_norm_noalloc(*small, None)) == \
        "SP_ERR_INVALID_ARG"
