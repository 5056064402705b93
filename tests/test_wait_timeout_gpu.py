"""Failure detection on the GPU without a fault: a bounded wait on a barrier that nothing
completes gives up after its limit, reports through the device error word, and the context stays
usable (the fused stage still runs and matches the oracle afterwards)."""
import time

import pytest
import torch

import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import synth

from parity_util import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    assert sp.sp_device_error(clear=True) == 0
    t0 = time.perf_counter()
    sp.sp_selftest_wait_timeout(20_000_000)  # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert sp.sp_device_error(clear=True) == 1  # SP_DEVICE_ERR_WAIT_TIMEOUT
    assert 0.015 <= elapsed < 1.5
    assert sp.sp_device_error(clear=False) == 0
    # the context is still usable
    inp = synth.make_inputs(synth.workload(1), device="cuda:0")
    compare(run_gpu(inp), run_oracle(inp), inp)
    assert sp.sp_device_error(clear=False) == 0


def test_selftest_rejects_bad_limits():
    with pytest.raises(sp.SpError):
        sp.sp_selftest_wait_timeout(0)
    with pytest.raises(sp.SpError):
        sp.sp_selftest_wait_timeout(3_000_000_000)
