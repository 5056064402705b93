"""Per-call status, the staged kernel's abort path, and the dynamic schedule's row counters, on
the GPU and without a fault.

* A call may pass a status word (options.status); a normal call leaves it zero.
* sp_selftest_fused_timeout runs the real staged kernel with a short wait limit while CTA 0's
  producer never fills one ring stage: the consumer warps' waits on it run out, all of them
  leave together, the drain of that stage runs out too, and the launch ends. The test checks the
  launch returns within a bounded time, the call's status word (or, for a call without one, the
  device error word) reads SP_DEVICE_ERR_WAIT_TIMEOUT while the other word stays clear, and the
  next normal call on the same context matches the oracle. Withholding a row's index stage (dynamic schedule) exercises the index wait's vote;
  withholding a segment mid-row exercises the segment waits' vote.
* A caller's own row counter (options.row_counter) gives the dynamic schedule on any stream and
  inside a captured graph; sp_last_launch tells which schedule a call ran, so the per-stream
  table's behaviour is visible: beyond its 256 slots a new stream takes over an idle slot, also
  while another host thread records a graph.
"""
import ctypes
import os
import subprocess
import sys
import time

import numpy as np
import pytest
import torch

import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import synth

from parity_util import bits_of, compare, run_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIMEOUT = 1  # SP_DEVICE_ERR_WAIT_TIMEOUT


def _small(w, rows, pad=5, **kw):
    tp = kw.get("tp", w["tp"])
    T_pad = tp * -(-rows // tp)
    return synth.make_inputs(w, device=DEV, T_pad=T_pad, T_valid=max(T_pad - pad, 0), **kw)


def _host(outs):
    return {k: (None if v is None else bits_of(v)) for k, v in outs.items()}


def _scale(inp):
    return None if inp["scale"] is None else torch.tensor([inp["scale"]], device=DEV)


def _call(inp, outs, options, stream=None):
    sp.sp_fused_reduce_norm_ex(options, inp["partials"], inp["weight"], outs["out"],
                               outs["residual_out"], residual=inp["residual"], bias=inp["bias"],
                               eps=inp["eps"], quant_mode=inp["mode"], scale=_scale(inp),
                               out_scales=outs["out_scales"], T_valid=inp["T_valid"],
                               stream=stream)


def _words(n):
    return torch.zeros(n, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("wi", [2, 3, 4, 5])
@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_status_word_stays_zero_on_normal_calls(wi, schedule):
    inp = _small(synth.workload(wi), rows=1024)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    status = _words(4)
    _call(inp, outs, sp.sp_options_init(schedule=schedule, status=status))
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert sp.sp_last_launch()["schedule"] == schedule
    compare(_host(outs), run_oracle(inp), inp)


# (workload, schedule, stage withheld in CTA 0). Workload 2 at 1024 rows: 5 segments per row.
# Static: the first stage, and a stage in the middle of CTA 0's second row. Dynamic: the first
# stage (row b's index and first segment), a mid-row segment, and the second row's index stage.
SELFTEST_CASES = [(2, "static", 0, True), (2, "static", 7, True), (2, "dynamic", 0, True),
                  (2, "dynamic", 3, True), (2, "dynamic", 5, True), (4, "dynamic", 2, True),
                  (5, "static", 4, True), (3, "static", 1, True), (2, "static", 2, False),
                  (5, "dynamic", 0, False)]


@pytest.mark.parametrize("wi,schedule,withhold,with_status", SELFTEST_CASES)
def test_staged_kernel_abort_path(wi, schedule, withhold, with_status):
    assert sp.sp_device_error(clear=True) == 0
    inp = _small(synth.workload(wi), rows=1024)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    status, counter = _words(4), _words(4)
    opts = sp.sp_options_init(schedule=schedule, status=status if with_status else None,
                              row_counter=counter if schedule == "dynamic" else None)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sp.sp_selftest_fused_timeout(20_000_000, withhold, opts, inp["partials"], inp["weight"],
                                 outs["out"], outs["residual_out"], residual=inp["residual"],
                                 bias=inp["bias"], eps=inp["eps"], quant_mode=inp["mode"],
                                 scale=_scale(inp), out_scales=outs["out_scales"],
                                 T_valid=inp["T_valid"])
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert sp.sp_last_launch()["config"]["kernel"] == 0  # the staged kernel ran
    assert sp.sp_last_launch()["schedule"] == schedule
    if with_status:  # the call's own word gets the report, the device word stays clear
        assert int(status[0]) == TIMEOUT
        assert sp.sp_device_error(clear=True) == 0
    else:
        assert sp.sp_device_error(clear=True) == TIMEOUT
    assert 0.015 <= elapsed < 1.5, elapsed
    # the context is usable and a normal call (fresh status, counter zeroed again) is right
    status.zero_()
    counter.zero_()
    outs2 = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    _call(inp, outs2, sp.sp_options_init(schedule=schedule, status=status,
                                         row_counter=counter if schedule == "dynamic" else None))
    torch.cuda.synchronize()
    assert int(status[0]) == 0 and sp.sp_device_error(clear=False) == 0
    assert not counter.any()
    compare(_host(outs2), run_oracle(inp), inp)


def test_withholding_a_stage_cta0_never_fills_changes_nothing():
    inp = _small(synth.workload(2), rows=1024)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    status = _words(4)
    sp.sp_selftest_fused_timeout(20_000_000, 10**9, sp.sp_options_init(status=status),
                                 inp["partials"], inp["weight"], outs["out"],
                                 outs["residual_out"], residual=inp["residual"], bias=inp["bias"],
                                 eps=inp["eps"], quant_mode=inp["mode"],
                                 out_scales=outs["out_scales"], T_valid=inp["T_valid"])
    torch.cuda.synchronize()
    assert int(status[0]) == 0 and sp.sp_device_error(clear=False) == 0
    compare(_host(outs), run_oracle(inp), inp)


def test_selftest_rejects_bad_arguments():
    inp = _small(synth.workload(2), rows=64)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    args = (inp["partials"], inp["weight"], outs["out"], outs["residual_out"])
    kw = dict(residual=inp["residual"], T_valid=inp["T_valid"])
    for limit, withhold in ((0, 0), (3_000_000_000, 0), (1_000_000, -1)):
        with pytest.raises(sp.SpError):
            sp.sp_selftest_fused_timeout(limit, withhold, None, *args, **kw)
    direct = sp.sp_options_init(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4))
    with pytest.raises(sp.SpError) as e:
        sp.sp_selftest_fused_timeout(1_000_000, 0, direct, *args, **kw)
    assert e.value.status == 2  # SP_ERR_UNSUPPORTED: the self-test runs the staged kernel


def test_caller_row_counter_on_streams_beyond_the_table():
    """More streams than the table's 256 slots: once the earlier streams' calls are done, a later
    stream takes over an idle slot and runs the dynamic schedule (sp_last_launch shows it) on a
    call that claims many rows from that slot; with a counter of its own it runs the dynamic
    schedule too. Both give the same bytes, and the caller's counter is zero again afterwards.
    Runs in a child process, so that this process's table is left as it was."""
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join(
        [os.path.dirname(here), here, os.environ.get("PYTHONPATH", "")]))
    proc = subprocess.run([sys.executable, os.path.abspath(__file__), "streams"], cwd=here,
                          env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-2000:]
    assert "streams ok" in proc.stdout


def _streams_beyond_the_table():
    inp = _small(synth.workload(3), rows=2048)
    rt = _cudart()
    handles = []
    for _ in range(257):
        h = ctypes.c_void_p()
        assert rt.cudaStreamCreateWithFlags(ctypes.byref(h), 1) == 0
        handles.append(h.value)
    try:
        small = _small(synth.workload(3), rows=16)
        so = sp.allocate_outputs(small["T_pad"], small["H"], small["mode"], DEV)
        torch.cuda.synchronize()  # inputs written on torch's stream before the raw streams read
        staged = dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=0)
        for h in handles:  # one dynamic staged call per stream takes (or finds) its slot
            _call(small, so, sp.sp_options_init(schedule="dynamic", launch=staged), stream=h)
        torch.cuda.synchronize()
        last = handles[-1]
        a = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
        _call(inp, a, sp.sp_options_init(schedule="dynamic"), stream=last)
        assert sp.sp_last_launch()["schedule"] == "dynamic"  # a reclaimed slot
        counter = _words(4)
        torch.cuda.synchronize()  # the counter's zeros written before `last` reads them
        b = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
        _call(inp, b, sp.sp_options_init(schedule="dynamic", row_counter=counter), stream=last)
        assert sp.sp_last_launch()["schedule"] == "dynamic"
        torch.cuda.synchronize()
        assert not counter.any()
        ha, hb = _host(a), _host(b)
        for k in ("out", "residual_out"):
            assert np.array_equal(ha[k].view(np.uint8), hb[k].view(np.uint8)), k
        compare(hb, run_oracle(inp), inp)
    finally:
        torch.cuda.synchronize()
        for h in handles:
            rt.cudaStreamDestroy(ctypes.c_void_p(h))
    print("streams ok")


def test_slot_reclaimed_while_another_thread_records_a_graph():
    """A call on a new stream that finds the counter table full reads the table back on the
    library's own stream. Made while another host thread records a CUDA graph in global capture
    mode (PyTorch's default), that read must neither fail nor break the recording: the call runs
    the dynamic schedule on a reclaimed slot and matches the oracle, and the graph, which holds
    a fused call of its own, replays to the oracle's result. Runs in a child process (it fills the
    table)."""
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join(
        [os.path.dirname(here), here, os.environ.get("PYTHONPATH", "")]))
    proc = subprocess.run([sys.executable, os.path.abspath(__file__), "capture"], cwd=here,
                          env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-2000:]
    assert "capture ok" in proc.stdout


def _reclaim_during_capture():
    import threading
    rt = _cudart()
    handles = []
    for _ in range(257):
        h = ctypes.c_void_p()
        assert rt.cudaStreamCreateWithFlags(ctypes.byref(h), 1) == 0
        handles.append(h.value)
    try:
        w = synth.workload(2)
        small = _small(w, rows=64)
        so = sp.allocate_outputs(small["T_pad"], small["H"], small["mode"], DEV)
        big = _small(w, rows=2048)
        bo = sp.allocate_outputs(big["T_pad"], big["H"], big["mode"], DEV)
        cap = _small(synth.workload(4), rows=330)
        co = sp.allocate_outputs(cap["T_pad"], cap["H"], cap["mode"], DEV)
        cap_stream = torch.cuda.Stream(device=DEV)
        dynamic, default = sp.sp_options_init(schedule="dynamic"), sp.sp_options_init()
        torch.cuda.synchronize()
        staged = sp.sp_options_init(schedule="dynamic", launch=dict(
            kernel=0, vec_per_thread=2, ctas_per_sm=1, stages=0))
        for h in handles[:256]:  # every slot of the table taken
            _call(small, so, staged, stream=h)
        _call(big, bo, dynamic, stream=handles[0])  # the big call's launch set up beforehand
        with torch.cuda.stream(cap_stream):
            _call(cap, co, default)  # and the captured call's
        torch.cuda.synchronize()  # every slot idle
        g = torch.cuda.CUDAGraph()
        inside, done, seen = threading.Event(), threading.Event(), {}

        def record():
            try:
                with torch.cuda.graph(g, stream=cap_stream):
                    _call(cap, co, default)
                    inside.set()
                    assert done.wait(120)
            except BaseException as e:  # reported by the main thread
                seen["error"] = e
                inside.set()

        t = threading.Thread(target=record)
        t.start()
        assert inside.wait(120)
        _call(big, bo, dynamic, stream=handles[256])
        schedule = sp.sp_last_launch()["schedule"]
        done.set()
        t.join(120)
        assert not t.is_alive()
        assert "error" not in seen, seen.get("error")
        assert schedule == "dynamic", schedule
        torch.cuda.synchronize()
        compare(_host(bo), run_oracle(big), big)
        for o in co.values():
            if o is not None:
                o.zero_()
        g.replay()
        torch.cuda.synchronize()
        compare(_host(co), run_oracle(cap), cap)
    finally:
        torch.cuda.synchronize()
        for h in handles:
            rt.cudaStreamDestroy(ctypes.c_void_p(h))
    print("capture ok")


def test_caller_row_counter_inside_a_captured_graph():
    """With its own counter a call keeps the dynamic schedule while its stream is captured; the
    graph replayed three times on refilled inputs gives the oracle's result each time."""
    w = synth.workload(4)
    inp = _small(w, rows=1024)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    counter = _words(4)
    s = torch.cuda.Stream(device=DEV)
    opts = sp.sp_options_init(schedule="dynamic", row_counter=counter)
    torch.cuda.synchronize()  # inputs written on torch's stream before `s` reads them
    with torch.cuda.stream(s):
        _call(inp, outs, opts)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _call(inp, outs, opts)
    assert sp.sp_last_launch()["schedule"] == "dynamic"
    for k in range(3):
        fresh = synth.make_inputs(w, device=DEV, T_pad=inp["T_pad"], T_valid=inp["T_valid"],
                                  seed=inp["seed"] + 17 * (k + 1))
        for name in ("partials", "residual", "weight", "bias"):
            inp[name].copy_(fresh[name])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert not counter.any()
        compare(_host(outs), run_oracle(fresh), fresh)


def test_last_launch_names_the_kernel():
    small = _small(synth.workload(1), rows=64, pad=0)
    outs = sp.allocate_outputs(small["T_pad"], small["H"], small["mode"], DEV)
    _call(small, outs, sp.sp_options_init())
    info = sp.sp_last_launch()
    want = sp.sp_select_launch(small["tp"], small["T_pad"], small["H"], small["mode"]).as_dict()
    assert info["config"]["kernel"] == want["kernel"] and info["schedule"] == "static"
    assert 0 < info["grid"] <= small["T_pad"] * max(1, want["split"])
    torch.cuda.synchronize()


def _cudart():
    import glob
    import os
    for name in ("libcudart.so", "libcudart.so.13", "libcudart.so.12"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    for path in glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart*.so*")):
        return ctypes.CDLL(path)
    pytest.skip("no CUDA runtime library to create raw streams")


if __name__ == "__main__" and sys.argv[1:] == ["streams"]:
    _streams_beyond_the_table()
if __name__ == "__main__" and sys.argv[1:] == ["capture"]:
    _reclaim_during_capture()
