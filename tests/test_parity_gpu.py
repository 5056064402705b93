"""GPU parity: the CUDA library against the fp64 oracle, element by element, through the C ABI.

Every case draws seeded inputs (padding rows NaN-filled), runs the library twice into
guard-banded outputs pre-filled with two different byte patterns (so an unwritten byte shows
up as a difference), checks the guard bands, and compares every output with the oracle under
the tolerances in parity_util. Cases cover every workload's tp / H / mode on a few hundred rows
(several rows per CTA, a ragged padded tail) under each launch configuration, the edge cases
(all padding, one row per shard, smallest and largest H, no residual / no bias, in-place
residual, odd tp, a side stream), and the five workloads at full size in the configuration the
bench launches.
"""
import ctypes

import numpy as np
import pytest
import torch

import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import synth

from parity_util import bits_of, compare, run_gpu, run_gpu_host, run_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _check(inp, config=None, inplace=False, stream=None, schedule="auto"):
    a = run_gpu(inp, config=config, fill=0xA5, inplace=inplace, stream=stream, schedule=schedule)
    b = run_gpu(inp, config=config, fill=0x5A, inplace=inplace, stream=stream, schedule=schedule)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), \
                f"{k}: bytes left unwritten or a non-deterministic result"
    ref = run_oracle(inp)
    return compare(a, ref, inp)


def _small(w, rows=330, pad=5, **kw):
    tp = kw.get("tp", w["tp"])
    T_pad = tp * -(-rows // tp)
    return synth.make_inputs(w, device=DEV, T_pad=T_pad, T_valid=max(T_pad - pad, 0), **kw)


CONFIGS = [
    None,
    dict(kernel=0, vec_per_thread=1, ctas_per_sm=1, stages=0),
    dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=0),
    dict(kernel=0, vec_per_thread=2, ctas_per_sm=1, stages=2),
    dict(kernel=0, vec_per_thread=4, ctas_per_sm=3, stages=3),
    dict(kernel=1, vec_per_thread=1, ctas_per_sm=2, stages=0),
    dict(kernel=1, vec_per_thread=2, ctas_per_sm=1, stages=0),
    dict(kernel=1, vec_per_thread=4, ctas_per_sm=4, stages=0),
]


def _supported(config, H):
    if config is None:
        return True
    threads = -(-(H // 8) // config["vec_per_thread"])
    return threads <= 512


@pytest.mark.parametrize("wi", range(1, 6))
@pytest.mark.parametrize("ci", range(len(CONFIGS)))
def test_workload_rows(wi, ci):
    w = synth.workload(wi)
    cfg = CONFIGS[ci]
    if not _supported(cfg, w["H"]):
        pytest.skip("vectors per thread too few for this H")
    try:
        stats = _check(_small(w), config=cfg)
    except sp.SpError as e:
        if e.status == 2:  # SP_ERR_UNSUPPORTED: this forced configuration does not fit this H
            pytest.skip(str(e))
        raise
    assert stats


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
def test_all_padding(mode):
    w = dict(synth.workload(2), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, T_pad=8, T_valid=0, tp=2, H=256)
    _check(inp)


@pytest.mark.parametrize("T_valid", [1, 15, 16])
@pytest.mark.parametrize("mode", ["none", "fp8_per_token", "nvfp4"])
def test_one_row_per_shard(T_valid, mode):
    w = dict(synth.workload(4), mode=mode)
    inp = synth.make_inputs(w, device=DEV, T_pad=16, T_valid=T_valid, H=2048)
    _check(inp)


@pytest.mark.parametrize("H,mode", [(8, "none"), (8, "fp8_static"), (8, "fp8_per_token"),
                                    (16, "nvfp4"), (1000, "none"), (1000, "fp8_per_token"),
                                    (1008, "nvfp4"), (2056, "fp8_static"), (16384, "none"),
                                    (16384, "nvfp4"), (12288, "fp8_per_token")])
def test_hidden_sizes(H, mode):
    w = dict(synth.workload(3), mode=mode, outliers=min(7, H // 8))
    if mode == "nvfp4":
        w["scale"] = None
    inp = synth.make_inputs(w, device=DEV, T_pad=200, T_valid=197, tp=4, H=H)
    for cfg in (None, dict(kernel=1, vec_per_thread=4, ctas_per_sm=1, stages=0)):
        _check(inp, config=cfg)


@pytest.mark.parametrize("with_residual,with_bias", [(False, True), (True, False), (False, False)])
@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
def test_optional_residual_and_bias(with_residual, with_bias, mode):
    w = dict(synth.workload(2), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, T_pad=400, T_valid=397, H=4096,
                            with_residual=with_residual, with_bias=with_bias)
    for cfg in (None, dict(kernel=1, vec_per_thread=2, ctas_per_sm=2, stages=0)):
        _check(inp, config=cfg)


@pytest.mark.parametrize("mode", ["none", "fp8_per_token", "nvfp4"])
def test_in_place_residual(mode):
    w = dict(synth.workload(5), mode=mode)
    inp = synth.make_inputs(w, device=DEV, T_pad=320, T_valid=317)
    _check(inp, inplace=True)


@pytest.mark.parametrize("tp", [1, 3, 5])
def test_odd_tp(tp):
    w = dict(synth.workload(3))
    inp = synth.make_inputs(w, device=DEV, T_pad=tp * 70, T_valid=tp * 70 - 2, tp=tp, H=3072)
    _check(inp)


def test_side_stream():
    w = synth.workload(2)
    inp = _small(w)
    s = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()  # the inputs are written on torch's stream; `s` does not wait for it
    with torch.cuda.stream(s):
        _check(inp, stream=s)


@pytest.mark.parametrize("wi", range(1, 6))
def test_full_size_workload(wi):
    """The workload at full size, launched exactly as the bench launches it."""
    w = synth.workload(wi)
    inp = synth.make_inputs(w, device=DEV)
    stats = _check(inp)
    print(w["name"], stats)


@pytest.mark.parametrize("wi,rows", [(1, None), (2, 330), (3, 330), (4, 330), (5, 330), (2, None)])
def test_host_buffers_zero_copy(wi, rows):
    """sp_fused_reduce_norm_host: inputs and outputs in pinned host memory."""
    w = synth.workload(wi)
    inp = synth.make_inputs(w, device=DEV) if rows is None else _small(w, rows=rows)
    a = run_gpu_host(inp, fill=0xA5)
    b = run_gpu_host(inp, fill=0x5A)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp), inp)


def test_host_entry_rejects_pageable_memory():
    w = synth.workload(1)
    inp = synth.make_inputs(w, device="cpu")  # pageable host tensors
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], "none", "cpu")
    # the binding refuses pageable tensors before calling the library ...
    with pytest.raises(ValueError, match="page-locked"):
        sp.sp_fused_reduce_norm_host(inp["partials"], inp["weight"], outs["out"],
                                     outs["residual_out"], residual=inp["residual"],
                                     bias=inp["bias"], T_valid=inp["T_valid"])
    # ... and the C entry point refuses their raw addresses itself
    p = lambda t: t.data_ptr()  # noqa: E731
    st = sp.load_library().sp_fused_reduce_norm_host(
        p(inp["partials"]), inp["tp"], inp["T_pad"], inp["T_valid"], inp["H"], p(inp["residual"]),
        p(inp["weight"]), p(inp["bias"]), ctypes.c_float(inp["eps"]), 0, None, p(outs["out"]),
        None, p(outs["residual_out"]), None)
    assert st == 1


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("c,with_addend,with_residual", [(0.5, True, True), (1.0 / 3.0, False, True),
                                                         (-1.25, True, False), (1.0, True, True)])
@pytest.mark.parametrize("host", [False, True])
def test_partial_scale_and_addend(mode, c, with_addend, with_residual, host):
    """sp_fused_reduce_norm_ex: h = c * sum_r p_r + bias + residual + addend."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, T_pad=336, T_valid=331, H=5120,
                            with_addend=with_addend, with_residual=with_residual)
    run = run_gpu_host if host else run_gpu
    a = run(inp, fill=0xA5, partial_scale=c)
    b = run(inp, fill=0x5A, partial_scale=c)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, partial_scale=c), inp)


@pytest.mark.parametrize("T_pad,H", [(336, 5120), (16, 80), (256, 1008), (136, 4096)])
@pytest.mark.parametrize("host", [False, True])
def test_swizzled_nvfp4_scales(T_pad, H, host):
    """NVFP4 block scales in the 128x4-tile layout: padded rows and columns zero, scales in place."""
    w = synth.workload(5)
    inp = synth.make_inputs(w, device=DEV, T_pad=T_pad, T_valid=T_pad - 3, H=H)
    run = run_gpu_host if host else run_gpu
    a = run(inp, fill=0xA5, scale_layout=1)
    b = run(inp, fill=0x5A, scale_layout=1)
    for k in ("out", "out_scales", "residual_out"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, scale_layout=1), inp)


E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _dequant_nvfp4(packed: torch.Tensor, scales_rm: torch.Tensor) -> torch.Tensor:
    lut = torch.tensor(E2M1_VALUES, dtype=torch.float64, device=packed.device)
    codes = torch.stack([packed & 0xF, packed >> 4], dim=-1).reshape(packed.shape[0], -1).long()
    sf = scales_rm.view(torch.float8_e4m3fn).to(torch.float64)
    return lut[codes] * sf.repeat_interleave(16, dim=1)


def test_swizzled_scales_feed_a_block_scaled_gemm():
    """cuBLASLt's NVFP4 block-scaled GEMM (torch._scaled_mm) reads the library's codes and swizzled
    scales; the product must equal the matmul of the values dequantised with the row-major
    scales of the same call."""
    M, K, N = 256, 1024, 256
    w = synth.workload(5)
    inp = synth.make_inputs(w, device=DEV, T_pad=M, T_valid=M, H=K)
    opts = lambda layout: sp.sp_options_init(scale_layout=layout)  # noqa: E731
    outs = {}
    for layout in (0, 1):
        o = sp.allocate_outputs(M, K, "nvfp4", DEV, scale_layout=layout)
        sp.sp_fused_reduce_norm_ex(opts(layout), inp["partials"], inp["weight"], o["out"],
                                   o["residual_out"], residual=inp["residual"], bias=inp["bias"],
                                   quant_mode="nvfp4",
                                   scale=torch.tensor([inp["scale"]], device=DEV),
                                   out_scales=o["out_scales"], T_valid=M)
        outs[layout] = o
    torch.cuda.synchronize()
    assert torch.equal(outs[0]["out"], outs[1]["out"])
    g = torch.Generator(device=DEV).manual_seed(9)
    b_codes = torch.randint(0, 256, (N, K // 2), generator=g, device=DEV, dtype=torch.uint8)
    b_codes[(b_codes & 0xF) == 0x8] ^= 0x8  # no negative zeros
    n_sb = 128 * -(-N // 128) * (-(-(K // 16) // 4) * 4)
    sb = torch.full((n_sb,), 0x38, dtype=torch.uint8, device=DEV)  # every B block scale = 1.0
    try:
        c = torch._scaled_mm(outs[1]["out"].view(torch.float4_e2m1fn_x2),
                             b_codes.view(torch.float4_e2m1fn_x2).t(),
                             scale_a=outs[1]["out_scales"].view(torch.float8_e4m3fn),
                             scale_b=sb.view(torch.float8_e4m3fn), out_dtype=torch.bfloat16)
    except (RuntimeError, NotImplementedError) as e:
        pytest.skip(f"no NVFP4 block-scaled GEMM in this torch build: {e}")
    a_deq = _dequant_nvfp4(outs[0]["out"], outs[0]["out_scales"])
    b_deq = _dequant_nvfp4(b_codes, torch.full((N, K // 16), 0x38, dtype=torch.uint8, device=DEV))
    ref = a_deq @ b_deq.t()
    err = (c.double() - ref).abs()
    tol = 1e-2 * ref.abs() + 1e-2 * ref.abs().max()
    assert bool((err <= tol).all()), f"max err {err.max().item()} vs scale {ref.abs().max().item()}"


def test_no_device_wait_ran_out():
    assert sp.sp_device_error(clear=False) == 0


def _call(inp, outs, stream=None):
    sc = None if inp["scale"] is None else torch.tensor([inp["scale"]], device=DEV)
    sp.sp_fused_reduce_norm(inp["partials"], inp["weight"], outs["out"], outs["residual_out"],
                            residual=inp["residual"], bias=inp["bias"], eps=inp["eps"],
                            quant_mode=inp["mode"], scale=sc, out_scales=outs["out_scales"],
                            T_valid=inp["T_valid"], stream=stream)


def _host(outs):
    from parity_util import bits_of
    return {k: (None if v is None else bits_of(v)) for k, v in outs.items()}


@pytest.mark.parametrize("wi", [2, 4, 5])
def test_cuda_graph_capture_and_replay(wi):
    """The call captured in a CUDA graph (with its programmatic-dependent-launch attribute) and
    replayed after the input buffers were refilled computes on the new contents."""
    w = synth.workload(wi)
    inp = _small(w)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    scale = None if inp["scale"] is None else torch.tensor([inp["scale"]], device=DEV)
    s = torch.cuda.Stream(device=DEV)
    g = torch.cuda.CUDAGraph()

    def call():
        sp.sp_fused_reduce_norm(inp["partials"], inp["weight"], outs["out"], outs["residual_out"],
                                residual=inp["residual"], bias=inp["bias"], eps=inp["eps"],
                                quant_mode=inp["mode"], scale=scale,
                                out_scales=outs["out_scales"], T_valid=inp["T_valid"])

    torch.cuda.synchronize()  # the inputs are written on torch's stream; `s` does not wait for it
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        call()
        call()  # two launches: a programmatic edge inside the graph
    fresh = synth.make_inputs(w, device=DEV, T_pad=inp["T_pad"], T_valid=inp["T_valid"],
                              seed=inp["seed"] + 77)
    for k in ("partials", "residual", "weight", "bias"):
        inp[k].copy_(fresh[k])
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    compare(_host(outs), run_oracle(fresh), fresh)


def test_two_streams_concurrently():
    """Calls on two streams at once, on different buffers, each give their own correct result."""
    w = synth.workload(3)
    a = _small(w)
    b = synth.make_inputs(w, device=DEV, T_pad=a["T_pad"], T_valid=a["T_valid"] - 4,
                          seed=a["seed"] + 5)
    oa = sp.allocate_outputs(a["T_pad"], a["H"], a["mode"], DEV)
    ob = sp.allocate_outputs(b["T_pad"], b["H"], b["mode"], DEV)
    sa, sb = torch.cuda.Stream(device=DEV), torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    for _ in range(20):
        _call(a, oa, stream=sa)
        _call(b, ob, stream=sb)
    torch.cuda.synchronize()
    compare(_host(oa), run_oracle(a), a)
    compare(_host(ob), run_oracle(b), b)


# ------------------------------------------------------------------------- row schedules
def _call_ex(inp, outs, stream=None, schedule="auto"):
    sc = None if inp["scale"] is None else torch.tensor([inp["scale"]], device=DEV)
    sp.sp_fused_reduce_norm_ex(sp.sp_options_init(schedule=schedule), inp["partials"],
                               inp["weight"], outs["out"], outs["residual_out"],
                               residual=inp["residual"], bias=inp["bias"], eps=inp["eps"],
                               quant_mode=inp["mode"], scale=sc, out_scales=outs["out_scales"],
                               T_valid=inp["T_valid"], stream=stream)


@pytest.mark.parametrize("wi", range(1, 6))
@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_schedule_forced(wi, schedule):
    """Each row schedule on every workload's shape (330 rows, a ragged padded tail). Each case
    runs twice on one stream, so the second dynamic call also checks that the first left its
    row counter at zero."""
    assert _check(_small(synth.workload(wi)), schedule=schedule)


@pytest.mark.parametrize("wi,rows", [(2, 4096), (3, 1024), (4, 1024), (5, 2048)])
def test_schedules_give_identical_bytes(wi, rows):
    """Static and dynamic schedules compute every row the same way: byte-identical outputs."""
    inp = _small(synth.workload(wi), rows=rows)
    a = run_gpu(inp, schedule="static")
    b = run_gpu(inp, schedule="dynamic")
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
def test_dynamic_schedule_with_options(mode):
    """Dynamic rows with a partial scale, an addend and (NVFP4) the swizzled scale layout, whose
    128-row padding adds rows beyond T_pad."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, T_pad=200, T_valid=197, H=5120, with_addend=True)
    layout = 1 if mode == "nvfp4" else 0
    a = run_gpu(inp, fill=0xA5, partial_scale=0.5, scale_layout=layout, schedule="dynamic")
    b = run_gpu(inp, fill=0x5A, partial_scale=0.5, scale_layout=layout, schedule="dynamic")
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, partial_scale=0.5, scale_layout=layout), inp)


def test_dynamic_schedule_on_two_streams_concurrently():
    """Dynamic calls on two streams at once use different row counters: both results correct."""
    w = synth.workload(3)
    a = _small(w, rows=1024)
    b = synth.make_inputs(w, device=DEV, T_pad=a["T_pad"], T_valid=a["T_valid"] - 4,
                          seed=a["seed"] + 5)
    oa = sp.allocate_outputs(a["T_pad"], a["H"], a["mode"], DEV)
    ob = sp.allocate_outputs(b["T_pad"], b["H"], b["mode"], DEV)
    sa, sb = torch.cuda.Stream(device=DEV), torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    for _ in range(50):
        _call_ex(a, oa, stream=sa, schedule="dynamic")
        _call_ex(b, ob, stream=sb, schedule="dynamic")
    torch.cuda.synchronize()
    compare(_host(oa), run_oracle(a), a)
    compare(_host(ob), run_oracle(b), b)


def test_dynamic_schedule_with_more_streams_than_counter_slots():
    """Streams beyond the 256-slot counter table take over idle slots: after 256 streams have
    each made a call and the device is idle, 44 new streams still run the dynamic schedule, with
    the same bytes. Then 300 more streams call without waiting, so that new streams find the
    table full while slots are busy (those calls may run either schedule; the bytes must not
    change). Runs in a child process, so that this process's table is left as it was."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join(
        [os.path.dirname(here), here, os.environ.get("PYTHONPATH", "")]))
    proc = subprocess.run([sys.executable, os.path.abspath(__file__), "streams"], cwd=here,
                          env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-2000:]
    assert "streams ok" in proc.stdout


def _more_streams_than_counter_slots():
    w = synth.workload(2)
    inp = _small(w, rows=64)
    n_first, n_reclaim, n_busy = 256, 44, 300
    n = n_first + n_reclaim + n_busy
    outs = [sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV) for _ in range(n)]
    # distinct CUDA streams (torch's stream pool would hand out the same few again)
    raw = [torch.cuda.ExternalStream(_new_raw_stream()) for _ in range(n)]
    torch.cuda.synchronize()
    staged = sp.sp_options_init(schedule="dynamic", launch=dict(
        kernel=0, vec_per_thread=2, ctas_per_sm=1, stages=0))  # the kernel with the schedule
    schedules = []
    for i, (o, st) in enumerate(zip(outs, raw)):
        if i in (n_first, n_first + n_reclaim):
            torch.cuda.synchronize()  # every slot idle
        sp.sp_fused_reduce_norm_ex(staged, inp["partials"], inp["weight"], o["out"],
                                   o["residual_out"], residual=inp["residual"], bias=inp["bias"],
                                   eps=inp["eps"], quant_mode=inp["mode"],
                                   out_scales=o["out_scales"], T_valid=inp["T_valid"], stream=st)
        schedules.append(sp.sp_last_launch()["schedule"])
    torch.cuda.synchronize()
    assert schedules[:n_first + n_reclaim] == ["dynamic"] * (n_first + n_reclaim), schedules
    assert set(schedules[n_first + n_reclaim:]) <= {"dynamic", "static"}
    ref = run_oracle(inp)
    for o in (outs[0], outs[n_first], outs[n - 1]):
        compare(_host(o), ref, inp)
    first = _host(outs[0])
    for o in outs[1:]:
        h = _host(o)
        for k in ("out", "residual_out"):
            assert np.array_equal(h[k].view(np.uint8), first[k].view(np.uint8))
    for st in raw:
        _destroy_raw_stream(st.cuda_stream)
    print("streams ok", schedules[n_first + n_reclaim:].count("static"), "static of", n_busy)


CHAIN_LAUNCHES = [
    dict(kernel=1, vec_per_thread=2, ctas_per_sm=4, stages=0, split=0),  # direct
    dict(kernel=1, vec_per_thread=1, ctas_per_sm=8, stages=0, split=8),  # direct, split rows
    dict(kernel=0, vec_per_thread=1, ctas_per_sm=8, stages=0, split=4),  # staged split rows
    dict(kernel=1, vec_per_thread=1, ctas_per_sm=8, stages=0, split=4),
    dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=0, split=0),  # staged (static)
    dict(kernel=0, vec_per_thread=1, ctas_per_sm=8, stages=0, split=2),
    dict(kernel=1, vec_per_thread=2, ctas_per_sm=8, stages=0, split=2),
    dict(kernel=0, vec_per_thread=1, ctas_per_sm=8, stages=0, split=8),
    dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=0, split=0),  # staged, dynamic rows
]


@pytest.mark.parametrize("mode", ["none", "fp8_per_token", "nvfp4"])
def test_chained_in_place_calls_match_one_at_a_time(mode):
    """63 calls that update one residual in place, each reading what the one before wrote,
    cycling through every kernel form (direct, split rows, staged, staged split rows, both row
    schedules) and queued back to back on one stream, where each lets the next start early. The
    same calls made one at a time, with the device idle in between, give the same bytes: no
    kernel reads its inputs before the kernel before it has written them."""
    w = dict(synth.workload(5 if mode == "nvfp4" else 4), mode=mode)
    if mode == "none":
        w["scale"] = None
    inp = synth.make_inputs(w, device=DEV, tp=8, T_pad=64, T_valid=61, H=8192)
    sc = None if inp["scale"] is None else torch.tensor([inp["scale"]], device=DEV)
    n = 7 * len(CHAIN_LAUNCHES)
    opts = [sp.sp_options_init(launch=c, schedule="dynamic" if i == len(CHAIN_LAUNCHES) - 1
                               else "static") for i, c in enumerate(CHAIN_LAUNCHES)]
    residual0 = inp["residual"].clone()

    def run(one_at_a_time: bool) -> list:
        residual = residual0.clone()
        outs = [sp.allocate_outputs(inp["T_pad"], inp["H"], mode, DEV) for _ in range(n)]
        s = torch.cuda.Stream(device=DEV)
        torch.cuda.synchronize()
        for i in range(n):
            o = outs[i]
            sp.sp_fused_reduce_norm_ex(opts[i % len(opts)], inp["partials"], inp["weight"],
                                       o["out"], residual, residual=residual, bias=inp["bias"],
                                       eps=inp["eps"], quant_mode=mode, scale=sc,
                                       out_scales=o["out_scales"], T_valid=inp["T_valid"],
                                       stream=s)
            if one_at_a_time:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return [bits_of(residual)] + [bits_of(o[k]) for o in outs for k in ("out", "out_scales")
                                      if o[k] is not None]

    chained, single = run(False), run(True)
    assert len(chained) == len(single)
    for i, (a, b) in enumerate(zip(chained, single)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"buffer {i} differs"


def _cudart():
    import ctypes
    for name in ("libcudart.so", "libcudart.so.13", "libcudart.so.12"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    import glob
    import os
    for path in glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart*.so*")):
        return ctypes.CDLL(path)
    pytest.skip("no CUDA runtime library to create raw streams")


def _new_raw_stream() -> int:
    import ctypes
    rt = _cudart()
    h = ctypes.c_void_p()
    assert rt.cudaStreamCreateWithFlags(ctypes.byref(h), 1) == 0  # non-blocking
    return h.value


def _destroy_raw_stream(h: int) -> None:
    import ctypes
    _cudart().cudaStreamDestroy(ctypes.c_void_p(h))


def test_dynamic_schedule_requested_under_graph_capture():
    """A dynamic call captured into a CUDA graph runs with the static schedule and replays
    correctly on refilled inputs."""
    w = synth.workload(4)
    inp = _small(w, rows=1024)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    s = torch.cuda.Stream(device=DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        _call_ex(inp, outs, schedule="dynamic")
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        _call_ex(inp, outs, schedule="dynamic")
    fresh = synth.make_inputs(w, device=DEV, T_pad=inp["T_pad"], T_valid=inp["T_valid"],
                              seed=inp["seed"] + 91)
    for k in ("partials", "residual", "weight", "bias"):
        inp[k].copy_(fresh[k])
    torch.cuda.synchronize()
    g.replay()
    with torch.cuda.stream(s):
        _call_ex(inp, outs, schedule="dynamic")  # the capturing stream, outside the graph
    torch.cuda.synchronize()
    compare(_host(outs), run_oracle(fresh), fresh)


# ------------------------------------------------------------------------- non-finite inputs
def _drop_rows(res: dict, rows) -> dict:
    out = {}
    for k, v in res.items():
        if isinstance(v, np.ndarray) and v.ndim >= 1 and k in ("out", "out_scales", "residual_out", "y"):
            out[k] = np.delete(v, rows, axis=0)
        else:
            out[k] = v
    return out


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_non_finite_inputs_stay_in_their_row(mode, schedule):
    """Inf and NaN in valid rows are outside the stage's contract (the pages define no such
    inputs), but they must not leak: every other row still matches the oracle exactly as usual,
    padding rows stay zero, and no device wait runs out."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, T_pad=64, T_valid=61, H=1024)
    poisoned = [3, 17, 40]
    inp["partials"][1, 3, 5] = float("inf")
    inp["residual"][17, 100] = float("nan")
    inp["partials"][0, 40, 7] = float("-inf")
    inp["partials"][2, 40, 7] = float("inf")
    a = run_gpu(inp, fill=0xA5, schedule=schedule)
    b = run_gpu(inp, fill=0x5A, schedule=schedule)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    ref = run_oracle(inp)
    clean = dict(inp, T_valid=inp["T_valid"] - len(poisoned))
    compare(_drop_rows(a, poisoned), _drop_rows(ref, poisoned), clean)
    assert sp.sp_device_error(clear=False) == 0


def test_dynamic_schedule_chained_with_other_kernels_on_one_stream():
    """A layer loop on one stream: each call's new residual feeds the next call (in place), with
    PyTorch kernels between the calls. Dynamic rows, so every call reuses the stream's row
    counter right after the previous call; the final residual matches the same loop run with the
    static schedule byte for byte."""
    w = synth.workload(4)
    inp = _small(w, rows=1024)
    s = torch.cuda.Stream(device=DEV)
    finals = []
    for schedule in ("dynamic", "static"):
        res = inp["residual"].clone()
        outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
        parts = inp["partials"].clone()
        with torch.cuda.stream(s):
            for layer in range(12):
                opts = sp.sp_options_init(schedule=schedule)
                sp.sp_fused_reduce_norm_ex(opts, parts, inp["weight"], outs["out"], res,
                                           residual=res, bias=inp["bias"], eps=inp["eps"],
                                           quant_mode=inp["mode"], out_scales=outs["out_scales"],
                                           T_valid=inp["T_valid"], stream=s)
                parts.mul_(0.5)  # a PyTorch kernel between two calls on the same stream
        torch.cuda.synchronize()
        finals.append((res.view(torch.int16).cpu().numpy(), outs["out"].cpu().numpy(),
                       outs["out_scales"].cpu().numpy()))
    for a, b in zip(finals[0], finals[1]):
        assert np.array_equal(a, b)


# ------------------------------------------------------------------------- exact ties
def _tie_inputs(weights: list[float], rows: int = 8, mode: str = "none", scale=None) -> dict:
    """tp = 1, no residual, no bias, every h = +-1 (so mean(h^2) = 1) and eps = 1e-30 (so
    mean + eps rounds to exactly 1 in fp32): y = h * w exactly when the kernel's rsqrt(1) is 1."""
    H = len(weights)
    g = torch.Generator(device="cpu").manual_seed(11)
    signs = (torch.randint(0, 2, (1, rows, H), generator=g) * 2 - 1).to(torch.bfloat16)
    return dict(partials=signs.to(DEV), residual=None, addend=None, bias=None,
                weight=torch.tensor(weights, dtype=torch.bfloat16, device=DEV),
                tp=1, T_pad=rows, T_valid=rows, H=H, eps=1e-30, mode=mode, scale=scale)


def _rsqrt_of_one_is_exact() -> bool:
    inp = _tie_inputs([1.0] * 16)
    out = run_gpu(inp)["out"].view(np.uint16)
    return bool(np.all((out == 0x3F80) | (out == 0xBF80)))  # +-1.0 in bf16


def test_fp8_codes_round_exact_ties_to_even():
    """E4M3 midpoints (values with one more mantissa bit than E4M3 holds) as quantiser inputs:
    the kernel's codes equal the oracle's ties-to-even codes bit for bit."""
    if not _rsqrt_of_one_is_exact():
        pytest.skip("rsqrt(1) is not exactly 1 on this device: no exact ties to feed")
    mids = []
    for e in (-6, -3, 0, 2, 7):              # normal binades of E4M3 (2^-6 .. 2^8)
        for k in range(8):                   # mantissa m/8, midpoint (2k+1)/16 above 1
            mids.append((1.0 + (2 * k + 1) / 16.0) * 2.0 ** e)
    mids += [-m for m in mids[:24]]
    mids += [0.5 * 2.0 ** -9, 1.5 * 2.0 ** -9, 2.5 * 2.0 ** -9]   # subnormal midpoints
    while len(mids) % 16:
        mids.append(1.0)
    inp = _tie_inputs(mids, mode="fp8_static", scale=1.0)
    got = run_gpu(inp)["out"]
    ref = run_oracle(inp)["out"]
    assert np.array_equal(got, ref)


def test_nvfp4_codes_round_exact_ties_to_even():
    """E2M1 midpoints in 16-element blocks whose largest magnitude is 6 (so with a global scale
    of 1 every block scale is exactly 1): codes equal the oracle's ties-to-even codes."""
    if not _rsqrt_of_one_is_exact():
        pytest.skip("rsqrt(1) is not exactly 1 on this device: no exact ties to feed")
    block = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5,
             -5.0, 1.0]
    inp = _tie_inputs(block * 4, mode="nvfp4", scale=1.0)
    got, ref = run_gpu(inp), run_oracle(inp)
    assert np.array_equal(got["out_scales"], ref["out_scales"])
    assert np.array_equal(got["out"], ref["out"])


def test_dynamic_schedule_soak_two_chained_streams():
    """100 calls in place on each of two streams at once, back to back (consecutive calls
    overlap through programmatic dependent launch): every call reads the residual the previous
    one wrote, so a row skipped or done twice anywhere would change the end result. Dynamic and
    static schedules must end byte-identical."""
    w = synth.workload(3)
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    inps = [synth.make_inputs(w, device=DEV, T_pad=4096, T_valid=4093, H=7168, seed=77 + k)
            for k in range(2)]
    scale = torch.tensor([w["scale"]], device=DEV)
    ends = []
    for schedule in ("dynamic", "static"):
        res = [i["residual"].clone() for i in inps]
        outs = [sp.allocate_outputs(4096, 7168, w["mode"], DEV) for _ in inps]
        torch.cuda.synchronize()
        for _ in range(100):
            for k, s in enumerate(streams):
                i = inps[k]
                sp.sp_fused_reduce_norm_ex(sp.sp_options_init(schedule=schedule), i["partials"],
                                           i["weight"], outs[k]["out"], res[k], residual=res[k],
                                           bias=i["bias"], eps=i["eps"], quant_mode=i["mode"],
                                           scale=scale, T_valid=i["T_valid"], stream=s)
        torch.cuda.synchronize()
        ends.append([(r.view(torch.int16).cpu().numpy(), o["out"].cpu().numpy())
                     for r, o in zip(res, outs)])
    for (ra, oa), (rb, ob) in zip(ends[0], ends[1]):
        assert np.array_equal(ra, rb) and np.array_equal(oa, ob)
    assert sp.sp_device_error(clear=False) == 0


# ------------------------------------------------------------------------- launch-rule bands
@pytest.mark.parametrize("tp,T,H,mode,band", [
    (4, 48, 8192, "fp8_per_token", (1, 2, 8, 0)),     # direct, two vectors per thread
    (4, 32, 5120, "fp8_per_token", (0, 1, 8, 0, 4)),  # staged split rows, tp <= 5, 17-32 rows
    (2, 24, 7168, "none", (0, 1, 8, 0, 8)),           # ... 8 per row for 17-24 rows, H >= 6144
    (16, 16, 5120, "nvfp4", (0, 1, 8, 0, 4)),         # ... NVFP4, tp >= 12, up to 16 rows
    (4, 128, 4096, "none", (1, 2, 16, 0)),            # direct, two vectors at tp <= 4
    (8, 384, 3072, "fp8_per_token", (1, 1, 16, 0)),   # direct up to 1.2 M at tp <= 8
    (16, 128, 2048, "fp8_static", (1, 1, 16, 0)),     # direct at tp >= 6
    (16, 16, 8192, "fp8_per_token", (1, 1, 8, 0, 8)), # split rows, 8 CTAs per row
    (8, 32, 5120, "nvfp4", (1, 1, 8, 0, 4)),          # split rows, 4 CTAs per row
    (8, 48, 5120, "fp8_per_token", (1, 1, 8, 0, 2)),  # split rows, 2 CTAs per row
    (8, 192, 5120, "nvfp4", (1, 1, 8, 0, 2)),         # split 2 up to 224 rows at H = 5120
    (6, 156, 6144, "fp8_static", (1, 1, 8, 0, 4)),    # split 4 up to 160 rows at H = 6144
    (16, 96, 5120, "nvfp4", (1, 1, 8, 0, 4)),         # split 4 for 65-128 rows, tp >= 12
    (16, 96, 7168, "fp8_static", (1, 2, 8, 0)),       # direct up to 128 rows below H = 8192
    (8, 16, 4096, "fp8_per_token", (1, 1, 8, 0, 4)),  # split 4 above H = 3072
    (4, 48, 4096, "none", (1, 1, 8, 0, 8)),           # split 8 up to 48 rows at tp <= 5
    (4, 8, 5120, "nvfp4", (1, 1, 8, 0, 4)),           # tp <= 5, NVFP4 below H = 6144
    (8, 80, 5120, "none", (1, 1, 8, 0, 4)),           # 65-96 rows at H <= 5120, tp >= 6
    (16, 48, 5120, "fp8_per_token", (1, 1, 8, 0, 2)), # 33-64 rows at H <= 5120, tp >= 12
    (12, 72, 7168, "none", (1, 1, 8, 0, 4)),          # 65-96 rows at H >= 7168, tp >= 12
    (4, 40, 16384, "fp8_per_token", (1, 1, 8, 0, 8)), # split 8 up to 64 rows above H = 12288
    (8, 144, 8192, "fp8_per_token", (1, 1, 8, 0, 4)), # 129-144 rows at H >= 7168: split 4
    (4, 152, 7168, "nvfp4", (1, 1, 8, 0, 2)),         # 145-152 rows at tp <= 5: split 2
    (16, 144, 5120, "none", (1, 1, 8, 0, 4)),         # tp >= 12, 129-144 rows: split 4
    (8, 152, 6144, "none", (1, 1, 8, 0, 2)),          # H 5121-6144, up to 152 rows: split 2
    (8, 160, 12288, "fp8_static", (1, 1, 8, 0, 8)),   # 153-160 rows at H <= 12288: split 8
    (16, 160, 4096, "nvfp4", (0, 1, 8, 0, 4)),        # staged split rows: tp >= 12, H = 4096
    (8, 224, 4096, "nvfp4", (0, 1, 8, 0, 2)),         # ... NVFP4 past 128 rows, 2 per row
    (8, 120, 5120, "fp8_per_token", (0, 1, 8, 0, 4)), # ... 97-128 rows at tp >= 6, H <= 5120
    (4, 256, 3072, "nvfp4", (0, 1, 8, 0, 2)),         # ... NVFP4 past 128 rows, H = 3072
    (8, 160, 7168, "none", (0, 1, 8, 0, 4)),          # ... H >= 7168, 145-160 rows at tp 6-11
    (4, 192, 8192, "fp8_static", (0, 1, 8, 0, 4)),    # ... H >= 7168, 161-192 rows at tp <= 5
    (2, 24, 12288, "fp8_static", (1, 1, 8, 0, 4)),    # split rows at H > 8192, tp <= 5
    (4, 96, 16384, "nvfp4", (1, 4, 8, 0)),            # direct, four vectors per thread
    (16, 48, 12288, "nvfp4", (1, 1, 8, 0, 4)),        # split rows at H > 8192
    (8, 80, 12288, "fp8_per_token", (1, 1, 8, 0, 8)), # 8 CTAs per row up to 80 rows
    (16, 112, 8192, "nvfp4", (0, 2, 1, 0)),           # staged, one CTA per SM
    (16, 320, 3072, "none", (0, 2, 3, 0)),            # one round of rows at H = 3072
    (6, 384, 6144, "fp8_per_token", (0, 2, 3, 0)),    # one round of rows at H = 6144
    (8, 256, 5120, "fp8_static", (0, 2, 2, 0)),       # one round of rows, fewest CTAs
    (4, 768, 4096, "none", (0, 2, 3, 0)),             # last round filled at 3 CTAs/SM
    (8, 512, 5120, "fp8_per_token", (0, 2, 2, 0)),    # last round filled at 2 CTAs/SM
    (4, 4096, 1024, "none", (1, 1, 16, 0)),           # direct up to 2^22 elements at H = 1024
    (8, 1536, 4096, "nvfp4", (0, 2, 4, 3)),           # the large-call launch
])
def test_default_launch_in_each_band(tp, T, H, mode, band):
    """Each band of the launch rule, checked to be the band and compared with the oracle."""
    c = sp.sp_select_launch(tp, T, H, mode)
    band = tuple(band) + (0,) * (5 - len(band))
    assert (c.kernel, c.vec_per_thread, c.ctas_per_sm, c.stages, c.split) == band
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=T, T_valid=T - 3, H=H)
    assert _check(inp)


# ------------------------------------------------------------------------- split rows
def _split_cfg(split, vec, ctas=2):
    return dict(kernel=1, vec_per_thread=vec, ctas_per_sm=ctas, stages=0, split=split)


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("split,vec", [(2, 1), (2, 2), (4, 1), (4, 2), (8, 1), (8, 2)])
@pytest.mark.parametrize("tp,T,H", [(8, 16, 8192), (4, 40, 4096), (3, 24, 1040), (2, 10, 16)])
def test_split_rows(mode, split, vec, tp, T, H):
    """Rows split across the CTAs of a cluster: every slice size, including CTAs whose slice is
    empty (H = 16 at split 8) and slices that end mid-warp (H = 1040)."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=T, T_valid=T - 3, H=H)
    assert _check(inp, config=_split_cfg(split, vec))


@pytest.mark.parametrize("mode", ["none", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("split,vec", [(2, 2), (4, 1), (4, 2), (8, 1), (8, 2)])
def test_split_rows_longest_hidden(mode, split, vec):
    """Split rows at the largest H the kernels take (16384: 256-1024 vectors per CTA)."""
    w = dict(synth.workload(3), mode=mode, scale=None)
    inp = synth.make_inputs(w, device=DEV, tp=4, T_pad=12, T_valid=10, H=sp.sp_max_hidden())
    assert _check(inp, config=_split_cfg(split, vec))


@pytest.mark.parametrize("mode", ["fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("tp,T_pad,T_valid,layout", [(1, 8, 8, 0), (4, 16, 0, 0), (4, 16, 0, 1),
                                                     (1, 1, 1, 1), (2, 130, 127, 1)])
def test_split_rows_edge_cases(mode, tp, T_pad, T_valid, layout):
    """Split rows at tp = 1, with every row padding (only zeros written, scales included), with
    a single row, and with the swizzled layout's padding rows beyond T_pad (NVFP4)."""
    if layout and mode != "nvfp4":
        pytest.skip("the swizzled layout is NVFP4-only")
    w = dict(synth.workload(3), mode=mode, scale=None)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=T_pad, T_valid=T_valid, H=2080)
    kw = dict(config=_split_cfg(8, 1), scale_layout=layout)
    a = run_gpu(inp, fill=0xA5, **kw)
    b = run_gpu(inp, fill=0x5A, **kw)
    for k in ("out", "out_scales", "residual_out"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, scale_layout=layout), inp)


@pytest.mark.parametrize("T,split", [(64, 0), (2048, 0), (48, 4), (4096, 2)])
@pytest.mark.parametrize("tp", [5, 8, 13])
def test_direct_kernel_batches_of_partials(tp, T, split):
    """One vector per thread with more than four partials: the variant with eight partial rows in
    flight (few rows, every CTA resident) and the one with four (more rows than fit at once),
    including a last batch that is only partly filled."""
    w = dict(synth.workload(4), tp=tp)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=tp * -(-T // tp), T_valid=T - 5, H=2048)
    cfg = dict(kernel=1, vec_per_thread=1, ctas_per_sm=16, stages=0, split=split)
    assert _check(inp, config=cfg)


@pytest.mark.parametrize("split,ctas", [(8, 1), (4, 1), (2, 1)])
def test_split_rows_many_rows_per_cluster(split, ctas):
    """Fewer clusters than rows: each cluster takes several rows in turn, reusing its two
    cross-CTA reduction slots on alternate rows."""
    w = synth.workload(4)  # per-token FP8 (the row max crosses the cluster too)
    inp = _small(w, rows=1000, H=2048)
    assert _check(inp, config=_split_cfg(split, 1, ctas))


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("split", [2, 8])
def test_split_rows_with_options(mode, split):
    """Split rows with a partial scale, an addend and (NVFP4) the swizzled scale layout, whose
    padding rows and columns the cluster's first CTA must zero."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, tp=4, T_pad=24, T_valid=21, H=1040, with_addend=True)
    layout = 1 if mode == "nvfp4" else 0
    kw = dict(config=_split_cfg(split, 1), partial_scale=0.5, scale_layout=layout)
    a = run_gpu(inp, fill=0xA5, **kw)
    b = run_gpu(inp, fill=0x5A, **kw)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, partial_scale=0.5, scale_layout=layout), inp)


@pytest.mark.parametrize("mode", ["fp8_per_token", "nvfp4"])
def test_split_rows_on_host_buffers(mode):
    """A forced split-row launch on page-locked host buffers (zero-copy), NVFP4 with the
    swizzled scale layout."""
    w = dict(synth.workload(3), mode=mode, scale=None)
    inp = synth.make_inputs(w, device=DEV, tp=8, T_pad=16, T_valid=13, H=4096)
    layout = 1 if mode == "nvfp4" else 0
    a = run_gpu_host(inp, fill=0xA5, scale_layout=layout, config=_split_cfg(8, 1))
    b = run_gpu_host(inp, fill=0x5A, scale_layout=layout, config=_split_cfg(8, 1))
    for k in ("out", "out_scales", "residual_out"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, scale_layout=layout), inp)


# ------------------------------------------------------------------------- staged split rows
def _slice_cfg(split):
    return dict(kernel=0, vec_per_thread=1, ctas_per_sm=8, stages=0, split=split)


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("tp,T,H", [(8, 16, 8192), (4, 40, 4096), (3, 24, 1040), (2, 10, 16),
                                    (16, 160, 4096)])
def test_slice_rows(mode, split, tp, T, H):
    """The staged kernel's split-row form: each CTA of a row's cluster brings its slice of the
    row's segments into shared memory with one bulk copy each. Every slice size, including CTAs
    whose slice is empty (H = 16 at split 8) and slices that end mid-warp (H = 1040)."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=T, T_valid=T - 3, H=H)
    assert _check(inp, config=_slice_cfg(split))


@pytest.mark.parametrize("mode", ["fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("tp,T_pad,T_valid,layout", [(1, 8, 8, 0), (4, 16, 0, 0), (4, 16, 0, 1),
                                                     (1, 1, 1, 1), (2, 130, 127, 1)])
def test_slice_rows_edge_cases(mode, tp, T_pad, T_valid, layout):
    """Staged split rows at tp = 1, with every row padding (only zeros written, scales
    included), with a single row, and with the swizzled layout's padding rows beyond T_pad."""
    if layout and mode != "nvfp4":
        pytest.skip("the swizzled layout is NVFP4-only")
    w = dict(synth.workload(3), mode=mode, scale=None)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=T_pad, T_valid=T_valid, H=2080)
    kw = dict(config=_slice_cfg(8), scale_layout=layout)
    a = run_gpu(inp, fill=0xA5, **kw)
    b = run_gpu(inp, fill=0x5A, **kw)
    for k in ("out", "out_scales", "residual_out"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, scale_layout=layout), inp)


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
@pytest.mark.parametrize("split", [2, 8])
def test_slice_rows_with_options(mode, split):
    """Staged split rows with a partial scale, an addend (one more segment in shared memory) and
    (NVFP4) the swizzled scale layout."""
    w = dict(synth.workload(3), mode=mode, scale=0.05 if mode == "fp8_static" else None)
    inp = synth.make_inputs(w, device=DEV, tp=4, T_pad=24, T_valid=21, H=1040, with_addend=True)
    layout = 1 if mode == "nvfp4" else 0
    kw = dict(config=_slice_cfg(split), partial_scale=0.5, scale_layout=layout)
    a = run_gpu(inp, fill=0xA5, **kw)
    b = run_gpu(inp, fill=0x5A, **kw)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    compare(a, run_oracle(inp, partial_scale=0.5, scale_layout=layout), inp)


@pytest.mark.parametrize("split", [4, 8])
def test_slice_rows_longest_hidden(split):
    """Staged split rows at the largest H the kernels take (slices of 256 and 512 vectors, one
    per thread; two CTAs per row would need 1024 threads and are refused)."""
    w = dict(synth.workload(3), mode="fp8_per_token", scale=None)
    inp = synth.make_inputs(w, device=DEV, tp=4, T_pad=12, T_valid=10, H=sp.sp_max_hidden())
    assert _check(inp, config=_slice_cfg(split))


@pytest.mark.parametrize("tp,H,split", [(32, 12288, 2), (4, 16384, 2)])
def test_slice_rows_refused_when_a_slice_does_not_fit(tp, H, split):
    """A CTA's slice must fit its shared memory and its threads: 33 segments of 768 vectors
    (tp = 32, H = 12288, two CTAs per row: 396 KB) and a slice of 1024 vectors (H = 16384, two
    CTAs per row) are refused before any launch."""
    w = dict(synth.workload(3), mode="none", scale=None)
    inp = synth.make_inputs(w, device=DEV, tp=tp, T_pad=tp, T_valid=tp, H=H)
    with pytest.raises(sp.SpError) as e:
        run_gpu(inp, config=_slice_cfg(split))
    assert e.value.status == 2  # SP_ERR_UNSUPPORTED


def test_split_rows_on_two_streams_concurrently():
    """Split-row launches (clusters of 8 and of 2 CTAs) on two streams at once, on different
    buffers, each give their own correct result."""
    w = synth.workload(4)
    a = synth.make_inputs(w, device=DEV, tp=16, T_pad=16, T_valid=14, H=8192)
    b = synth.make_inputs(w, device=DEV, tp=16, T_pad=64, T_valid=61, H=8192, seed=a["seed"] + 3)
    oa = sp.allocate_outputs(a["T_pad"], a["H"], a["mode"], DEV)
    ob = sp.allocate_outputs(b["T_pad"], b["H"], b["mode"], DEV)
    sa, sb = torch.cuda.Stream(device=DEV), torch.cuda.Stream(device=DEV)

    def call(inp, outs, cfg, stream):
        sp.sp_fused_reduce_norm_ex(sp.sp_options_init(launch=cfg), inp["partials"], inp["weight"],
                                   outs["out"], outs["residual_out"], residual=inp["residual"],
                                   bias=inp["bias"], eps=inp["eps"], quant_mode=inp["mode"],
                                   out_scales=outs["out_scales"], T_valid=inp["T_valid"],
                                   stream=stream)

    torch.cuda.synchronize()
    for _ in range(20):
        call(a, oa, _split_cfg(8, 1), sa)
        call(b, ob, _split_cfg(2, 1), sb)
    torch.cuda.synchronize()
    compare(_host(oa), run_oracle(a), a)
    compare(_host(ob), run_oracle(b), b)


def test_split_rows_captured_in_a_graph_after_other_kernels():
    """Split-row launches (clusters with the programmatic-dependent-launch attribute) inside a
    CUDA graph, each after a PyTorch kernel that rewrites its partials: every replay computes on
    the new contents."""
    w = synth.workload(4)
    inp = synth.make_inputs(w, device=DEV, tp=8, T_pad=16, T_valid=13, H=8192)
    outs = sp.allocate_outputs(inp["T_pad"], inp["H"], inp["mode"], DEV)
    src = inp["partials"].clone()
    opts = sp.sp_options_init(launch=_split_cfg(8, 1))
    s = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()  # the inputs are written on torch's stream; `s` does not wait for it

    def step():
        inp["partials"].copy_(src)
        inp["partials"].mul_(0.5)
        sp.sp_fused_reduce_norm_ex(opts, inp["partials"], inp["weight"], outs["out"],
                                   outs["residual_out"], residual=inp["residual"],
                                   bias=inp["bias"], eps=inp["eps"], quant_mode=inp["mode"],
                                   out_scales=outs["out_scales"], T_valid=inp["T_valid"])

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
        step()
    fresh = synth.make_inputs(w, device=DEV, tp=8, T_pad=16, T_valid=13, H=8192,
                              seed=inp["seed"] + 9)
    src.copy_(fresh["partials"])
    for k in ("residual", "weight", "bias"):
        inp[k].copy_(fresh[k])
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    fresh["partials"] = (fresh["partials"].float() * 0.5).to(torch.bfloat16)
    compare(_host(outs), run_oracle(fresh), fresh)


if __name__ == "__main__":
    import sys
    if sys.argv[1:] == ["streams"]:
        _more_streams_than_counter_slots()
