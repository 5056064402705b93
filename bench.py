"""Benchmark of the fused reduce + bias/residual add + RMSNorm + quant stage on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME|INDEX] [--no-extras]

A step is one call of the whole per-token stage (sum of tp partials, bias + residual add, new
residual, RMSNorm, output in the workload's form, padding rows zeroed) over one batch of
synthetic, seeded input already resident in HBM. The default workload is the largest one: tp=8,
16384 tokens, H=5120, Student-t partials, NVFP4 output (1.72 GB moved per step). Every step's
inputs are larger than the 129 MB L2, and the timed loop also rotates over resident sets, so every
step reads its inputs from HBM. The timed launches are queued behind a short GPU-side sleep placed
before the start event, so the GPU never waits on the Python loop inside the timed region.

Printed: one JSON line (rank 0) with the headline HBM GB/s (algorithmic bytes / time), Mtokens/s,
the roofline of the kernel against the measured HBM copy peak, the end-to-end figure through the
public API with host buffers (host->device copies and device->host reads in the timed region),
the oracle timed on the host cores as a CPU baseline, SM clocks sampled during the timed region,
and per-workload figures for the other four workloads.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent replicas;
nothing is exchanged between ranks) and the value is the sum over ranks divided by the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fused reduce+add-RMSNorm+quant HBM GB/s and Mtokens/s; % of GB300 HBM peak"
DEFAULT_WORKLOAD = "tp8_T16384_H5120_nvfp4"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (for context; `peak` is the measured copy)
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------------------ workload math
def algorithmic_bytes(tp: int, T_valid: int, T_pad: int, H: int, mode: str,
                      residual: bool = True, addend: bool = False) -> int:
    """Bytes one call must move: per valid row tp partial rows + the residual row (+ the addend
    row) read (2H each) and residual_out + out (+ scales) written; per padding row the zero writes
    only. Weight and bias (2H each, read once per CTA and L2-resident) are left out."""
    out_row = {"none": 2 * H, "fp8_static": H, "fp8_per_token": H + 4,
               "nvfp4": H // 2 + H // 16}[mode]
    read_row = 2 * H * (tp + (1 if residual else 0) + (1 if addend else 0))
    write_row = 2 * H + out_row
    return T_valid * (read_row + write_row) + (T_pad - T_valid) * write_row


def workload_config(w: dict, world: int) -> dict:
    """The `config` object of the JSON line; identical in both arms for the same workload."""
    one = algorithmic_bytes(w["tp"], w["T_valid"], w["T_pad"], w["H"], w["mode"])
    return {"workload": w["name"], "tp": w["tp"], "T_valid": w["T_valid"], "T_pad": w["T_pad"],
            "H": w["H"], "quant": w["mode"], "bytes_per_step": one,
            "l2": f"inputs larger than L2 ({one / 1e6:.0f} MB per step, L2 129 MB)",
            "parallelism": f"replicas x{world}"}


KERNEL_SOURCES = ("sp_device.cuh", "sp_kernels.cuh")  # the device code of every kernel


def kernel_source_hash() -> str:
    """Hash of the device code the fused kernels compile from: comments and blank lines are left
    out, so only a change to the code itself marks recorded ncu counters as stale."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sequence_reduce_add_gb300", "csrc", rel)) as f:
            code = [line.split("//", 1)[0].rstrip() for line in f]
        h.update(rel.encode() + "\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def measured_peak() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload: str, launch: dict) -> int | None:
    """DRAM bytes per launch from a committed ncu capture, if it was taken on the current device
    code with the same launch configuration (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            data = json.load(f)
    except Exception:
        return None
    entry = data.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    if entry.get("launch") != launch:
        return None
    return int(entry["dram_bytes_per_launch"])


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_start: float, t_end: float) -> dict:
        del t_start, t_end
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ our arm
VARIANTS = {
    # "First" layer of the quant-aware SP patterns: no incoming residual
    "first": dict(with_residual=False),
    # a scale on every partial before the reduction plus a per-shard addend after it
    "scaled_addend": dict(with_addend=True, partial_scale=0.5),
    # NVFP4 block scales written in the 128x4-tile layout block-scaled GEMMs read
    "swizzled_scales": dict(scale_layout=1),
}
# (workload, variant) pairs measured beside the other workloads
# Decode-sized calls (tp, tokens, H) of the per-token FP8 workload's kind: latency-bound, so each
# is also timed replayed from a CUDA graph.
DECODE_RUNS = [(8, 8, 8192), (8, 64, 8192), (8, 256, 8192), (8, 16, 4096), (8, 144, 8192)]

VARIANT_RUNS = [("tp4_T4093p4096_H4096_bf16", "first"),
                ("tp4_T4093p4096_H4096_bf16", "scaled_addend"),
                ("tp8_T16384_H5120_nvfp4", "swizzled_scales")]


class Problem:
    """One resident input/output set of a workload, with prebuilt C-ABI argument tuples."""

    def __init__(self, w: dict, seed: int, device, sp, variant: str | None = None):
        from sequence_reduce_add_gb300 import synth
        v = dict(VARIANTS.get(variant, {}))
        partial_scale = v.pop("partial_scale", 1.0)
        scale_layout = v.pop("scale_layout", 0)
        self.inp = synth.make_inputs(w, seed=seed, device=device, **v)
        i = self.inp
        self.outs = sp.allocate_outputs(i["T_pad"], i["H"], i["mode"], device,
                                        scale_layout=scale_layout)
        self.scale = (torch.tensor([i["scale"]], dtype=torch.float32, device=device)
                      if i["scale"] is not None else None)
        p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        self.args = (p(i["partials"]), i["tp"], i["T_pad"], i["T_valid"], i["H"], p(i["residual"]),
                     p(i["weight"]), p(i["bias"]), ctypes.c_float(i["eps"]),
                     sp.QUANT_MODES[i["mode"]], p(self.scale), p(self.outs["out"]),
                     p(self.outs["out_scales"]), p(self.outs["residual_out"]))
        self.fn_name = "sp_fused_reduce_norm"
        if variant is not None:  # the options entry point
            self.options = sp.sp_options_init(partial_scale=partial_scale, addend=i["addend"],
                                              scale_layout=scale_layout)
            self.args = (ctypes.byref(self.options),) + self.args
            self.fn_name = "sp_fused_reduce_norm_ex"
        self.bytes = algorithmic_bytes(i["tp"], i["T_valid"], i["T_pad"], i["H"], i["mode"],
                                       i["residual"] is not None, i["addend"] is not None)

    def nbytes(self) -> int:
        ts = [self.inp["partials"], self.inp["residual"], self.inp["addend"], self.outs["out"],
              self.outs["out_scales"], self.outs["residual_out"]]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)


# Host time to enqueue one call (ctypes + checks + launch) is a few microseconds; the gate that
# holds the GPU while the timed launches are queued is sized from this, generously.
ENQUEUE_US_PER_CALL = 10.0
GATE_MAX_LAUNCHES = 1024
SLEEP_CYCLES_PER_US = 2100  # at most ~2.1 GHz SM clock: a sleep of n cycles lasts >= n/2100 us


def gate_stream(stream, launches: int) -> None:
    """Hold `stream` in a short device-side sleep long enough for the host to enqueue `launches`
    calls behind it (at most GATE_MAX_LAUNCHES), so the timed launches start back to back instead
    of waiting for the Python loop. The sleep runs before the start event: it is not timed."""
    us = 100.0 + ENQUEUE_US_PER_CALL * min(launches, GATE_MAX_LAUNCHES)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * SLEEP_CYCLES_PER_US))


def time_kernel_loop(lib, problems, steps: int, stream, per_launch_events: bool,
                     gate: bool = False, end_events: bool = False):
    """Launch `steps` calls rotating over `problems` on `stream`; returns (total_ms, [launch ms],
    info). per_launch_events: an event pair around every launch (isolated launches). end_events:
    one event after every launch (consecutive differences = per-launch times in a chain). gate:
    queue everything behind gate_stream; info["host_ahead"] says whether the host had queued every
    launch before the GPU reached the start event."""
    handle = ctypes.c_void_p(stream.cuda_stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)] if per_launch_events else None)
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if end_events else None
    fn = getattr(lib, problems[0].fn_name)
    n = len(problems)
    if gate:
        gate_stream(stream, steps)
    start.record(stream)
    for s in range(steps):
        if ev:
            ev[s][0].record(stream)
        st = fn(*problems[s % n].args, handle)
        if st != 0:
            raise RuntimeError(f"{problems[0].fn_name} returned {st}")
        if ev:
            ev[s][1].record(stream)
        if ends:
            ends[s].record(stream)
    end.record(stream)
    host_ahead = not start.query() if gate else None
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    launches = [a.elapsed_time(b) for a, b in ev] if ev else []
    if ends:
        marks = [start] + ends
        launches = [a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:])]
    return total, launches, {"host_ahead": host_ahead}


def e2e_loop(sp, w: dict, problem: Problem, steps: int, warmup: int, stream) -> dict:
    """The same call through the public API with host buffers. Inputs live in pinned host
    memory and outputs are written to pinned host memory; every step moves all input bytes
    host->device and all output bytes device->host.

    zero_copy: ``sp_fused_reduce_norm_host`` -- the kernel reads the inputs across the host link
    and writes the outputs back as it computes (both directions overlap).
    staged_copies: host->device copies of the inputs, the device call, device->host copies of the
    outputs, in order on one stream (reported beside it)."""
    i, o = problem.inp, problem.outs
    host_in = {k: i[k].cpu().pin_memory() for k in ("partials", "residual", "weight", "bias")
               if i[k] is not None}
    host_out = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in o.items()
                if v is not None}
    host_scale = problem.scale.cpu().pin_memory() if problem.scale is not None else None
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    def zero_copy():
        sp.sp_fused_reduce_norm_host(host_in["partials"], host_in["weight"], host_out["out"],
                                     host_out["residual_out"], residual=host_in.get("residual"),
                                     bias=host_in.get("bias"), eps=i["eps"], quant_mode=i["mode"],
                                     scale=host_scale, out_scales=host_out.get("out_scales"),
                                     T_valid=i["T_valid"], stream=stream)

    def staged_copies():
        with torch.cuda.stream(stream):
            for k, t in host_in.items():
                i[k].copy_(t, non_blocking=True)
            sp.sp_fused_reduce_norm(i["partials"], i["weight"], o["out"], o["residual_out"],
                                    residual=i["residual"], bias=i["bias"], eps=i["eps"],
                                    quant_mode=i["mode"], scale=problem.scale,
                                    out_scales=o["out_scales"], T_valid=i["T_valid"],
                                    stream=stream)
            for k, t in host_out.items():
                t.copy_(o[k], non_blocking=True)

    def timed(step):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()  # the host may now read every output of every step
        return a.elapsed_time(b) / steps

    return {"ms_per_step": timed(zero_copy), "staged_ms_per_step": timed(staged_copies),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "host_inputs": host_in}


class OracleRunner:
    """The oracle as it stands, on row samples of one workload, on all host cores."""

    def __init__(self, w: dict, host_in: dict):
        import oracle
        from sequence_reduce_add_gb300 import synth
        b = synth.bf16_bits
        self.oracle = oracle
        self.w = w
        self.parts = b(host_in["partials"])
        self.res = b(host_in["residual"]) if "residual" in host_in else None
        self.wt = b(host_in["weight"])
        self.bs = b(host_in["bias"]) if "bias" in host_in else None
        self.scale = host_in.get("scale")
        self.cores = os.cpu_count() or 1
        self.buffers = None
        self.next_row = 0

    def run(self, nrows: int, threads: int | None = None) -> tuple[float, int]:
        """Compute `nrows` valid rows (cycling through the workload) on `threads` threads (default:
        all cores); returns (seconds, bytes)."""
        Tv = self.w["T_valid"]
        nrows = max(1, min(nrows, Tv))
        if self.next_row + nrows > Tv:
            self.next_row = 0
        rows = (self.next_row, self.next_row + nrows)
        self.next_row += nrows
        t0 = time.perf_counter()
        r = self.oracle.fused_reduce_norm(self.parts, self.res, self.wt, self.bs, 1e-6,
                                          self.w["mode"], self.scale, Tv, rows=rows,
                                          threads=min(threads or self.cores, nrows),
                                          buffers=self.buffers)
        dt = time.perf_counter() - t0
        assert r["status"] == 0
        self.buffers = r
        tp, _, H = self.parts.shape
        return dt, algorithmic_bytes(tp, nrows, nrows, H, self.w["mode"], self.res is not None)

    def rows_for(self, seconds: float, threads: int | None = None) -> int:
        """Rows that take about `seconds`, from a probe of 8 rows per thread."""
        probe = min(self.w["T_valid"], 8 * (threads or self.cores))
        self.run(probe, threads)  # warm caches and the library
        dt, _ = self.run(probe, threads)
        return max(1, int(probe * seconds / max(dt, 1e-6)))


def cpu_baseline(w: dict, host_in: dict, target_s: float = 12.0,
                 single_thread_s: float = 3.0) -> dict:
    """The oracle as it stands, on all host cores, over a bounded sample of about `target_s`
    seconds: consecutive valid rows of the workload, wrapping around when the sample is larger
    than the workload. Beside it, the same on one thread over about `single_thread_s` seconds."""
    runner = OracleRunner(w, host_in)

    def sample(seconds: float, threads: int | None) -> tuple[int, float, int]:
        want = runner.rows_for(seconds, threads)
        runner.next_row = 0
        done, secs, nbytes = 0, 0.0, 0
        while done < want:
            n = min(w["T_valid"], want - done)
            dt, b = runner.run(n, threads)
            done, secs, nbytes = done + n, secs + dt, nbytes + b
        return done, secs, nbytes

    done, secs, nbytes = sample(target_s, None)
    d1, s1, b1 = sample(single_thread_s, 1)
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": runner.cores, "kind": "oracle",
            "sample": f"{done} valid rows ({done / w['T_valid']:.2f} passes over the workload's "
                      f"{w['T_valid']} rows, {nbytes / 1e6:.0f} MB algorithmic), "
                      f"{runner.cores} threads, {secs:.1f} s",
            "mtokens_per_s": done / secs / 1e6,
            "single_thread": {"value": b1 / s1 / 1e9, "unit": "GB/s",
                              "sample": f"{d1} valid rows, 1 thread, {s1:.1f} s"}}


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over the ranks of the default process group (the slowest rank's
    time); the value itself when no group is initialised."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """GB/s over all ranks: every rank moves bytes_per_step per step (independent replicas),
    divided by the slowest rank's timed region."""
    return bytes_per_step * steps * world / (max_ms / 1e3) / 1e9


def run_ours(args) -> None:
    import sequence_reduce_add_gb300 as sp
    from sequence_reduce_add_gb300 import build as sp_build
    from sequence_reduce_add_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0 or world == 1:
        sp_build.build()
    if dist:
        dist.barrier()
    lib = sp.load_library()

    w = synth.workload(args.workload if not str(args.workload).isdigit() else int(args.workload))
    one = algorithmic_bytes(w["tp"], w["T_valid"], w["T_pad"], w["H"], w["mode"])
    # enough resident sets that one full rotation is far above L2
    probe = Problem(w, synth.BASE_SEED + 1 + synth.WORKLOADS.index(
        next(x for x in synth.WORKLOADS if x["name"] == w["name"])), device, sp)
    sets = max(2, min(8, -(-(4 * L2_BYTES) // probe.nbytes())))
    problems = [probe] + [Problem(w, probe.inp["seed"] + 1000 * k, device, sp)
                          for k in range(1, sets)]
    rotation_bytes = sum(p.nbytes() for p in problems)
    stream = torch.cuda.Stream(device=device)

    # The clock sampler starts first, so that the GPU does not idle between the warm-up and the
    # timed region; then warm-up, then the timed region (barrier + synchronize on both sides).
    # The timed launches are queued behind a device-side sleep that ends before the start event.
    with ClockSampler(local) as clocks:
        time_kernel_loop(lib, problems, max(args.warmup, 3), stream, False)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        total_ms, _, info = time_kernel_loop(lib, problems, args.steps, stream, False, gate=True)
        t1 = time.time()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
        total_ms = max_over_ranks(total_ms, device)
    ms_per_step = total_ms / args.steps
    value = whole_job_throughput(one, args.steps, world, total_ms)
    mtok = w["T_valid"] * args.steps * world / (total_ms / 1e3) / 1e6
    # The timed loop is one kernel per step launched back to back (consecutive launches overlap
    # their launch latency and prologue through programmatic dependent launch), so the kernel's
    # average launch duration is the timed region over the launches. Beside it: the same chain
    # with an event after every launch (per-launch times of the first launches, to show the
    # timed region is steady from its start), and event-bracketed launches (no overlap with
    # their neighbours).
    kernel_ms = ms_per_step
    _, chain, _ = time_kernel_loop(lib, problems, min(args.steps, 20), stream, False, gate=True,
                                   end_events=True)
    _, isolated, _ = time_kernel_loop(lib, problems, min(args.steps, 300), stream, True)
    isolated_ms = float(np.mean(isolated))
    isolated_median_ms, isolated_min_ms = float(np.median(isolated)), float(np.min(isolated))
    peak, peak_kind = measured_peak()
    achieved = one / (kernel_ms / 1e3) / 1e9

    e2e = e2e_loop(sp, w, problems[0], steps=max(5, min(50, args.steps // 100)),
                   warmup=2, stream=stream)
    host_in = e2e.pop("host_inputs")
    if problems[0].inp["scale"] is not None:
        host_in["scale"] = problems[0].inp["scale"]
    e2e_value = one / (e2e["ms_per_step"] / 1e3) / 1e9

    extras = {}
    if not args.no_extras:
        for other in synth.WORKLOADS:
            if other["name"] == w["name"]:
                continue
            extras[other["name"]] = bench_extra(lib, sp, synth, other, device, stream, peak)
        for name, variant in VARIANT_RUNS:
            extras[f"{name}+{variant}"] = bench_extra(lib, sp, synth, synth.workload(name),
                                                      device, stream, peak, variant)
        for tp, T, H in DECODE_RUNS:
            dw = dict(synth.workload("tp16_T3500p3504_H8192_fp8pertoken"), tp=tp, T_valid=T,
                      T_pad=T, H=H, name=f"decode_tp{tp}_T{T}_H{H}_fp8pertoken")
            extras[dw["name"]] = bench_extra(lib, sp, synth, dw, device, stream, peak,
                                             seed=synth.BASE_SEED + 100 + T)
        extras["fc2_reorganize_G8_otp2_N8192_H7168_bf16"] = bench_fc2(lib, device, stream, peak)

    if rank != 0:
        return
    cpu = cpu_baseline(w, host_in) if world == 1 or rank == 0 else None
    cfg = sp.sp_select_launch(w["tp"], w["T_pad"], w["H"], w["mode"]).as_dict()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; bf16 inputs as in the workload definition)",
        "mtokens_per_s": round(mtok, 3),
        "config": workload_config(w, world),
        "launch": cfg,
        "rotation": f"{len(problems)} resident input/output sets rotated, "
                    f"{rotation_bytes / 1e6:.0f} MB per rotation",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": ncu_traffic(w["name"], cfg), "kernel_ms": round(kernel_ms, 6),
                     "isolated_launch_ms": round(isolated_ms, 6),
                     "isolated_launch_ms_median": round(isolated_median_ms, 6),
                     "isolated_launch_ms_min": round(isolated_min_ms, 6),
                     "isolated_frac": round(one / (isolated_ms / 1e3) / 1e9 / peak, 4),
                     "kernel": "k_staged" if cfg["kernel"] == 0 else "k_direct",
                     "peak_note": "peak = measured HBM copy (torch copy_, read + write bytes)",
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "host_ahead": info["host_ahead"],
                     "chain_launch_us": [round(x * 1e3, 2) for x in chain]},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "ms_per_step": round(e2e["ms_per_step"], 4),
                "api": "sp_fused_reduce_norm_host (zero-copy over the host link)",
                "staged_copies_value": round(one / (e2e["staged_ms_per_step"] / 1e3) / 1e9, 2),
                "staged_copies_ms_per_step": round(e2e["staged_ms_per_step"], 4)},
        "cpu_baseline": cpu,
        "clocks": clocks.summary(t0, t1),
        "gpu_launches": args.steps,
        "workloads": extras,
    }
    print(json.dumps(line), flush=True)


def bench_extra(lib, sp, synth, w, device, stream, peak, variant: str | None = None,
                seed: int | None = None) -> dict:
    """Per-workload kernel figures for the other workloads (rotating sets, CUDA events)."""
    if seed is None:
        seed = synth.BASE_SEED + 1 + synth.WORKLOADS.index(w)
    base = Problem(w, seed, device, sp, variant)
    sets = max(2, min(6, -(-(4 * L2_BYTES) // base.nbytes())))
    problems = [base] + [Problem(w, base.inp["seed"] + 1000 * k, device, sp, variant)
                         for k in range(1, sets)]
    one = base.bytes
    # about 50 ms of timed launches at ~6.5 TB/s (at least 20, at most 4000 launches)
    steps = int(min(4000, max(20, 0.05 * 6.5e12 / max(one, 1))))
    time_kernel_loop(lib, problems, 10, stream, False)
    total, _, _ = time_kernel_loop(lib, problems, steps, stream, False, gate=True)
    _, launches, _ = time_kernel_loop(lib, problems, min(steps, 100), stream, True)
    k = total / steps
    gbs = one / (k / 1e3) / 1e9
    graph_us = None
    if one < 64e6:  # small enough to be launch-bound: also time launches replayed from a graph
        g = torch.cuda.CUDAGraph()
        fn = getattr(lib, problems[0].fn_name)
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                hh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
                for i in range(100):
                    fn(*problems[i % len(problems)].args, hh)
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(20):
                g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        graph_us = round(a.elapsed_time(b) / 2000 * 1e3, 2)
        del g
    res = {"GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
           "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
           "mtokens_per_s": round(w["T_valid"] / (k / 1e3) / 1e6, 3), "kernel_us": round(k * 1e3, 2),
           "isolated_launch_us": round(float(np.mean(launches)) * 1e3, 2), "steps": steps,
           "bytes": one, "cuda_graph_us_per_launch": graph_us,
           "sets": len(problems),
           "launch": sp.sp_select_launch(w["tp"], w["T_pad"], w["H"], w["mode"]).as_dict()}
    del problems
    torch.cuda.empty_cache()
    return res


FC2_WORKLOAD = "fc2_reorganize_G8_otp2_N8192_H7168_bf16"
REFERENCE_ROWS = 4096  # rows of the workload the reference arm draws on the host


def run_kernel_only(args) -> None:
    """Warm-up and timed launches of the workload's kernel only, rotating over resident sets;
    prints a short JSON line (the launch sequence that profiler captures are taken from).
    --rows R keeps the workload's shape and mode but only its first R padded rows (a smaller
    capture of the same kernel)."""
    import sequence_reduce_add_gb300 as sp
    from sequence_reduce_add_gb300 import build as sp_build
    from sequence_reduce_add_gb300 import synth
    sp_build.build()
    lib = sp.load_library()
    device = torch.device("cuda", 0)
    if args.workload == FC2_WORKLOAD:
        stream = torch.cuda.Stream(device=device)
        r = bench_fc2(lib, device, stream, measured_peak()[0])
        print(json.dumps({"workload": FC2_WORKLOAD, **r}), flush=True)
        return
    w = synth.workload(args.workload if not str(args.workload).isdigit() else int(args.workload))
    if args.shape:  # tp,T,H[,mode]: the workload's distributions at another shape (all rows valid)
        parts = args.shape.split(",")
        tp, T, H = (int(x) for x in parts[:3])
        w.update(tp=tp, T_pad=T, T_valid=T, H=H, name=f"{w['name']}@tp{tp}_T{T}_H{H}")
        if len(parts) > 3:
            w["mode"] = parts[3]
    if args.rows:  # a multiple of tp, with as many padding rows as the full workload
        pad = w["T_pad"] - w["T_valid"]
        w["T_pad"] = max(w["tp"], min(w["T_pad"], args.rows) // w["tp"] * w["tp"])
        w["T_valid"] = max(0, w["T_pad"] - pad)
    base_name = w["name"].split("@")[0]
    base = Problem(w, synth.BASE_SEED + 1 + synth.WORKLOADS.index(
        next(x for x in synth.WORKLOADS if x["name"] == base_name)), device, sp)
    sets = max(2, min(8, -(-(4 * L2_BYTES) // base.nbytes())))
    problems = [base] + [Problem(w, base.inp["seed"] + 1000 * k, device, sp)
                         for k in range(1, sets)]
    stream = torch.cuda.Stream(device=device)
    if args.warmup:
        time_kernel_loop(lib, problems, args.warmup, stream, False)
    total_ms, launches, _ = time_kernel_loop(lib, problems, args.steps, stream, True)
    one = algorithmic_bytes(w["tp"], w["T_valid"], w["T_pad"], w["H"], w["mode"])
    k = float(np.mean(launches))
    print(json.dumps({"workload": w["name"], "launches": args.steps, "sets": len(problems),
                      "kernel_us": round(k * 1e3, 2), "GB_per_s": round(one / k / 1e6, 1),
                      "launch": sp.sp_select_launch(w["tp"], w["T_pad"], w["H"],
                                                    w["mode"]).as_dict()}), flush=True)


def bench_fc2(lib, device, stream, peak, G=8, P=2, N=8192, H=7168) -> dict:
    """FlashComm2 token reorganisation of [G][N][H/G] bf16 (a pure permutation: algorithmic
    bytes = read x + write y = 2 * N * H * 2)."""
    nbytes = N * H * 2
    sets = max(2, -(-(4 * L2_BYTES) // (2 * nbytes)))
    g = torch.Generator(device=device).manual_seed(7)
    xs = [torch.randn((G, N, H // G), generator=g, device=device).to(torch.bfloat16)
          for _ in range(sets)]
    ys = [torch.empty((G, N // (G // P), H // P), dtype=torch.bfloat16, device=device)
          for _ in range(sets)]
    h = ctypes.c_void_p(stream.cuda_stream)
    args = [(x.data_ptr(), G, P, N, H, 2, y.data_ptr(), h) for x, y in zip(xs, ys)]
    one = 2 * nbytes
    steps = int(min(4000, max(20, 0.05 * 6.5e12 / one)))
    for k in range(10):
        lib.sp_fc2_reorganize(*args[k % sets])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gate_stream(stream, steps)
    a.record(stream)
    for k in range(steps):
        st = lib.sp_fc2_reorganize(*args[k % sets])
        if st != 0:
            raise RuntimeError(f"sp_fc2_reorganize returned {st}")
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    gbs = one / (ms / 1e3) / 1e9
    del xs, ys
    torch.cuda.empty_cache()
    return {"GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
            "kernel_us": round(ms * 1e3, 2), "steps": steps, "bytes": one, "sets": sets,
            "mtokens_per_s": round(N / (ms / 1e3) / 1e6, 3)}


# ------------------------------------------------------------------------------ reference arm
def run_reference(args) -> None:
    """The oracle (fp64 C++ on the host cores), timed as the reference arm on our workload.

    Each step computes a bounded sample of rows of the workload, sized so that the whole
    --warmup W --steps K run takes about --reference-budget-s seconds."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import build as oracle_build
    from sequence_reduce_add_gb300 import synth
    oracle_build.build()
    w = synth.workload(args.workload if not str(args.workload).isdigit() else int(args.workload))
    # The oracle computes a bounded row sample per step, so only the first REFERENCE_ROWS rows of
    # the workload are drawn (same shape, mode and distributions; a multiple of tp).
    rows_drawn = min(w["T_pad"], max(w["tp"], REFERENCE_ROWS // w["tp"] * w["tp"]))
    inp = synth.make_inputs(w, device="cpu", T_pad=rows_drawn)
    host_in = {k: inp[k] for k in ("partials", "residual", "weight", "bias") if inp[k] is not None}
    if inp["scale"] is not None:
        host_in["scale"] = inp["scale"]
    runner = OracleRunner(dict(w, T_pad=rows_drawn, T_valid=inp["T_valid"]), host_in)
    total_steps = max(args.warmup, 0) + args.steps
    rows = runner.rows_for(args.reference_budget_s / max(total_steps, 1))
    for _ in range(max(args.warmup, 0)):
        runner.run(rows)
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        dt, b = runner.run(rows)
        secs += dt
        nbytes += b
    value = nbytes / secs / 1e9
    rows = min(rows, inp["T_valid"])
    tok = rows * args.steps
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": runner.cores, "kind": "oracle",
           "sample": f"{rows} valid rows per step (of the workload's first {rows_drawn} rows, "
                     f"drawn as in the workload), {args.steps} timed steps, {secs:.1f} s, "
                     f"{runner.cores} threads"}
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "mtokens_per_s": round(tok / secs / 1e6, 4),
        "config": workload_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--kernel-only", action="store_true",
                    help="only warm-up + timed kernel launches of the workload (for profilers)")
    ap.add_argument("--rows", type=int, default=0,
                    help="with --kernel-only: use only the first ROWS padded rows")
    ap.add_argument("--shape", default="",
                    help="with --kernel-only: tp,T,H[,mode] at the workload's distributions")
    ap.add_argument("--reference-budget-s", type=float, default=60.0,
                    help="CPU seconds for the whole reference-arm run (bounded row samples)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel_only:
        run_kernel_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
