"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (the hot path's contract):
* layout, padding, shard indexing: bit-exact; every byte of a padding row is zero.
* bf16 outputs (out, residual_out): |gpu - ref| <= 2 bf16 ulp(|ref|) + floor, where ref is the
  oracle's fp64 y (out) or its correctly rounded bf16 value (residual_out), and
  floor = 2^-18 * max_j |ref_row|. The floor covers fp32 cancellation in h: the kernel adds up to
  tp + 2 bf16 terms in fp32, an absolute error of at most (tp + 2) * 2^-24 * sum|terms| per
  element, which is below 2^-18 of the row's largest output for the workloads' distributions.
* FP8 / FP4 codes: >= 99.9 % identical, every other one at most one code step away (+0 and -0
  are the same step).
* fp32 per-token scales: relative 1e-5.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import synth

GUARD = 4096
CANARY = 0xC3
CORES = os.cpu_count() or 1


def guarded_empty(nbytes: int, device, fill: int) -> tuple[torch.Tensor, torch.Tensor]:
    """A uint8 buffer with GUARD canary bytes on each side; returns (whole, middle)."""
    whole = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
    mid = whole[GUARD:GUARD + nbytes]
    mid.fill_(fill)
    return whole, mid


def _view(mid: torch.Tensor, shape, dtype) -> torch.Tensor:
    return mid.view(dtype).view(shape)


def _pinned(t):
    return None if t is None else t.cpu().pin_memory()


def run_gpu_host(inp: dict, *, fill: int = 0xA5, stream=None, partial_scale: float = 1.0,
                 scale_layout: int = 0, config: dict | None = None) -> dict:
    """Run the zero-copy entry point on pinned host copies of ``inp`` into guard-banded pinned
    host outputs pre-filled with ``fill``; returns numpy results."""
    T_pad, H, mode = inp["T_pad"], inp["H"], inp["mode"]
    hin = {k: _pinned(inp.get(k)) for k in ("partials", "residual", "weight", "bias", "addend")}
    o_bytes = sp.sp_out_bytes(T_pad, H, mode)
    s_bytes = sp.sp_out_scales_bytes_ex(T_pad, H, mode, scale_layout)
    oshape, odt, sshape, sdt = oracle.out_layout(T_pad, H, mode, scale_layout)
    tdt = {np.uint16: torch.bfloat16, np.uint8: torch.uint8, np.float32: torch.float32}

    def guarded(nbytes):
        whole = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8).pin_memory()
        whole[GUARD:GUARD + nbytes].fill_(fill)
        return whole, whole[GUARD:GUARD + nbytes]

    out_w, out_m = guarded(o_bytes)
    out = _view(out_m, oshape, tdt[odt])
    sc_w = sc = None
    if s_bytes:
        sc_w, sc_m = guarded(s_bytes)
        sc = _view(sc_m, sshape, tdt[sdt])
    res_w, res_m = guarded(T_pad * H * 2)
    res_out = _view(res_m, (T_pad, H), torch.bfloat16)
    scale_t = (torch.tensor([inp["scale"]], dtype=torch.float32).pin_memory()
               if inp["scale"] is not None else None)
    if partial_scale == 1.0 and hin["addend"] is None and scale_layout == 0 and config is None:
        sp.sp_fused_reduce_norm_host(hin["partials"], hin["weight"], out, res_out,
                                     residual=hin["residual"], bias=hin["bias"], eps=inp["eps"],
                                     quant_mode=mode, scale=scale_t, out_scales=sc,
                                     T_valid=inp["T_valid"], stream=stream)
    else:
        opts = sp.sp_options_init(partial_scale=partial_scale, addend=hin["addend"],
                                  scale_layout=scale_layout, host_buffers=True, launch=config)
        sp.sp_fused_reduce_norm_ex(opts, hin["partials"], hin["weight"], out, res_out,
                                   residual=hin["residual"], bias=hin["bias"], eps=inp["eps"],
                                   quant_mode=mode, scale=scale_t, out_scales=sc,
                                   T_valid=inp["T_valid"], stream=stream)
    torch.cuda.synchronize()
    for w in (out_w, sc_w, res_w):
        if w is not None:
            g = torch.cat([w[:GUARD], w[-GUARD:]])
            assert bool((g == CANARY).all()), "write outside an output buffer"
    return {"out": bits_of(out), "out_scales": None if sc is None else bits_of(sc),
            "residual_out": bits_of(res_out)}


def run_gpu(inp: dict, *, config: dict | None = None, fill: int = 0xA5, inplace: bool = False,
            stream=None, partial_scale: float = 1.0, scale_layout: int = 0,
            schedule: str = "auto") -> dict:
    """Run the library once on inputs ``inp`` (device tensors from synth.make_inputs) into
    guard-banded outputs pre-filled with ``fill``; returns host numpy results."""
    dev = inp["partials"].device
    T_pad, H, mode = inp["T_pad"], inp["H"], inp["mode"]
    o_bytes = sp.sp_out_bytes(T_pad, H, mode)
    s_bytes = sp.sp_out_scales_bytes_ex(T_pad, H, mode, scale_layout)
    out_w, out_m = guarded_empty(o_bytes, dev, fill)
    oshape, odt, sshape, sdt = oracle.out_layout(T_pad, H, mode, scale_layout)
    tdt = {np.uint16: torch.bfloat16, np.uint8: torch.uint8, np.float32: torch.float32}
    out = _view(out_m, oshape, tdt[odt])
    sc_w = sc = None
    if s_bytes:
        sc_w, sc_m = guarded_empty(s_bytes, dev, fill)
        sc = _view(sc_m, sshape, tdt[sdt])
    residual = inp["residual"]
    if inplace:
        assert residual is not None
        res_w, res_m = guarded_empty(T_pad * H * 2, dev, 0)
        res_out = _view(res_m, (T_pad, H), torch.bfloat16)
        res_out.copy_(residual)
        residual = res_out
    else:
        res_w, res_m = guarded_empty(T_pad * H * 2, dev, fill)
        res_out = _view(res_m, (T_pad, H), torch.bfloat16)
    scale_t = None
    if inp["scale"] is not None:
        scale_t = torch.tensor([inp["scale"]], dtype=torch.float32, device=dev)
    kw = dict(residual=residual, bias=inp["bias"], eps=inp["eps"], quant_mode=mode, scale=scale_t,
              out_scales=sc, T_valid=inp["T_valid"], stream=stream)
    if (partial_scale != 1.0 or inp.get("addend") is not None or scale_layout != 0
            or schedule != "auto"):
        opts = sp.sp_options_init(partial_scale=partial_scale, addend=inp.get("addend"),
                                  scale_layout=scale_layout, schedule=schedule, launch=config)
        sp.sp_fused_reduce_norm_ex(opts, inp["partials"], inp["weight"], out, res_out, **kw)
    elif config is None:
        sp.sp_fused_reduce_norm(inp["partials"], inp["weight"], out, res_out, **kw)
    else:
        sp.sp_fused_reduce_norm_with_config(config, inp["partials"], inp["weight"], out, res_out,
                                            **kw)
    torch.cuda.synchronize(dev)
    for w in (out_w, sc_w, res_w):
        if w is not None:
            g = torch.cat([w[:GUARD], w[-GUARD:]])
            assert bool((g == CANARY).all()), "write outside an output buffer"
    return {"out": bits_of(out), "out_scales": None if sc is None else bits_of(sc),
            "residual_out": bits_of(res_out)}


def bits_of(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def run_oracle(inp: dict, want_y: bool = True, rows=None, partial_scale: float = 1.0,
               scale_layout: int = 0) -> dict:
    to = synth.bf16_bits
    add = inp.get("addend")
    res = oracle.fused_reduce_norm(
        to(inp["partials"]), None if inp["residual"] is None else to(inp["residual"]),
        to(inp["weight"]), None if inp["bias"] is None else to(inp["bias"]), inp["eps"],
        inp["mode"], inp["scale"], inp["T_valid"], want_y=want_y, threads=CORES, rows=rows,
        partial_scale=partial_scale, addend=None if add is None else to(add),
        scale_layout=scale_layout)
    assert res["status"] == 0
    return res


def _bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.exp2(e - 7)


def check_bf16(gpu: np.ndarray, ref: np.ndarray, rows: slice, what: str) -> float:
    g = _bf16_to_f64(gpu[rows])
    r = ref[rows]
    floor = np.exp2(-18) * np.abs(r).max(axis=1, keepdims=True)
    tol = 2 * _bf16_ulp(r) + floor
    bad = ~(np.abs(g - r) <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance; first at "
                           f"{np.argwhere(bad)[0]}: gpu {g[bad][0]!r} ref {r[bad][0]!r}")
    return float(np.abs(g - r).max()) if g.size else 0.0


def _ordinal(codes: np.ndarray, sign_bit: int) -> np.ndarray:
    c = codes.astype(np.int32)
    mag = c & (sign_bit - 1)
    return np.where(c & sign_bit, -mag, mag)


def check_codes(gpu: np.ndarray, ref: np.ndarray, sign_bit: int, what: str) -> float:
    og, orf = _ordinal(gpu, sign_bit), _ordinal(ref, sign_bit)
    d = np.abs(og - orf)
    if d.size == 0:
        return 1.0
    match = float((d == 0).mean())
    assert d.max() <= 1, f"{what}: a code {int(d.max())} steps away"
    assert match >= 0.999, f"{what}: only {match:.6f} of codes identical"
    return match


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def compare(gpu: dict, ref: dict, inp: dict) -> dict:
    """Assert parity of one call; returns summary statistics."""
    Tv, mode = inp["T_valid"], inp["mode"]
    valid = slice(0, Tv)
    stats = {}
    swizzled = mode == "nvfp4" and gpu["out_scales"] is not None and gpu["out_scales"].ndim == 1
    # padding rows: all zero bytes (swizzled scales: compared whole against the oracle below)
    for k in ("out", "out_scales", "residual_out"):
        if gpu[k] is not None and not (k == "out_scales" and swizzled):
            pad = gpu[k][Tv:]
            assert not pad.view(np.uint8).any(), f"{k}: padding rows not zero"
    stats["residual_max_abs"] = check_bf16(gpu["residual_out"], _bf16_to_f64(ref["residual_out"]),
                                           valid, "residual_out")
    if mode == "none":
        stats["out_max_abs"] = check_bf16(gpu["out"], ref["y"], valid, "out")
    elif mode in ("fp8_static", "fp8_per_token"):
        stats["code_match"] = check_codes(gpu["out"][valid], ref["out"][valid], 0x80, "e4m3 out")
        if mode == "fp8_per_token":
            g, r = gpu["out_scales"][valid].astype(np.float64), ref["out_scales"][valid].astype(np.float64)
            rel = np.abs(g - r) / np.where(r > 0, r, 1.0)
            assert np.all((rel <= 1e-5) | ((g == 0) & (r == 0))), "per-token scales"
            stats["scale_max_rel"] = float(rel.max()) if rel.size else 0.0
    elif mode == "nvfp4":
        if swizzled:  # the whole padded buffer: scales in place, padding bytes zero
            stats["scale_code_match"] = check_codes(gpu["out_scales"], ref["out_scales"], 0x80,
                                                    "e4m3 block scales (swizzled)")
        else:
            stats["scale_code_match"] = check_codes(gpu["out_scales"][valid],
                                                    ref["out_scales"][valid], 0x80,
                                                    "e4m3 block scales")
        stats["code_match"] = check_codes(unpack_e2m1(gpu["out"][valid]),
                                          unpack_e2m1(ref["out"][valid]), 0x8, "e2m1 out")
    return stats
