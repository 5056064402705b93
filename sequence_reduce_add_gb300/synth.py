"""Seeded synthetic inputs for the fused reduce + bias/residual add + RMSNorm + quant stage.

This module is the one piece that both the CUDA path's tests/bench and the CPU oracle see: it
draws input tensors and nothing else. It holds none of the method's arithmetic (no sums,
norms, scales or codes) and imports nothing else from this package.

Workloads (one per row of the hot path's configuration list; the pages publish no data, so all
values are drawn from the stated distributions with ``torch.Generator(seed)``):

* partials: ``tp`` tensors [T_pad, H], normal with variance 1/tp (so their sum has unit
  variance), or Student-t with 3 degrees of freedom divided by 8 (heavy tails);
* residual: N(0, 1) [T_pad, H]; optionally a seeded 0.1 % of the hidden channels scaled x50
  (outlier channels);
* weight ``1 + 0.1 N(0,1)`` and bias ``0.01 N(0,1)``, each [H];
* every input row at or beyond ``T_valid`` (padding) is filled with NaN, so any read of a padding
  row would surface in the outputs.

All tensors are rounded once to bf16 from fp32 draws.
"""
from __future__ import annotations

import math

import torch

BASE_SEED = 20261202

# The five workloads, in order. ``T_pad`` is stated, not computed: 4093 tokens pad to 4096 for
# tp=4, 3500 pad to 3504 for tp=16 (16 shards of 219 rows).
WORKLOADS = [
    dict(name="tp2_T64_H1024_bf16", tp=2, T_valid=64, T_pad=64, H=1024, mode="none",
         partial_dist="normal", outliers=0, scale=None),
    dict(name="tp4_T4093p4096_H4096_bf16", tp=4, T_valid=4093, T_pad=4096, H=4096, mode="none",
         partial_dist="normal", outliers=0, scale=None),
    dict(name="tp8_T8192_H7168_fp8static", tp=8, T_valid=8192, T_pad=8192, H=7168,
         mode="fp8_static", partial_dist="normal", outliers=7, scale=0.05),
    dict(name="tp16_T3500p3504_H8192_fp8pertoken", tp=16, T_valid=3500, T_pad=3504, H=8192,
         mode="fp8_per_token", partial_dist="normal", outliers=0, scale=None),
    # NVFP4 global scale: 2688 / amax(y) over the first 256 rows of this workload's seed data,
    # taken from the oracle by tests/golden/calibrate_nvfp4_global_scale.py (3 significant digits).
    dict(name="tp8_T16384_H5120_nvfp4", tp=8, T_valid=16384, T_pad=16384, H=5120, mode="nvfp4",
         partial_dist="student_t3", outliers=0, scale=None),
]

NVFP4_GLOBAL_SCALE_FILE = "tests/golden/nvfp4_global_scale.json"


def workload(index_or_name) -> dict:
    """Workload by 1-based index or by name (a copy)."""
    if isinstance(index_or_name, int):
        return dict(WORKLOADS[index_or_name - 1])
    for w in WORKLOADS:
        if w["name"] == index_or_name:
            return dict(w)
    raise KeyError(index_or_name)


def _normal(g: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def make_inputs(w: dict, *, seed: int | None = None, device="cpu", T_valid: int | None = None,
                T_pad: int | None = None, H: int | None = None, tp: int | None = None,
                with_residual: bool = True, with_bias: bool = True, with_addend: bool = False,
                nan_padding: bool = True) -> dict:
    """Draw one problem of workload ``w`` (sizes may be overridden to shrink it).

    Returns a dict of tensors on ``device``: ``partials`` bf16 [tp, T_pad, H], ``residual`` bf16
    [T_pad, H] or None, ``weight`` bf16 [H], ``bias`` bf16 [H] or None, ``addend`` bf16
    [T_pad, H] (0.5 N(0,1), drawn last) or None, plus the scalars
    ``tp, T_pad, T_valid, H, eps, mode, scale`` (``scale`` is a Python float or None).
    """
    tp = tp or w["tp"]
    T_pad = T_pad if T_pad is not None else w["T_pad"]
    T_valid = T_valid if T_valid is not None else min(w["T_valid"], T_pad)
    H = H or w["H"]
    if seed is None:
        seed = BASE_SEED + WORKLOADS.index(next(x for x in WORKLOADS if x["name"] == w["name"])) + 1
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    partials = torch.empty((tp, T_pad, H), dtype=torch.bfloat16, device=device)
    for r in range(tp):
        if w["partial_dist"] == "normal":
            x = _normal(g, (T_pad, H), device) * math.sqrt(1.0 / tp)
        elif w["partial_dist"] == "student_t3":
            z = _normal(g, (T_pad, H), device)
            chi2 = _normal(g, (T_pad, H), device).square_()
            chi2 += _normal(g, (T_pad, H), device).square_()
            chi2 += _normal(g, (T_pad, H), device).square_()
            x = z / torch.sqrt(chi2 / 3.0) / 8.0
            del z, chi2
        else:
            raise ValueError(w["partial_dist"])
        partials[r] = x.to(torch.bfloat16)
        del x

    residual = None
    if with_residual:
        res = _normal(g, (T_pad, H), device)
        n_out = w.get("outliers", 0)
        if n_out:
            channels = torch.randperm(H, generator=g, device=device)[:n_out]
            res[:, channels] *= 50.0
        residual = res.to(torch.bfloat16)
        del res
    weight = (1.0 + 0.1 * _normal(g, (H,), device)).to(torch.bfloat16)
    bias = (0.01 * _normal(g, (H,), device)).to(torch.bfloat16) if with_bias else None

    addend = (0.5 * _normal(g, (T_pad, H), device)).to(torch.bfloat16) if with_addend else None

    if nan_padding and T_valid < T_pad:
        partials[:, T_valid:] = float("nan")
        for t in (residual, addend):
            if t is not None:
                t[T_valid:] = float("nan")

    scale = w.get("scale")
    if w["mode"] == "nvfp4":
        scale = nvfp4_global_scale()
    return dict(partials=partials, residual=residual, weight=weight, bias=bias, addend=addend,
                tp=tp, T_pad=T_pad,
                T_valid=T_valid, H=H, eps=1e-6, mode=w["mode"], scale=scale, seed=seed)


def nvfp4_global_scale() -> float:
    """The static NVFP4 global scale of the NVFP4 workload (a stored calibration constant)."""
    import json
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, NVFP4_GLOBAL_SCALE_FILE)) as f:
        return float(json.load(f)["global_scale"])


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's 16-bit patterns as a C-contiguous numpy uint16 array (on the host)."""
    import numpy as np
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
