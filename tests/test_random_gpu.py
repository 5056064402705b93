"""GPU parity on seeded random problems: shapes, modes, optional inputs, options, launch
configurations (split rows of both kernels included) and row schedules drawn together, so that combinations the hand-picked cases do not list are
covered too. Each problem is compared with the oracle element by element under the tolerances
of parity_util, after two runs into differently pre-filled, guard-banded outputs. Random
FlashComm2 reorganisations are compared byte for byte.
"""
import random

import numpy as np
import pytest
import torch

import oracle

import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import synth

from parity_util import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CASES = 128
SLICE_CASES = 32
FC2_CASES = 48
MODES = ["none", "fp8_static", "fp8_per_token", "nvfp4"]


def _draw(i: int) -> dict:
    """Problem i: sizes kept to at most ~2^21 row elements so the oracle stays fast."""
    r = random.Random(7919 * i + 17)
    mode = r.choice(MODES)
    step = 16 if mode == "nvfp4" else 8
    H = step * r.choice([1, 2, 3, r.randint(1, 64), r.randint(64, 512), r.randint(512, 1024)])
    tp = r.choice([1, 2, 3, 4, 5, 8, 16, r.randint(1, 24)])
    max_rows = max(tp, min(700, (1 << 21) // H))
    T_pad = tp * r.randint(1, max(1, max_rows // tp))
    T_valid = r.choice([T_pad, T_pad - r.randint(0, tp - 1), r.randint(0, T_pad)])
    p = dict(mode=mode, H=H, tp=tp, T_pad=T_pad, T_valid=max(0, T_valid),
             partial_dist=r.choice(["normal", "student_t3"]),
             outliers=r.choice([0, 0, min(H, 3)]),
             with_residual=r.random() < 0.8, with_bias=r.random() < 0.7,
             with_addend=r.random() < 0.25, inplace=False, config=None,
             partial_scale=1.0, scale_layout=0, schedule="auto", seed=1000 + i)
    if r.random() < 0.25:
        p["partial_scale"] = r.choice([0.5, 1.0 / 3.0, -2.0, 0.125])
    if mode == "nvfp4" and r.random() < 0.4:
        p["scale_layout"] = 1
    if r.random() < 0.3:
        p["schedule"] = r.choice(["static", "dynamic"])
    options = (p["with_addend"] or p["partial_scale"] != 1.0 or p["scale_layout"] != 0
               or p["schedule"] != "auto")
    if not options and p["with_residual"] and r.random() < 0.2:
        p["inplace"] = True
    if r.random() < 0.6:  # a forced launch (passed in the options when there are any)
        kernel = r.choice([0, 1])
        vec = r.choice([1, 2, 4])
        while -(-(H // 8) // vec) > 512:
            vec *= 2
        if vec <= 4:
            p["config"] = dict(kernel=kernel, vec_per_thread=vec, ctas_per_sm=r.randint(1, 8),
                               stages=r.choice([0, 2, 3, 4]) if kernel == 0 else 0)
            if kernel == 1 and vec <= 2 and r.random() < 0.5:
                p["config"]["split"] = r.choice([2, 4, 8])
            elif kernel == 0 and vec == 1 and r.random() < 0.5:  # staged split rows
                p["config"]["split"] = r.choice([2, 4, 8])
    return p


def _inputs(p: dict) -> dict:
    w = dict(name=f"random_{p['seed']}", tp=p["tp"], T_valid=p["T_valid"], T_pad=p["T_pad"],
             H=p["H"], mode=p["mode"], partial_dist=p["partial_dist"], outliers=p["outliers"],
             scale=0.05 if p["mode"] == "fp8_static" else None)
    return synth.make_inputs(w, seed=p["seed"], device=DEV, with_residual=p["with_residual"],
                             with_bias=p["with_bias"], with_addend=p["with_addend"])


def _check(p: dict) -> None:
    inp = _inputs(p)
    kw = dict(config=p["config"], inplace=p["inplace"], partial_scale=p["partial_scale"],
              scale_layout=p["scale_layout"], schedule=p["schedule"])
    try:
        a = run_gpu(inp, fill=0xA5, **kw)
    except sp.SpError as e:
        if e.status != 2 or p["config"] is None:  # only a forced launch may not fit
            raise
        kw["config"] = None
        a = run_gpu(inp, fill=0xA5, **kw)
    b = run_gpu(inp, fill=0x5A, **kw)
    for k in ("out", "out_scales", "residual_out"):
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), \
                f"{k}: bytes left unwritten or a non-deterministic result ({p})"
    ref = run_oracle(inp, partial_scale=p["partial_scale"], scale_layout=p["scale_layout"])
    compare(a, ref, inp)


@pytest.mark.parametrize("i", range(CASES))
def test_random_problem(i):
    _check(_draw(i))


@pytest.mark.parametrize("i", range(SLICE_CASES))
def test_random_staged_split_rows(i):
    """Random problems forced onto the staged kernel with rows split across a cluster."""
    p = _draw(CASES + i)
    r = random.Random(31 * i + 5)
    p["config"] = dict(kernel=0, vec_per_thread=1, ctas_per_sm=8, stages=0,
                       split=r.choice([2, 4, 8]))
    _check(p)


def test_draws_cover_every_mode_and_option():
    """The seeded draws include every mode, each option, forced launches and in-place updates."""
    ps = [_draw(i) for i in range(CASES)]
    assert {p["mode"] for p in ps} == set(MODES)
    assert any(p["with_addend"] for p in ps)
    assert any(p["partial_scale"] != 1.0 for p in ps)
    assert any(p["scale_layout"] == 1 for p in ps)
    assert any(p["inplace"] for p in ps)
    assert any(p["config"] and p["config"]["kernel"] == 0 for p in ps)
    assert any(p["config"] and p["config"]["kernel"] == 1 for p in ps)
    assert any(not p["with_residual"] for p in ps) and any(not p["with_bias"] for p in ps)
    assert any(p["T_valid"] < p["T_pad"] for p in ps)
    assert {p["schedule"] for p in ps} == {"auto", "static", "dynamic"}
    splits = [p for p in ps if p["config"] and p["config"].get("split", 0) > 1]
    assert {p["config"]["split"] for p in splits} == {2, 4, 8}
    assert {p["mode"] for p in splits} == set(MODES)
    staged_splits = [p for p in splits if p["config"]["kernel"] == 0]
    assert {p["config"]["split"] for p in staged_splits} == {2, 4, 8}
    assert len({p["mode"] for p in staged_splits}) >= 3
    assert any(p["scale_layout"] == 1 for p in splits)
    assert any(p["config"] and p["with_addend"] for p in ps)


def _draw_fc2(i: int) -> dict:
    r = random.Random(104729 * i + 3)
    G = r.choice([1, 2, 4, 8, 16, 32])
    P = r.choice([d for d in range(1, G + 1) if G % d == 0])
    eb = r.choice([1, 2, 4])
    # piece bytes F * eb: a multiple of 16, from one vector to past the 24 KB bulk-copy tile
    piece = 16 * r.choice([1, 2, r.randint(1, 64), r.randint(64, 512), r.randint(1536, 2048)])
    F = piece // eb
    N = G * r.randint(1, max(1, (1 << 23) // (G * G * piece)))
    return dict(G=G, P=P, eb=eb, F=F, N=N, seed=5000 + i)


@pytest.mark.parametrize("i", range(FC2_CASES))
def test_random_fc2_reorganisation(i):
    q = _draw_fc2(i)
    G, P, N, F, eb = q["G"], q["P"], q["N"], q["F"], q["eb"]
    D = G // P
    g = torch.Generator(device=DEV).manual_seed(q["seed"])
    x = torch.randint(0, 256, (G, N, F * eb), generator=g, device=DEV, dtype=torch.uint8)
    dt = {1: torch.uint8, 2: torch.bfloat16, 4: torch.float32}[eb]
    xv = x.view(dt)
    ys = []
    for fill in (0xA5, 0x5A):
        y = torch.full((G, N // D, D * F * eb), fill, dtype=torch.uint8, device=DEV)
        sp.sp_fc2_reorganize(xv, P, y.view(dt))
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy())
    assert np.array_equal(ys[0], ys[1]), f"bytes left unwritten ({q})"
    ref = oracle.fc2_reorganize(x.cpu().numpy(), P)
    assert np.array_equal(ys[0].reshape(ref.shape[0], ref.shape[1], -1),
                          ref.reshape(ref.shape[0], ref.shape[1], -1)), q
