"""The Python binding refuses tensors the call would misuse, before anything reaches the library.

The C entry points can check only what their shape arguments imply; a buffer that is too small,
non-contiguous, of the wrong element type or on another device would turn into out-of-bounds or
wrong-row accesses on the GPU. These CPU tests stand a CPU device in for the current CUDA device
and a recording fake in for the library: every valid call reaches the fake, and every bad tensor
raises ValueError with the fake untouched.
"""
import pytest
import torch

import sequence_reduce_add_gb300 as sp


class FakeLib:
    """Records calls; every entry point returns SP_OK."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append(name)
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(sp, "load_library", lambda: lib)
    monkeypatch.setattr(sp, "_current_device", lambda: torch.device("cpu"))
    return lib


TP, T, H = 2, 8, 64


def problem(mode="none", scale_layout=0):
    bf = torch.bfloat16
    p = dict(partials=torch.zeros((TP, T, H), dtype=bf), weight=torch.ones(H, dtype=bf),
             residual=torch.zeros((T, H), dtype=bf), bias=torch.zeros(H, dtype=bf))
    outs = sp.allocate_outputs(T, H, "none" if mode == "none" else "fp8_static", "cpu")
    if mode == "fp8_per_token":
        outs["out_scales"] = torch.zeros(T, dtype=torch.float32)
    if mode == "nvfp4":
        outs["out"] = torch.zeros((T, H // 2), dtype=torch.uint8)
        n = 128 * 4 if scale_layout == 1 else T * (H // 16)
        outs["out_scales"] = torch.zeros(n, dtype=torch.uint8)
    p.update(outs)
    p["scale"] = torch.ones(1, dtype=torch.float32) if mode in ("fp8_static", "nvfp4") else None
    return p


def call(p, mode="none", entry=sp.sp_fused_reduce_norm, **extra):
    entry(p["partials"], p["weight"], p["out"], p["residual_out"], residual=p["residual"],
          bias=p["bias"], quant_mode=mode, scale=p["scale"], out_scales=p["out_scales"],
          stream=0, **extra)


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
def test_valid_calls_reach_the_library(fake, mode):
    call(problem(mode), mode)
    assert fake.calls == ["sp_fused_reduce_norm"]


BAD = {
    "partials_dtype": lambda p: p.update(partials=p["partials"].float()),
    "partials_2d": lambda p: p.update(partials=p["partials"][0]),
    "partials_strided": lambda p: p.update(partials=p["partials"].transpose(1, 2)),
    "residual_short": lambda p: p.update(residual=p["residual"][: T - 1]),
    "residual_transposed": lambda p: p.update(residual=p["residual"].t()),
    "residual_dtype": lambda p: p.update(residual=p["residual"].half()),
    "weight_short": lambda p: p.update(weight=p["weight"][: H - 8]),
    "bias_dtype": lambda p: p.update(bias=p["bias"].float()),
    "out_short": lambda p: p.update(out=p["out"][: T - 1]),
    "out_dtype": lambda p: p.update(out=p["out"].float()),
    "residual_out_short": lambda p: p.update(residual_out=p["residual_out"][1:]),
    "residual_out_strided": lambda p: p.update(
        residual_out=torch.zeros((H, T), dtype=torch.bfloat16).t()),
    "other_device": lambda p: p.update(weight=torch.ones(H, dtype=torch.bfloat16, device="meta")),
    "not_a_tensor": lambda p: p.update(bias=[0.0] * H),
}


@pytest.mark.parametrize("name", sorted(BAD))
def test_bad_tensor_is_refused_before_the_library(fake, name):
    p = problem()
    BAD[name](p)
    with pytest.raises(ValueError):
        call(p)
    assert fake.calls == []


@pytest.mark.parametrize("mode,bad", [
    ("fp8_per_token", lambda p: p.update(out_scales=p["out_scales"][: T - 1])),
    ("fp8_per_token", lambda p: p.update(out_scales=p["out_scales"].double())),
    ("nvfp4", lambda p: p.update(out_scales=p["out_scales"][:-1])),
    ("nvfp4", lambda p: p.update(out=p["out"][:, : H // 4])),
    ("fp8_static", lambda p: p.update(scale=p["scale"].double())),
    ("fp8_static", lambda p: p.update(scale=torch.ones(0, dtype=torch.float32))),
])
def test_bad_mode_buffers_are_refused(fake, mode, bad):
    p = problem(mode)
    bad(p)
    with pytest.raises(ValueError):
        call(p, mode)
    assert fake.calls == []


def test_swizzled_scales_need_the_padded_size(fake):
    p = problem("nvfp4", scale_layout=1)
    opts = sp.sp_options_init(scale_layout=1)
    call(p, "nvfp4", entry=lambda *a, **k: sp.sp_fused_reduce_norm_ex(opts, *a, **k))
    assert fake.calls == ["sp_options_init", "sp_fused_reduce_norm_ex"]
    fake.calls.clear()
    p["out_scales"] = p["out_scales"][: T * (H // 16)]  # the row-major size is too small here
    with pytest.raises(ValueError):
        call(p, "nvfp4", entry=lambda *a, **k: sp.sp_fused_reduce_norm_ex(opts, *a, **k))
    assert fake.calls == []


def test_addend_is_checked(fake):
    p = problem()
    opts = sp.sp_options_init(addend=torch.zeros((T - 1, H), dtype=torch.bfloat16))
    fake.calls.clear()
    with pytest.raises(ValueError, match="addend"):
        call(p, entry=lambda *a, **k: sp.sp_fused_reduce_norm_ex(opts, *a, **k))
    assert fake.calls == []


def test_host_entry_needs_page_locked_memory(fake):
    with pytest.raises(ValueError, match="page-locked"):
        call(problem(), entry=sp.sp_fused_reduce_norm_host)
    assert fake.calls == []


def test_fc2_buffers_are_checked(fake):
    x = torch.zeros((4, 16, 8), dtype=torch.bfloat16)
    sp.sp_fc2_reorganize(x, 2, torch.zeros((4, 8, 16), dtype=torch.bfloat16), stream=0)
    assert fake.calls == ["sp_fc2_reorganize"]
    fake.calls.clear()
    for y in (torch.zeros((4, 8, 16), dtype=torch.float16),     # another element type
              torch.zeros((4, 8, 15), dtype=torch.bfloat16),    # too small
              torch.zeros((4, 16, 8), dtype=torch.bfloat16).transpose(1, 2)):  # strided
        with pytest.raises(ValueError):
            sp.sp_fc2_reorganize(x, 2, y, stream=0)
    assert fake.calls == []
