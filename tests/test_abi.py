"""The C boundary without a GPU: the library loads, exports every function include/*.h declares,
its host-only helpers follow the pages' layout rules, and its argument checks return the same
statuses as the oracle's rules. Nothing here launches a kernel or touches device memory."""
import ctypes
import glob
import json
import os
import re

import pytest

import oracle
import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import build as sp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sp_build.build()
    return sp.load_library()


def declared_functions() -> list[str]:
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(sp_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("sp_fused_reduce_norm", "sp_check_args", "sp_pad_tokens", "sp_shard_rows",
                     "sp_status_string", "sp_device_error"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert [sp.sp_status_string(s) for s in range(5)] == [
        "SP_OK", "SP_ERR_INVALID_ARG", "SP_ERR_UNSUPPORTED", "SP_ERR_ALIGNMENT", "SP_ERR_CUDA"]
    assert sp.sp_status_string(99) == "SP_UNKNOWN_STATUS"


def test_padding_and_shards_match_the_pr_example(lib):
    with open(os.path.join(ROOT, "tests", "golden", "shard_layout_tp16_t3500.json")) as f:
        gold = json.load(f)
    tp = gold["tp"]
    assert sp.sp_pad_tokens(gold["num_tokens"], tp) == gold["num_tokens_pad"]
    for r in range(tp):
        assert sp.sp_shard_rows(gold["num_tokens_pad"], tp, r) == (gold["shard_starts"][r],
                                                                    gold["local_tokens"])
    assert sp.sp_pad_tokens(4093, 4) == 4096 and sp.sp_pad_tokens(0, 4) == 0
    assert sp.sp_pad_tokens(8192, 8) == 8192 and sp.sp_pad_tokens(7, 1) == 7
    assert sp.sp_pad_tokens(-1, 4) == -1 and sp.sp_pad_tokens(5, 0) == -1
    with pytest.raises(sp.SpError):
        sp.sp_shard_rows(3500, 16, 0)
    with pytest.raises(sp.SpError):
        sp.sp_shard_rows(3504, 16, 16)


def test_swizzled_scale_sizes(lib):
    # rows padded to 128, block columns to 4
    assert sp.sp_out_scales_bytes_ex(16384, 5120, "nvfp4", 1) == 16384 * 320
    assert sp.sp_out_scales_bytes_ex(3500, 5120, "nvfp4", 1) == 3584 * 320
    assert sp.sp_out_scales_bytes_ex(1, 16, "nvfp4", 1) == 128 * 4
    assert sp.sp_out_scales_bytes_ex(200, 1008, "nvfp4", 1) == 256 * 64
    assert sp.sp_out_scales_bytes_ex(16, 64, "nvfp4", 0) == 16 * 4
    assert sp.sp_out_scales_bytes_ex(16, 64, "fp8_per_token", 1) == -1
    assert sp.sp_out_scales_bytes_ex(16, 64, "nvfp4", 3) == -1


def test_output_sizes(lib):
    assert sp.sp_out_bytes(4096, 4096, "none") == 4096 * 4096 * 2
    assert sp.sp_out_bytes(8192, 7168, "fp8_static") == 8192 * 7168
    assert sp.sp_out_bytes(16384, 5120, "nvfp4") == 16384 * 2560
    assert sp.sp_out_scales_bytes(3504, 8192, "fp8_per_token") == 3504 * 4
    assert sp.sp_out_scales_bytes(16384, 5120, "nvfp4") == 16384 * 320
    assert sp.sp_out_scales_bytes(10, 64, "none") == 0
    assert sp.sp_out_bytes(10, 64, 9) == -1
    assert sp.sp_max_hidden() >= 8192


def test_launch_selection(lib):
    for tp, T, H in ((2, 64, 1024), (4, 4096, 4096), (8, 8192, 7168), (16, 3504, 8192),
                     (8, 16384, 5120), (1, 8, 16384), (3, 9, 8)):
        cfg = sp.sp_select_launch(tp, T, H, "none")
        assert cfg.kernel in (0, 1) and cfg.vec_per_thread in (1, 2, 4)
        assert cfg.ctas_per_sm >= 1
    with pytest.raises(sp.SpError):
        sp.sp_select_launch(2, 8, sp.sp_max_hidden() + 8, "none")


@pytest.mark.parametrize("tp,T,H,want", [
    # H <= 4096: direct while T * H <= 2^20 (2^22 for H <= 1024), one vector per thread ...
    (2, 64, 1024, (1, 1, 16, 0)),
    (8, 64, 4096, (1, 1, 16, 0)),
    (16, 64, 4096, (1, 1, 16, 0)),
    (16, 256, 2048, (1, 1, 16, 0)),
    (8, 512, 2048, (1, 1, 16, 0)),
    (4, 4096, 1024, (1, 1, 16, 0)),
    (4, 8192, 1024, (0, 2, 16, 4)),
    (8, 16, 3072, (1, 1, 16, 0)),       # no split up to H = 3072
    # 3072 < H <= 4096: split 4 up to 16 rows (24 rows, 32 at tp <= 5), split 8 up to 48 rows at
    # tp <= 5 (the longer bands not for NVFP4)
    (8, 8, 4096, (1, 1, 8, 0, 4)),
    (8, 24, 4096, (1, 1, 8, 0, 4)),
    (8, 32, 4096, (1, 1, 16, 0)),
    (4, 32, 4096, (1, 1, 8, 0, 4)),
    (4, 48, 4096, (1, 1, 8, 0, 8)),
    # ... two at tp <= 4 for 2^18 <= T * H <= 800 K, and up to 1.4 M (tp <= 4) / 1.2 M (tp <= 8)
    (4, 64, 4096, (1, 2, 16, 0)),
    (4, 128, 4096, (1, 2, 16, 0)),
    (5, 160, 4096, (1, 1, 16, 0)),
    (4, 320, 4096, (1, 1, 16, 0)),
    (8, 384, 3072, (1, 1, 16, 0)),
    # then one round of rows (H >= 3072): ceil(T / 152) CTAs per SM, deepest ring
    (16, 320, 3072, (0, 2, 3, 0)),
    (4, 768, 4096, (0, 2, 3, 0)),       # 1.3 rounds at 4 CTAs/SM: 3 fill it better
    (4, 1024, 4096, (0, 2, 4, 3)),      # fewer CTAs would leave each more than 3 rows
    # 4096 < H <= 8192: split rows, a cluster of 8, 4 or 2 CTAs per row, one vector per thread
    (8, 8, 8192, (1, 1, 8, 0, 8)),
    (6, 12, 8192, (1, 1, 8, 0, 8)),
    (8, 32, 5120, (1, 1, 8, 0, 4)),
    (8, 40, 5120, (1, 1, 8, 0, 2)),     # 33-64 rows at H = 5120, 6 <= tp < 12: 2 per row
    (6, 48, 5120, (1, 1, 8, 0, 2)),
    (16, 16, 7168, (1, 1, 8, 0, 8)),
    (16, 64, 8192, (1, 1, 8, 0, 4)),
    (2, 8, 7168, (1, 1, 8, 0, 8)),
    (4, 8, 5120, (1, 1, 8, 0, 8)),      # tp <= 5: 8 per row up to 16 rows (NVFP4 below 6144: 4)
    (4, 32, 5120, (0, 1, 8, 0, 4)),     # tp <= 5: staged split rows for 17-32 rows below
    (4, 24, 8192, (0, 1, 8, 0, 8)),     # H = 6144 (4 per row), 17-24 rows above (8 per row)
    (4, 16, 8192, (1, 1, 8, 0, 8)),
    (1, 8, 8192, (1, 2, 8, 0)),         # a single partial: no split
    # then direct, two vectors per thread, up to 128 rows (tp >= 12: 96, or 128 below 7168)
    (4, 32, 8192, (1, 2, 8, 0)),
    (4, 40, 8192, (1, 2, 8, 0)),
    (4, 64, 8192, (1, 2, 8, 0)),
    (8, 72, 5120, (1, 1, 8, 0, 4)),     # 65-96 rows at H <= 5120, tp >= 6: 4 per row
    (12, 96, 5120, (1, 1, 8, 0, 4)),
    (16, 48, 5120, (1, 1, 8, 0, 2)),    # tp >= 12, 33-64 rows at H <= 5120: 2 per row
    (8, 72, 8192, (1, 2, 8, 0)),
    (4, 128, 7168, (1, 2, 8, 0)),
    (2, 160, 8192, (1, 2, 8, 0)),       # tp <= 3 at H >= 7168: up to 160 rows
    (16, 80, 8192, (1, 1, 8, 0, 4)),    # tp >= 12, 65-96 rows at H >= 7168: 4 per row
    (16, 112, 5120, (0, 1, 8, 0, 4)),   # 97-128 rows, tp >= 6, H <= 5120: staged split rows
    (8, 128, 8192, (1, 2, 8, 0)),
    (16, 320, 2048, (1, 1, 16, 0)),
    (16, 160, 4096, (0, 1, 8, 0, 4)),   # tp >= 12, 145-192 rows at H = 4096: staged split rows
    (8, 160, 8192, (0, 1, 8, 0, 4)),    # H >= 7168, 6 <= tp < 12, 145-160 rows
    (4, 192, 8192, (0, 1, 8, 0, 4)),    # H >= 7168, tp <= 5, 161-192 rows
    (16, 112, 8192, (0, 2, 1, 0)),      # tp >= 12, 97-128 rows at H = 8192: deep ring, 1/SM
    (16, 112, 7168, (1, 2, 8, 0)),
    (8, 192, 5120, (1, 1, 8, 0, 2)),    # split 2 up to 224 rows at H = 5120
    (6, 160, 6144, (1, 1, 8, 0, 4)),    # split 4 up to 160 rows at H = 6144
    (8, 256, 5120, (0, 2, 2, 0)),       # one round of rows at H <= 6144, deepest ring
    (8, 384, 5120, (0, 2, 3, 0)),
    (6, 384, 6144, (0, 2, 3, 0)),
    (8, 512, 5120, (0, 2, 2, 0)),       # 1.1 rounds at 3 CTAs/SM: 2 CTAs/SM fill the last one
    (16, 144, 8192, (1, 1, 8, 0, 4)),   # tp >= 12, 129-144 rows: 4 per row
    (16, 160, 6144, (1, 1, 8, 0, 4)),   # ... and up to 160 rows at H <= 6144
    (16, 160, 8192, (0, 2, 2, 4)),
    (8, 144, 8192, (1, 1, 8, 0, 4)),    # H >= 7168, tp >= 4, 129-144 rows: 4 per row
    (4, 152, 8192, (1, 1, 8, 0, 2)),    # ... 2 per row for 145-152 at tp <= 5
    (4, 160, 7168, (1, 1, 8, 0, 4)),    # ... and 4 again up to 160 rows at tp <= 5
    (8, 152, 6144, (1, 1, 8, 0, 2)),    # H 5121-6144: 2 per row up to 152 rows
    (8, 160, 12288, (1, 1, 8, 0, 8)),   # H 8193-12288, 153-160 rows: 8 per row
    (16, 256, 7168, (0, 2, 2, 4)),
    (8, 384, 7168, (0, 2, 1, 0)),       # 1.3 rounds at 2 CTAs/SM; long rows: one CTA per SM
    (4, 384, 7168, (0, 2, 2, 4)),       # ... but not at tp = 4
    # H > 8192: split rows, else (tp <= 5) direct with four vectors per thread, for few rows
    (2, 16, 16384, (1, 1, 8, 0, 8)),
    (2, 32, 16384, (1, 1, 8, 0, 8)),    # H > 12288, tp <= 5: 8 per row up to 64 rows
    (8, 24, 16384, (1, 1, 8, 0, 8)),
    (4, 32, 12288, (1, 1, 8, 0, 4)),
    (4, 64, 12288, (1, 1, 8, 0, 4)),
    (8, 32, 12288, (1, 1, 8, 0, 4)),
    (8, 64, 16384, (1, 1, 8, 0, 4)),
    (16, 64, 16384, (1, 1, 8, 0, 4)),
    (8, 80, 12288, (1, 1, 8, 0, 8)),
    (4, 96, 16384, (1, 4, 8, 0)),
    (4, 128, 12288, (1, 4, 8, 0)),
    (4, 128, 16384, (0, 4, 1, 4)),
    (8, 72, 16384, (0, 4, 1, 4)),
    (16, 128, 16384, (0, 4, 1, 4)),
    # large calls: staged, CTAs/SM = 16384 / H
    (4, 4096, 4096, (0, 2, 4, 3)),
    (8, 8192, 7168, (0, 2, 2, 4)),
    (8, 16384, 5120, (0, 2, 3, 4)),
])
def test_launch_rule(lib, tp, T, H, want):
    c = sp.sp_select_launch(tp, T, H, "none")
    want = tuple(want) + (0,) * (5 - len(want))
    assert (c.kernel, c.vec_per_thread, c.ctas_per_sm, c.stages, c.split) == want


@pytest.mark.parametrize("mode,tp,T,H,split", [
    # NVFP4 output: split 4 (not 8) for few rows below H = 6144, and the longer split bands only
    # from H = 4609 (at H = 4608 a split lost there); per-token FP8 follows bf16
    ("nvfp4", 4, 8, 5120, 4),
    ("fp8_per_token", 4, 8, 5120, 8),
    ("nvfp4", 8, 8, 4096, 4),
    ("nvfp4", 4, 32, 4096, 0),
    ("fp8_per_token", 4, 32, 4096, 4),
    ("nvfp4", 8, 96, 4608, 0),
    ("fp8_per_token", 8, 96, 4608, 4),
    ("nvfp4", 12, 96, 5120, 4),
    ("nvfp4", 16, 112, 5120, 4),
    ("fp8_per_token", 16, 112, 5120, 4),
    ("nvfp4", 8, 224, 4096, 2),         # NVFP4 in the direct band past 128 rows, H >= 3072
    ("fp8_per_token", 8, 224, 4096, 0),
    ("nvfp4", 4, 192, 3072, 2),
    ("nvfp4", 16, 192, 4096, 4),
    ("nvfp4", 16, 48, 5120, 4),
    ("fp8_per_token", 16, 48, 5120, 2),
])
def test_launch_rule_by_mode(lib, mode, tp, T, H, split):
    c = sp.sp_select_launch(tp, T, H, mode)
    assert c.split == split
    if split:
        assert (c.vec_per_thread, c.ctas_per_sm) == (1, 8)


A = 1 << 20  # fake 16-byte-aligned addresses: compared, never dereferenced


def _base():
    return dict(partials=A, tp=4, T_pad=16, T_valid=13, H=64, residual=A * 8, weight=A * 9,
                bias=A * 10, eps=1e-6, quant_mode="fp8_per_token", scale=None, out=A * 11,
                out_scales=A * 12, residual_out=A * 13)


CASES = [
    ({}, "SP_OK"),
    ({"quant_mode": "fp8_dynamic_per_tensor"}, "SP_ERR_UNSUPPORTED"),
    ({"quant_mode": 7}, "SP_ERR_INVALID_ARG"),
    ({"quant_mode": -1}, "SP_ERR_INVALID_ARG"),
    ({"tp": 0}, "SP_ERR_INVALID_ARG"),
    ({"T_pad": 18}, "SP_ERR_INVALID_ARG"),
    ({"T_pad": -4}, "SP_ERR_INVALID_ARG"),
    ({"T_valid": 17}, "SP_ERR_INVALID_ARG"),
    ({"T_valid": -1}, "SP_ERR_INVALID_ARG"),
    ({"H": 60}, "SP_ERR_INVALID_ARG"),
    ({"H": 0}, "SP_ERR_INVALID_ARG"),
    ({"H": 72, "quant_mode": "nvfp4", "scale": A * 14}, "SP_ERR_INVALID_ARG"),
    ({"eps": 0.0}, "SP_ERR_INVALID_ARG"),
    ({"eps": -1e-6}, "SP_ERR_INVALID_ARG"),
    ({"eps": float("nan")}, "SP_ERR_INVALID_ARG"),
    ({"partials": None}, "SP_ERR_INVALID_ARG"),
    ({"weight": None}, "SP_ERR_INVALID_ARG"),
    ({"out": None}, "SP_ERR_INVALID_ARG"),
    ({"residual_out": None}, "SP_ERR_INVALID_ARG"),
    ({"out_scales": None}, "SP_ERR_INVALID_ARG"),
    ({"quant_mode": "fp8_static", "out_scales": None}, "SP_ERR_INVALID_ARG"),  # no scale
    ({"quant_mode": "nvfp4", "scale": None}, "SP_ERR_INVALID_ARG"),
    ({"residual": None}, "SP_OK"),
    ({"bias": None}, "SP_OK"),
    ({"residual_out": A * 8}, "SP_OK"),
    ({"residual_out": A * 8 + 16}, "SP_ERR_INVALID_ARG"),
    ({"out": A + 64}, "SP_ERR_INVALID_ARG"),
    ({"out": A * 13 + 32}, "SP_ERR_INVALID_ARG"),
    ({"out_scales": A * 11 + 16}, "SP_ERR_INVALID_ARG"),
    ({"T_pad": 0, "T_valid": 0, "partials": None, "out": None}, "SP_OK"),
    ({"partials": A + 8}, "SP_ERR_ALIGNMENT"),
    ({"out": A * 11 + 4}, "SP_ERR_ALIGNMENT"),
    ({"residual": A * 8 + 2, "residual_out": A * 13}, "SP_ERR_ALIGNMENT"),
    ({"H": 1 << 16}, "SP_ERR_UNSUPPORTED"),
    # the partials would exceed 2^62 bytes (4 x T_pad x H x 2): a shape error, checked before
    # any size is computed from the shapes (so nothing overflows int64), and before max H
    ({"T_pad": (1 << 53) + 4, "T_valid": 0}, "SP_ERR_INVALID_ARG"),
    ({"T_pad": 1 << 61, "T_valid": 0}, "SP_ERR_INVALID_ARG"),
    ({"T_pad": 1 << 50, "T_valid": 0, "H": 1 << 16}, "SP_ERR_INVALID_ARG"),
]


@pytest.mark.parametrize("kw,want", CASES)
def test_argument_checks(lib, kw, want):
    a = {**_base(), **kw}
    st = sp.sp_check_args(**a)
    assert sp.sp_status_string(st) == want
    # the oracle applies the same shape, mode and pointer rules (alignment and the largest H
    # are device-path limits, and the oracle reads the scale value, so those cases are skipped)
    if want not in ("SP_ERR_ALIGNMENT",) and not (kw.get("H", 0) > 16384) and "scale" not in kw:
        ost = oracle.check_args(a["partials"], a["tp"], a["T_pad"], a["T_valid"], a["H"],
                                a["residual"], a["weight"], a["bias"], a["eps"],
                                sp._mode(a["quant_mode"]), None, a["out"], a["out_scales"],
                                a["residual_out"])
        assert ost == st


def test_main_entry_rejects_before_any_cuda_call(lib):
    # invalid arguments: the status comes back from the checks, no CUDA call is made
    a = _base()
    f = lib.sp_fused_reduce_norm
    st = f(a["partials"], 4, 18, 13, 64, a["residual"], a["weight"], a["bias"], ctypes.c_float(1e-6),
           2, None, a["out"], a["out_scales"], a["residual_out"], None)
    assert sp.sp_status_string(st) == "SP_ERR_INVALID_ARG"
    st = f(a["partials"], 4, 16, 13, 64, a["residual"], a["weight"], a["bias"], ctypes.c_float(1e-6),
           4, None, a["out"], a["out_scales"], a["residual_out"], None)
    assert sp.sp_status_string(st) == "SP_ERR_UNSUPPORTED"


def test_product_path_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "sequence_reduce_add_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(path).read()
            assert "import oracle" not in src and "from oracle" not in src, path
            assert "sp_oracle" not in src and "libsporacle" not in src, path


OPTION_CASES = [
    (dict(), {}, "SP_OK"),
    (dict(partial_scale=0.5), {}, "SP_OK"),
    (dict(partial_scale=float("inf")), {}, "SP_ERR_INVALID_ARG"),
    (dict(partial_scale=float("nan")), {}, "SP_ERR_INVALID_ARG"),
    (dict(addend=A * 20), {}, "SP_OK"),
    (dict(addend=A * 20 + 8), {}, "SP_ERR_ALIGNMENT"),
    (dict(addend=A * 11 + 64), {}, "SP_ERR_INVALID_ARG"),          # inside `out`
    (dict(addend=A * 13), {}, "SP_ERR_INVALID_ARG"),                # is residual_out
    (dict(scale_layout=1), {}, "SP_ERR_INVALID_ARG"),               # swizzle is NVFP4-only
    (dict(scale_layout=2), {}, "SP_ERR_UNSUPPORTED"),
    (dict(scale_layout=1), {"quant_mode": "nvfp4", "scale": A * 14}, "SP_OK"),
    # 16 x 64 NVFP4 scales: 64 bytes row-major, 128 x 4 = 512 bytes swizzled
    (dict(scale_layout=0), {"quant_mode": "nvfp4", "scale": A * 14,
                            "out_scales": A * 13 - 256}, "SP_OK"),
    (dict(scale_layout=1), {"quant_mode": "nvfp4", "scale": A * 14,
                            "out_scales": A * 13 - 256}, "SP_ERR_INVALID_ARG"),
    (dict(host_buffers=2), {}, "SP_ERR_UNSUPPORTED"),
    (dict(schedule=1), {}, "SP_OK"),
    (dict(schedule=2), {}, "SP_OK"),
    (dict(schedule=3), {}, "SP_ERR_UNSUPPORTED"),
    (dict(schedule=-1), {}, "SP_ERR_UNSUPPORTED"),
    (dict(addend=A * 20), {"T_pad": 18}, "SP_ERR_INVALID_ARG"),     # shape rule first
    # an explicit launch configuration: the checks of sp_fused_reduce_norm_with_config
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4)), {}, "SP_OK"),
    (dict(launch=dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=3)), {}, "SP_OK"),
    (dict(launch=dict(kernel=2, vec_per_thread=1, ctas_per_sm=4)), {}, "SP_ERR_INVALID_ARG"),
    (dict(launch=dict(kernel=1, vec_per_thread=3, ctas_per_sm=4)), {}, "SP_ERR_INVALID_ARG"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=0)), {}, "SP_ERR_INVALID_ARG"),
    (dict(launch=dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=1)), {},
     "SP_ERR_UNSUPPORTED"),
    # split rows: 0/1 (whole rows), 2, 4, 8 with the direct kernel and 1-2 vectors per thread
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=1)), {}, "SP_OK"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=2)), {}, "SP_OK"),
    (dict(launch=dict(kernel=1, vec_per_thread=2, ctas_per_sm=4, split=4)), {}, "SP_OK"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=8)), {}, "SP_OK"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=3)), {},
     "SP_ERR_INVALID_ARG"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=16)), {},
     "SP_ERR_INVALID_ARG"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=-2)), {},
     "SP_ERR_INVALID_ARG"),
    (dict(launch=dict(kernel=1, vec_per_thread=4, ctas_per_sm=4, split=2)), {},
     "SP_ERR_UNSUPPORTED"),
    (dict(launch=dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=3, split=2)), {},
     "SP_ERR_UNSUPPORTED"),
    (dict(launch=dict(kernel=1, vec_per_thread=1, ctas_per_sm=4, split=8), scale_layout=1),
     {"quant_mode": "nvfp4", "scale": A * 14}, "SP_OK"),
    (dict(launch=dict(kernel=1, vec_per_thread=2, ctas_per_sm=4), host_buffers=1), {}, "SP_OK"),
    (dict(launch=dict(kernel=0, vec_per_thread=2, ctas_per_sm=2, stages=3), host_buffers=1), {},
     "SP_ERR_UNSUPPORTED"),
    # the caller's row counter (8 bytes) and status word (4 bytes): aligned, overlapping nothing
    (dict(row_counter=A * 21, status=A * 22), {}, "SP_OK"),
    (dict(row_counter=A * 21 + 8), {}, "SP_ERR_ALIGNMENT"),
    (dict(status=A * 22 + 4), {}, "SP_ERR_ALIGNMENT"),
    (dict(row_counter=A * 11), {}, "SP_ERR_INVALID_ARG"),           # inside `out`
    (dict(status=A * 8 + 16), {}, "SP_ERR_INVALID_ARG"),            # inside the residual
    (dict(row_counter=A * 21, status=A * 21), {}, "SP_ERR_INVALID_ARG"),  # the same bytes
    (dict(status=A * 9), {}, "SP_ERR_INVALID_ARG"),                 # is the weight
]


@pytest.mark.parametrize("opt,kw,want", OPTION_CASES)
def test_option_checks(lib, opt, kw, want):
    o = sp.Options()
    lib.sp_options_init(ctypes.byref(o))
    assert o.partial_scale == 1.0 and o.addend is None and o.scale_layout == 0
    assert o.host_buffers == 0 and o.schedule == 0  # SP_SCHEDULE_AUTO
    assert not o.launch  # NULL: the library's own choice
    assert o.row_counter is None and o.status is None
    cfg = None
    for k, v in opt.items():
        if k == "launch":
            cfg = sp.LaunchConfig(**v)
            o.launch = ctypes.pointer(cfg)
        else:
            setattr(o, k, v)
    a = {**_base(), **kw}
    st = sp.sp_check_args_ex(o, a["partials"], a["tp"], a["T_pad"], a["T_valid"], a["H"],
                             a["residual"], a["weight"], a["bias"], a["eps"], a["quant_mode"],
                             a["scale"], a["out"], a["out_scales"], a["residual_out"])
    assert sp.sp_status_string(st) == want


def test_fc2_batch_ids_match_the_page(lib):
    with open(os.path.join(ROOT, "tests", "golden", "fc2_reorganize_tp4_otp2.json")) as f:
        gold = json.load(f)
    assert sp.sp_fc2_batch_ids(gold["global_tp"], gold["otp_size"]) == gold["batch_ids"]
    assert sp.sp_fc2_batch_ids(8, 2) == [[0, 4], [1, 5], [2, 6], [3, 7]]
    assert sp.sp_fc2_batch_ids(8, 8) == [[0, 1, 2, 3, 4, 5, 6, 7]]
    with pytest.raises(sp.SpError):
        sp.sp_fc2_batch_ids(6, 4)


FC2_CASES = [
    (dict(), "SP_OK"),
    (dict(global_tp=0), "SP_ERR_INVALID_ARG"),
    (dict(otp_size=3), "SP_ERR_INVALID_ARG"),          # 8 % 3
    (dict(N=100), "SP_ERR_INVALID_ARG"),               # 100 % 8
    (dict(H=1020), "SP_ERR_INVALID_ARG"),              # 1020 % 8
    (dict(elem_bytes=3), "SP_ERR_INVALID_ARG"),
    (dict(x=None), "SP_ERR_INVALID_ARG"),
    (dict(y=A + 4096), "SP_ERR_INVALID_ARG"),          # overlaps x
    (dict(y=A * 64 + 8), "SP_ERR_ALIGNMENT"),
    (dict(H=8 * 4), "SP_ERR_ALIGNMENT"),               # 4 bf16 per slice = 8 bytes
    (dict(N=0, x=None, y=None), "SP_OK"),
    (dict(N=1 << 56), "SP_ERR_INVALID_ARG"),           # x would exceed 2^62 bytes
]


@pytest.mark.parametrize("kw,want", FC2_CASES)
def test_fc2_argument_checks(lib, kw, want):
    a = dict(x=A, global_tp=8, otp_size=2, N=128, H=1024, elem_bytes=2, y=A * 64)
    a.update(kw)
    st = sp.sp_fc2_check_args(a["x"], a["global_tp"], a["otp_size"], a["N"], a["H"],
                              a["elem_bytes"], a["y"])
    assert sp.sp_status_string(st) == want


def test_every_selected_launch_passes_the_launch_checks(lib):
    """Over a grid of tp, H, T and modes, the configuration sp_select_launch picks passes the
    checks a forced configuration gets (kernel, vector count, threads, ring depth, split), so the
    default path never picks a launch the library would refuse."""
    G = 1 << 40  # fake, far-apart 16-byte-aligned addresses: compared, never dereferenced
    checked = 0
    for mode in ("none", "fp8_static", "fp8_per_token", "nvfp4"):
        for tp in (1, 2, 3, 4, 5, 6, 8, 12, 16, 24, 32):
            for H in (8, 16, 24, 512, 1000, 1024, 2048, 2056, 3072, 4096, 4608, 5120, 6144,
                      7168, 8192, 12288, 16376, 16384):
                if mode == "nvfp4" and H % 16:
                    continue
                for T in (1, 2, 7, 8, 16, 24, 32, 33, 48, 64, 80, 96, 100, 120, 128, 144, 152,
                          160, 192, 224, 256, 304, 500, 1024, 4096, 9999):
                    T_pad = sp.sp_pad_tokens(T, tp)
                    cfg = sp.sp_select_launch(tp, T_pad, H, mode)
                    o = sp.Options()
                    lib.sp_options_init(ctypes.byref(o))
                    o.launch = ctypes.pointer(cfg)
                    st = sp.sp_check_args_ex(o, G, tp, T_pad, T, H, 2 * G, 3 * G, 4 * G, 1e-6, mode,
                                             5 * G if mode in ("fp8_static", "nvfp4") else None,
                                             6 * G, 7 * G if mode in ("fp8_per_token", "nvfp4") else None,
                                             8 * G)
                    assert sp.sp_status_string(st) == "SP_OK", (mode, tp, H, T, cfg.as_dict())
                    checked += 1
    assert checked > 9000


def test_each_declared_call_cites_its_passage():
    """Every exported call's comment (the comment block nearest before its declaration) names
    the passage of the pages it restates (a section mark), or says it has no counterpart there."""
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        # comment blocks that open a line (argument notes inside a declaration are not blocks)
        pieces = re.split(r"(^[ \t]*/\*.*?\*/)", src, flags=re.S | re.M)
        last_comment = ""
        for piece in pieces:
            if piece.lstrip().startswith("/*"):
                last_comment = piece
                continue
            for name in re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(sp_\w+)\s*\(", piece,
                                   flags=re.M):
                assert "§" in last_comment or "no counterpart on the pages" in last_comment, name
