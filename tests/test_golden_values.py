"""Stored values under tests/golden/ are reproduced by their committed writers."""
import importlib.util
import json
import os

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_nvfp4_global_scale_is_reproduced():
    spec = importlib.util.spec_from_file_location(
        "calibrate", os.path.join(GOLDEN, "calibrate_nvfp4_global_scale.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    gs, amax = mod.calibrate()
    with open(os.path.join(GOLDEN, "nvfp4_global_scale.json")) as f:
        stored = json.load(f)
    assert stored["global_scale"] == gs
    assert abs(stored["amax_y"] - amax) <= 1e-9 * amax
