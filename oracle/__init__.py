"""fp64 CPU oracle for the fused reduce + bias/residual add + RMSNorm + quant stage.

TEST INFRASTRUCTURE ONLY. The product path (the CUDA library and its Python binding) never
imports, loads or calls anything in this package. Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.

The arithmetic lives in ``sp_oracle.cpp`` (plain fp64 C++, one row at a time). This module only
marshals numpy arrays into it. bf16 tensors travel as their 16-bit patterns (``np.uint16``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

MODES = {"none": 0, "fp8_static": 1, "fp8_per_token": 2, "nvfp4": 3, "fp8_dynamic_per_tensor": 4}
STATUS = {0: "ok", 1: "invalid_arg", 2: "unsupported", 3: "alignment", 4: "cuda"}

_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64

_ARGS = [_u16p, ctypes.c_int, _i64, _i64, _i64, _u16p, _u16p, _u16p, ctypes.c_float, ctypes.c_int,
         _f32p, _vp, _vp, _u16p]

_loaded: dict[str, ctypes.CDLL] = {}


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library at ``path`` (default: the in-tree one)."""
    if path is None:
        # SP_ORACLE_LIBRARY lets the mutation test point the pin suites at a planted-bug build
        path = os.environ.get("SP_ORACLE_LIBRARY") or _build.build()
    if path in _loaded:
        return _loaded[path]
    lib = ctypes.CDLL(path)
    lib.sp_oracle_fused_reduce_norm.argtypes = _ARGS
    lib.sp_oracle_fused_reduce_norm.restype = ctypes.c_int
    lib.sp_oracle_check_args.argtypes = _ARGS
    lib.sp_oracle_check_args.restype = ctypes.c_int
    lib.sp_oracle_fused_reduce_norm_rows.argtypes = _ARGS + [_f64p, _i64, _i64]
    lib.sp_oracle_fused_reduce_norm_rows.restype = ctypes.c_int
    lib.sp_oracle_fused_reduce_norm_rows_ex.argtypes = _ARGS + [_f64p, _i64, _i64, ctypes.c_float,
                                                                 _u16p, ctypes.c_int]
    lib.sp_oracle_out_scales_bytes.argtypes = [_i64, _i64, ctypes.c_int, ctypes.c_int]
    lib.sp_oracle_out_scales_bytes.restype = _i64
    lib.sp_oracle_fused_reduce_norm_rows_ex.restype = ctypes.c_int
    for name, cin, cout in (("bf16_encode", _f64p, _u16p), ("bf16_decode", _u16p, _f64p),
                            ("e4m3_encode", _f64p, _u8p), ("e4m3_decode", _u8p, _f64p),
                            ("e2m1_encode", _f64p, _u8p), ("e2m1_decode", _u8p, _f64p)):
        fn = getattr(lib, "sp_oracle_" + name)
        fn.argtypes = [cin, cout, _i64]
        fn.restype = None
    lib.sp_oracle_fc2_batch_ids.argtypes = [ctypes.c_int, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_int)]
    lib.sp_oracle_fc2_batch_ids.restype = None
    lib.sp_oracle_fc2_reorganize.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _i64, _i64,
                                             ctypes.c_int, _u8p]
    lib.sp_oracle_fc2_reorganize.restype = ctypes.c_int
    _loaded[path] = lib
    return lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def out_layout(T_pad: int, H: int, mode: str, scale_layout: int = 0):
    """(out shape, out dtype, scales shape or None, scales dtype or None) for a mode (the
    swizzled NVFP4 scale layout is a flat byte buffer)."""
    if mode == "nvfp4" and scale_layout == 1:
        n = -(-T_pad // 128) * 128 * (-(-(H // 16) // 4) * 4)
        return (T_pad, H // 2), np.uint8, (n,), np.uint8
    if mode == "none":
        return (T_pad, H), np.uint16, None, None
    if mode == "fp8_static":
        return (T_pad, H), np.uint8, None, None
    if mode == "fp8_per_token":
        return (T_pad, H), np.uint8, (T_pad,), np.float32
    if mode == "nvfp4":
        return (T_pad, H // 2), np.uint8, (T_pad, H // 16), np.uint8
    raise ValueError(mode)


def fused_reduce_norm(partials: np.ndarray, residual: np.ndarray | None, weight: np.ndarray,
                      bias: np.ndarray | None, eps: float, mode: str, scale: float | None,
                      T_valid: int, *, want_y: bool = False, rows: tuple[int, int] | None = None,
                      threads: int = 1, lib: ctypes.CDLL | None = None,
                      buffers: dict | None = None, partial_scale: float = 1.0,
                      addend: np.ndarray | None = None, scale_layout: int = 0) -> dict:
    """Run the oracle over rows ``rows`` (default all) of a [tp, T_pad, H] problem.

    Returns a dict with ``status``, ``out``, ``out_scales`` (or None), ``residual_out`` and, when
    ``want_y``, the unrounded fp64 ``y`` [T_pad, H]. Rows outside ``rows`` are left zero, unless
    ``buffers`` (a previous result) is given: its arrays are then reused and only ``rows`` of
    them are rewritten. ``partial_scale`` multiplies every partial before the reduction;
    ``addend`` (bf16 bits [T_pad, H]) is added after it, before the norm.
    """
    lib = lib or load()
    tp, T_pad, H = partials.shape
    oshape, odt, sshape, sdt = out_layout(T_pad, H, mode, scale_layout)
    if buffers is not None:
        out, out_scales = buffers["out"], buffers["out_scales"]
        residual_out, y = buffers["residual_out"], buffers["y"] if want_y else None
        assert out.shape == oshape and residual_out.shape == (T_pad, H)
        assert (out_scales is None) == (sshape is None) and (not want_y or y is not None)
    else:
        out = np.zeros(oshape, odt)
        out_scales = np.zeros(sshape, sdt) if sshape else None
        residual_out = np.zeros((T_pad, H), np.uint16)
        y = np.zeros((T_pad, H), np.float64) if want_y else None
    scale_arr = np.array([scale], np.float32) if scale is not None else None
    args = [_ptr(partials, ctypes.c_uint16), tp, T_pad, T_valid, H,
            _ptr(residual, ctypes.c_uint16), _ptr(weight, ctypes.c_uint16),
            _ptr(bias, ctypes.c_uint16), ctypes.c_float(eps), MODES[mode],
            _ptr(scale_arr, ctypes.c_float), out.ctypes.data_as(_vp),
            out_scales.ctypes.data_as(_vp) if out_scales is not None else None,
            _ptr(residual_out, ctypes.c_uint16)]
    begin, end = rows if rows is not None else (0, T_pad)
    status = [0]

    extended = partial_scale != 1.0 or addend is not None or scale_layout != 0

    def run(b, e, slot):
        if extended:
            st = lib.sp_oracle_fused_reduce_norm_rows_ex(
                *args, _ptr(y, ctypes.c_double), b, e, ctypes.c_float(partial_scale),
                _ptr(addend, ctypes.c_uint16), scale_layout)
        else:
            st = lib.sp_oracle_fused_reduce_norm_rows(*args, _ptr(y, ctypes.c_double), b, e)
        if st != 0:
            status[slot] = st

    if threads <= 1 or end - begin < 2:
        run(begin, end, 0)
    else:
        n = min(threads, end - begin)
        bounds = np.linspace(begin, end, n + 1).astype(np.int64)
        status = [0] * n
        pool = [threading.Thread(target=run, args=(int(bounds[i]), int(bounds[i + 1]), i))
                for i in range(n)]
        for th in pool:
            th.start()
        for th in pool:
            th.join()
    st = next((s for s in status if s != 0), 0)
    return {"status": st, "out": out, "out_scales": out_scales, "residual_out": residual_out,
            "y": y}


def check_args(partials_ptr, tp, T_pad, T_valid, H, residual_ptr, weight_ptr, bias_ptr, eps, mode,
               scale: float | None, out_ptr, out_scales_ptr, residual_out_ptr,
               lib: ctypes.CDLL | None = None) -> int:
    """Argument rules alone, on raw addresses (integers or None); nothing is dereferenced except
    the scale value, which is passed here as a number."""
    lib = lib or load()
    scale_arr = np.array([scale], np.float32) if scale is not None else None
    c = lambda p, t: ctypes.cast(p, ctypes.POINTER(t))  # noqa: E731
    return lib.sp_oracle_check_args(
        c(partials_ptr, ctypes.c_uint16), tp, T_pad, T_valid, H, c(residual_ptr, ctypes.c_uint16),
        c(weight_ptr, ctypes.c_uint16), c(bias_ptr, ctypes.c_uint16), ctypes.c_float(eps),
        mode if isinstance(mode, int) else MODES[mode], _ptr(scale_arr, ctypes.c_float),
        out_ptr, out_scales_ptr, c(residual_out_ptr, ctypes.c_uint16))


def _codec(name: str, x: np.ndarray, in_dt, out_dt, lib=None) -> np.ndarray:
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=in_dt)
    y = np.empty(x.shape, out_dt)
    ctype_in = {np.float64: ctypes.c_double, np.uint16: ctypes.c_uint16, np.uint8: ctypes.c_uint8}
    getattr(lib, "sp_oracle_" + name)(_ptr(x, ctype_in[in_dt]), _ptr(y, ctype_in[out_dt]), x.size)
    return y


def bf16_encode(x, lib=None):
    return _codec("bf16_encode", x, np.float64, np.uint16, lib)


def bf16_decode(c, lib=None):
    return _codec("bf16_decode", c, np.uint16, np.float64, lib)


def e4m3_encode(x, lib=None):
    return _codec("e4m3_encode", x, np.float64, np.uint8, lib)


def e4m3_decode(c, lib=None):
    return _codec("e4m3_decode", c, np.uint8, np.float64, lib)


def e2m1_encode(x, lib=None):
    return _codec("e2m1_encode", x, np.float64, np.uint8, lib)


def e2m1_decode(c, lib=None):
    return _codec("e2m1_decode", c, np.uint8, np.float64, lib)


def fc2_batch_ids(global_tp: int, otp_size: int, lib=None) -> list[list[int]]:
    """The reorganised batch ids: odp_size lists of otp_size token-segment indices."""
    lib = lib or load()
    D = global_tp // otp_size
    ids = (ctypes.c_int * (D * otp_size))()
    lib.sp_oracle_fc2_batch_ids(global_tp, otp_size, ids)
    return [list(ids[j * otp_size:(j + 1) * otp_size]) for j in range(D)]


def fc2_reorganize(x: np.ndarray, otp_size: int, lib=None) -> np.ndarray:
    """FlashComm2 token reorganisation of x [G][N][H/G] (any dtype) into [G][N/D][H/P]."""
    lib = lib or load()
    G, N, F = x.shape
    D = G // otp_size
    x = np.ascontiguousarray(x)
    y = np.zeros((G, N // D, F * D), x.dtype)
    st = lib.sp_oracle_fc2_reorganize(x.view(np.uint8).ctypes.data_as(_u8p), G, otp_size, N,
                                      F * G, x.dtype.itemsize, y.view(np.uint8).ctypes.data_as(_u8p))
    if st != 0:
        raise ValueError(f"oracle fc2_reorganize: status {st}")
    return y
