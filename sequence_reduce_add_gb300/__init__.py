"""GB300 (sm_103a) fused reduce + bias/residual add + RMSNorm + quant for sequence parallelism.

The per-token stage of the rewrite AllReduce -> RMSNorm -> quant  ==>  ReduceScatter -> RMSNorm
-> quant -> AllGather, run on one GPU: the tp partial-sum buffers are summed, bias and residual
added, RMSNorm applied with a weight, the new residual written, and bf16 / FP8-E4M3 (static or
per-token) / NVFP4 output produced, with padding rows zeroed (vllm-ascend SP/FlashComm notes
§2.3; vLLM SP/AsyncTP/quant notes §四; PR #18671 notes §5.2-5.3).

Every computation runs in the CUDA library ``libspfused.so`` (include/sp_fused.h). This module
only marshals arguments: it turns torch tensors into device pointers and sizes, calls the C
entry point of the same name, and raises ``SpError`` on a non-OK status. There is no fallback:
without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "SpError", "QUANT_MODES", "load_library", "sp_fused_reduce_norm", "sp_fused_reduce_norm_host",
    "sp_fused_reduce_norm_with_config", "sp_check_args", "sp_select_launch", "sp_pad_tokens",
    "sp_shard_rows", "sp_out_bytes", "sp_out_scales_bytes", "sp_max_hidden", "sp_status_string",
    "sp_device_error", "allocate_outputs", "LaunchConfig", "Options", "sp_options_init",
    "sp_fused_reduce_norm_ex", "sp_check_args_ex", "sp_out_scales_bytes_ex", "sp_fc2_reorganize",
    "sp_fc2_check_args", "sp_fc2_batch_ids", "sp_selftest_wait_timeout",
    "sp_selftest_fused_timeout", "sp_last_launch", "LaunchInfo", "sp_fused_reduce_norm_noalloc",
]

QUANT_MODES = {"none": 0, "fp8_static": 1, "fp8_per_token": 2, "nvfp4": 3,
               "fp8_dynamic_per_tensor": 4}
STATUS_NAMES = {0: "SP_OK", 1: "SP_ERR_INVALID_ARG", 2: "SP_ERR_UNSUPPORTED",
                3: "SP_ERR_ALIGNMENT", 4: "SP_ERR_CUDA"}
KERNELS = {"staged": 0, "direct": 1}

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


class SpError(RuntimeError):
    """A non-OK status from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class LaunchConfig(ctypes.Structure):
    """sp_launch_config: kernel (0 staged, 1 direct), vec_per_thread, ctas_per_sm, stages,
    split (CTAs of a cluster per row; 0 or 1 = one CTA per row)."""
    _fields_ = [("kernel", ctypes.c_int), ("vec_per_thread", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("stages", ctypes.c_int), ("split", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class Options(ctypes.Structure):
    """sp_fused_options: partial_scale, addend (device address or None), scale_layout,
    host_buffers, schedule, launch (a LaunchConfig or None), row_counter (the caller's own
    dynamic-schedule counter, 8 bytes, or None), status (a per-call error word or None)."""
    _fields_ = [("partial_scale", ctypes.c_float), ("addend", ctypes.c_void_p),
                ("scale_layout", ctypes.c_int), ("host_buffers", ctypes.c_int),
                ("schedule", ctypes.c_int), ("launch", ctypes.POINTER(LaunchConfig)),
                ("row_counter", ctypes.c_void_p), ("status", ctypes.c_void_p)]


class LaunchInfo(ctypes.Structure):
    """sp_launch_info: the configuration a call launched, its grid and its row schedule."""
    _fields_ = [("config", LaunchConfig), ("grid", ctypes.c_int), ("schedule", ctypes.c_int)]


SCHEDULES = {"auto": 0, "static": 1, "dynamic": 2}


_MAIN_ARGS = [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, _vp, ctypes.c_float, ctypes.c_int,
              _vp, _vp, _vp, _vp]

_lib: ctypes.CDLL | None = None


def library_path() -> str:
    return _build.LIBRARY


def load_library() -> ctypes.CDLL:
    """Load libspfused.so (built by ``__graft_entry__.build()`` / ``build.py``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    lib = ctypes.CDLL(path)
    lib.sp_fused_reduce_norm.argtypes = _MAIN_ARGS + [_vp]
    lib.sp_fused_reduce_norm.restype = ctypes.c_int
    lib.sp_fused_reduce_norm_with_config.argtypes = [ctypes.POINTER(LaunchConfig)] + _MAIN_ARGS + [_vp]
    lib.sp_fused_reduce_norm_with_config.restype = ctypes.c_int
    lib.sp_options_init.argtypes = [ctypes.POINTER(Options)]
    lib.sp_options_init.restype = None
    lib.sp_fused_reduce_norm_ex.argtypes = [ctypes.POINTER(Options)] + _MAIN_ARGS + [_vp]
    lib.sp_fused_reduce_norm_ex.restype = ctypes.c_int
    lib.sp_check_args_ex.argtypes = [ctypes.POINTER(Options)] + _MAIN_ARGS
    lib.sp_check_args_ex.restype = ctypes.c_int
    lib.sp_fused_reduce_norm_host.argtypes = _MAIN_ARGS + [_vp]
    lib.sp_fused_reduce_norm_host.restype = ctypes.c_int
    lib.sp_check_args.argtypes = _MAIN_ARGS
    lib.sp_check_args.restype = ctypes.c_int
    lib.sp_select_launch.argtypes = [ctypes.c_int, _i64, _i64, ctypes.c_int,
                                     ctypes.POINTER(LaunchConfig)]
    lib.sp_select_launch.restype = ctypes.c_int
    lib.sp_pad_tokens.argtypes = [_i64, ctypes.c_int]
    lib.sp_pad_tokens.restype = _i64
    lib.sp_shard_rows.argtypes = [_i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_i64),
                                  ctypes.POINTER(_i64)]
    lib.sp_shard_rows.restype = ctypes.c_int
    lib.sp_out_bytes.argtypes = [_i64, _i64, ctypes.c_int]
    lib.sp_out_bytes.restype = _i64
    lib.sp_out_scales_bytes.argtypes = [_i64, _i64, ctypes.c_int]
    lib.sp_out_scales_bytes.restype = _i64
    lib.sp_out_scales_bytes_ex.argtypes = [_i64, _i64, ctypes.c_int, ctypes.c_int]
    lib.sp_out_scales_bytes_ex.restype = _i64
    lib.sp_fc2_reorganize.argtypes = [_vp, ctypes.c_int, ctypes.c_int, _i64, _i64, ctypes.c_int,
                                      _vp, _vp]
    lib.sp_fc2_reorganize.restype = ctypes.c_int
    lib.sp_fc2_check_args.argtypes = [_vp, ctypes.c_int, ctypes.c_int, _i64, _i64, ctypes.c_int,
                                      _vp]
    lib.sp_fc2_check_args.restype = ctypes.c_int
    lib.sp_fc2_batch_ids.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.sp_fc2_batch_ids.restype = ctypes.c_int
    lib.sp_max_hidden.argtypes = []
    lib.sp_max_hidden.restype = _i64
    lib.sp_status_string.argtypes = [ctypes.c_int]
    lib.sp_status_string.restype = ctypes.c_char_p
    lib.sp_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.sp_device_error.restype = ctypes.c_int
    lib.sp_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp]
    lib.sp_selftest_wait_timeout.restype = ctypes.c_int
    lib.sp_selftest_fused_timeout.argtypes = ([ctypes.c_uint64, _i64, ctypes.POINTER(Options)]
                                              + _MAIN_ARGS + [_vp])
    lib.sp_selftest_fused_timeout.restype = ctypes.c_int
    lib.sp_last_launch.argtypes = [ctypes.POINTER(LaunchInfo)]
    lib.sp_last_launch.restype = ctypes.c_int
    lib.sp_fused_reduce_norm_noalloc.argtypes = _MAIN_ARGS + [_vp]
    lib.sp_fused_reduce_norm_noalloc.restype = ctypes.c_int
    _lib = lib
    return lib


def _mode(quant_mode) -> int:
    return QUANT_MODES[quant_mode] if isinstance(quant_mode, str) else int(quant_mode)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _current_device():
    """The device the library launches on (torch's current CUDA device)."""
    import torch
    return torch.device("cuda", torch.cuda.current_device())


# Element types each buffer may have (one byte per code for FP8 / packed FP4 / block scales).
def _dtypes():
    import torch
    byte = [torch.uint8, torch.int8]
    for name in ("float8_e4m3fn", "float4_e2m1fn_x2"):
        if hasattr(torch, name):
            byte.append(getattr(torch, name))
    return {"bf16": (torch.bfloat16,), "f32": (torch.float32,), "byte": tuple(byte)}


def _check_tensor(name: str, t, dtypes, min_bytes: int, device, host: bool) -> None:
    """Raise ValueError unless `t` is a contiguous tensor of one of `dtypes`, at least
    `min_bytes` long, on `device` (or, with host=True, page-locked host memory)."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if host and t.device.type == "cpu":
        if not t.is_pinned():
            raise ValueError(f"{name}: host tensors must be page-locked (tensor.pin_memory())")
    elif t.device != device:
        raise ValueError(f"{name}: expected a tensor on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not one of {[str(d) for d in dtypes]}")
    nbytes = t.numel() * t.element_size()
    if nbytes < min_bytes:
        raise ValueError(f"{name}: {nbytes} bytes, the call needs at least {min_bytes}")


def _main_args(partials, residual, weight, bias, eps, quant_mode, scale, out, out_scales,
               residual_out, T_valid, *, host: bool = False, addend=None, scale_layout: int = 0):
    """Check every tensor against what the call will read and write, then marshal the C
    arguments. The library can only check sizes derived from the shape arguments, so a buffer
    that is too small, non-contiguous, of the wrong type or on another device is refused here,
    before anything is launched."""
    import torch
    dev = _current_device()
    dt = _dtypes()
    if not isinstance(partials, torch.Tensor) or partials.dim() != 3:
        raise ValueError("partials: expected a bf16 tensor [tp, T_pad, H]")
    tp, T_pad, H = partials.shape
    mode = _mode(quant_mode)
    if T_valid is None:
        T_valid = T_pad
    _check_tensor("partials", partials, dt["bf16"], 0, dev, host)
    rows = T_pad * H * 2
    for name, t, need in (("residual", residual, rows), ("addend", addend, rows),
                          ("bias", bias, H * 2)):
        if t is not None:
            _check_tensor(name, t, dt["bf16"], need, dev, host)
    _check_tensor("weight", weight, dt["bf16"], H * 2, dev, host)
    _check_tensor("residual_out", residual_out, dt["bf16"], rows, dev, host)
    if scale is not None:
        _check_tensor("scale", scale, dt["f32"], 4, dev, host)
    if mode in (0, 1, 2, 3):
        out_bytes = {0: rows, 1: T_pad * H, 2: T_pad * H, 3: T_pad * (H // 2)}[mode]
        _check_tensor("out", out, dt["bf16"] if mode == 0 else dt["byte"], out_bytes, dev, host)
        if out_scales is not None and mode in (2, 3):
            if mode == 2:
                _check_tensor("out_scales", out_scales, dt["f32"], T_pad * 4, dev, host)
            else:
                need = (-(-T_pad // 128) * 128 * (-(-(H // 16) // 4) * 4) if scale_layout == 1
                        else T_pad * (H // 16))
                _check_tensor("out_scales", out_scales, dt["byte"], need, dev, host)
    return [_ptr(partials), tp, T_pad, T_valid, H, _ptr(residual), _ptr(weight), _ptr(bias),
            ctypes.c_float(eps), mode, _ptr(scale), _ptr(out), _ptr(out_scales),
            _ptr(residual_out)]


def sp_fused_reduce_norm(partials, weight, out, residual_out, *, residual=None, bias=None,
                         eps: float = 1e-6, quant_mode="none", scale=None, out_scales=None,
                         T_valid: int | None = None, stream=None) -> None:
    """Enqueue the fused stage (see include/sp_fused.h) on ``stream`` (default: torch's current).

    partials: bf16 CUDA tensor [tp, T_pad, H]; residual: bf16 [T_pad, H] or None; weight, bias:
    bf16 [H] (bias may be None); scale: fp32 CUDA tensor with one element or None; out,
    out_scales, residual_out: preallocated CUDA tensors (``allocate_outputs``). T_valid defaults
    to T_pad.
    """
    args = _main_args(partials, residual, weight, bias, eps, quant_mode, scale, out, out_scales,
                      residual_out, T_valid)
    st = load_library().sp_fused_reduce_norm(*args, _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_fused_reduce_norm")


def sp_fused_reduce_norm_noalloc(partials, weight, out, residual_out, *, residual=None,
                                 bias=None, eps: float = 1e-6, quant_mode="none", scale=None,
                                 out_scales=None, T_valid: int | None = None,
                                 stream=None) -> None:
    """``sp_fused_reduce_norm`` for callers that may not allocate device memory (inside a graph
    capture, in a framework that owns every buffer, in an allocation-free serving loop): the
    dynamic row schedule's counter lives in the library's own static device memory. Calls that
    overlap on the GPU share that counter: order them (see include/sp_fused.h)."""
    args = _main_args(partials, residual, weight, bias, eps, quant_mode, scale, out, out_scales,
                      residual_out, T_valid)
    st = load_library().sp_fused_reduce_norm_noalloc(*args, _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_fused_reduce_norm_noalloc")


def sp_options_init(*, partial_scale: float = 1.0, addend=None, scale_layout: int = 0,
                    host_buffers: bool = False, schedule="auto", launch=None, row_counter=None,
                    status=None) -> Options:
    """An sp_fused_options initialised by the library, then set from the keywords (``addend`` is a
    tensor or None; ``schedule`` is "auto", "static", "dynamic" or the enum value; ``launch`` a
    LaunchConfig, a dict of its fields, or None for the library's choice; ``row_counter`` an
    int32/uint32 tensor of two zeroed elements or None; ``status`` an int32/uint32 tensor of one
    element or None)."""
    o = Options()
    load_library().sp_options_init(ctypes.byref(o))
    o.partial_scale = partial_scale
    o.addend = _ptr(addend)
    o._addend_ref = addend  # checked (and kept alive) by the call that uses these options
    o.row_counter = _ptr(row_counter)
    o._row_counter_ref = row_counter
    o.status = _ptr(status)
    o._status_ref = status
    o.scale_layout = scale_layout
    o.host_buffers = 1 if host_buffers else 0
    o.schedule = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    if launch is not None:
        cfg = LaunchConfig(**launch) if isinstance(launch, dict) else launch
        o._launch_ref = cfg  # the struct must outlive the options that point at it
        o.launch = ctypes.pointer(cfg)
    return o


def sp_fused_reduce_norm_ex(options: Options | None, partials, weight, out, residual_out, *,
                            residual=None, bias=None, eps: float = 1e-6, quant_mode="none",
                            scale=None, out_scales=None, T_valid: int | None = None,
                            stream=None) -> None:
    """``sp_fused_reduce_norm`` with options (``sp_options_init``): a scale applied to every
    partial before the reduction, an addend after it, host buffers."""
    args = _options_args(options, partials, residual, weight, bias, eps, quant_mode, scale, out,
                         out_scales, residual_out, T_valid)
    st = load_library().sp_fused_reduce_norm_ex(
        ctypes.byref(options) if options is not None else None, *args, _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_fused_reduce_norm_ex")


def _options_args(options, partials, residual, weight, bias, eps, quant_mode, scale, out,
                  out_scales, residual_out, T_valid):
    """_main_args for the options-taking calls: the options' tensors are checked too."""
    host = bool(options is not None and options.host_buffers)
    args = _main_args(partials, residual, weight, bias, eps, quant_mode, scale, out, out_scales,
                      residual_out, T_valid, host=host,
                      addend=getattr(options, "_addend_ref", None),
                      scale_layout=options.scale_layout if options is not None else 0)
    import torch
    words = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    for name, need in (("row_counter", 8), ("status", 4)):
        t = getattr(options, f"_{name}_ref", None)
        if t is not None:
            _check_tensor(name, t, words, need, _current_device(), host)
    return args


def sp_selftest_fused_timeout(limit_ns: int, withhold: int, options: Options | None, partials,
                              weight, out, residual_out, *, residual=None, bias=None,
                              eps: float = 1e-6, quant_mode="none", scale=None, out_scales=None,
                              T_valid: int | None = None, stream=None) -> None:
    """The staged kernel's abort path, forced without a fault (see include/sp_fused.h): waits
    give up after ``limit_ns`` and CTA 0 never fills ring stage ``withhold``."""
    args = _options_args(options, partials, residual, weight, bias, eps, quant_mode, scale, out,
                         out_scales, residual_out, T_valid)
    st = load_library().sp_selftest_fused_timeout(
        limit_ns, withhold, ctypes.byref(options) if options is not None else None, *args,
        _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_selftest_fused_timeout")


def sp_last_launch() -> dict:
    """The calling thread's last fused-stage launch: {"config": {...}, "grid", "schedule"}
    (schedule "static" or "dynamic"; None before the first call)."""
    info = LaunchInfo()
    st = load_library().sp_last_launch(ctypes.byref(info))
    if st != 0:
        raise SpError(st, "sp_last_launch")
    names = {1: "static", 2: "dynamic"}
    return {"config": info.config.as_dict(), "grid": info.grid,
            "schedule": names.get(info.schedule)}


def sp_check_args_ex(options: Options | None, partials, tp, T_pad, T_valid, H, residual, weight,
                     bias, eps, quant_mode, scale, out, out_scales, residual_out) -> int:
    """The checks of sp_fused_reduce_norm_ex on raw addresses; returns the status."""
    return load_library().sp_check_args_ex(
        ctypes.byref(options) if options is not None else None, partials, tp, T_pad, T_valid, H,
        residual, weight, bias, ctypes.c_float(eps), _mode(quant_mode), scale, out, out_scales,
        residual_out)


def sp_fused_reduce_norm_host(partials, weight, out, residual_out, *, residual=None, bias=None,
                              eps: float = 1e-6, quant_mode="none", scale=None, out_scales=None,
                              T_valid: int | None = None, stream=None) -> None:
    """The stage on page-locked HOST tensors (``tensor.pin_memory()``): the kernel reads inputs
    and writes outputs across the host link (zero-copy). ``scale`` is a pinned fp32 tensor with
    one element, or None. Asynchronous on ``stream`` (default: torch's current CUDA stream);
    synchronise before reading the outputs."""
    args = _main_args(partials, residual, weight, bias, eps, quant_mode, scale, out, out_scales,
                      residual_out, T_valid, host=True)
    st = load_library().sp_fused_reduce_norm_host(*args, _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_fused_reduce_norm_host")


def sp_fused_reduce_norm_with_config(config: LaunchConfig | dict, partials, weight, out,
                                     residual_out, *, residual=None, bias=None, eps: float = 1e-6,
                                     quant_mode="none", scale=None, out_scales=None,
                                     T_valid: int | None = None, stream=None) -> None:
    """Like ``sp_fused_reduce_norm`` with an explicit launch configuration."""
    if isinstance(config, dict):
        config = LaunchConfig(**config)
    args = _main_args(partials, residual, weight, bias, eps, quant_mode, scale, out, out_scales,
                      residual_out, T_valid)
    st = load_library().sp_fused_reduce_norm_with_config(ctypes.byref(config), *args,
                                                         _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_fused_reduce_norm_with_config")


def sp_check_args(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode, scale,
                  out, out_scales, residual_out) -> int:
    """The library's argument checks on raw addresses (ints or None); returns the status."""
    return load_library().sp_check_args(partials, tp, T_pad, T_valid, H, residual, weight, bias,
                                        ctypes.c_float(eps), _mode(quant_mode), scale, out,
                                        out_scales, residual_out)


def sp_select_launch(tp: int, T_pad: int, H: int, quant_mode="none") -> LaunchConfig:
    cfg = LaunchConfig()
    st = load_library().sp_select_launch(tp, T_pad, H, _mode(quant_mode), ctypes.byref(cfg))
    if st != 0:
        raise SpError(st, "sp_select_launch")
    return cfg


def sp_pad_tokens(T: int, tp: int) -> int:
    return load_library().sp_pad_tokens(T, tp)


def sp_shard_rows(T_pad: int, tp: int, rank: int) -> tuple[int, int]:
    start, length = _i64(), _i64()
    st = load_library().sp_shard_rows(T_pad, tp, rank, ctypes.byref(start), ctypes.byref(length))
    if st != 0:
        raise SpError(st, "sp_shard_rows")
    return start.value, length.value


def sp_out_bytes(T_pad: int, H: int, quant_mode) -> int:
    return load_library().sp_out_bytes(T_pad, H, _mode(quant_mode))


def sp_out_scales_bytes(T_pad: int, H: int, quant_mode) -> int:
    return load_library().sp_out_scales_bytes(T_pad, H, _mode(quant_mode))


def sp_out_scales_bytes_ex(T_pad: int, H: int, quant_mode, scale_layout: int) -> int:
    return load_library().sp_out_scales_bytes_ex(T_pad, H, _mode(quant_mode), scale_layout)


def sp_fc2_reorganize(x, otp_size: int, y, stream=None) -> None:
    """FlashComm2 token reorganisation of x [G, N, H/G] into y [G, N/D, H/P] (CUDA tensors of
    the same dtype; D = G / otp_size)."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError("x: expected a tensor [G, N, H/G]")
    G, N, F = x.shape
    dev = _current_device()
    _check_tensor("x", x, (x.dtype,), 0, dev, False)
    _check_tensor("y", y, (x.dtype,), x.numel() * x.element_size(), dev, False)
    st = load_library().sp_fc2_reorganize(x.data_ptr(), G, otp_size, N, F * G, x.element_size(),
                                          y.data_ptr(), _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_fc2_reorganize")


def sp_fc2_check_args(x, global_tp, otp_size, N, H, elem_bytes, y) -> int:
    return load_library().sp_fc2_check_args(x, global_tp, otp_size, N, H, elem_bytes, y)


def sp_fc2_batch_ids(global_tp: int, otp_size: int) -> list[list[int]]:
    D = global_tp // otp_size if otp_size > 0 else 0
    ids = (ctypes.c_int * max(1, D * otp_size))()
    st = load_library().sp_fc2_batch_ids(global_tp, otp_size, ids)
    if st != 0:
        raise SpError(st, "sp_fc2_batch_ids")
    return [list(ids[j * otp_size:(j + 1) * otp_size]) for j in range(D)]


def sp_max_hidden() -> int:
    return load_library().sp_max_hidden()


def sp_status_string(status: int) -> str:
    return load_library().sp_status_string(status).decode()


def sp_device_error(clear: bool = True) -> int:
    flags = ctypes.c_uint32()
    st = load_library().sp_device_error(ctypes.byref(flags), 1 if clear else 0)
    if st != 0:
        raise SpError(st, "sp_device_error")
    return flags.value


def sp_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Run the bounded-wait timeout self-test (see include/sp_fused.h)."""
    st = load_library().sp_selftest_wait_timeout(limit_ns, _stream_handle(stream))
    if st != 0:
        raise SpError(st, "sp_selftest_wait_timeout")


def allocate_outputs(T_pad: int, H: int, quant_mode, device, residual_out: bool = True,
                     scale_layout: int = 0) -> dict:
    """Uninitialised output tensors for a call: ``out``, ``out_scales`` (or None) and
    ``residual_out`` (the kernel writes every byte of each). With the swizzled NVFP4 scale
    layout ``out_scales`` is a flat uint8 buffer of sp_out_scales_bytes_ex bytes."""
    import torch
    mode = _mode(quant_mode)
    if mode == 0:
        out = torch.empty((T_pad, H), dtype=torch.bfloat16, device=device)
    elif mode in (1, 2):
        out = torch.empty((T_pad, H), dtype=torch.uint8, device=device)
    elif mode == 3:
        out = torch.empty((T_pad, H // 2), dtype=torch.uint8, device=device)
    else:
        raise ValueError(f"unsupported quant mode {quant_mode}")
    scales = None
    if mode == 2:
        scales = torch.empty((T_pad,), dtype=torch.float32, device=device)
    elif mode == 3 and scale_layout == 1:
        scales = torch.empty((sp_out_scales_bytes_ex(T_pad, H, mode, 1),), dtype=torch.uint8,
                             device=device)
    elif mode == 3:
        scales = torch.empty((T_pad, H // 16), dtype=torch.uint8, device=device)
    res = torch.empty((T_pad, H), dtype=torch.bfloat16, device=device) if residual_out else None
    return {"out": out, "out_scales": scales, "residual_out": res}
