"""Thin ctypes binding of libarfusion (include/ar_fusion.h).

Argument marshalling only: every function has the name of the C entry point,
turns torch tensors into device pointers / sizes, calls the library, and raises
:class:`ArFusionError` on a non-zero status.  No compute happens here and
there is no fallback: if the library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libarfusion.so")

# enum ar_dtype
AR_DT_BF16 = 0
AR_DT_FP16 = 1
AR_DT_FP32 = 2
# enum ar_pattern
AR_RESIDUAL_OUT = 1
AR_NORM_OUT = 2
AR_QUANT_FP8 = 4
AR_QUANT_NVFP4 = 8
# enum ar_status
AR_OK = 0
AR_ERR_INVALID = -1
AR_ERR_UNSUPPORTED = -2
AR_ERR_CUDA = -3
AR_ERR_TIMEOUT = -4
AR_ERR_CAPACITY = -5
# enum ar_mode
AR_MODE_AUTO = 0
AR_MODE_LAMPORT = 1
AR_MODE_BUFFER = 2
# enum ar_variant
AR_VARIANT_AUTO = 0
AR_VARIANT_WARP_ROW = 1
AR_VARIANT_CTA_ROW = 2
AR_VARIANT_BULK_PIPE = 3

# enum ar_scale_layout
AR_SF_LINEAR = 0
AR_SF_SWIZZLED = 1
# enum ar_accumulate
AR_ACC_FP32 = 0
AR_ACC_ELEMENT = 1

AR_MAX_RANKS = 16
AR_ONESHOT_MAX_TOKENS = 128
AR_BARRIER_FLAG_COUNT = 256
AR_MAX_HIDDEN = 32768
AR_NOALLOC_SLOT_BYTES = 4 << 20

PATTERNS = {
    "res_norm": AR_RESIDUAL_OUT | AR_NORM_OUT,
    "norm": AR_NORM_OUT,
    "res_fp8": AR_RESIDUAL_OUT | AR_QUANT_FP8,
    "res_nvfp4": AR_RESIDUAL_OUT | AR_QUANT_NVFP4,
    "res_norm_fp8": AR_RESIDUAL_OUT | AR_NORM_OUT | AR_QUANT_FP8,
    "res_norm_nvfp4": AR_RESIDUAL_OUT | AR_NORM_OUT | AR_QUANT_NVFP4,
}


class ArFusionError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ar_fusion error {code}: {msg}")
        self.code = code


class WsInfo(ctypes.Structure):
    _fields_ = [
        ("tp_size", ctypes.c_int32), ("max_token_num", ctypes.c_int32),
        ("hidden_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32), ("oneshot_max_tokens", ctypes.c_int32),
        ("total_bytes", ctypes.c_uint64), ("buffer_bytes", ctypes.c_uint64),
        ("flag_bytes", ctypes.c_uint64), ("lamport_comm_bytes", ctypes.c_uint64),
        ("lamport_buffer_bytes", ctypes.c_uint64), ("state_bytes", ctypes.c_uint64),
        ("base", ctypes.c_void_p), ("buffer", ctypes.c_void_p), ("flags", ctypes.c_void_p),
        ("lamport", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("last_variant", ctypes.c_int32), ("last_cluster", ctypes.c_int32),
    ]


class State(ctypes.Structure):
    _fields_ = [
        ("counter", ctypes.c_uint32), ("flag", ctypes.c_uint32),
        ("lamport_flag", ctypes.c_uint32), ("clear_elem_bytes", ctypes.c_uint32),
        ("comm_size", ctypes.c_uint64), ("clear_size", ctypes.c_uint64),
        ("status", ctypes.c_int32), ("detail", ctypes.c_int32), ("calls", ctypes.c_uint64),
    ]


_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libarfusion.so (built in-tree by ``build.py``) and declare its
    signatures.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    L.ar_fusion_version.restype = _i
    L.ar_fusion_version.argtypes = []
    L.ar_fusion_last_error.restype = ctypes.c_char_p
    L.ar_fusion_last_error.argtypes = []
    L.ar_fusion_workspace_bytes.argtypes = [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]
    L.ar_fusion_workspace_create.argtypes = [_i, _i, _i, _i, _vp, ctypes.c_size_t, _vp,
                                             ctypes.POINTER(_vp)]
    L.ar_fusion_workspace_destroy.argtypes = [_vp]
    L.ar_fusion_workspace_info.argtypes = [_vp, ctypes.POINTER(WsInfo)]
    L.ar_fusion_workspace_copy_state.argtypes = [_vp, _vp, ctypes.POINTER(State)]
    L.ar_fusion_workspace_status.argtypes = [_vp, _vp, ctypes.POINTER(_i)]
    L.ar_fusion_workspace_reset.argtypes = [_vp, _vp]
    L.ar_fusion_workspace_set_timeout_ns.argtypes = [_vp, ctypes.c_uint64]
    L.ar_fusion_workspace_set_variant.argtypes = [_vp, _i]
    L.ar_fusion_workspace_set_mode.argtypes = [_vp, _i]
    L.ar_fusion_workspace_set_launch.argtypes = [_vp, _i, _i]
    L.ar_fusion_workspace_set_accumulate.argtypes = [_vp, _i]
    L.ar_fusion_workspace_set_scale_layout.argtypes = [_vp, _i]
    L.ar_fusion_sum_ex.argtypes = [ctypes.POINTER(_vp), _i, ctypes.c_size_t, _i, _i, _vp, _vp]
    L.ar_fusion_workspace_stage.argtypes = [_vp, _i, _vp, _i, _i, _vp]
    L.ar_fusion_workspace_partial_ptr.argtypes = [_vp, _i, _i, _i, _vp, ctypes.POINTER(_vp)]
    L.ar_fusion_run.argtypes = [_vp, ctypes.POINTER(_vp), _i, _i, _i, _i, _vp, _vp,
                                ctypes.c_float, _i, _vp, _vp, _vp, _vp, _vp, _vp]
    L.ar_fusion_norm_amax.argtypes = [_vp, ctypes.POINTER(_vp), _i, _i, _i, _i, _vp, _vp,
                                      ctypes.c_float, _vp, _vp]
    L.ar_fusion_sum.argtypes = [ctypes.POINTER(_vp), _i, ctypes.c_size_t, _i, _vp, _vp]
    L.ar_fusion_run_noalloc.argtypes = [ctypes.POINTER(_vp), _i, _i, _i, _i, _vp, _vp,
                                        ctypes.c_float, _i, _vp, _vp, _vp, _vp, _vp, _vp]
    L.ar_fusion_noalloc_status.argtypes = [_vp, ctypes.POINTER(_i)]
    for name in ("ar_fusion_workspace_bytes", "ar_fusion_workspace_create",
                 "ar_fusion_workspace_destroy", "ar_fusion_workspace_info",
                 "ar_fusion_workspace_copy_state", "ar_fusion_workspace_status",
                 "ar_fusion_workspace_reset", "ar_fusion_workspace_set_timeout_ns",
                 "ar_fusion_workspace_set_variant", "ar_fusion_workspace_set_mode",
                 "ar_fusion_workspace_set_launch", "ar_fusion_workspace_set_accumulate",
                 "ar_fusion_workspace_set_scale_layout",
                 "ar_fusion_sum_ex",
                 "ar_fusion_workspace_stage", "ar_fusion_workspace_partial_ptr",
                 "ar_fusion_run", "ar_fusion_norm_amax",
                 "ar_fusion_sum", "ar_fusion_run_noalloc", "ar_fusion_noalloc_status"):
        getattr(L, name).restype = _i
    _lib = L
    return L


def lib() -> ctypes.CDLL:
    return load()


def _check(rc: int) -> int:
    if rc != AR_OK:
        raise ArFusionError(rc, ar_fusion_last_error())
    return rc


def _dtype_id(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return AR_DT_BF16
    if t.dtype == torch.float16:
        return AR_DT_FP16
    if t.dtype == torch.float32:
        return AR_DT_FP32
    raise TypeError(f"unsupported element type {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr_array(ts):
    arr = (_vp * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t)
    return arr


class Workspace:
    """Handle of an ``ar_fusion_ws``; keeps caller-supplied memory alive."""

    def __init__(self, handle: int, mem, tp_size, max_token_num, hidden_dim, dtype):
        self.handle = handle
        self.mem = mem
        self.tp_size = tp_size
        self.max_token_num = max_token_num
        self.hidden_dim = hidden_dim
        self.dtype = dtype

    def __del__(self):
        try:
            if self.handle:
                ar_fusion_workspace_destroy(self)
        except Exception:
            pass


# ------------------------------------------------------------------- calls

def ar_fusion_version() -> int:
    return lib().ar_fusion_version()


def ar_fusion_last_error() -> str:
    return lib().ar_fusion_last_error().decode()


def ar_fusion_workspace_bytes(tp_size: int, max_token_num: int, hidden_dim: int,
                              dtype: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().ar_fusion_workspace_bytes(tp_size, max_token_num, hidden_dim, dtype,
                                           ctypes.byref(n)))
    return n.value


def ar_fusion_workspace_create(tp_size: int, max_token_num: int, hidden_dim: int, dtype: int,
                               device_mem: torch.Tensor | None = None, stream=None) -> Workspace:
    h = _vp()
    mem_ptr = _ptr(device_mem) if device_mem is not None else None
    mem_bytes = device_mem.numel() * device_mem.element_size() if device_mem is not None else 0
    _check(lib().ar_fusion_workspace_create(tp_size, max_token_num, hidden_dim, dtype, mem_ptr,
                                            mem_bytes, _stream(stream), ctypes.byref(h)))
    return Workspace(h.value, device_mem, tp_size, max_token_num, hidden_dim, dtype)


def ar_fusion_workspace_destroy(ws: Workspace) -> None:
    if ws.handle:
        h, ws.handle = ws.handle, None
        _check(lib().ar_fusion_workspace_destroy(h))


def ar_fusion_workspace_info(ws: Workspace) -> dict:
    info = WsInfo()
    _check(lib().ar_fusion_workspace_info(ws.handle, ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in WsInfo._fields_}


def ar_fusion_workspace_copy_state(ws: Workspace, stream=None) -> dict:
    st = State()
    _check(lib().ar_fusion_workspace_copy_state(ws.handle, _stream(stream), ctypes.byref(st)))
    return {name: getattr(st, name) for name, _ in State._fields_}


def ar_fusion_workspace_status(ws: Workspace, stream=None):
    """Returns (status code, detail); does not raise on a device error."""
    d = _i(-1)
    rc = lib().ar_fusion_workspace_status(ws.handle, _stream(stream), ctypes.byref(d))
    return rc, d.value


def ar_fusion_workspace_reset(ws: Workspace, stream=None) -> None:
    _check(lib().ar_fusion_workspace_reset(ws.handle, _stream(stream)))


def ar_fusion_workspace_set_timeout_ns(ws: Workspace, ns: int) -> None:
    _check(lib().ar_fusion_workspace_set_timeout_ns(ws.handle, int(ns)))


def ar_fusion_workspace_set_variant(ws: Workspace, variant: int) -> None:
    _check(lib().ar_fusion_workspace_set_variant(ws.handle, int(variant)))


def ar_fusion_workspace_set_mode(ws: Workspace, mode: int) -> None:
    _check(lib().ar_fusion_workspace_set_mode(ws.handle, int(mode)))


def ar_fusion_workspace_set_launch(ws: Workspace, cluster_size: int = 0, pdl: int = 0) -> None:
    _check(lib().ar_fusion_workspace_set_launch(ws.handle, int(cluster_size), int(pdl)))


def ar_fusion_workspace_set_accumulate(ws: Workspace, accumulate: int) -> None:
    _check(lib().ar_fusion_workspace_set_accumulate(ws.handle, int(accumulate)))


def ar_fusion_workspace_set_scale_layout(ws: Workspace, layout: int) -> None:
    _check(lib().ar_fusion_workspace_set_scale_layout(ws.handle, int(layout)))


def swizzled_scale_bytes(tokens: int, hidden: int) -> int:
    """Size of an AR_SF_SWIZZLED scale buffer (whole 128 x 4 tiles)."""
    kb = hidden // 16
    return (tokens + 127) // 128 * 128 * ((kb + 3) // 4) * 4


def ar_fusion_workspace_stage(ws: Workspace, rank: int, src: torch.Tensor, tokens: int | None = None,
                              mode: int = AR_MODE_AUTO, stream=None) -> None:
    if tokens is None:
        tokens = src.shape[0] if src.dim() >= 2 else src.numel() // ws.hidden_dim
    _check(lib().ar_fusion_workspace_stage(ws.handle, rank, _ptr(src), tokens, mode,
                                           _stream(stream)))


def ar_fusion_workspace_partial_ptr(ws: Workspace, rank: int, tokens: int,
                                    mode: int = AR_MODE_AUTO, stream=None) -> int:
    """Device address where rank `rank`'s [tokens, hidden] partial is staged."""
    out = ctypes.c_void_p()
    _check(lib().ar_fusion_workspace_partial_ptr(ws.handle, rank, tokens, mode, _stream(stream),
                                                 ctypes.byref(out)))
    return out.value


def ar_fusion_run(ws: Workspace, partials, residual_in: torch.Tensor, gamma: torch.Tensor,
                  eps: float, pattern: int, residual_out=None, norm_out=None, quant_out=None,
                  scale_out=None, scale_factor=None, stream=None, nranks: int | None = None) -> None:
    """partials: list of R [tokens, hidden] CUDA tensors, or None for the
    partials staged in ``ws``."""
    tokens, hidden = residual_in.shape[0], residual_in.shape[-1]
    if partials is None:
        parr = None
        R = ws.tp_size if nranks is None else nranks
    else:
        parr = _ptr_array(partials)
        R = len(partials) if nranks is None else nranks
    _check(lib().ar_fusion_run(ws.handle, parr, R, tokens, hidden, _dtype_id(residual_in),
                               _ptr(residual_in), _ptr(gamma), ctypes.c_float(eps), pattern,
                               _ptr(residual_out), _ptr(norm_out), _ptr(quant_out),
                               _ptr(scale_out), _ptr(scale_factor), _stream(stream)))


def bound_run(ws: Workspace, partials, residual_in: torch.Tensor, gamma: torch.Tensor,
              eps: float, pattern: int, residual_out=None, norm_out=None, quant_out=None,
              scale_out=None, scale_factor=None, stream=None, nranks: int | None = None):
    """ar_fusion_run with every argument marshalled once: returns a callable
    that launches the call (same tensors, same stream) with no per-call
    Python work beyond the C call itself, for loops that repeat one call.
    The tensors must stay alive while the callable is used."""
    tokens, hidden = residual_in.shape[0], residual_in.shape[-1]
    if partials is None:
        parr = None
        R = ws.tp_size if nranks is None else nranks
    else:
        parr = _ptr_array(partials)
        R = len(partials) if nranks is None else nranks
    fn = lib().ar_fusion_run
    args = (ws.handle, parr, R, tokens, hidden, _dtype_id(residual_in), _ptr(residual_in),
            _ptr(gamma), ctypes.c_float(eps), pattern, _ptr(residual_out), _ptr(norm_out),
            _ptr(quant_out), _ptr(scale_out), _ptr(scale_factor), _stream(stream))

    def call():
        rc = fn(*args)
        if rc != AR_OK:
            _check(rc)

    return call


def ar_fusion_norm_amax(ws: Workspace, partials, residual_in: torch.Tensor, gamma: torch.Tensor,
                        eps: float, amax_out: torch.Tensor, stream=None,
                        nranks: int | None = None) -> None:
    tokens, hidden = residual_in.shape[0], residual_in.shape[-1]
    if partials is None:
        parr = None
        R = ws.tp_size if nranks is None else nranks
    else:
        parr = _ptr_array(partials)
        R = len(partials) if nranks is None else nranks
    _check(lib().ar_fusion_norm_amax(ws.handle, parr, R, tokens, hidden, _dtype_id(residual_in),
                                     _ptr(residual_in), _ptr(gamma), ctypes.c_float(eps),
                                     _ptr(amax_out), _stream(stream)))


def ar_fusion_sum_ex(bufs, out: torch.Tensor, accumulate: int, n: int | None = None,
                     stream=None) -> None:
    if n is None:
        n = out.numel()
    _check(lib().ar_fusion_sum_ex(_ptr_array(bufs), len(bufs), n, _dtype_id(out), int(accumulate),
                                  _ptr(out), _stream(stream)))


def ar_fusion_sum(bufs, out: torch.Tensor, n: int | None = None, stream=None) -> None:
    if n is None:
        n = out.numel()
    _check(lib().ar_fusion_sum(_ptr_array(bufs), len(bufs), n, _dtype_id(out), _ptr(out),
                               _stream(stream)))


def ar_fusion_run_noalloc(partials, residual_in: torch.Tensor, gamma: torch.Tensor, eps: float,
                          pattern: int, residual_out=None, norm_out=None, quant_out=None,
                          scale_out=None, scale_factor=None, stream=None) -> None:
    """The one-shot fused call without a workspace (no device allocation):
    scratch lives in a fixed device array inside the library."""
    tokens, hidden = residual_in.shape[0], residual_in.shape[-1]
    _check(lib().ar_fusion_run_noalloc(_ptr_array(partials), len(partials), tokens, hidden,
                                       _dtype_id(residual_in), _ptr(residual_in), _ptr(gamma),
                                       ctypes.c_float(eps), pattern, _ptr(residual_out),
                                       _ptr(norm_out), _ptr(quant_out), _ptr(scale_out),
                                       _ptr(scale_factor), _stream(stream)))


def ar_fusion_noalloc_status(stream=None):
    """(status, detail) of the no-allocation call on the current device: the
    first device-side error since the previous query (AR_OK if none), which
    the query clears.  Synchronises the stream."""
    d = ctypes.c_int(-1)
    rc = lib().ar_fusion_noalloc_status(_stream(stream), ctypes.byref(d))
    if rc not in (AR_OK, AR_ERR_TIMEOUT):
        _check(rc)
    return rc, d.value
