"""ctypes wrapper around the C oracle in ``ar_oracle.c``.

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the product library.

Arrays of 16-bit elements (bf16 / fp16) travel as ``numpy.uint16`` bit
patterns so that no conversion happens outside the C code.  Row-parallel entry
points split rows over a thread pool; ctypes releases the GIL during each C
call and every row is computed identically, so results do not depend on the
thread count.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "BF16", "FP16", "build_oracle", "lib", "load_library",
    "bf16_round", "f16_round", "bf16_to_f32", "f16_to_f32",
    "e4m3_encode", "e4m3_decode", "e2m1_encode", "e2m1_decode",
    "lamport_flip", "fused", "amax", "fp8_inv_scale", "quant_fp8",
    "nvfp4_global_scale", "quant_nvfp4", "vector_sum", "workspace_sizes",
    "lamport_step", "host_threads", "swizzle_scales", "fused_f32", "amax_f32",
    "quant_fp8_f32", "quant_nvfp4_f32", "vector_sum_f32",
]

BF16 = 0
FP16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ar_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")


def build_oracle(force: bool = False) -> str:
    """Compile ``ar_oracle.c`` into ``liboracle.so`` beside it (strict IEEE)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-o", tmp, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def load_library(path: str) -> ctypes.CDLL:
    """Load a compiled oracle from ``path`` and declare its signatures."""
    L = ctypes.CDLL(path)
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_f32.restype = ctypes.c_float
    L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_f16.restype = ctypes.c_uint16
    L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_f32.restype = ctypes.c_float
    L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    L.oracle_e2m1_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_to_f32.restype = ctypes.c_float
    L.oracle_f32_to_e2m1.argtypes = [ctypes.c_float]
    L.oracle_f32_to_e2m1.restype = ctypes.c_uint8
    L.oracle_lamport_flip.argtypes = [_u32p, ctypes.c_int64]
    L.oracle_lamport_flip.restype = None
    L.oracle_fused_rows.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _u16p, _u16p, _u16p, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.oracle_fused_rows.restype = None
    L.oracle_amax.argtypes = [ctypes.c_int, _u16p, ctypes.c_int64]
    L.oracle_amax.restype = ctypes.c_float
    L.oracle_fp8_inv_scale.argtypes = [ctypes.c_float]
    L.oracle_fp8_inv_scale.restype = ctypes.c_float
    L.oracle_quant_fp8.argtypes = [ctypes.c_int, _u16p, ctypes.c_int64, ctypes.c_float, _u8p]
    L.oracle_quant_fp8.restype = None
    L.oracle_nvfp4_global_scale.argtypes = [ctypes.c_float]
    L.oracle_nvfp4_global_scale.restype = ctypes.c_float
    L.oracle_quant_nvfp4.argtypes = [ctypes.c_int, _u16p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_float, _u8p, _u8p]
    L.oracle_quant_nvfp4.restype = None
    L.oracle_sum.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                             ctypes.c_int64, _u16p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]
    L.oracle_sum.restype = None
    L.oracle_workspace_sizes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p]
    L.oracle_workspace_sizes.restype = None
    L.oracle_lamport_step.argtypes = [_i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
    L.oracle_swizzle_scales.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
    L.oracle_swizzle_scales.restype = None
    L.oracle_fused_rows_f32.argtypes = [
        ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _f32p, _f32p, _f32p,
        ctypes.c_float, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p]
    L.oracle_fused_rows_f32.restype = None
    L.oracle_amax_f32.argtypes = [_f32p, ctypes.c_int64]
    L.oracle_amax_f32.restype = ctypes.c_float
    L.oracle_quant_fp8_f32.argtypes = [_f32p, ctypes.c_int64, ctypes.c_float, _u8p]
    L.oracle_quant_fp8_f32.restype = None
    L.oracle_quant_nvfp4_f32.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                         _u8p, _u8p]
    L.oracle_quant_nvfp4_f32.restype = None
    L.oracle_sum_f32.argtypes = [ctypes.c_int, ctypes.c_int64, _f32p, ctypes.c_void_p,
                                 ctypes.c_int64, ctypes.c_int64]
    L.oracle_sum_f32.restype = None
    L.oracle_lamport_step.restype = None
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library(build_oracle())
    return _lib


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _chunks(n: int, parts: int):
    parts = max(1, min(parts, n)) if n > 0 else 1
    step = (n + parts - 1) // parts if n > 0 else 0
    return [(b, min(n, b + step)) for b in range(0, n, step)] if n > 0 else []


# ------------------------------------------------------------ scalar codecs --

def _vec(fn, arr, out_dtype):
    flat = np.asarray(arr).ravel()
    return np.array([fn(x) for x in flat.tolist()], dtype=out_dtype).reshape(np.shape(arr))


def bf16_round(x):
    """fp32 values -> bf16 bit patterns (uint16), round to nearest even."""
    return _vec(lib().oracle_f32_to_bf16, np.asarray(x, dtype=np.float32), np.uint16)


def f16_round(x):
    return _vec(lib().oracle_f32_to_f16, np.asarray(x, dtype=np.float32), np.uint16)


def bf16_to_f32(b):
    return _vec(lib().oracle_bf16_to_f32, np.asarray(b, dtype=np.uint16), np.float32)


def f16_to_f32(b):
    return _vec(lib().oracle_f16_to_f32, np.asarray(b, dtype=np.uint16), np.float32)


def e4m3_encode(x):
    return _vec(lib().oracle_f32_to_e4m3, np.asarray(x, dtype=np.float32), np.uint8)


def e4m3_decode(c):
    return _vec(lib().oracle_e4m3_to_f32, np.asarray(c, dtype=np.uint8), np.float32)


def e2m1_encode(x):
    return _vec(lib().oracle_f32_to_e2m1, np.asarray(x, dtype=np.float32), np.uint8)


def e2m1_decode(c):
    return _vec(lib().oracle_e2m1_to_f32, np.asarray(c, dtype=np.uint8), np.float32)


# ----------------------------------------------------------- array kernels --

def lamport_flip(bits16: np.ndarray) -> np.ndarray:
    """Copy of a uint16 array (even length per 32-bit word) with every 32-bit
    word equal to the -0.0f sentinel rewritten to +0.0f."""
    a = np.ascontiguousarray(bits16, dtype=np.uint16).copy()
    words = a.reshape(-1).view(np.uint32)
    lib().oracle_lamport_flip(words, words.size)
    return a


def fused(dtype: int, partials: np.ndarray, residual_in: np.ndarray, gamma: np.ndarray,
          eps: float, rows=None, want_residual=True, want_norm=True, threads: int | None = None,
          acc: int = 0):
    """Residual add + RMSNorm of the rank sum.

    partials: uint16 [R, T, H]; residual_in: uint16 [T, H]; gamma: uint16 [H].
    ``rows``: optional (begin, end) row range; outputs cover only those rows.
    ``acc``: 0 = fp32 rank sum rounded once; 1 = rounded to the element type
    after every addition.
    Returns (residual_out uint16 [n, H] | None, norm_out uint16 [n, H] | None,
    rstd float32 [n]).
    """
    partials = np.ascontiguousarray(partials, dtype=np.uint16)
    residual_in = np.ascontiguousarray(residual_in, dtype=np.uint16)
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    R, T, H = partials.shape
    assert residual_in.shape == (T, H) and gamma.shape == (H,)
    b, e = (0, T) if rows is None else rows
    n = e - b
    res = np.zeros((T, H), np.uint16) if want_residual else None
    nrm = np.zeros((T, H), np.uint16) if want_norm else None
    rstd = np.zeros(T, np.float32)
    L = lib()

    def run(rb, re_):
        L.oracle_fused_rows(dtype, acc, R, T, H, T * H, partials, residual_in, gamma,
                            ctypes.c_float(eps), rb, re_,
                            res.ctypes.data if res is not None else None,
                            nrm.ctypes.data if nrm is not None else None,
                            rstd.ctypes.data)

    nt = threads or host_threads()
    spans = [(b + x, b + y) for x, y in _chunks(n, nt * 4)]
    if nt > 1 and len(spans) > 1:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(lambda s: run(*s), spans))
    else:
        for s in spans:
            run(*s)
    return (res[b:e] if res is not None else None,
            nrm[b:e] if nrm is not None else None, rstd[b:e])


def amax(dtype: int, x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return float(lib().oracle_amax(dtype, x.reshape(-1), x.size))


def fp8_inv_scale(a: float) -> np.float32:
    return np.float32(lib().oracle_fp8_inv_scale(ctypes.c_float(a)))


def quant_fp8(dtype: int, n_bits: np.ndarray, inv_scale: float) -> np.ndarray:
    n_bits = np.ascontiguousarray(n_bits, dtype=np.uint16)
    q = np.zeros(n_bits.shape, np.uint8)
    lib().oracle_quant_fp8(dtype, n_bits.reshape(-1), n_bits.size, ctypes.c_float(inv_scale),
                           q.reshape(-1))
    return q


def nvfp4_global_scale(a: float) -> np.float32:
    return np.float32(lib().oracle_nvfp4_global_scale(ctypes.c_float(a)))


def quant_nvfp4(dtype: int, n_bits: np.ndarray, gs: float):
    """Returns (quant uint8 [T, H/2], scale uint8 [T, H/16])."""
    n_bits = np.ascontiguousarray(n_bits, dtype=np.uint16)
    T, H = n_bits.shape
    assert H % 16 == 0
    q = np.zeros((T, H // 2), np.uint8)
    s = np.zeros((T, H // 16), np.uint8)
    lib().oracle_quant_nvfp4(dtype, n_bits, T, H, ctypes.c_float(gs), q, s)
    return q, s


def vector_sum(dtype: int, ins: np.ndarray, threads: int | None = None, acc: int = 0) -> np.ndarray:
    """ins: uint16 [R, N] -> uint16 [N], fp32 rank-order sum rounded once
    (acc = 1: rounded to the element type after every addition)."""
    ins = np.ascontiguousarray(ins, dtype=np.uint16)
    R, N = ins.shape
    out = np.zeros(N, np.uint16)
    L = lib()
    nt = threads or host_threads()
    spans = _chunks(N, nt * 4)
    run = lambda s: L.oracle_sum(dtype, acc, R, N, N, ins, out.ctypes.data, s[0], s[1])  # noqa: E731
    if nt > 1 and len(spans) > 1:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, spans))
    else:
        for s in spans:
            run(s)
    return out


def workspace_sizes(R: int, max_tokens: int, H: int, elem_bytes: int, oneshot_max: int,
                    flag_count: int):
    out = np.zeros(4, np.int64)
    lib().oracle_workspace_sizes(R, max_tokens, H, elem_bytes, oneshot_max, flag_count, out)
    return tuple(int(v) for v in out)


def lamport_step(flag: int, clear_size: int, R: int, T: int, H: int):
    """Returns (new_flag, new_clear_size, slot_read, slot_cleared)."""
    io = np.array([flag, clear_size, 0, 0], np.int64)
    lib().oracle_lamport_step(io, R, T, H)
    return int(io[0]), int(io[1]), int(io[2]), int(io[3])


def swizzle_scales(linear: np.ndarray) -> np.ndarray:
    """[T, KB] uint8 block scales -> the 128 x 4 tile layout (zero padding)."""
    linear = np.ascontiguousarray(linear, dtype=np.uint8)
    T, KB = linear.shape
    out = np.zeros((T + 127) // 128 * 128 * ((KB + 3) // 4) * 4, np.uint8)
    lib().oracle_swizzle_scales(linear, T, KB, out)
    return out


# ------------------------------------------------------ fp32 element type --

def fused_f32(partials, residual_in, gamma, eps, threads: int | None = None):
    """fp32 elements: partials float32 [R, T, H] -> (residual_out, norm_out,
    rstd) float32."""
    partials = np.ascontiguousarray(partials, dtype=np.float32)
    residual_in = np.ascontiguousarray(residual_in, dtype=np.float32)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    R, T, H = partials.shape
    res = np.zeros((T, H), np.float32)
    nrm = np.zeros((T, H), np.float32)
    rstd = np.zeros(T, np.float32)
    L = lib()

    def run(rb, re_):
        L.oracle_fused_rows_f32(R, T, H, T * H, partials, residual_in, gamma, ctypes.c_float(eps),
                                rb, re_, res.ctypes.data, nrm.ctypes.data, rstd.ctypes.data)

    nt = threads or host_threads()
    spans = _chunks(T, nt * 4)
    if nt > 1 and len(spans) > 1:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(lambda s: run(*s), spans))
    else:
        for s in spans:
            run(*s)
    return res, nrm, rstd


def amax_f32(x) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().oracle_amax_f32(x.reshape(-1), x.size))


def quant_fp8_f32(n, inv_scale):
    n = np.ascontiguousarray(n, dtype=np.float32)
    q = np.zeros(n.shape, np.uint8)
    lib().oracle_quant_fp8_f32(n.reshape(-1), n.size, ctypes.c_float(inv_scale), q.reshape(-1))
    return q


def quant_nvfp4_f32(n, gs):
    n = np.ascontiguousarray(n, dtype=np.float32)
    T, H = n.shape
    q = np.zeros((T, H // 2), np.uint8)
    s = np.zeros((T, H // 16), np.uint8)
    lib().oracle_quant_nvfp4_f32(n, T, H, ctypes.c_float(gs), q, s)
    return q, s


def vector_sum_f32(ins) -> np.ndarray:
    ins = np.ascontiguousarray(ins, dtype=np.float32)
    R, N = ins.shape
    out = np.zeros(N, np.float32)
    lib().oracle_sum_f32(R, N, ins, out.ctypes.data, 0, N)
    return out
