"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects invalid arguments before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    BUILD.build()
    return B.load()


def declared_symbols():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s+(ar_\w+)\s*\(", src,
                                    flags=re.M))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 16
    for n in sorted(names):
        assert hasattr(L, n), n


def test_version_and_last_error(L):
    assert B.ar_fusion_version() == 10000
    assert isinstance(B.ar_fusion_last_error(), str)


def _err(rc):
    return rc, B.ar_fusion_last_error()


def test_workspace_bytes_validation(L):
    n = ctypes.c_size_t()
    assert L.ar_fusion_workspace_bytes(8, 8192, 7168, B.AR_DT_BF16, ctypes.byref(n)) == B.AR_OK
    # regions: buffer, flags, 3 lamport slots, state -- each 256-byte aligned
    buf = 8 * 8192 * 7168 * 2
    flags = 8 * B.AR_BARRIER_FLAG_COUNT * 4
    slot = 8 * 8192 * 7168 * 2
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert n.value == up(up(up(buf) + flags) + 3 * slot + 56)
    assert L.ar_fusion_workspace_bytes(8, 16, 7168, B.AR_DT_BF16, ctypes.byref(n)) == B.AR_OK
    # Lamport slots hold at least the one-shot token capacity
    assert n.value >= 3 * 8 * B.AR_ONESHOT_MAX_TOKENS * 7168 * 2
    for args, code in [((0, 16, 512, 0), B.AR_ERR_UNSUPPORTED), ((17, 16, 512, 0), B.AR_ERR_UNSUPPORTED),
                       ((2, 0, 512, 0), B.AR_ERR_INVALID), ((2, 16, 500, 0), B.AR_ERR_INVALID),
                       ((2, 16, 0, 0), B.AR_ERR_INVALID), ((2, 16, 65536, 0), B.AR_ERR_UNSUPPORTED),
                       ((2, 16, 512, 7), B.AR_ERR_UNSUPPORTED)]:
        rc = L.ar_fusion_workspace_bytes(*args, ctypes.byref(n))
        assert rc == code, (args, _err(rc))
        assert B.ar_fusion_last_error()
    assert L.ar_fusion_workspace_bytes(2, 16, 512, 0, None) == B.AR_ERR_INVALID
    # fp32 elements: the same regions with 4-byte elements
    assert L.ar_fusion_workspace_bytes(8, 8192, 7168, B.AR_DT_FP32, ctypes.byref(n)) == B.AR_OK
    assert n.value == up(up(up(2 * buf) + flags) + 3 * 2 * slot + 56)


def test_create_rejects_bad_shapes_before_cuda(L):
    h = ctypes.c_void_p()
    assert L.ar_fusion_workspace_create(2, 16, 12, 0, None, 0, None, ctypes.byref(h)) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_create(99, 16, 512, 0, None, 0, None, ctypes.byref(h)) == B.AR_ERR_UNSUPPORTED
    assert L.ar_fusion_workspace_create(2, 16, 512, 0, None, 0, None, None) == B.AR_ERR_INVALID
    # caller memory too small
    assert L.ar_fusion_workspace_create(2, 16, 512, 0, ctypes.c_void_p(1 << 20), 16, None,
                                        ctypes.byref(h)) == B.AR_ERR_INVALID


def test_run_and_calls_reject_null_workspace(L):
    rc = L.ar_fusion_run(None, None, 2, 16, 512, 0, None, None, ctypes.c_float(1e-6), 3,
                         None, None, None, None, None, None)
    assert rc == B.AR_ERR_INVALID
    rc = L.ar_fusion_norm_amax(None, None, 2, 16, 512, 0, None, None, ctypes.c_float(1e-6),
                               None, None)
    assert rc == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_stage(None, 0, None, 16, 0, None) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_info(None, None) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_reset(None, None) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_set_variant(None, 1) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_set_mode(None, 1) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_set_launch(None, 2, 1) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_set_accumulate(None, 1) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_set_timeout_ns(None, 5) == B.AR_ERR_INVALID
    assert L.ar_fusion_workspace_destroy(None) == B.AR_OK


def test_sum_validation(L):
    arr = (ctypes.c_void_p * 2)(16, 32)
    assert L.ar_fusion_sum(arr, 0, 10, 0, ctypes.c_void_p(64), None) == B.AR_ERR_UNSUPPORTED
    assert L.ar_fusion_sum(arr, 17, 10, 0, ctypes.c_void_p(64), None) == B.AR_ERR_UNSUPPORTED
    assert L.ar_fusion_sum(arr, 2, 10, 3, ctypes.c_void_p(64), None) == B.AR_ERR_UNSUPPORTED
    assert L.ar_fusion_sum(arr, 2, 0, 0, ctypes.c_void_p(64), None) == B.AR_OK     # empty: no launch
    assert L.ar_fusion_sum_ex(arr, 2, 10, 0, 7, ctypes.c_void_p(64), None) == B.AR_ERR_INVALID
    # fp32 needs 4-byte element alignment
    assert L.ar_fusion_sum(arr, 2, 10, B.AR_DT_FP32, ctypes.c_void_p(66), None) == B.AR_ERR_INVALID
    odd = (ctypes.c_void_p * 2)(16, 34)
    assert L.ar_fusion_sum(odd, 2, 10, B.AR_DT_FP32, ctypes.c_void_p(64), None) == B.AR_ERR_INVALID
    assert L.ar_fusion_sum(arr, 2, 10, 0, None, None) == B.AR_ERR_INVALID
    bad = (ctypes.c_void_p * 2)(16, 33)
    assert L.ar_fusion_sum(bad, 2, 10, 0, ctypes.c_void_p(64), None) == B.AR_ERR_INVALID


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("allreduce_residual_rmsnorm_gb300.binding")
    saved = mod._lib
    mod._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            mod.load(str(tmp_path / "nope.so"))
    finally:
        mod._lib = saved


def test_plain_c_program_uses_the_library(L, tmp_path):
    # the header compiles as C99 with a C compiler and the library links and
    # answers from C (entry points that need no GPU)
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_abi_check.c")
    exe = tmp_path / "c_abi_check"
    libdir = os.path.dirname(B.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", HEADER_DIR, src,
                        "-o", str(exe), "-L", libdir, "-larfusion", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_partial_ptr_rejects_bad_arguments_before_cuda(L):
    out = ctypes.c_void_p()
    assert L.ar_fusion_workspace_partial_ptr(None, 0, 16, 0, None, ctypes.byref(out)) == B.AR_ERR_INVALID


def test_last_error_is_per_thread(L):
    # each host thread reads the message of its own last failure
    import threading
    n = ctypes.c_size_t()
    results = {}
    barrier = threading.Barrier(4)

    def worker(k):
        hidden = 480 + k                   # not a multiple of 8: AR_ERR_INVALID naming it
        barrier.wait()
        for _ in range(200):
            rc = L.ar_fusion_workspace_bytes(2, 16, hidden, 0, ctypes.byref(n))
            msg = L.ar_fusion_last_error().decode()
            if rc != B.AR_ERR_INVALID or str(hidden) not in msg:
                results[k] = (rc, msg)
                return
        results[k] = "ok"

    ts = [threading.Thread(target=worker, args=(k,)) for k in range(1, 5)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert all(v == "ok" for v in results.values()), results
