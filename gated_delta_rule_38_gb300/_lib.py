"""ctypes view of the C ABI declared in include/gdr.h (argument marshalling only)."""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgdr.so")

GDR_BF16, GDR_FP16, GDR_FP32 = 0, 1, 2
GDR_L2NORM_QK = 1 << 0
GDR_STATE_V_FIRST = 1 << 1
GDR_GATE_IN_KERNEL = 1 << 8
GDR_BETA_SIGMOID_IN_KERNEL = 1 << 9
GDR_ALLOW_NEG_EIGVAL = 1 << 10
GDR_INTER_CARD_CP = 1 << 11
GDR_CHUNK = 64

STATUS_NAMES = {
    0: "GDR_OK", 1: "GDR_ERR_NULL", 2: "GDR_ERR_SHAPE", 3: "GDR_ERR_DTYPE", 4: "GDR_ERR_UNSUPPORTED",
    5: "GDR_ERR_DEVICE", 6: "GDR_ERR_ALIGN", 7: "GDR_ERR_WORKSPACE", 8: "GDR_ERR_CUSEQLENS",
    9: "GDR_ERR_TIMEOUT", 10: "GDR_ERR_CUDA", 11: "GDR_ERR_INTERNAL",
}

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ["gdr_max_chunks", "gdr_prepare_chunks", "gdr_fwd_workspace_size", "gdr_bwd_workspace_size",
           "gdr_fwd", "gdr_bwd", "gdr_get_error", "gdr_status_string", "gdr_version", "gdr_profile_enable",
           "gdr_profile_read", "gdr_fwd_noalloc", "gdr_saved_bytes", "gdr_saved_workspace_size", "gdr_fwd_ex",
           "gdr_bwd_ex", "gdr_decode", "gdr_debug_set_wait_polls", "gdr_last_cuda_error"]


class Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("Hq", ctypes.c_int), ("Hv", ctypes.c_int),
        ("K", ctypes.c_int), ("V", ctypes.c_int), ("dtype", ctypes.c_int), ("gate_dtype", ctypes.c_int),
        ("scale", ctypes.c_float), ("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
        ("flags", ctypes.c_uint), ("num_segments", ctypes.c_int),
    ]


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = "%s failed: %s (%s)" % (where, STATUS_NAMES.get(status, status), status_string(status))
        if status == 10:  # GDR_ERR_CUDA: name the runtime error behind it
            msg += ": " + last_cuda_error()
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libgdr.so; fails loudly when the CUDA library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("the CUDA library %s is missing: run gated_delta_rule_38_gb300.build.build() "
                               "(there is no CPU fallback)" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        PP = ctypes.POINTER(Problem)
        i32 = ctypes.c_int
        lib.gdr_max_chunks.argtypes = [PP]
        lib.gdr_max_chunks.restype = ctypes.c_int64
        lib.gdr_prepare_chunks.argtypes = [P, i32, i32, i32, P, ctypes.c_int64, P, P, P]
        lib.gdr_prepare_chunks.restype = i32
        lib.gdr_fwd_workspace_size.argtypes = [PP, ctypes.POINTER(ctypes.c_size_t)]
        lib.gdr_fwd_workspace_size.restype = i32
        lib.gdr_bwd_workspace_size.argtypes = [PP, ctypes.POINTER(ctypes.c_size_t)]
        lib.gdr_bwd_workspace_size.restype = i32
        lib.gdr_fwd.argtypes = [PP] + [P] * 12 + [ctypes.c_size_t, P]
        lib.gdr_fwd.restype = i32
        lib.gdr_bwd.argtypes = [PP] + [P] * 16 + [ctypes.c_size_t, P]
        lib.gdr_bwd.restype = i32
        lib.gdr_saved_bytes.argtypes = [PP, ctypes.POINTER(ctypes.c_size_t)]
        lib.gdr_saved_bytes.restype = i32
        lib.gdr_saved_workspace_size.argtypes = [PP, i32, ctypes.POINTER(ctypes.c_size_t)]
        lib.gdr_saved_workspace_size.restype = i32
        lib.gdr_decode.argtypes = [PP] + [P] * 9
        lib.gdr_decode.restype = i32
        lib.gdr_fwd_ex.argtypes = [PP] + [P] * 12 + [ctypes.c_size_t, P, P]
        lib.gdr_fwd_ex.restype = i32
        lib.gdr_bwd_ex.argtypes = [PP] + [P] * 16 + [ctypes.c_size_t, P, P]
        lib.gdr_bwd_ex.restype = i32
        lib.gdr_fwd_noalloc.argtypes = [PP] + [P] * 9
        lib.gdr_fwd_noalloc.restype = i32
        lib.gdr_get_error.argtypes = [P]
        lib.gdr_get_error.restype = i32
        lib.gdr_status_string.argtypes = [i32]
        lib.gdr_status_string.restype = ctypes.c_char_p
        lib.gdr_last_cuda_error.argtypes = []
        lib.gdr_last_cuda_error.restype = ctypes.c_char_p
        lib.gdr_profile_enable.argtypes = [i32]
        lib.gdr_profile_enable.restype = i32
        lib.gdr_profile_read.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_longlong),
                                         ctypes.POINTER(ctypes.c_double)]
        lib.gdr_profile_read.restype = i32
        lib.gdr_debug_set_wait_polls.argtypes = [ctypes.c_longlong]
        lib.gdr_debug_set_wait_polls.restype = i32
        lib.gdr_version.argtypes = []
        lib.gdr_version.restype = i32
        _lib = lib
    return _lib


def status_string(st: int) -> str:
    try:
        return load().gdr_status_string(int(st)).decode()
    except Exception:  # pragma: no cover
        return "?"


def last_cuda_error() -> str:
    """Name of the CUDA runtime error behind this thread's latest GDR_ERR_CUDA."""
    try:
        return load().gdr_last_cuda_error().decode()
    except Exception:  # pragma: no cover
        return "?"


def check(st: int, where: str) -> None:
    if st != 0:
        raise GdrError(st, where)


def profile_enable(on: bool) -> None:
    load().gdr_profile_enable(1 if on else 0)


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} of the launches timed since profile_enable(True)."""
    lib = load()
    cap = 32
    names = (ctypes.c_char_p * cap)()
    cnt = (ctypes.c_longlong * cap)()
    ms = (ctypes.c_double * cap)()
    n = lib.gdr_profile_read(cap, names, cnt, ms)
    if n < 0:
        raise RuntimeError("gdr_profile_read failed")
    return {names[i].decode(): (int(cnt[i]), float(ms[i])) for i in range(min(n, cap))}
