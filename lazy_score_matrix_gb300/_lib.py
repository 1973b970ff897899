"""ctypes binding of libtp's C ABI (include/tp.h): the same names, argument marshalling only.

Loading fails loudly when ``libtp.so`` has not been built: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtp.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "tp.h")

TP_OK, TP_ERR_INVALID_ARG, TP_ERR_UNSUPPORTED, TP_ERR_CUDA, TP_ERR_WORKSPACE, TP_ERR_TIMEOUT = range(6)
TP_F32, TP_F64 = 0, 1
METRICS = {"sqeuclidean": 0, "linear": 1, "rbf": 2}


PAIR_MASKS = {"all": 0, "causal": 1, "band": 2, "same_group": 3}


class tp_score(ctypes.Structure):
    _fields_ = [("metric", ctypes.c_int), ("gamma", ctypes.c_double), ("scale", ctypes.c_double),
                ("apply_exp", ctypes.c_int),
                ("row_bias", ctypes.c_void_p), ("col_bias", ctypes.c_void_p),
                ("row_weight", ctypes.c_void_p), ("col_weight", ctypes.c_void_p),
                ("pair_mask", ctypes.c_int), ("band", ctypes.c_int64),
                ("row_group", ctypes.c_void_p), ("col_group", ctypes.c_void_p)]


class tp_pairs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("N", ctypes.c_int64), ("M", ctypes.c_int64), ("D", ctypes.c_int64),
                ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int
_PAIRS = ctypes.POINTER(tp_pairs)
_SCORE = ctypes.POINTER(tp_score)

SIGNATURES = {
    "tp_pairwise_matmul": ([_PAIRS, _SCORE, _P, _I64, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_logsumexp": ([_PAIRS, _SCORE, _INT, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_logsumexp_noalloc": ([_PAIRS, _SCORE, _INT, _P, _P], _INT),
    "tp_pairwise_softmax_matmul": ([_PAIRS, _SCORE, _P, _I64, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_displacement": ([_PAIRS, _SCORE, _P, _P, _SZ, _P], _INT),
    "tp_svgd_direction": ([_PAIRS, ctypes.c_double, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_topk": ([_PAIRS, _SCORE, _INT, _INT, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_matmul_backward": ([_PAIRS, _SCORE, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_logsumexp_backward": ([_PAIRS, _SCORE, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_softmax_matmul_backward": (
        [_PAIRS, _SCORE, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_displacement_backward": ([_PAIRS, _SCORE, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _INT),
    "tp_pairwise_topk_backward": ([_PAIRS, _SCORE, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _INT),
    "tp_workspace_size": ([ctypes.c_char_p, _PAIRS, _I64, _INT], _SZ),
    "tp_status_string": ([_INT], ctypes.c_char_p),
    "tp_last_error": ([], ctypes.c_char_p),
    "tp_launch_count": ([_INT], _I64),
    "tp_set_launch_hook": ([_P, _P], None),
    "tp_timer_start": ([_I64], _INT),
    "tp_timer_stop": ([], _I64),
    "tp_timer_read": ([_I64, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)], _INT),
    "tp_device_status": ([_INT], _INT),
    "tp_selftest_bounded_wait": ([_I64, _P], _INT),
    "tp_selftest_exp64": ([_P, _P, _I64, _P], _INT),
}

LAUNCH_HOOK = ctypes.CFUNCTYPE(None, ctypes.c_char_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p)

_lock = threading.Lock()
_lib = None


class TPError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {detail}")


def header_symbols() -> list[str]:
    """Every function the public header declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^TP_API\s+[\w\s\*]+?\b(tp_\w+)\s*\(", text, flags=re.M)))


def load(path: str | None = None):
    """Load libtp.so (built in-tree by lazy_score_matrix_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libtp is not built ({p} missing): run `python -m lazy_score_matrix_gb300.build` "
                              "or __graft_entry__.build(); there is no CPU fallback")
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        if path is None:
            _lib = lib
        return lib


def status_text(status: int) -> str:
    lib = load()
    return (lib.tp_status_string(status) or b"").decode()


def check(status: int, where: str) -> None:
    if status != TP_OK:
        lib = load()
        raise TPError(status, where, f"{status_text(status)} ({(lib.tp_last_error() or b'').decode()})")


def launch_count(reset: bool = False) -> int:
    return int(load().tp_launch_count(1 if reset else 0))


def __getattr__(name):
    if name in SIGNATURES:
        return getattr(load(), name)
    raise AttributeError(name)
