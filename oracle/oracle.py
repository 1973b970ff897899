"""Oracle for the streamed pairwise score consumers: TEST INFRASTRUCTURE ONLY.

ctypes binding of ``tp_oracle.c`` (plain fp64 CPU loops). Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this module; the
product package never imports it and has no CPU fallback through it.

Every input is promoted to fp64 here and every output is fp64 (numpy arrays). The C library is
compiled with gcc on first use (or by ``build()``) into ``oracle/_build/libtp_oracle.so``.

What each function computes is stated in ``tp_oracle.c`` with the passages of
"Using Torchpairwise in Models" (torchpairwise guide) it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tp_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libtp_oracle.so")
_lock = threading.Lock()
_lib = None

METRICS = {"sqeuclidean": 0, "linear": 1, "rbf": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only: it also builds on the Arm GPU host)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", "-Wno-unused-parameter",
               "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Score(ctypes.Structure):
    _fields_ = [("metric", ctypes.c_int), ("gamma", ctypes.c_double), ("scale", ctypes.c_double),
                ("apply_exp", ctypes.c_int),
                ("row_bias", ctypes.c_void_p), ("col_bias", ctypes.c_void_p),
                ("row_weight", ctypes.c_void_p), ("col_weight", ctypes.c_void_p),
                ("pair_mask", ctypes.c_int), ("band", ctypes.c_int64),
                ("row_group", ctypes.c_void_p), ("col_group", ctypes.c_void_p)]


PAIR_MASKS = {"all": 0, "causal": 1, "band": 2, "same_group": 3}


class _Pairs(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("M", ctypes.c_int64), ("D", ctypes.c_int64)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            for name, args in {
                "or_matmul": [P, P, P, I64, P],
                "or_logsumexp": [P, P, ctypes.c_int, P],
                "or_softmax_matmul": [P, P, P, I64, P, P],
                "or_displacement": [P, P, P],
                "or_svgd_direction": [P, ctypes.c_double, P, P],
                "or_topk": [P, P, ctypes.c_int, ctypes.c_int, P, P],
                "or_matmul_backward": [P, P, P, I64, P, P, P, P, P, P, P, P],
                "or_logsumexp_backward": [P, P, ctypes.c_int, P, P, P, P, P, P, P, P],
                "or_softmax_matmul_backward": [P, P, P, I64, P, P, P, P, P, P, P, P, P, P],
                "or_displacement_backward": [P, P, P, P, P, P, P, P, P],
                "or_topk_backward": [P, P, ctypes.c_int, P, P, P, P, P, P, P, P],
            }.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            lib.or_pair_score.argtypes = [P, P, I64, I64]
            lib.or_pair_score.restype = ctypes.c_double
            lib.or_set_threads.argtypes = [ctypes.c_int]
            lib.or_set_threads.restype = None
            lib.or_get_threads.argtypes = []
            lib.or_get_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def set_threads(n: int) -> None:
    """Number of host threads the oracle uses (0 = every online core)."""
    _load().or_set_threads(int(n))


def get_threads() -> int:
    return int(_load().or_get_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Problem:
    """fp64 copies of X, Y and the score parameters, kept alive for the C calls."""

    def __init__(self, X, Y, metric="linear", gamma=1.0, scale=1.0, apply_exp=False,
                 row_bias=None, col_bias=None, row_weight=None, col_weight=None,
                 pair_mask="all", band=0, row_group=None, col_group=None):
        self.X = _f64(X)
        self.Y = _f64(Y)
        if self.X.ndim != 2 or self.Y.ndim != 2 or self.X.shape[1] != self.Y.shape[1]:
            raise ValueError("X [N,D] and Y [M,D] expected")
        self.N, self.D = self.X.shape
        self.M = self.Y.shape[0]
        self.rb, self.cb = _f64(row_bias), _f64(col_bias)
        self.rw, self.cw = _f64(row_weight), _f64(col_weight)
        # pair masks ("Score Expressions": tp.masks causal, band, same_group), group ids as int32
        self.rg = None if row_group is None else np.ascontiguousarray(np.asarray(row_group), dtype=np.int32)
        self.cg = None if col_group is None else np.ascontiguousarray(np.asarray(col_group), dtype=np.int32)
        if pair_mask == "same_group" and (self.rg is None or self.cg is None):
            raise ValueError("same_group needs row_group and col_group")
        gp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
        self.score = _Score(METRICS[metric], float(gamma), float(scale), int(bool(apply_exp)),
                            _ptr(self.rb), _ptr(self.cb), _ptr(self.rw), _ptr(self.cw),
                            PAIR_MASKS[pair_mask], int(band), gp(self.rg), gp(self.cg))
        self.pairs = _Pairs(_ptr(self.X), _ptr(self.Y), self.N, self.M, self.D)

    def _args(self):
        return ctypes.byref(self.pairs), ctypes.byref(self.score)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name} rejected its arguments (code {rc})")


def pair_score(pb: Problem, i: int, j: int) -> float:
    return float(_load().or_pair_score(*pb._args(), int(i), int(j)))


def matmul(pb: Problem, V):
    V = _f64(V)
    out = np.zeros((pb.N, V.shape[1]))
    _check(_load().or_matmul(*pb._args(), _ptr(V), V.shape[1], _ptr(out)), "matmul")
    return out


def logsumexp(pb: Problem, exclude_self=False):
    out = np.zeros(pb.N)
    _check(_load().or_logsumexp(*pb._args(), int(bool(exclude_self)), _ptr(out)), "logsumexp")
    return out


def softmax_matmul(pb: Problem, V):
    V = _f64(V)
    out = np.zeros((pb.N, V.shape[1]))
    lse = np.zeros(pb.N)
    _check(_load().or_softmax_matmul(*pb._args(), _ptr(V), V.shape[1], _ptr(out), _ptr(lse)),
           "softmax_matmul")
    return out, lse


def displacement(pb: Problem):
    out = np.zeros((pb.N, pb.D))
    _check(_load().or_displacement(*pb._args(), _ptr(out)), "displacement")
    return out


def svgd_direction(x, score, gamma, y=None):
    """phi for the particles x (rows) against the particles y (default x), score given at y."""
    pb = Problem(x, x if y is None else y, metric="rbf", gamma=gamma)
    sc = _f64(score)
    out = np.zeros((pb.N, pb.D))
    _check(_load().or_svgd_direction(ctypes.byref(pb.pairs), float(gamma), _ptr(sc), _ptr(out)),
           "svgd_direction")
    return out


def topk(pb: Problem, k, largest=False):
    vals = np.zeros((pb.N, k))
    idx = np.zeros((pb.N, k), dtype=np.int64)
    rc = _load().or_topk(*pb._args(), int(k), int(bool(largest)), _ptr(vals), _ptr(idx))
    if rc == 2:
        raise MemoryError("oracle topk ran out of host memory")
    _check(rc, "topk")
    return vals, idx


def _grads(pb: Problem, want_V=None):
    dX = np.zeros((pb.N, pb.D))
    dY = np.zeros((pb.M, pb.D))
    dV = None if want_V is None else np.zeros((pb.M, want_V))
    dbr = np.zeros(pb.N) if pb.rb is not None else None
    dbc = np.zeros(pb.M) if pb.cb is not None else None
    dwr = np.zeros(pb.N) if pb.rw is not None else None
    dwc = np.zeros(pb.M) if pb.cw is not None else None
    return dict(dX=dX, dY=dY, dV=dV, d_row_bias=dbr, d_col_bias=dbc, d_row_weight=dwr,
                d_col_weight=dwc)


def _gp(g):
    return [_ptr(g["d_row_bias"]), _ptr(g["d_col_bias"]), _ptr(g["d_row_weight"]),
            _ptr(g["d_col_weight"])]


def matmul_backward(pb: Problem, V, grad_out):
    V, go = _f64(V), _f64(grad_out)
    g = _grads(pb, V.shape[1])
    _check(_load().or_matmul_backward(*pb._args(), _ptr(V), V.shape[1], _ptr(go), _ptr(g["dX"]),
                                      _ptr(g["dY"]), _ptr(g["dV"]), *_gp(g)), "matmul_backward")
    return g


def logsumexp_backward(pb: Problem, lse, grad_lse, exclude_self=False):
    lse, gl = _f64(lse), _f64(grad_lse)
    g = _grads(pb)
    _check(_load().or_logsumexp_backward(*pb._args(), int(bool(exclude_self)), _ptr(lse), _ptr(gl),
                                         _ptr(g["dX"]), _ptr(g["dY"]), *_gp(g)),
           "logsumexp_backward")
    return g


def softmax_matmul_backward(pb: Problem, V, out, lse, grad_out):
    V, out, lse, go = _f64(V), _f64(out), _f64(lse), _f64(grad_out)
    g = _grads(pb, V.shape[1])
    _check(_load().or_softmax_matmul_backward(*pb._args(), _ptr(V), V.shape[1], _ptr(out), _ptr(lse),
                                              _ptr(go), _ptr(g["dX"]), _ptr(g["dY"]), _ptr(g["dV"]),
                                              *_gp(g)), "softmax_matmul_backward")
    return g


def displacement_backward(pb: Problem, grad_out):
    go = _f64(grad_out)
    g = _grads(pb)
    _check(_load().or_displacement_backward(*pb._args(), _ptr(go), _ptr(g["dX"]), _ptr(g["dY"]),
                                            *_gp(g)), "displacement_backward")
    return g


def topk_backward(pb: Problem, k, indices, grad_values):
    idx = np.ascontiguousarray(np.asarray(indices), dtype=np.int64)
    gv = _f64(grad_values)
    g = _grads(pb)
    _check(_load().or_topk_backward(*pb._args(), int(k), idx.ctypes.data_as(ctypes.c_void_p),
                                    _ptr(gv), _ptr(g["dX"]), _ptr(g["dY"]), *_gp(g)),
           "topk_backward")
    return g
