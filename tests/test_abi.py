"""The C-ABI library on the CPU: it loads, exports every symbol include/tp.h declares, sizes its
workspace from the shapes alone, and rejects invalid arguments before launching anything.

Every call made here is invalid on purpose and returns before any CUDA work is enqueued, so the
fake device addresses are never touched (on a machine with or without a GPU).
"""
import ctypes
import subprocess

import pytest

from lazy_score_matrix_gb300 import _lib
from lazy_score_matrix_gb300 import build as tpbuild


@pytest.fixture(scope="module")
def lib():
    tpbuild.build()
    return _lib.load()


FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced


def pairs(N=10, M=12, D=3, dtype=_lib.TP_F32, X=FAKE, Y=FAKE + 0x100000):
    return _lib.tp_pairs(dtype, N, M, D, X, Y)


def score(metric=1, **kw):
    return _lib.tp_score(metric, kw.get("gamma", 1.0), kw.get("scale", 1.0), 0, kw.get("rb"), kw.get("cb"),
                         kw.get("rw"), kw.get("cw"))


def test_exports_every_header_symbol(lib):
    declared = _lib.header_symbols()
    assert len(declared) == 23, declared
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    for s in declared:
        assert getattr(lib, s) is not None
    assert set(declared) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    for s in range(6):
        assert lib.tp_status_string(s)
    assert b"INVALID" in lib.tp_status_string(_lib.TP_ERR_INVALID_ARG)


def test_timer_argument_checks(lib):
    # host-only paths: no CUDA call is made before these checks
    assert lib.tp_timer_start(0) == _lib.TP_ERR_INVALID_ARG
    assert lib.tp_timer_stop() == 0
    name, ms = ctypes.c_char_p(), ctypes.c_float()
    assert lib.tp_timer_read(0, ctypes.byref(name), ctypes.byref(ms)) == _lib.TP_ERR_INVALID_ARG
    assert lib.tp_timer_read(-1, ctypes.byref(name), ctypes.byref(ms)) == _lib.TP_ERR_INVALID_ARG


def ws(lib, entry, p, C=0, k=0):
    return lib.tp_workspace_size(entry.encode(), ctypes.byref(p), C, k)


def test_workspace_sizes_from_shapes(lib):
    big = ctypes.c_size_t(-1).value
    p2 = pairs(8192, 8192, 64)
    a = ws(lib, "pairwise_logsumexp", p2)
    assert 0 < a < (1 << 30) and a % 256 == 0
    assert ws(lib, "pairwise_logsumexp", p2) == a  # deterministic
    assert ws(lib, "pairwise_logsumexp_backward", p2) >= a
    # a streamed set of one tile needs no split, hence no workspace
    assert ws(lib, "pairwise_matmul", pairs(100, 20, 3), C=4) == 0
    assert ws(lib, "pairwise_topk", pairs(1000, 5000, 16), k=16) > 0
    assert ws(lib, "pairwise_topk", pairs(1000, 5000, 16), k=0) == big
    assert ws(lib, "pairwise_matmul", pairs(), C=65) == big
    assert ws(lib, "no_such_entry", pairs()) == big
    assert ws(lib, "pairwise_matmul", pairs(D=65), C=4) == big
    # fp64 partial states are twice the fp32 ones (D = 32: no tensor-core path)
    a32 = ws(lib, "pairwise_logsumexp", pairs(8192, 8192, 32))
    assert ws(lib, "pairwise_logsumexp", pairs(8192, 8192, 32, _lib.TP_F64)) >= 2 * a32 - 512
    # fp32, D = 64: room for the tensor-core path's fp16 hi/lo split (256 bytes per distinct point)
    assert a >= 2 * 8192 * 256
    # Y = X: one split, plus the triangle sweep's column partials (2 KB per tile of the upper triangle of
    # 64 x 64 tiles of 128 points)
    same = ws(lib, "pairwise_logsumexp", pairs(8192, 8192, 64, X=FAKE, Y=FAKE))
    tri = 64 * 65 // 2 * 128 * 4 * 4
    assert 8192 * 256 + tri <= same and same - tri < a


def call_matmul(lib, p, s, V=FAKE + 0x200000, C=4, out=FAKE + 0x300000, w=None, n=0):
    return lib.tp_pairwise_matmul(ctypes.byref(p) if p is not None else None, ctypes.byref(s), V, C, out, w, n,
                                  None)


@pytest.mark.parametrize("case", ["null_pairs", "D0", "D65", "C0", "C65", "N0", "dtype", "metric", "unaligned",
                                  "alias_out_X", "ws_small"])
def test_invalid_arguments_rejected(lib, case):
    p, s, kw = pairs(), score(), {}
    if case == "null_pairs":
        p = None
    elif case == "D0":
        p = pairs(D=0)
    elif case == "D65":
        p = pairs(D=65)
    elif case == "C0":
        kw["C"] = 0
    elif case == "C65":
        kw["C"] = 65
    elif case == "N0":
        p = pairs(N=0)
    elif case == "dtype":
        p = pairs(dtype=7)
    elif case == "metric":
        s = score(metric=9)
    elif case == "unaligned":
        p = pairs(X=FAKE + 2)
    elif case == "alias_out_X":
        kw["out"] = FAKE + 8
    elif case == "ws_small":
        p = pairs(N=100, M=5000, D=3)
        kw["w"], kw["n"] = FAKE + 0x400000, 16
    assert call_matmul(lib, p, s, **kw) == _lib.TP_ERR_INVALID_ARG
    assert lib.tp_last_error()


@pytest.mark.parametrize("case,msg", [("unknown", "unknown pair mask"), ("negative_band", "band must be >= 0"),
                                      ("no_groups", "needs row_group and col_group"),
                                      ("unaligned_groups", "not aligned to 4 bytes")])
def test_pair_mask_arguments_rejected(lib, case, msg):
    # the pair-mask fields of the score are checked on the host before anything is launched
    s = score()
    if case == "unknown":
        s.pair_mask = 7
    elif case == "negative_band":
        s.pair_mask, s.band = _lib.PAIR_MASKS["band"], -1
    elif case == "no_groups":
        s.pair_mask, s.row_group = _lib.PAIR_MASKS["same_group"], FAKE + 0x700000
    else:
        s.pair_mask = _lib.PAIR_MASKS["same_group"]
        s.row_group, s.col_group = FAKE + 0x700000, FAKE + 0x710002
    p = pairs(N=12, M=12, D=64)
    assert call_matmul(lib, p, s) == _lib.TP_ERR_INVALID_ARG
    assert msg in lib.tp_last_error().decode()
    assert lib.tp_pairwise_softmax_matmul(ctypes.byref(p), ctypes.byref(s), FAKE + 0x200000, 64, FAKE + 0x300000,
                                          FAKE + 0x380000, None, 0, None) == _lib.TP_ERR_INVALID_ARG
    assert msg in lib.tp_last_error().decode()


def test_other_entries_reject(lib):
    p = pairs(N=10, M=12)
    s = score()
    # exclude_self needs N == M
    assert lib.tp_pairwise_logsumexp(ctypes.byref(p), ctypes.byref(s), 1, FAKE + 0x300000, None, 0, None) == \
        _lib.TP_ERR_INVALID_ARG
    # k out of range
    for k in (0, 13, 200):
        assert lib.tp_pairwise_topk(ctypes.byref(p), ctypes.byref(s), k, 0, FAKE + 0x300000, FAKE + 0x380000, None,
                                    0, None) == _lib.TP_ERR_INVALID_ARG
    # k above the compiled list length: unsupported, not invalid
    pbig = pairs(N=10, M=500)
    assert lib.tp_pairwise_topk(ctypes.byref(pbig), ctypes.byref(s), 64, 0, FAKE + 0x300000, FAKE + 0x380000, None,
                                0, None) == _lib.TP_ERR_UNSUPPORTED
    # dX and dY may only coincide when X and Y are the same points
    g = FAKE + 0x500000
    assert lib.tp_pairwise_logsumexp_backward(ctypes.byref(pairs(N=12, M=12)), ctypes.byref(s), 0, FAKE + 0x300000,
                                              FAKE + 0x310000, g, g, None, None, None, None, None, 0, None) == \
        _lib.TP_ERR_INVALID_ARG
    # a parameter gradient for a parameter the score does not have
    assert lib.tp_pairwise_logsumexp_backward(ctypes.byref(pairs(N=12, M=12)), ctypes.byref(s), 0, FAKE + 0x300000,
                                              FAKE + 0x310000, g, None, FAKE + 0x600000, None, None, None, None, 0,
                                              None) == _lib.TP_ERR_INVALID_ARG
    # outputs overlapping each other
    assert lib.tp_pairwise_softmax_matmul(ctypes.byref(p), ctypes.byref(s), FAKE + 0x200000, 4, FAKE + 0x300000,
                                          FAKE + 0x300010, None, 0, None) == _lib.TP_ERR_INVALID_ARG


def test_product_path_has_no_fallback():
    """The package refuses CPU tensors instead of computing on the host."""
    import torch

    import lazy_score_matrix_gb300 as tp
    x = torch.randn(4, 3)
    with pytest.raises((ValueError, ImportError)):
        tp.lazy(x, x, "linear").logsumexp(-1)


def test_package_does_not_import_the_oracle():
    import pathlib
    import re
    pkg = pathlib.Path(_lib.PKG)
    for f in list(pkg.glob("*.py")) + list(pkg.glob("csrc/*")):
        text = f.read_text()
        assert not re.search(r"^\s*(from|import)\s+oracle", text, flags=re.M), f
        assert "tp_oracle" not in text and "or_matmul" not in text, f


def test_fault_injection_fails_the_named_entry_before_launch(lib, monkeypatch):
    """TP_FAULT_INJECT=<entry>: that entry validates its arguments, then returns TP_ERR_CUDA without
    launching anything (the fake device addresses are never touched); invalid arguments still win."""
    p = pairs(10, 10, 3)
    sc = score()
    monkeypatch.setenv("TP_FAULT_INJECT", "pairwise_logsumexp")
    _lib.launch_count(reset=True)
    st = lib.tp_pairwise_logsumexp(ctypes.byref(p), ctypes.byref(sc), 0, FAKE + 0x200000, None, 0, None)
    assert st == _lib.TP_ERR_CUDA
    assert b"fault injected" in lib.tp_last_error()
    assert _lib.launch_count() == 0
    # validation runs first: a NULL output is still an invalid argument
    assert lib.tp_pairwise_logsumexp(ctypes.byref(p), ctypes.byref(sc), 0, None, None, 0, None) == \
        _lib.TP_ERR_INVALID_ARG
    # the no-alloc entry point goes through the same entry (the shape needs no scratch here)
    st = lib.tp_pairwise_logsumexp_noalloc(ctypes.byref(p), ctypes.byref(sc), 0, FAKE + 0x200000, None)
    assert st == _lib.TP_ERR_CUDA and b"fault injected" in lib.tp_last_error()
    for name, call in (
            ("pairwise_matmul", lambda: lib.tp_pairwise_matmul(ctypes.byref(p), ctypes.byref(sc), FAKE + 0x300000, 4,
                                                               FAKE + 0x400000, None, 0, None)),
            ("pairwise_topk", lambda: lib.tp_pairwise_topk(ctypes.byref(p), ctypes.byref(sc), 3, 0, FAKE + 0x300000,
                                                           FAKE + 0x400000, FAKE + 0x1000000, 1 << 30, None))):
        monkeypatch.setenv("TP_FAULT_INJECT", name)
        assert call() == _lib.TP_ERR_CUDA, name
        assert b"fault injected" in lib.tp_last_error()
    assert _lib.launch_count() == 0


def test_selftest_limit_is_checked_on_the_host(lib):
    assert lib.tp_selftest_bounded_wait(0, None) == _lib.TP_ERR_INVALID_ARG
    assert lib.tp_selftest_bounded_wait(3 * 10 ** 9, None) == _lib.TP_ERR_INVALID_ARG


def test_noalloc_rejects_problems_beyond_its_fixed_array(lib):
    """The no-alloc entry point checks the scratch it needs against its fixed 16 MiB before anything
    else: fp32 D = 64 beyond N = 54542 with Y the same array is rejected with a message, on the host."""
    lim = 16 << 20
    for N, same in ((54542, True), (54543, True), (30000, False)):
        p = pairs(N, N, 64, X=FAKE, Y=FAKE if same else FAKE + (1 << 36))
        need = ws(lib, "pairwise_logsumexp", p)
        assert (need <= lim) == (N == 54542), (N, same, need)
    for N, same in ((54543, True), (30000, False)):
        p = pairs(N, N, 64, X=FAKE, Y=FAKE if same else FAKE + (1 << 36))
        st = lib.tp_pairwise_logsumexp_noalloc(ctypes.byref(p), ctypes.byref(score()), 1, FAKE + (1 << 37), None)
        assert st == _lib.TP_ERR_INVALID_ARG
        assert b"fixed array" in lib.tp_last_error()
    # any other shape fits: the streamed path needs at most 2 MiB
    for D, dt in ((32, _lib.TP_F32), (64, _lib.TP_F64), (3, _lib.TP_F64)):
        for N in (1000, 65536, 10 ** 6):
            assert ws(lib, "pairwise_logsumexp", pairs(N, 10 ** 6, D, dtype=dt)) <= 2 << 20


def test_exp64_table_is_correctly_rounded():
    """The 64-entry table 2^(j/64) of the fp64 exp (csrc/tp_device.cuh), recomputed here in 60-digit
    decimal arithmetic (ln 2 from its series, exp from its series) and rounded to the nearest double."""
    import os
    import re
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    src = open(os.path.join(os.path.dirname(_lib.PKG), "lazy_score_matrix_gb300", "csrc", "tp_device.cuh")).read()
    body = src[src.index("kExp2Tab64[64] = {"):]
    body = body[body.index("{") + 1:body.index("};")]
    tab = [float.fromhex(v) for v in re.findall(r"0x[0-9a-f.]+p[+-]\d+", body)]
    assert len(tab) == 64
    ln2 = sum(Decimal(1) / (k * Decimal(2) ** k) for k in range(1, 400))

    def dexp(x):
        s, t = Decimal(1), Decimal(1)
        for k in range(1, 120):
            t = t * x / k
            s += t
        return s

    for j, v in enumerate(tab):
        exact = dexp(ln2 * j / 64)
        assert v == float(exact), j
        # correctly rounded: no double is closer
        import math
        assert abs(Decimal(v) - exact) <= Decimal(math.ulp(v)) / 2, j
