"""Shared test helpers: the error measure the tolerances are stated in, and array conversion."""
import os

import numpy as np

# Tolerances (max relative error, see rel_err): fp32 forward, fp32 gradients, fp64 anything.
TOL_F32_FWD = 1e-4
TOL_F32_GRAD = 5e-4
TOL_F64 = 1e-10


def to_np(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        return t.detach().double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


# Floor of the relative error, as a fraction of the tensor's largest magnitude.
FLOOR = 1e-3


def rel_err(got, want, floor_frac=FLOOR, abs_floor=0.0):
    """max_e |got_e - want_e| / (|want_e| + floor): elementwise relative error with a floor of
    floor_frac of the tensor's largest magnitude (or abs_floor if larger), so entries that cancel to
    ~0 do not dominate."""
    g, w = to_np(got), to_np(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    if w.size == 0:
        return 0.0
    fin = np.isfinite(w)
    assert (np.isfinite(g) == fin).all(), "non-finite pattern differs"
    assert (g[~fin] == w[~fin]).all(), "infinite entries differ"
    if not fin.any():
        return 0.0
    g, w = g[fin], w[fin]
    floor = max(floor_frac * np.abs(w).max(), abs_floor)
    if floor == 0:
        return float(np.abs(g - w).max())
    return float((np.abs(g - w) / (np.abs(w) + floor)).max())


def other_errors(got, want):
    """The two measures reported beside rel_err when a check fails: the normwise error |a - b| / |b| over
    the finite entries and the elementwise relative error without a floor."""
    g, w = to_np(got), to_np(want)
    fin = np.isfinite(w) & np.isfinite(g)
    g, w = g[fin], w[fin]
    nw = float(np.linalg.norm(g - w) / np.linalg.norm(w)) if np.linalg.norm(w) > 0 else float(np.abs(g).max(initial=0))
    with np.errstate(divide="ignore", invalid="ignore"):
        ew = np.where(w != 0, np.abs(g - w) / np.abs(w), np.where(g == w, 0.0, np.inf))
    return nw, float(ew.max(initial=0.0))


def assert_close(got, want, tol, what="", floor_frac=FLOOR, abs_floor=0.0):
    e = rel_err(got, want, floor_frac, abs_floor)
    log = os.environ.get("TP_TEST_ERROR_LOG")
    if log:  # one line per check: the error and the bound it was held to (for reviewing the margins)
        with open(log, "a") as f:
            f.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '?').split(' ')[0]}\t{what}\t{e:.4g}\t{tol:.4g}\n")
    if e > tol:
        nw, ew = other_errors(got, want)
        raise AssertionError(f"{what}: max relative error {e:.3g} > {tol:g} (normwise {nw:.3g}, elementwise "
                             f"without a floor {ew:.3g})")
    return e
