"""Shared test helpers: the error measure the tolerances are stated in, and array conversion."""
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


def rel_err(got, want):
    """max_e |got_e - want_e| / (|want_e| + 1e-3 * max|want|): elementwise relative error with a
    floor of 1e-3 of the tensor's largest magnitude, so entries that cancel to ~0 do not dominate."""
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
    floor = 1e-3 * np.abs(w).max()
    if floor == 0:
        return float(np.abs(g - w).max())
    return float((np.abs(g - w) / (np.abs(w) + floor)).max())


def assert_close(got, want, tol, what=""):
    e = rel_err(got, want)
    assert e <= tol, f"{what}: max relative error {e:.3g} > {tol:g}"
    return e
