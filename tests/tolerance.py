"""The acceptance bar for a GPU result against the fp64 oracle.

Per element: |Y - Y_ref| <= 1e-3 * sum_k |x w| + 1e-6, and per output tensor:
||Y - Y_ref||_2 / max(||Y_ref||_2, 1e-30) <= 1e-4.  The per-element bound
scales with the magnitude of the terms because fp32 accumulation error does;
relative L2 per destination tensor is the measure "ninfer-3080
docs/performance.md" (A8 prefill routes section) reports against its FP64
oracle.
"""
import numpy as np

ELEM_REL = 1e-3
ELEM_ABS = 1e-6
REL_L2 = 1e-4


def rel_l2(Y, Yref) -> float:
    return float(np.linalg.norm(Y - Yref) / max(np.linalg.norm(Yref), 1e-30))


def assert_close(Y, Yref, A, what: str = "") -> float:
    Y = np.asarray(Y, np.float64)
    assert Y.shape == Yref.shape, (what, Y.shape, Yref.shape)
    assert np.all(np.isfinite(Y)), f"{what}: non-finite output"
    err = np.abs(Y - Yref)
    bound = ELEM_REL * A + ELEM_ABS
    bad = err > bound
    if bad.any():
        t, n = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside the bound, first at t={t} n={n}: "
                             f"Y={Y[t, n]!r} ref={Yref[t, n]!r} bound={bound[t, n]!r}")
    r = rel_l2(Y, Yref)
    assert r <= REL_L2, f"{what}: relative L2 {r:.3e} > {REL_L2}"
    return r
