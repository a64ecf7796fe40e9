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

# bf16 output: the fp32 result rounded to nearest bf16 (8 significant bits)
# moves by at most half an ulp, 2^-8 of its magnitude; relative L2 then
# stays below 2^-8 as well.
BF16_HALF_ULP = 2.0 ** -8
REL_L2_BF16 = 4e-3

# SwiGLU of a gate/up pair: g and u each within the bound above (e = 1e-3 A
# + 1e-6), silu(z) = z sigmoid(z) has |silu'| <= 1.1, and the fp32 silu and
# product add a few ulps (1e-6 relative):
#   |out - ref| <= 1.1 e_g (|u| + e_u) + |silu(g)| e_u + 1e-6 |ref| + 1e-6
SILU_LIPSCHITZ = 1.1


def rel_l2(Y, Yref) -> float:
    return float(np.linalg.norm(Y - Yref) / max(np.linalg.norm(Yref), 1e-30))


def assert_close(Y, Yref, A, what: str = "", bf16: bool = False) -> float:
    return _check(Y, Yref, ELEM_REL * A + ELEM_ABS, what, bf16)


def swiglu_bound(ref, g, u, Ag, Au):
    """Per-element bound of a SwiGLU output (see SILU_LIPSCHITZ above)."""
    eg = ELEM_REL * Ag + ELEM_ABS
    eu = ELEM_REL * Au + ELEM_ABS
    silu = g / (1.0 + np.exp(-np.clip(g, -700, 700)))
    return SILU_LIPSCHITZ * eg * (np.abs(u) + eu) + np.abs(silu) * eu + 1e-6 * np.abs(ref) + ELEM_ABS


def assert_close_swiglu(Y, ref, g, u, Ag, Au, what: str = "", bf16: bool = False) -> float:
    return _check(Y, ref, swiglu_bound(ref, g, u, Ag, Au), what, bf16)


def _check(Y, Yref, bound, what, bf16):
    Y = np.asarray(Y, np.float64)
    assert Y.shape == Yref.shape, (what, Y.shape, Yref.shape)
    assert np.all(np.isfinite(Y)), f"{what}: non-finite output"
    err = np.abs(Y - Yref)
    if bf16:
        bound = bound + BF16_HALF_ULP * (np.abs(Yref) + bound)
    bad = err > bound
    if bad.any():
        t, n = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside the bound, first at t={t} n={n}: "
                             f"Y={Y[t, n]!r} ref={Yref[t, n]!r} bound={bound[t, n]!r}")
    r = rel_l2(Y, Yref)
    lim = REL_L2_BF16 if bf16 else REL_L2
    assert r <= lim, f"{what}: relative L2 {r:.3e} > {lim}"
    return r
