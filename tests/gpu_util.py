"""Shared helpers of the GPU parity tests (comparison and tolerances).

Tolerances are the stated acceptance bar for bf16 inputs with fp32
accumulation: max |O - O_oracle| <= 2e-2 and max |L - L_oracle| <= 1e-3.
"""
import numpy as np

O_TOL = 2e-2
L_TOL = 1e-3


def compare(name, O_gpu, L_gpu, O_ref, L_ref, o_tol=O_TOL, l_tol=L_TOL):
    """Element-wise check; -inf in the reference L must be matched exactly."""
    O_gpu = np.asarray(O_gpu, dtype=np.float64)
    O_ref = np.asarray(O_ref, dtype=np.float64)
    assert O_gpu.shape == O_ref.shape, (name, O_gpu.shape, O_ref.shape)
    assert np.all(np.isfinite(O_gpu)), f"{name}: non-finite O"
    eo = np.abs(O_gpu - O_ref)
    worst = np.unravel_index(np.argmax(eo), eo.shape) if eo.size else None
    msg = f"{name}: max|dO| = {eo.max() if eo.size else 0:.3e} at {worst}, mean {eo.mean() if eo.size else 0:.2e}"
    assert (eo.max() if eo.size else 0.0) <= o_tol, msg
    if L_gpu is not None:
        L_gpu = np.asarray(L_gpu, dtype=np.float64)
        L_ref = np.asarray(L_ref, dtype=np.float64)
        ninf = np.isneginf(L_ref)
        assert np.array_equal(np.isneginf(L_gpu), ninf), f"{name}: -inf rows of L differ"
        fin = ~ninf
        assert np.all(np.isfinite(L_gpu[fin])), f"{name}: non-finite L"
        el = np.abs(L_gpu[fin] - L_ref[fin])
        assert (el.max() if el.size else 0.0) <= l_tol, f"{name}: max|dL| = {el.max():.3e}"
    return float(eo.max()) if eo.size else 0.0
