"""Error metrics shared by the parity tests.

The contract's metric is err = max|y_gpu - y_oracle| / rms(y_oracle). Tolerances:
1e-5 for fp32 I/O and 2e-2 for bf16 I/O. A bf16 output cannot be closer to the exact
value than its own rounding (half a unit in the last place, at most 2^-8 |y|), and
for large heavy-tailed outputs that rounding alone can exceed 2e-2 * rms. So bf16
outputs are checked element by element against 2e-2 * rms(y_oracle) + 2^-8 |y_oracle|
(tolerance plus the output's own quantum), and the computation itself is checked at
the plain metric through the fp32-output variant of the same call.
"""
import numpy as np
import torch

TOL_F32 = 1e-5
TOL_BF16 = 2e-2
BF16_HALF_ULP_REL = 2.0 ** -8


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, np.float64)


def rms(a):
    a = to64(a)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def rel_err(gpu, ref):
    """max|gpu - ref| / rms(ref)."""
    g, r = to64(gpu), to64(ref)
    if r.size == 0:
        return 0.0
    s = rms(r)
    return float(np.max(np.abs(g - r)) / (s if s > 0 else 1.0))


def check(gpu, ref, tol, bf16_out=False, what=""):
    """Assert parity; returns the plain metric."""
    g, r = to64(gpu), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    e = rel_err(g, r)
    if bf16_out:
        bound = tol * rms(r) + BF16_HALF_ULP_REL * np.abs(r)
        bad = np.abs(g - r) > bound
        assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tol*rms + bf16 half-ulp (metric {e:.3g})"
    else:
        assert e <= tol, f"{what}: max|err|/rms = {e:.3g} > {tol}"
    return e
