"""Numerical bounds of the parity tests (no GPU imports)."""
import numpy as np

# Tolerances: max-abs on float outputs, and the top-2 gap below which either
# greedy token is accepted.
TOL = {"f32": 1e-4, "bf16": 2e-2}
GAP = {"f32": 1e-4, "bf16": 1e-2}
# The top-2 gap is the difference of two logits, each within TOL, and both the
# largest and the second-largest logit move by at most max|dlogit|: the gap's
# bound is twice the logit bound.
GAP_TOL = {k: 2 * v for k, v in TOL.items()}

# Outputs that pass through several bf16 rounding points (a stack of layers)
# differ from the oracle by the bf16 noise floor rather than by one rounding:
# a fraction f of elements flipped by one ulp at one rounding point, fed
# through a linear layer of fan-in K, perturbs its outputs by about
# sqrt(f) * 2^-8 relative, which flips a fraction ~sqrt(f) at the next
# rounding point, so after a few points most elements sit one ulp apart.  The
# bounds: relative Frobenius error <= 2^-6 (a few ulps rms) and max-abs <=
# 2^-4 * rms(ref).
STACK_FRO = 2.0 ** -6
STACK_PEAK = 2.0 ** -4


def stack_error(got, ref):
    """(relative Frobenius error, max-abs error / rms(ref)) of got against ref."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    d = got - ref
    fro = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))
    rms = float(np.sqrt(np.mean(ref * ref)))
    return fro, float(np.max(np.abs(d)) / max(rms, 1e-300))
