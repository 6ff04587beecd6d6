"""Numerical bounds of the parity tests (no GPU imports)."""
import json
import os

import numpy as np

# Stated bounds: max-abs on float outputs, and the top-2 gap below which either
# greedy token is accepted.
TOL = {"f32": 1e-4, "bf16": 2e-2}
GAP = {"f32": 1e-4, "bf16": 1e-2}
# The top-2 gap is the difference of two logits, each within TOL, and both the
# largest and the second-largest logit move by at most max|dlogit|: the gap's
# bound is twice the logit bound.
GAP_TOL = {k: 2 * v for k, v in TOL.items()}

# ---------------------------------------------------------------------------
# The bf16 noise floor at full width (tests/golden/noise_floor.json, written by
# tests/golden/noise_floor.py with the oracle alone).
#
# Two emulations that round to bf16 at the same points and differ only in
# float64 vs float32 accumulation of their products are both correct; their
# disagreement after a stack of layers is the floor below which no
# float32-accumulating implementation can be held.  At the benchmarked widths
# that floor exceeds the stated 2e-2 / 1e-2 on outputs of a layer stack
# (captured states, deep keys/values, logits, near-tie tokens).  For those
# outputs, and only where the floor exceeds the stated bound, the bound is
# FLOOR_MARGIN times the floor; everywhere else the stated bound holds.
# ---------------------------------------------------------------------------
FLOOR_MARGIN = 2.0
_FLOOR_JSON = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "noise_floor.json")
with open(_FLOOR_JSON) as _f:
    FLOORS = json.load(_f)["floors"]


def floor_of(workload, stage, output, stat="max_abs"):
    """The measured floor of one output (0 if the workload was not measured)."""
    return float(FLOORS.get(workload, {}).get(stage, {}).get(output, {}).get(stat, 0.0))


def floor_bound(workload, stage, output, stated, stat="max_abs"):
    """max(stated bound, FLOOR_MARGIN x the measured floor)."""
    return max(stated, FLOOR_MARGIN * floor_of(workload, stage, output, stat))


def token_gap_bound(workload, stage, dtype="bf16"):
    """Greedy tokens must agree where the oracle's top-2 gap exceeds this:
    the stated near-tie bound, or FLOOR_MARGIN x the largest top-2 gap change
    between the two emulations (a token can only flip where the gap is below
    the change)."""
    return max(GAP[dtype], FLOOR_MARGIN * floor_of(workload, stage, "tokens", "max_gap_change"))


# Outputs that pass through several bf16 rounding points at the small test
# widths: relative Frobenius error and max-abs relative to rms (used where a
# test compares a whole stacked tensor).
STACK_FRO = 2.0 ** -6
STACK_PEAK = 2.0 ** -4


def stack_error(got, ref):
    """(relative Frobenius error, max-abs error / rms(ref)) of got against ref."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    d = got - ref
    fro = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))
    rms = float(np.sqrt(np.mean(ref * ref)))
    return fro, float(np.max(np.abs(d)) / max(rms, 1e-300))
