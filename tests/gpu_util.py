"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Model, Session, desc_of
from conftest import oracle_models
from oracle import dflash_oracle as O

from tolerances import GAP, GAP_TOL, STACK_FRO, STACK_PEAK, TOL, stack_error  # noqa: F401

_TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def dev():
    return torch.device("cuda:0")


def to_dev(a, dtype):
    return torch.as_tensor(np.ascontiguousarray(a)).to(device=dev(), dtype=_TDT[dtype] if isinstance(dtype, str)
                                                       else dtype)


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rounder(wl):
    return O.Rounder("bf16" if wl.dtype == "bf16" else "none")


def build_model(wl, weights=None):
    w = weights if weights is not None else synth.workload_weights(wl)
    m = Model(wl.target, wl.draft_layers, wl.dtype)
    m.load(w)
    tg, dr = oracle_models(wl, w)
    return m, tg, dr, w


def check_tokens(gpu, ref, gap, dtype, what, bound=None):
    """Greedy tokens must agree wherever the oracle's top-2 gap exceeds the
    near-tie bound (GAP, or ``bound``); returns the number of exempted
    positions."""
    gpu, ref, gap = np.asarray(gpu), np.asarray(ref), np.asarray(gap)
    bad = (gpu != ref) & (gap > (GAP[dtype] if bound is None else bound))
    assert not bad.any(), f"{what}: mismatch at {np.nonzero(bad)[0][:10]} (gaps {gap[bad][:5]})"
    return int(((gpu != ref) & ~bad).sum())


def check_tokens_vs_logits(gpu_tok, ref_tok, ref_gap, gpu_logits, ref_logits, dtype, what):
    """Greedy tokens against the oracle's, given both sides' logits: if the GPU
    picks b where the oracle picks a, then ref[a] - ref[b] <= 2 max|gpu - ref|
    over the row, so a row's tokens must agree wherever the oracle's top-2 gap
    exceeds max(GAP, 2 x that row's largest logit difference).  The logits
    themselves are bounded by a separate check.  Returns the number of rows
    exempted and the number whose tokens differ while the oracle's gap exceeds
    the stated GAP."""
    gpu_tok, ref_tok, ref_gap = np.asarray(gpu_tok), np.asarray(ref_tok), np.asarray(ref_gap)
    dl = np.max(np.abs(np.asarray(gpu_logits, np.float64) - np.asarray(ref_logits, np.float64)), axis=-1)
    bound = np.maximum(GAP[dtype], 2.0 * dl)
    differ = gpu_tok != ref_tok
    bad = differ & (ref_gap > bound)
    assert not bad.any(), f"{what}: mismatch at {np.nonzero(bad)[0][:10]} (gaps {ref_gap[bad][:5]}, bounds {bound[bad][:5]})"
    return int((differ & ~bad).sum()), int((differ & (ref_gap > GAP[dtype])).sum())


def assert_close(gpu, ref, dtype, what, tol=None):
    gpu, ref = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    err = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    t = TOL[dtype] if tol is None else tol
    assert err <= t, f"{what}: max-abs {err:.3e} > {t:.1e}"
    return err


def bf16_ulp(x):
    """Spacing of bfloat16 values at |x| (8 significant bits): 2^(e-7) for
    2^e <= |x| < 2^(e+1)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return np.exp2(e - 7)


def assert_close_rounded(gpu, ref, what, tol=TOL["bf16"]):
    """A single bf16 rounding of values that the two sides compute with
    different accumulation order: each element within the stated bound or
    within one bf16 ulp of the reference value, whichever is larger (two
    correct results a hair apart can round to adjacent bf16 values, and above
    |x| = 2.56 one ulp exceeds 2e-2)."""
    gpu, ref = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    d = np.abs(gpu - ref)
    bound = np.maximum(tol, bf16_ulp(ref))
    bad = d > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} values off by more than max({tol:.0e}, 1 ulp); worst {d.max():.3e}"
    return float(d.max()) if d.size else 0.0


def assert_close_stack(gpu, ref, what):
    """Stacked outputs: within the bf16 noise-floor bounds (tolerances.py)."""
    fro, peak = stack_error(gpu, ref)
    assert fro <= STACK_FRO and peak <= STACK_PEAK, \
        f"{what}: relative Frobenius {fro:.3e} (bound {STACK_FRO:.1e}), max-abs/rms {peak:.3e} (bound {STACK_PEAK:.1e})"
    return fro, peak


def oracle_logits_along(tg, prompt, stream, rnd):
    """Oracle greedy tokens and gaps for every emitted position, given the
    prefix the GPU actually produced (one causal forward over prompt+stream)."""
    seq = np.concatenate([prompt, stream[:-1]]).astype(np.int64)
    sh = tg.shape
    out = O.target_forward(tg, seq, O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim), rnd, keep_logits=False)
    P0 = len(prompt)
    return out.argmax[P0 - 1:], out.gap[P0 - 1:]


__all__ = ["Model", "Session", "desc_of", "capi", "synth", "O"]
