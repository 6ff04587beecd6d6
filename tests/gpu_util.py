"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Model, Session, desc_of
from conftest import oracle_models
from oracle import dflash_oracle as O

# Tolerances: max-abs on float outputs, and the top-2 gap below which either
# greedy token is accepted.
TOL = {"f32": 1e-4, "bf16": 2e-2}
GAP = {"f32": 1e-4, "bf16": 1e-2}

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


def check_tokens(gpu, ref, gap, dtype, what):
    """Greedy tokens must agree wherever the oracle's top-2 gap exceeds the
    near-tie bound; returns the number of exempted positions."""
    gpu, ref, gap = np.asarray(gpu), np.asarray(ref), np.asarray(gap)
    bad = (gpu != ref) & (gap > GAP[dtype])
    assert not bad.any(), f"{what}: mismatch at {np.nonzero(bad)[0][:10]} (gaps {gap[bad][:5]})"
    return int(((gpu != ref) & ~bad).sum())


def assert_close(gpu, ref, dtype, what, tol=None):
    gpu, ref = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    err = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    t = TOL[dtype] if tol is None else tol
    assert err <= t, f"{what}: max-abs {err:.3e} > {t:.1e}"
    return err


def oracle_logits_along(tg, prompt, stream, rnd):
    """Oracle greedy tokens and gaps for every emitted position, given the
    prefix the GPU actually produced (one causal forward over prompt+stream)."""
    seq = np.concatenate([prompt, stream[:-1]]).astype(np.int64)
    sh = tg.shape
    out = O.target_forward(tg, seq, O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim), rnd, keep_logits=False)
    P0 = len(prompt)
    return out.argmax[P0 - 1:], out.gap[P0 - 1:]


__all__ = ["Model", "Session", "desc_of", "capi", "synth", "O"]
