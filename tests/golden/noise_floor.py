"""The bf16 noise floor at the benchmarked widths, measured with the oracle alone.

Two emulations of the same bf16 computation that round at exactly the same
points (the oracle's ``Rounder("bf16")``) and differ only in the precision of
their matrix products -- float64 products against float32-accumulated
products -- are both correct implementations of the method.  Where they
disagree, no bound tighter than their disagreement can be met by an
implementation that accumulates in float32, as the GPU does.  This module
measures that disagreement for every output the full-width GPU parity tests
compare, at the widths of the benchmarked workloads:

  verify : a causal target forward of one block (16 or 15 tokens) over a
           seeded synthetic 4096-position cache through 6 target layers
           (the fewest that hold the 5 capture points), the LM head and the
           argmax -- logits, top-2 gaps, captured states, each layer's keys
           and values;
  draft  : the non-causal drafter forward of one block through the full 5
           drafter layers over a seeded synthetic 4096-position injected
           context -- logits and top-2 gaps of slots 1..B-1.

``python tests/golden/noise_floor.py`` writes ``noise_floor.json`` beside it,
which ``tests/tolerances.py`` reads.  Only ``oracle/`` and ``synth`` (seeded
draws) are called.
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402

FLOOR_JSON = os.path.join(HERE, "noise_floor.json")
CTX = 4096          # synthetic context of the measurement
N_TARGET_LAYERS = 6
SEED = 64           # synthetic cache and token draws


def _f32_linear(x, w):
    """The same product with float32 inputs (exact: they are bf16 values) and
    float32 accumulation."""
    return (np.asarray(x, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)


def _models(wl: synth.Workload, n_layers: int):
    """Oracle target (n_layers) and drafter at the workload's widths.  Weights
    are seeded N(0, 0.02) bf16 values drawn per canonical name; the embedding
    table holds only the rows the measurement uses (row 0: anchor, row 1:
    mask, rows 2..: block tokens)."""
    t = wl.target
    specs = synth.weight_specs(t, wl.draft_layers)
    idx = synth.spec_index(specs)

    def get(name):
        i = idx[name]
        return synth.host_tensor(i, specs[i][1], specs[i][2], "bf16")

    def layers(prefix, n):
        return [O.Layer(*(get(f"{prefix}{i}.{p}") for p in synth.LAYER_PARTS)) for i in range(n)]

    emb = synth.to_bf16_f32(synth.gaussian((2 + wl.block, t.hidden), seed=SEED, stream=900, scale=synth.INIT_STD))
    sh = O.Shape(n_layers, t.hidden, t.n_q, t.n_kv, t.head_dim, t.ffn, t.vocab, t.rope_theta, t.eps)
    dsh = O.Shape(wl.draft_layers, t.hidden, t.n_q, t.n_kv, t.head_dim, t.ffn, t.vocab, t.rope_theta, t.eps)
    lm = get("lm_head")
    tg = O.Target(sh, emb, layers("layers.", n_layers), get("final_norm"), lm, tuple(O.layer_indices(n_layers)))
    dr = O.Draft(dsh, get("draft.w_fc"), get("draft.fc_norm"), layers("draft.layers.", wl.draft_layers),
                 get("draft.final_norm"), 1)
    return tg, dr


def _cache(n_layers, sh, stream0):
    kv = O.KV.empty(n_layers, sh.n_kv, sh.head_dim)
    for li in range(n_layers):
        kv.k[li] = synth.to_bf16_f32(synth.gaussian((sh.n_kv, CTX, sh.head_dim), seed=SEED,
                                                    stream=stream0 + 2 * li)).astype(np.float64)
        kv.v[li] = synth.to_bf16_f32(synth.gaussian((sh.n_kv, CTX, sh.head_dim), seed=SEED,
                                                    stream=stream0 + 2 * li + 1)).astype(np.float64)
    return kv


def _diff(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    d = a - b
    rms = float(np.sqrt(np.mean(a * a)))
    return {"max_abs": float(np.max(np.abs(d))), "rel_fro": float(np.linalg.norm(d) / max(np.linalg.norm(a), 1e-300)),
            "max_abs_over_rms": float(np.max(np.abs(d)) / max(rms, 1e-300)), "rms": rms,
            "frac_differ": float(np.mean(a != b))}


def _tokens(am_a, gap_a, am_b, gap_b):
    """Largest gap (of either emulation) at which the two greedy choices differ,
    and the largest change of a top-2 gap."""
    differ = am_a != am_b
    worst = float(np.max(np.maximum(gap_a, gap_b)[differ])) if differ.any() else 0.0
    return {"differ": int(differ.sum()), "max_gap_where_differ": worst,
            "max_gap_change": float(np.max(np.abs(gap_a - gap_b)))}


def measure(wl: synth.Workload, what=("verify", "draft")) -> dict:
    """Floors of one workload's widths (see the module docstring)."""
    tg, dr = _models(wl, N_TARGET_LAYERS)
    rnd = O.Rounder("bf16")
    out = {"workload": wl.name, "hidden": wl.target.hidden, "heads": [wl.target.n_q, wl.target.n_kv],
           "ffn": wl.target.ffn, "vocab": wl.target.vocab, "block": wl.block, "context": CTX,
           "target_layers": N_TARGET_LAYERS, "draft_layers": wl.draft_layers}
    lin = O.linear
    try:
        if "verify" in what:
            kv = _cache(N_TARGET_LAYERS, tg.shape, 0)
            toks = np.arange(2, 2 + wl.block)
            runs = []
            for f in (lin, _f32_linear):
                O.linear = f
                runs.append(O.target_forward(tg, toks, kv, rnd))
            a, b = runs
            v = {"logits": _diff(a.logits, b.logits), "hcap": _diff(a.hcap, b.hcap),
                 "tokens": _tokens(a.argmax, a.gap, b.argmax, b.gap)}
            for li in range(N_TARGET_LAYERS):
                v[f"k{li}"] = _diff(a.new_k[li], b.new_k[li])
                v[f"v{li}"] = _diff(a.new_v[li], b.new_v[li])
            out["verify"] = v
        if "draft" in what:
            kv = _cache(wl.draft_layers, dr.shape, 1000)
            runs = []
            for f in (lin, _f32_linear):
                O.linear = f
                runs.append(O.draft_logits(dr, tg, 0, wl.block, kv, rnd))
            a, b = runs
            am_a, gap_a = O.argmax_top2(a)
            am_b, gap_b = O.argmax_top2(b)
            out["draft"] = {"logits": _diff(a, b), "tokens": _tokens(am_a, gap_a, am_b, gap_b)}
    finally:
        O.linear = lin
    return out


WIDTHS = ("small-bf16-gqa4", "small-bf16-gqa5", "qwen3-8b-4k", "dense27b-36k")


def main():
    res = {"what": "bf16 noise floor: oracle with float64 products vs the same oracle with float32-accumulated "
                   "products, identical rounding points; written by tests/golden/noise_floor.py",
           "floors": {}}
    for name in WIDTHS:
        t0 = time.time()
        res["floors"][name] = measure(synth.WORKLOADS[name])
        print(f"{name}: {time.time() - t0:.0f} s", flush=True)
    with open(FLOOR_JSON, "w") as f:
        json.dump(res, f, indent=1, sort_keys=True)
        f.write("\n")
    print(FLOOR_JSON)


if __name__ == "__main__":
    main()
