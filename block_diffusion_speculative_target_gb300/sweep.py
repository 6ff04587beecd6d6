"""Context/block sweep of the DFlash step on the Qwen3-8B shapes.

For each context length P0 the target and drafter caches are filled with
seeded N(0, 1) bf16 keys/values at positions 0..P0-1 (the step's cost does not
depend on the cached values, and a real prefill at 98K positions would
dominate the run), the greedy AR stream from that state is decoded on a copy
of the target cache, and then for each block size B the teacher-forced step
is captured in one CUDA graph and timed with CUDA events.  Per point: step
time, emitted tokens/s, per-stage time (eager, events between stages) and the
fraction of the HBM roofline (weights + keys/values read per step).

    python -m block_diffusion_speculative_target_gb300.sweep [--contexts 512 4096 ...] [--blocks 2 8 ...]

Prints one JSON object per point and a markdown table at the end."""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

import numpy as np
import torch

from . import capi
from .engine import Model, Session

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

STAGES = ("fuse", "inject", "draft", "teacher", "verify", "accept")


def build_model(wl, dev):
    m = Model(wl.target, wl.draft_layers, wl.dtype, device=dev)
    views = m.views()
    for i, (name, shape, kind) in enumerate(synth.weight_specs(wl.target, wl.draft_layers)):
        synth.fill_torch(views[name], i, kind)
    m.finalize()
    torch.cuda.synchronize()
    return m


def fill_cache(cache, n_layers, P, shape, seed):
    """Seeded N(0,1) bf16 keys/values at positions 0..P-1 of every layer."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    k = torch.empty(shape.n_kv, P, shape.head_dim, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    for li in range(n_layers):
        k.normal_(generator=g)
        v.normal_(generator=g)
        capi.dflash_cache_write(cache, li, 0, 0, P, k, v)
    capi.dflash_cache_set_lengths(cache, [P])


def step_bytes(shape, draft_layers, P, window=0, kv="bf16"):
    """Weights once (the injection's W_k/W_v are the drafter layers' own) plus
    the keys/values read: the target's over P positions (bf16, or with the
    8-bit cache one byte per entry plus a 4-byte scale per row), the
    drafter's over min(P, window) positions when a cross-context window is
    set."""
    d = shape.head_dim
    layer = 2 * (shape.hidden * (shape.n_q + 2 * shape.n_kv) * d + shape.n_q * d * shape.hidden
                 + 3 * shape.hidden * shape.ffn)
    lm = 2 * shape.vocab * shape.hidden
    fc = 2 * shape.hidden * 5 * shape.hidden
    Pd = min(P, window) if window > 0 else P
    tpos = 2 * shape.n_kv * (d + 4) if kv == "q8" else 2 * 2 * shape.n_kv * d
    kvb = shape.n_layers * P * tpos + draft_layers * Pd * 2 * 2 * shape.n_kv * d
    return shape.n_layers * layer + lm + draft_layers * layer + lm + fc + kvb


def run(contexts, blocks, steps, warmup, stage_passes, peak, window=0, kv="bf16"):
    wl = synth.WORKLOADS["qwen3-8b-4k"]
    s = wl.target
    dev = torch.device("cuda", 0)
    m = build_model(wl, dev)
    m.set_cross_ctx(window)
    tgc, drc = m.structs()
    Bmax = max(blocks)
    n_steps = 2 + warmup + steps + stage_passes
    n_ref = (n_steps + 2) * Bmax
    out = []
    for P0 in contexts:
        cap = P0 + n_ref + 64
        sess = Session(m, batch=1, capacity=cap, block=Bmax, stream_cap=n_ref + 8, kv_format=kv)
        fill_cache(sess.tcache, s.n_layers, P0, s, seed=100 + P0)
        fill_cache(sess.dcache, wl.draft_layers, P0, s, seed=200 + P0)
        anchor = int(synth.prompt_tokens(1, s.vocab, stream=P0)[0])
        sess.anchor.fill_(anchor)
        sess.stream[0, 0] = anchor
        sess.stream_len.fill_(1)
        sess.n_pend.zero_()
        ar = Session(m, batch=1, capacity=cap, block=Bmax, with_draft=False, stream_cap=n_ref + 8, kv_format=kv)
        ar.copy_target_from(sess)
        for _ in range(n_ref - 1):
            ar.ar_step()
        G = ar.emitted()[0]
        assert len(G) == n_ref and ar.status() == 0
        ar.close()
        for B in blocks:
            # back to the state after the synthetic prefill
            capi.dflash_cache_set_lengths(sess.tcache, [P0])
            capi.dflash_cache_set_lengths(sess.dcache, [P0])
            sess.anchor.fill_(anchor)
            sess.stream_len.fill_(1)
            sess.n_pend.zero_()
            sess.block = B
            k_draw, r_draw = synth.acceptance_draws(n_steps + 2, s.vocab)
            sess.set_teacher(G[None, :], k_draw, r_draw)
            sess.step(teacher=True)
            graph = sess.capture_graph(lambda: sess.step(teacher=True))
            for _ in range(warmup):
                graph.replay()
            len0 = int(sess.stream_len.item())
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
            torch.cuda.synchronize()
            evs[0].record()
            for i in range(steps):
                graph.replay()
                evs[i + 1].record()
            torch.cuda.synchronize()
            ms = statistics.median(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
            total = evs[0].elapsed_time(evs[steps]) / 1e3
            tokens = int(sess.stream_len.item()) - len0
            stage = {k: [] for k in STAGES}
            for _ in range(stage_passes):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
                ev[0].record()
                capi.dflash_fuse_features(drc, sess.hcap, B, sess.fused, sess.ws)
                ev[1].record()
                capi.dflash_inject_kv(drc, sess.fused, 1, B, sess.n_pend, sess.dcache, sess.ws)
                ev[2].record()
                capi.dflash_draft_block(drc, tgc, sess.anchor, 1, B, sess.dcache, sess.draft, sess.ws)
                ev[3].record()
                capi.dflash_teacher_force(sess.draft, 1, B, sess.ref, sess.ref.shape[1], sess.ref.shape[1],
                                          sess.stream_len, sess.k_draw, sess.r_draw, sess.k_draw.shape[0],
                                          sess.step_ctr, s.vocab, sess.ws)
                ev[4].record()
                capi.target_verify(tgc, sess.draft, 1, B, 0, sess.tcache, sess.argmax, sess.gap, sess.hcap, None,
                                   None, None, None, 0, sess.ws)
                ev[5].record()
                capi.dflash_accept_rollback(sess.draft, sess.argmax, 1, B, sess.tcache, sess.anchor, sess.n_pend,
                                            sess.accept_len, sess.stream, sess.stream_len, sess.stream_cap, sess.ws)
                ev[6].record()
                torch.cuda.synchronize()
                for j, k in enumerate(STAGES):
                    stage[k].append(ev[j].elapsed_time(ev[j + 1]))
            assert sess.status() == 0
            E = sess.emitted()[0]
            assert np.array_equal(E, G[:len(E)]), "speculative stream left the greedy stream"
            P_mid = P0 + 0.5 * (len0 + int(sess.stream_len.item())) - 1
            by = step_bytes(s, wl.draft_layers, P_mid, window, kv)
            rec = {"P0": P0, "block": B, "cross_ctx": window, "target_kv": kv, "ms_per_step": ms, "tokens_per_s": tokens / total, "tau": tokens / steps,
                   "bytes_per_step": by, "roofline_frac": by / (ms / 1e3) / (peak * 1e9),
                   "stage_ms": {k: statistics.median(v) for k, v in stage.items()}}
            print(json.dumps(rec), flush=True)
            out.append(rec)
            del graph
        sess.close()
    return out


def table(recs, peak):
    lines = [f"| P0 | B | ms/step | tok/s | tau | GB/step | % of {peak:.0f} GB/s | "
             + " | ".join(f"{k} ms" for k in STAGES) + " |",
             "|" + "---|" * (7 + len(STAGES))]
    for r in recs:
        lines.append(f"| {r['P0']} | {r['block']} | {r['ms_per_step']:.3f} | {r['tokens_per_s']:.0f} | {r['tau']:.2f} "
                     f"| {r['bytes_per_step'] / 1e9:.2f} | {100 * r['roofline_frac']:.1f} | "
                     + " | ".join(f"{r['stage_ms'][k]:.3f}" for k in STAGES) + " |")
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--contexts", type=int, nargs="+", default=[512, 4096, 12288, 36864, 98304])
    ap.add_argument("--blocks", type=int, nargs="+", default=[2, 8, 12, 15, 16])
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--stage-passes", type=int, default=2)
    ap.add_argument("--cross-ctx", type=int, default=0, help="the drafter's cross-context window (0: whole context)")
    ap.add_argument("--kv", choices=["bf16", "q8"], default="bf16", help="the target's K/V cache storage")
    args = ap.parse_args()
    capi.load()
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(p)).get("hbm_gbs", 6800.0) if os.path.exists(p) else 6800.0
    recs = run(args.contexts, args.blocks, args.steps, args.warmup, args.stage_passes, peak, args.cross_ctx, args.kv)
    print(table(recs, peak), flush=True)


if __name__ == "__main__":
    main()
