#!/usr/bin/env python
"""Throughput of the DFlash speculative-decoding step on GB300.

One step = fuse + inject + draft (one non-causal drafter forward over the
block) + teacher forcing + verify (one causal target forward over the block)
+ accept/rollback, for a Qwen3-8B-shaped bf16 target (36 layers, hidden 4096,
32/8 heads x 128, FFN 12288, vocab 151936) with a 5-layer drafter, block 16,
after a 4096-token random prompt.  Random-init weights give ~0 natural
acceptance, so drafts are teacher-forced to the target's own greedy stream
with a geometric number of accepted tokens (mean 7): exactly min(k, 15)
drafts are accepted per step and the emitted stream stays the greedy one.

Prints one JSON line.  --impl reference times the CPU oracle instead (the
reference arm: a bounded sample of the same workload on the host cores).
Under torchrun each rank runs an independent replica (the step does not
shard); value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "emitted tokens/s per step (draft block+verify) at 4K/36K ctx; % of HBM roofline"
UNIT = "tokens/s"

# DRAM bytes (read + write) per gemm_cl_kernel launch, averaged over the 168
# weight-product launches of one step of the 4K workload: ncu
# (dram__bytes_read.sum + dram__bytes_write.sum, two launches per shape) on
# `kernel_bench gemm` for each of the step's seven product shapes, weighted by
# how often the step launches each (1 fusion, 1 injection, 41 each of QKV, O,
# gate/up and down, 2 LM heads).  None whenever the kernel has changed since
# the counters were taken.
GEMM_TRAFFIC = {"workload": "qwen3-8b-4k", "bytes_per_launch": 111515896}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3-8b-4k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="bound on the CPU-baseline sample")
    ap.add_argument("--also", nargs="*", default=["dense27b-36k", "dense27b-36k-q8"],
                    help="further workloads measured after the main one (one GPU only); empty to skip")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------


def layer_weight_bytes(s, es=2):
    d = s.head_dim
    return es * (s.hidden * (s.n_q + 2 * s.n_kv) * d + s.n_q * d * s.hidden + 3 * s.hidden * s.ffn)


def step_bytes(wl: synth.Workload, P_mean: float, batch=1):
    """Algorithmic bytes of one step: every weight matrix once plus the
    keys/values read, bf16.

    verify: every target layer + LM head; draft: every drafter layer + LM head;
    fuse: W_fc; attention: target and drafter keys+values for P positions (per
    sequence).  The injection projects with the drafter layers' own W_k/W_v,
    which the drafter layers already count, so it adds no bytes (the library
    streams a packed copy of them, which the roofline does not credit)."""
    s = wl.target
    Wl = layer_weight_bytes(s)
    lm = 2 * s.vocab * s.hidden
    fc = 2 * s.hidden * 5 * s.hidden
    weights = s.n_layers * Wl + lm + wl.draft_layers * Wl + lm + fc
    kv = batch * P_mean * (s.n_layers * kv_pos_bytes(wl, target=True) + wl.draft_layers * kv_pos_bytes(wl, False))
    return weights + kv, weights, kv


def kv_pos_bytes(wl: synth.Workload, target: bool):
    """Keys and values of one layer at one position: bf16, or (the target's
    8-bit cache) one byte per entry plus a float32 scale per row."""
    s = wl.target
    if target and wl.kv == "q8":
        return 2 * s.n_kv * (s.head_dim + 4)
    return 2 * 2 * s.n_kv * s.head_dim


def stage_bytes(wl: synth.Workload, P_mean: float, batch=1):
    """Algorithmic bytes of each stage of one step (the terms of step_bytes):
    fuse reads W_fc; inject nothing of its own (the drafter layers' W_k/W_v
    are counted with the draft stage); draft every drafter
    layer, the LM head and the drafter's keys/values; verify every target
    layer, the LM head and the target's keys/values.  Teacher forcing and
    accept move bytes per row only (counted 0)."""
    s = wl.target
    Wl = layer_weight_bytes(s)
    lm = 2 * s.vocab * s.hidden
    return {"fuse": 2 * s.hidden * 5 * s.hidden,
            "inject": 0,
            "draft": wl.draft_layers * Wl + lm + batch * wl.draft_layers * P_mean * kv_pos_bytes(wl, False),
            "teacher": 0,
            "verify": s.n_layers * Wl + lm + batch * s.n_layers * P_mean * kv_pos_bytes(wl, True), "accept": 0}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (barrier + max only; the data path has no collective)
# ---------------------------------------------------------------------------


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group("nccl" if self._cuda() else "gloo")
            self.pg = dist

    @staticmethod
    def _cuda():
        import torch

        return torch.cuda.is_available()

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device="cuda" if self._cuda() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device="cuda" if self._cuda() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(dist: Dist, units: float, seconds: float) -> float:
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    return dist.sum(units) / dist.max(seconds)


# ---------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------


def oracle_step_sample(wl: synth.Workload, seconds: float, tau: float, P: int, weights_dev=None, repeats=None,
                       batch=1):
    """Time the oracle on a bounded sample of one DFlash step at the workload's
    shapes: fusion + injection of B rows, one drafter layer and one target
    layer over a P-position synthetic context (B block rows), and one LM head
    (B rows).  The step time is extrapolated by layer count and, for a batch,
    by the number of sequences (the oracle runs them one after another):
        t_step = batch * (t_fuse + t_inject + Ld*t_dlayer + L*t_tlayer + 2*t_lmhead).
    ``tau`` is the emitted tokens per step of the whole batch.
    Returns (tokens/s, seconds per step, description, threads)."""
    from oracle import dflash_oracle as O

    s = wl.target
    B = wl.block
    rnd = O.Rounder("bf16" if wl.dtype == "bf16" else "none")
    specs = synth.weight_specs(s, wl.draft_layers)
    idx = synth.spec_index(specs)
    need = ["embed", "lm_head", "final_norm", "draft.w_fc", "draft.fc_norm"]
    need += [f"layers.0.{p}" for p in synth.LAYER_PARTS] + [f"draft.layers.0.{p}" for p in synth.LAYER_PARTS]
    w = {}
    for name in need:
        shape, kind = specs[idx[name]][1], specs[idx[name]][2]
        w[name] = _host_weight(name, idx[name], shape, kind, weights_dev)
    sh = O.Shape(1, s.hidden, s.n_q, s.n_kv, s.head_dim, s.ffn, s.vocab, s.rope_theta, s.eps)
    tl = O.Layer(*(w[f"layers.0.{p}"] for p in synth.LAYER_PARTS))
    dl = O.Layer(*(w[f"draft.layers.0.{p}"] for p in synth.LAYER_PARTS))
    dr = O.Draft(sh, w["draft.w_fc"], w["draft.fc_norm"], [dl], w["final_norm"], s.vocab - 1)
    rng = np.random.default_rng(5)
    hcap = O.round_bf16(rng.standard_normal((B, 5 * s.hidden)))
    ctx_k = O.round_bf16(rng.standard_normal((s.n_kv, P, s.head_dim)))
    ctx_v = O.round_bf16(rng.standard_normal((s.n_kv, P, s.head_dim)))
    x = rng.standard_normal((B, s.hidden))
    times = {"fuse": [], "inject": [], "dlayer": [], "tlayer": [], "lm": []}
    t_start = time.perf_counter()
    it = 0
    while True:
        t0 = time.perf_counter()
        f = O.fuse_features(dr, hcap, rnd)
        t1 = time.perf_counter()
        O.inject_kv(dr, f, np.arange(P, P + B), rnd)
        t2 = time.perf_counter()
        O.decoder_layer(x, dl, sh, ctx_k, ctx_v, P, False, rnd)
        t3 = time.perf_counter()
        O.decoder_layer(x, tl, sh, ctx_k, ctx_v, P, True, rnd)
        t4 = time.perf_counter()
        z = rnd(O.rmsnorm(x, w["final_norm"], s.eps))
        O.argmax_top2(O.linear(z, w["lm_head"]))
        t5 = time.perf_counter()
        for k, v in zip(times, (t1 - t0, t2 - t1, t3 - t2, t4 - t3, t5 - t4)):
            times[k].append(v)
        it += 1
        if repeats is not None and it >= repeats:
            break
        if repeats is None and time.perf_counter() - t_start >= seconds:
            break
    med = {k: statistics.median(v) for k, v in times.items()}
    t_seq = med["fuse"] + med["inject"] + wl.draft_layers * med["dlayer"] + s.n_layers * med["tlayer"] + 2 * med["lm"]
    t_step = batch * t_seq
    desc = (f"{it} sample(s) of: fuse+inject of {B} rows, 1 drafter + 1 target layer over a {P}-position context, "
            f"1 LM head; step time extrapolated to {wl.draft_layers} drafter + {s.n_layers} target layers + 2 LM heads"
            + (f" x {batch} sequences" if batch > 1 else "") + f" ({t_step:.2f} s/step), tokens/step = {tau:.2f}")
    return tau / t_step, t_step, desc, _blas_threads()


def _host_weight(name, index, shape, kind, weights_dev):
    if weights_dev is not None and name in weights_dev:
        return weights_dev[name].float().cpu().numpy()
    import torch

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    synth.fill_torch(t, index, kind)
    return t.float().cpu().numpy()


def _blas_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# ---------------------------------------------------------------------------
# reference arm
# ---------------------------------------------------------------------------


def timed_tau(wl: synth.Workload, steps: int, warmup: int, rank: int = 0) -> float:
    """Emitted tokens per step (summed over the batch) of the GPU arm's timed
    steps for the same --steps/--warmup: its first, eager step takes draw 0 and
    the warm-up replays draws 1..warmup, so the timed steps take the next
    `steps` draws; a step emits min(k, B - 1) + 1 tokens per sequence.  The
    reference arm divides by this, so both arms count the same tokens."""
    k, _ = synth.acceptance_draws(1 + warmup + steps, wl.target.vocab, batch=wl.batch,
                                  seed=synth.ACCEPT_SEED + rank)
    k = k[1 + warmup:]
    return float(np.mean(np.sum(np.minimum(k, wl.block - 1) + 1, axis=1)))


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    B = wl.block
    tau = timed_tau(wl, max(args.steps, 1), args.warmup)
    P = int(round(np.mean(synth.prompt_lengths(wl))))
    for _ in range(args.warmup):
        oracle_step_sample(wl, 0.0, tau, P, repeats=1, batch=wl.batch)
    t0 = time.perf_counter()
    vals = []
    desc = ""
    for _ in range(args.steps):
        v, t_step, desc, thr = oracle_step_sample(wl, 0.0, tau, P, repeats=1, batch=wl.batch)
        vals.append(t_step)
    wall = time.perf_counter() - t0
    t_step = statistics.median(vals)
    value = tau / t_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / max(args.steps, 1) * 1e3,
        "extrapolated_ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "block": B, "context": P, "target_layers": wl.target.n_layers,
                   "draft_layers": wl.draft_layers},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                         "extrapolated": True,
                         "sample": desc + f"; {args.steps} timed samples, wall {wall:.1f} s"},
        "extrapolated": True,
        "extrapolation": "value = tokens per step / extrapolated_ms_per_step, the layer-count extrapolation of "
                         "one timed sample per step to a whole step (see cpu_baseline.sample); ms_per_step is the "
                         "wall time actually timed per step (one sample)",
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def build_model(wl, device):
    import torch

    from block_diffusion_speculative_target_gb300.engine import Model

    m = Model(wl.target, wl.draft_layers, wl.dtype, device=device)
    specs = synth.weight_specs(wl.target, wl.draft_layers)
    views = m.views()
    for i, (name, shape, kind) in enumerate(specs):
        synth.fill_torch(views[name], i, kind)
    m.finalize()
    torch.cuda.synchronize()
    return m


def measure_ours(wl: synth.Workload, args, dist: Dist) -> dict:
    """Build the workload's model, prefill, decode the greedy reference stream,
    then time K teacher-forced steps replayed from one CUDA graph (device
    timing), the same steps with host buffers (e2e), and eager passes per
    stage and per weight product.  Returns the JSON line's fields; every
    device allocation is released before returning."""
    import torch

    from block_diffusion_speculative_target_gb300 import capi
    from block_diffusion_speculative_target_gb300.engine import Session

    dev = torch.device("cuda", dist.local)
    s = wl.target
    B, V, nb = wl.block, s.vocab, wl.batch
    lens0 = synth.prompt_lengths(wl)
    K, W, PS = args.steps, max(args.warmup, 3), args.profile_steps
    n_steps = 1 + W + K + K + 2 * PS + 2          # eager, warm-up, timed, e2e, profile passes, margin
    n_ref = 1 + n_steps * B + B
    cap = max(lens0) + n_ref + 64

    t_setup = time.perf_counter()
    m = build_model(wl, dev)
    prompts = [synth.prompt_tokens(P, V, stream=1000 * dist.rank + b) for b, P in enumerate(lens0)]

    # the speculative session: prefill (target forward over the prompts, fusion and injection)
    sess = Session(m, batch=nb, capacity=cap, block=B, stream_cap=n_ref + 8, kv_format=wl.kv)
    sess.prefill(prompts)
    torch.cuda.synchronize()
    t_prefill = time.perf_counter() - t_setup

    # greedy AR reference stream from the same committed state (and the plain
    # AR decode rate on this GPU)
    ar = Session(m, batch=nb, capacity=cap, block=B, with_draft=False, stream_cap=n_ref + 8, kv_format=wl.kv)
    ar.copy_target_from(sess)
    ar.ar_step()
    g_ar = ar.capture_graph(ar.ar_step)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n_ref - 2):
        g_ar.replay()
    e1.record()
    torch.cuda.synchronize()
    ar_tok_s = nb * (n_ref - 2) / (e0.elapsed_time(e1) / 1e3)
    G = ar.emitted()
    assert all(len(g) == n_ref for g in G) and ar.status() == 0
    ar.close()
    del g_ar

    k_draw, r_draw = synth.acceptance_draws(n_steps, V, batch=nb, seed=synth.ACCEPT_SEED + dist.rank)
    sess.set_teacher(np.stack(G), k_draw, r_draw)
    sess.step(teacher=True)                      # eager first step
    launches0 = capi.dflash_launch_count()
    graph = sess.capture_graph(lambda: sess.step(teacher=True))
    kernels_per_step = capi.dflash_launch_count() - launches0
    for _ in range(W):
        graph.replay()
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    # ---------------------------------------------------------------- timed region
    len0 = int(sess.stream_len.sum().item())
    P_before = sess.target_len()
    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.4)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    evs[0].record()
    for i in range(K):
        graph.replay()
        evs[i + 1].record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    dist.barrier()
    clk = clocks.stop()
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(K)]
    total_s = evs[0].elapsed_time(evs[K]) / 1e3
    tokens = int(sess.stream_len.sum().item()) - len0
    P_after = sess.target_len()
    assert sess.status() == 0, "device status set during the timed region"

    # ---------------------------------------------------------------- end to end (host buffers)
    pin_k = torch.from_numpy(k_draw.astype(np.int32)).pin_memory()
    pin_r = torch.from_numpy(r_draw.astype(np.int32)).pin_memory()
    # results come back into two pinned buffers: step i+1 is queued before the
    # host waits for step i's copy, as a serving loop streaming tokens one step
    # behind would do (the step itself needs nothing from the host)
    out_acc = [torch.zeros(nb, dtype=torch.int32).pin_memory() for _ in range(2)]
    out_tok = [torch.zeros(nb * B, dtype=torch.int32).pin_memory() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    st_host = int(sess.step_ctr.item())
    torch.cuda.synchronize()
    e2e_tokens = 0
    t_e2e = time.perf_counter()
    for i in range(K + 1):
        if i < K:
            si = st_host + i
            # this step's inputs from pinned host memory, its emitted tokens back
            sess.k_draw[si].copy_(pin_k[si], non_blocking=True)
            sess.r_draw[si].copy_(pin_r[si], non_blocking=True)
            graph.replay()
            out_acc[i % 2].copy_(sess.accept_len, non_blocking=True)
            out_tok[i % 2].copy_(sess.argmax[:nb * B], non_blocking=True)
            done[i % 2].record()
        if i >= 1:  # the previous step's results, read on the host
            done[(i - 1) % 2].synchronize()
            e2e_tokens += int(out_acc[(i - 1) % 2].sum()) + nb
    e2e_s = time.perf_counter() - t_e2e
    h2d = 2 * 4 * nb
    d2h = 4 * nb + 4 * nb * B

    # ---------------------------------------------------------------- kernel timing pass (eager)
    stage_ms = {k: [] for k in ("fuse", "inject", "draft", "teacher", "verify", "accept")}
    tgt, drc = m.structs()
    for _ in range(PS):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        rows = sess.batch * B
        ev[0].record()
        capi.dflash_fuse_features(drc, sess.hcap, rows, sess.fused, sess.ws)
        ev[1].record()
        capi.dflash_inject_kv(drc, sess.fused, sess.batch, B, sess.n_pend, sess.dcache, sess.ws)
        ev[2].record()
        capi.dflash_draft_block(drc, tgt, sess.anchor, sess.batch, B, sess.dcache, sess.draft, sess.ws)
        ev[3].record()
        capi.dflash_teacher_force(sess.draft, sess.batch, B, sess.ref, sess.ref.shape[1], sess.ref.shape[1],
                                  sess.stream_len, sess.k_draw, sess.r_draw, sess.k_draw.shape[0], sess.step_ctr, V,
                                  sess.ws)
        ev[4].record()
        capi.target_verify(tgt, sess.draft, sess.batch, B, 0, sess.tcache, sess.argmax, sess.gap, sess.hcap, None,
                           None, None, None, 0, sess.ws)
        ev[5].record()
        capi.dflash_accept_rollback(sess.draft, sess.argmax, sess.batch, B, sess.tcache, sess.anchor, sess.n_pend,
                                    sess.accept_len, sess.stream, sess.stream_len, sess.stream_cap, sess.ws)
        ev[6].record()
        torch.cuda.synchronize()
        for j, k in enumerate(stage_ms):
            stage_ms[k].append(ev[j].elapsed_time(ev[j + 1]))
    capi.dflash_profile_begin(4096)
    for _ in range(PS):
        sess.step(teacher=True)
    recs = capi.dflash_profile_end(4096)
    assert sess.status() == 0
    chains = [(ms, kb) for (ms, kind, rows, kb) in recs if kind == 1]
    gemm_bytes = sum(kb * 1024.0 for _, kb in chains)
    gemm_ms = sum(ms for ms, _ in chains)
    gemm_gbs = gemm_bytes / (gemm_ms / 1e3) / 1e9 if gemm_ms > 0 else None
    gemm_bytes_step = gemm_bytes / PS
    gemm_graph = products_graph_gbs(m, wl, B * nb, sess.ws, torch)

    # ---------------------------------------------------------------- results
    P_mean = 0.5 * (float(np.mean(P_before)) + float(np.mean(P_after)))
    bytes_step, w_bytes, kv_bytes = step_bytes(wl, P_mean, batch=nb)
    stage_med = {k: statistics.median(v) for k, v in stage_ms.items()}
    stage_by = stage_bytes(wl, P_mean, batch=nb)
    assert abs(sum(stage_by.values()) - bytes_step) < 1e-6 * bytes_step
    ms_step = statistics.median(step_ms)
    peak, peak_kind = measured_peaks()
    step_gbs = bytes_step / (ms_step / 1e3) / 1e9
    value = aggregate(dist, tokens, total_s)
    e2e_val = aggregate(dist, e2e_tokens, e2e_s)
    tau = tokens / K

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        try:
            views = m.views()
            need = {n: views[n] for n in ["embed", "lm_head", "final_norm", "draft.w_fc", "draft.fc_norm"]
                    + [f"layers.0.{p}" for p in synth.LAYER_PARTS]
                    + [f"draft.layers.0.{p}" for p in synth.LAYER_PARTS]}
            v, t_step, desc, thr = oracle_step_sample(wl, args.cpu_seconds, tau, int(round(np.mean(lens0))),
                                                      weights_dev=need, batch=nb)
            cpu = {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle", "extrapolated": True, "sample": desc}
        except Exception as e:  # the baseline is reported, never required
            cpu = {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"failed: {type(e).__name__}: {e}"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random-init weights N(0,0.02), uniform random prompt, teacher-forced acceptance)",
        "config": {"workload": wl.name, "batch": nb, "block": B,
                   "context": lens0[0] if nb == 1 else lens0, "context_mean_timed": P_mean,
                   "target_layers": s.n_layers, "draft_layers": wl.draft_layers, "hidden": s.hidden,
                   "vocab": V, "target_kv": wl.kv, "parallelism": f"replicas{dist.world}",
                   "l2": "inputs larger than L2 (weights+KV read per step >> 129 MB)", "graph": "one CUDA graph per step"},
        "tau": tau,
        "bytes_per_step": bytes_step, "weight_bytes_per_step": w_bytes, "kv_bytes_per_step": kv_bytes,
        "step_roofline": {"achieved_gbs": step_gbs, "peak_gbs": peak, "frac": step_gbs / peak, "peak_kind": peak_kind,
                          "frac_of_8tbs": step_gbs / 8000.0},
        "stage_ms": stage_med,
        "stage_gbs": {k: (stage_by[k] / (stage_med[k] / 1e3) / 1e9 if stage_by[k] and stage_med[k] > 0 else None)
                      for k in stage_med},
        "ar_tokens_per_s": ar_tok_s,
        "roofline": {"bound": "hbm", "kernel": "gemm_cl_kernel", "achieved": gemm_graph["gbs"], "peak": peak,
                     "unit": "GB/s", "frac": gemm_graph["gbs"] / peak,
                     "traffic": GEMM_TRAFFIC["bytes_per_launch"] if wl.name == GEMM_TRAFFIC["workload"] else None,
                     "algorithmic_bytes_per_launch": gemm_graph["bytes"] / gemm_graph["launches"],
                     "peak_kind": peak_kind, "timing": "graph",
                     "achieved_eager": gemm_gbs, "frac_eager": (gemm_gbs / peak) if gemm_gbs else None,
                     "frac_in_graph_lower_bound": gemm_bytes_step / (ms_step / 1e3) / 1e9 / peak,
                     "note": f"achieved = weight bytes per launch / the average launch duration of the step's "
                             f"{gemm_graph['launches']} weight products replayed back to back in one CUDA graph "
                             f"(CUDA events around the replay on its stream; the model's weights, a float-store "
                             f"epilogue): {gemm_graph['bytes'] / 1e9:.2f} GB in {gemm_graph['ms']:.3f} ms per "
                             f"replay. achieved_eager = the same bytes over {len(chains)} launches timed one by one "
                             f"with events around each in {PS} eager steps (no overlap with the neighbours: an upper "
                             f"bound on the kernel's time in the graph). frac_in_graph_lower_bound = the products' "
                             f"bytes per step / the whole graph-timed step. traffic = ncu DRAM read+write bytes per "
                             f"launch over the step's product shapes (null for other workloads)"},
        "clocks": clk,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(kernels_per_step * K),
        "kernels_per_step": int(kernels_per_step),
        "cpu_baseline": cpu,
        "setup_s": setup_s,
        "prefill_s": t_prefill,
    }
    sess.close()
    del graph, sess, m
    import gc

    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


# Keys of a second workload's measurement carried in the main line.
SUB_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "tau", "bytes_per_step", "step_roofline",
            "stage_ms", "stage_gbs", "roofline", "clocks", "e2e", "gpu_launches", "kernels_per_step", "cpu_baseline",
            "ar_tokens_per_s", "setup_s", "prefill_s")


def step_products(m, wl: synth.Workload):
    """(weight, M, K) of every weight product of one step in issue order: fusion, injection, the
    drafter's layers and LM head, the target's layers and LM head."""
    s = wl.target
    H, V = s.hidden, s.vocab
    out = [(m.w_fc, H, 5 * H), (m.w_kv_all, m.w_kv_all.shape[0], H)]
    for layers in (m.dlayers, None, m.layers, None):
        if layers is None:
            out.append((m.lm_head, V, H))
            continue
        for lw in layers:
            out += [(lw["wqkv"], lw["wqkv"].shape[0], H), (lw["wo"], H, lw["wo"].shape[1]),
                    (lw["w_gate_up"], lw["w_gate_up"].shape[0], H), (lw["w_down"], H, lw["w_down"].shape[1])]
    return out


def products_graph_gbs(m, wl: synth.Workload, rows, ws, torch, reps=20):
    """The step's weight products alone, back to back in one CUDA graph (the library's product kernel
    with a float-store epilogue, the model's own weights): their weight bytes over the graph-timed
    replay.  An in-graph figure for the product kernel, which the per-launch eager events overstate."""
    from block_diffusion_speculative_target_gb300 import capi

    prods = step_products(m, wl)
    dev = m.lm_head.device
    xs = {K: torch.zeros(rows, K, dtype=torch.bfloat16, device=dev) for _, _, K in prods}
    y = torch.empty(rows, max(M for _, M, _ in prods), dtype=torch.float32, device=dev)

    def run():
        for W, M, K in prods:
            capi.dflash_linear(capi.BF16, xs[K], W, y, rows, M, K, ws)

    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=st):
        run()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    wbytes = sum(W.numel() * W.element_size() for W, _, _ in prods)
    del g, xs, y
    return {"gbs": wbytes / (ms / 1e3) / 1e9, "ms": ms, "launches": len(prods), "bytes": wbytes}


def run_ours(args, dist: Dist):
    import torch

    from block_diffusion_speculative_target_gb300 import capi

    torch.cuda.set_device(dist.local)
    capi.load()
    line = measure_ours(synth.WORKLOADS[args.workload], args, dist)
    # the metric is quoted at 4K and 36K: one GPU also measures the 27B-class
    # shapes at a 36K context, after the first model has been released
    if dist.world == 1:
        for name in args.also:
            if name and name != args.workload:
                sub = measure_ours(synth.WORKLOADS[name], args, dist)
                line.setdefault("also", {})[name] = {k: sub[k] for k in SUB_KEYS if k in sub}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
