"""Host-side bookkeeping of bench.py: the algorithmic bytes a step reads and
the tokens per step the reference arm divides by.  CPU only."""
import importlib.util
import os

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_step_bytes_qwen3_8b_by_hand(bench):
    """Qwen3-8B shapes (H 4096, 32/8 heads of 128, FFN 12288, V 151936, 36 + 5
    layers): one decoder layer's bf16 weights are 2 (H (nq + 2 nkv) d + nq d H
    + 3 H F) = 385,875,968 B; a step reads 41 layers, the LM head twice and
    W_fc [H, 5H], plus K and V of every layer at every context position.  The
    injection's K/V projections are the drafter layers' own W_k/W_v, already
    counted once with those layers."""
    wl = synth.WORKLOADS["qwen3-8b-4k"]
    layer = 2 * (4096 * (32 + 2 * 8) * 128 + 32 * 128 * 4096 + 3 * 4096 * 12288)
    assert layer == 385_875_968
    lm = 2 * 151936 * 4096
    fc = 2 * 4096 * 5 * 4096
    weights = 41 * layer + 2 * lm + fc
    kv_per_pos = 41 * 2 * 2 * 8 * 128
    total, w, kv = bench.step_bytes(wl, 4096.0)
    assert w == weights == 18_478_006_272
    assert kv == kv_per_pos * 4096
    assert total == weights + kv_per_pos * 4096


def test_step_bytes_q8_cache_by_hand(bench):
    """The 27B-class shapes with the target's cache in 8 bits: per target
    layer and position, K and V are 8 heads x (128 one-byte codes + a 4-byte
    scale); the drafter's 5 layers stay bf16 (8 heads x 128 x 2 B each)."""
    q8, bf = synth.WORKLOADS["dense27b-36k-q8"], synth.WORKLOADS["dense27b-36k"]
    P = 36864.0
    t8, w8, kv8 = bench.step_bytes(q8, P)
    tb, wb, kvb = bench.step_bytes(bf, P)
    assert w8 == wb
    assert kv8 == P * (64 * 2 * 8 * (128 + 4) + 5 * 2 * 2 * 8 * 128)
    assert kvb == P * 69 * 2 * 2 * 8 * 128


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
@pytest.mark.parametrize("P", [0.0, 512.0, 4120.5, 36871.0])
def test_stage_bytes_partition_the_step(bench, name, P):
    wl = synth.WORKLOADS[name]
    total, _, _ = bench.step_bytes(wl, P, batch=wl.batch)
    stages = bench.stage_bytes(wl, P, batch=wl.batch)
    assert set(stages) == {"fuse", "inject", "draft", "teacher", "verify", "accept"}
    assert sum(stages.values()) == pytest.approx(total, rel=1e-12)
    assert stages["verify"] > stages["draft"] > stages["fuse"] > stages["inject"] == 0


@pytest.mark.parametrize("name,steps,warmup", [("qwen3-8b-4k", 40, 5), ("qwen3-8b-4k", 3, 3),
                                               ("dense27b-36k", 20, 5), ("qwen3-8b-batch8", 20, 5)])
def test_reference_tau_is_the_gpu_arms_timed_window(bench, name, steps, warmup):
    """The GPU arm runs one eager step, `warmup` graph replays, then `steps`
    timed replays, each step taking the next acceptance draw of every sequence
    and emitting min(k, B - 1) + 1 tokens for it.  Walk that sequence of calls
    with a step counter and count the timed tokens."""
    wl = synth.WORKLOADS[name]
    k, _ = synth.acceptance_draws(1 + warmup + steps + 4, wl.target.vocab, batch=wl.batch)
    ctr = 0
    ctr += 1                        # eager first step
    ctr += warmup                   # warm-up replays
    timed = 0
    for _ in range(steps):          # timed replays
        timed += sum(min(int(k[ctr, b]), wl.block - 1) + 1 for b in range(wl.batch))
        ctr += 1
    assert bench.timed_tau(wl, steps, warmup) == pytest.approx(timed / steps, rel=1e-12)
    # more than one token per step on average, at most a full block per sequence
    assert wl.batch < bench.timed_tau(wl, steps, warmup) <= wl.batch * wl.block
