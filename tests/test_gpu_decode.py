"""Whole-decode parity on the GPU: emitted streams against the oracle,
losslessness (speculative stream == greedy autoregressive stream, bit-exact),
teacher-forced acceptance, CUDA-graph replay, and ragged batches."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300.engine import Session
from gpu_util import build_model, check_tokens, oracle_logits_along, rounder
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


def gpu_ar(m, prompts, n_tokens, capacity):
    s = Session(m, batch=len(prompts), capacity=capacity, block=16, with_draft=False, stream_cap=n_tokens + 8)
    s.prefill(prompts, inject=False)
    for _ in range(n_tokens - 1):
        s.ar_step()
    out = s.emitted()
    assert s.status() == 0
    s.close()
    return out


def spec_run(m, prompts, block, steps, capacity, teacher=None, graph=False):
    s = Session(m, batch=len(prompts), capacity=capacity, block=block, stream_cap=1 + (steps + 2) * block)
    s.prefill(prompts)
    if teacher is not None:
        s.set_teacher(*teacher)
    accepts = []
    if graph:
        s.step(teacher=teacher is not None)  # warm-up step outside the graph
        accepts.append(s.accept_len.cpu().numpy().copy())
        g = s.capture_graph(lambda: s.step(teacher=teacher is not None))
        for _ in range(steps - 1):
            g.replay()
            torch.cuda.synchronize()
            accepts.append(s.accept_len.cpu().numpy().copy())
    else:
        for _ in range(steps):
            s.step(teacher=teacher is not None)
            accepts.append(s.accept_len.cpu().numpy().copy())
    out = s.emitted()
    assert s.status() == 0
    tl, dl = s.target_len(), s.draft_len()
    s.close()
    return out, np.array(accepts), tl, dl


@pytest.mark.parametrize("name", ["tiny-f32", "small-bf16-gqa4", "small-bf16-gqa5"])
def test_natural_stream_matches_oracle(name):
    """Natural drafting (random drafter): every emitted token is the oracle's
    greedy token given the GPU's own prefix (near-ties excepted), and the
    stream equals the oracle's speculative stream up to the first near-tie."""
    wl = synth.WORKLOADS[name]
    m, tg, dr, _ = build_model(wl)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    steps = 10
    out, acc, tl, dl = spec_run(m, [prompt], wl.block, steps, wl.prompt_len + (steps + 2) * wl.block + 16)
    gpu = out[0]
    assert len(gpu) == 1 + int(acc.sum()) + steps
    assert tl == [wl.prompt_len + len(gpu) - 1]
    rnd = rounder(wl)
    ref_tok, ref_gap = oracle_logits_along(tg, prompt, gpu, rnd)
    check_tokens(gpu, ref_tok, ref_gap, wl.dtype, f"{name} stream")
    ora, steps_o = O.spec_decode(tg, dr, prompt, len(gpu), wl.block, rnd, max_steps=steps)
    n = min(len(ora), len(gpu))
    first_tie = np.argmax(np.r_[ref_gap[:n] <= 1e-2, True])
    assert np.array_equal(gpu[:first_tie], ora[:first_tie])


@pytest.mark.parametrize("name", ["tiny-f32", "small-bf16-gqa4", "small-bf16-gqa5"])
def test_teacher_forced_lossless(name):
    """Teacher-forced drafts: accepted counts equal min(k, B-1) exactly and the
    speculative stream is bit-identical to the GPU's greedy AR stream, which
    itself agrees with the oracle's greedy decode."""
    wl = synth.WORKLOADS[name]
    m, tg, dr, _ = build_model(wl)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    B, steps = wl.block, 8
    n_ref = 1 + steps * B + B
    cap = wl.prompt_len + n_ref + 16
    G = gpu_ar(m, [prompt], n_ref, cap)[0]
    rnd = rounder(wl)
    ref_tok, ref_gap = oracle_logits_along(tg, prompt, G, rnd)
    check_tokens(G, ref_tok, ref_gap, wl.dtype, f"{name} AR stream")
    k, r = synth.acceptance_draws(steps, wl.target.vocab)
    out, acc, tl, dl = spec_run(m, [prompt], B, steps, cap, teacher=(G[None, :], k, r))
    assert np.array_equal(acc[:, 0], np.minimum(k[:, 0], B - 1))
    assert np.array_equal(out[0], G[:len(out[0])])
    # the drafter cache lags by the rows accepted in the last step (injected next step)
    assert dl[0] + int(acc[-1, 0]) + 1 == tl[0]
    # oracle teacher-forced run agrees on the accepted counts
    Gor, _ = O.greedy_ar(tg, prompt, n_ref, rnd)
    if np.array_equal(Gor, G):
        _, st = O.spec_decode(tg, dr, prompt, len(out[0]), B, rnd, forcing=(k[:, 0], r[:, 0]), ref=Gor,
                              max_steps=steps)
        assert [x.accept for x in st] == acc[:, 0].tolist()


def test_graph_replay_equals_eager():
    wl = synth.WORKLOADS["small-bf16-gqa4"]
    m, tg, dr, _ = build_model(wl)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    B, steps = wl.block, 6
    cap = wl.prompt_len + (steps + 3) * B + 16
    G = gpu_ar(m, [prompt], 1 + (steps + 1) * B + B, cap)[0]
    k, r = synth.acceptance_draws(steps, wl.target.vocab)
    eager = spec_run(m, [prompt], B, steps, cap, teacher=(G[None, :], k, r))
    graph = spec_run(m, [prompt], B, steps, cap, teacher=(G[None, :], k, r), graph=True)
    assert np.array_equal(eager[0][0], graph[0][0])
    assert np.array_equal(eager[1], graph[1])
    nat_e = spec_run(m, [prompt], B, steps, cap)
    nat_g = spec_run(m, [prompt], B, steps, cap, graph=True)
    assert np.array_equal(nat_e[0][0], nat_g[0][0])


def test_ragged_batch_equals_single():
    """Several sequences of unequal prompt lengths in one launch per stage,
    with independent acceptance draws, give each sequence exactly its
    single-sequence result."""
    wl = synth.WORKLOADS["small-bf16-gqa4"]
    m, tg, dr, _ = build_model(wl)
    lens = [96, 33, 150, 64]
    prompts = [synth.prompt_tokens(L, wl.target.vocab, stream=40 + i) for i, L in enumerate(lens)]
    B, steps = wl.block, 5
    n_ref = 1 + steps * B + B
    cap = max(lens) + n_ref + 16
    G = gpu_ar(m, prompts, n_ref, cap)
    for i, p in enumerate(prompts):
        assert np.array_equal(G[i], gpu_ar(m, [p], n_ref, cap)[0])
    k, r = synth.acceptance_draws(steps, wl.target.vocab, batch=len(lens))
    out, acc, tl, dl = spec_run(m, prompts, B, steps, cap, teacher=(np.stack(G), k, r))
    assert np.array_equal(acc, np.minimum(k, B - 1))
    for i in range(len(lens)):
        assert np.array_equal(out[i], G[i][:len(out[i])])
        assert tl[i] == lens[i] + len(out[i]) - 1
    # natural drafting: batch == each sequence alone
    nat, nacc, _, _ = spec_run(m, prompts, B, steps, cap)
    for i, p in enumerate(prompts):
        single, sacc, _, _ = spec_run(m, [p], B, steps, cap)
        assert np.array_equal(nat[i], single[0])
        assert np.array_equal(nacc[:, i], sacc[:, 0])
