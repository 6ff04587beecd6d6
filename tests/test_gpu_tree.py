"""Tree verification (DDTree reading) on the GPU against the oracle: the
drafter's top-K candidates and the best-first tree, the ancestor-masked target
forward at depth positions, the walk with the compaction of the accepted
path's keys/values and captured rows, and whole tree decodes (the chain tree
equal to linear verification bit for bit, branching trees equal to the
oracle's greedy stream)."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Session
from gpu_util import assert_close, build_model, check_tokens, check_tokens_vs_logits, dev, oracle_logits_along, \
    rounder, to_dev, to_np
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


def _mask_bits(tree):
    anc = O.tree_ancestors(tree)
    return np.array([sum(1 << j for j in range(anc.shape[1]) if anc[i, j]) for i in range(anc.shape[0])],
                    dtype=np.uint64)


@pytest.mark.parametrize("B,batch,topk,budget", [(8, 2, 3, 20), (16, 1, 4, 63), (4, 3, 2, 9), (16, 2, 1, 15)])
def test_draft_tree_matches_oracle(B, batch, topk, budget):
    V = 4096
    d = capi.ModelDesc(1, 256, 4, 4, 64, 768, V, 1e6, 1e-6, capi.F32)
    ws = capi.dflash_workspace_alloc(d, None, 128, 256)
    try:
        rng = np.random.default_rng(B * 100 + budget)
        z = (rng.standard_normal((batch, B, V)) * 3.0).astype(np.float32)
        capi.dflash_workspace_logits(ws, batch * B, V, which=1).copy_(to_dev(z.reshape(batch * B, V), "f32"))
        anchors = rng.integers(0, V, batch).astype(np.int32)
        n = budget + 1
        i32 = dict(dtype=torch.int32, device=dev())
        tt, tp, td = (torch.zeros(batch, n, **i32) for _ in range(3))
        tm = torch.zeros(batch, n, dtype=torch.int64, device=dev())
        capi.dflash_draft_tree(to_dev(anchors, torch.int32), batch, B, V, topk, budget, tt, tp, td, tm, ws)
        for b in range(batch):
            ct, cl = O.topk_candidates(z[b, 1:].astype(np.float64), topk)
            tree = O.build_tree(int(anchors[b]), ct, cl, budget)
            assert tt[b].cpu().numpy().tolist() == tree.tokens.tolist(), b
            assert tp[b].cpu().numpy().tolist() == tree.parent.tolist(), b
            assert td[b].cpu().numpy().tolist() == tree.depth.tolist(), b
            assert tm[b].cpu().numpy().astype(np.uint64).tolist() == _mask_bits(tree).tolist(), b
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_workspace_free(ws)


@pytest.fixture(scope="module", params=["tiny-f32", "small-bf16-gqa4"])
def setup(request):
    wl = synth.WORKLOADS[request.param]
    m, tg, dr, _ = build_model(wl)
    return wl, m, tg, dr


def _greedy_tree(anchor, greedy, vocab):
    """A tree whose branch 0 follows the greedy continuation greedy[0..2]
    and that carries distractors beside and below it."""
    alt = lambda t, k: int((t + 1 + 17 * k) % (vocab - 1))
    tokens = [anchor, alt(greedy[0], 1), greedy[0], alt(greedy[1], 2), greedy[1], alt(greedy[0], 3), greedy[2],
              alt(greedy[2], 4), alt(greedy[3], 5)]
    parent = [-1, 0, 0, 2, 2, 1, 4, 4, 6]
    depth = [0, 1, 1, 2, 2, 2, 3, 3, 4]
    return O.Tree(np.array(tokens), np.array(parent), np.array(depth), np.zeros(len(tokens)))


def test_tree_verify_and_accept(setup):
    wl, m, tg, dr = setup
    sh = wl.target
    P = 150
    rnd = rounder(wl)
    s = Session(m, batch=1, capacity=P + 80, block=wl.block, tree_budget=16)
    kv = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    mk = synth.to_bf16_f32 if wl.dtype == "bf16" else (lambda a: a.astype(np.float32))
    for li in range(sh.n_layers):
        k = mk(synth.gaussian((sh.n_kv, P, sh.head_dim), seed=110, stream=2 * li))
        v = mk(synth.gaussian((sh.n_kv, P, sh.head_dim), seed=110, stream=2 * li + 1))
        capi.dflash_cache_write(s.tcache, li, 0, 0, P, to_dev(k, wl.dtype), to_dev(v, wl.dtype))
        kv.k[li], kv.v[li] = k.astype(np.float64), v.astype(np.float64)
    capi.dflash_cache_set_lengths(s.tcache, [P])
    anchor = int(synth.prompt_tokens(1, sh.vocab, stream=111)[0])
    # the oracle's greedy continuation from the anchor
    greedy, ctx = [], kv.copy()
    tok = anchor
    for _ in range(4):
        out = O.target_forward(tg, [tok], ctx, rnd)
        O.commit(ctx, out, 1)
        tok = int(out.argmax[0])
        greedy.append(tok)
    tree = _greedy_tree(anchor, greedy, sh.vocab)
    n = len(tree.tokens)
    i32 = dict(dtype=torch.int32, device=dev())
    tt = torch.as_tensor(tree.tokens.astype(np.int32), device=dev())[None]
    tp = torch.as_tensor(tree.parent.astype(np.int32), device=dev())[None]
    td = torch.as_tensor(tree.depth.astype(np.int32), device=dev())[None]
    tm = torch.as_tensor(_mask_bits(tree).astype(np.int64), device=dev())[None]
    tgc, _ = m.structs()
    capi.target_verify_tree(tgc, tt, td, tm, 1, n, s.tcache, s.argmax, s.gap, s.hcap, s.ws)
    lg = to_np(capi.dflash_workspace_logits(s.ws, n, sh.vocab))
    ref = O.target_forward_tree(tg, tree, kv, rnd)
    assert_close(lg, ref.logits, wl.dtype, "tree verify logits")
    am = s.argmax[:n].cpu().numpy()
    check_tokens_vs_logits(am, ref.argmax, ref.gap, lg, ref.logits, wl.dtype, "tree verify argmax")
    # the nodes' keys/values at their scratch slots, and their captured rows, before the walk
    before_k, before_v = [], []
    for li in range(sh.n_layers):
        k = torch.empty(sh.n_kv, n, sh.head_dim, dtype=s.fused.dtype, device=dev())
        v = torch.empty_like(k)
        capi.dflash_cache_read(s.tcache, li, 0, P, n, k, v)
        before_k.append(k.clone())
        before_v.append(v.clone())
        kr = np.transpose(to_np(k), (1, 0, 2))
        assert_close(kr, ref.new_k[li], wl.dtype, f"tree node keys layer {li}")
    hcap_before = s.hcap[:n].clone()
    s.anchor.fill_(anchor)
    s.stream_len.fill_(3)
    capi.dflash_accept_tree(tgc, tt, tp, s.argmax, 1, n, s.tcache, s.hcap, s.anchor, s.n_pend, s.accept_len, s.stream,
                            s.stream_len, s.stream_cap, s.ws)
    path, em = O.accept_tree(tree, am)  # the walk over the GPU's own greedy tokens
    a = len(path) - 1
    assert a == 3  # the greedy branch is accepted to its end
    assert s.accept_len.item() == a and s.n_pend.item() == a + 1 and s.anchor.item() == em[-1]
    assert s.stream[0, 3:3 + a + 1].cpu().numpy().tolist() == em.tolist()
    assert s.target_len() == [P + a + 1]
    for li in range(sh.n_layers):
        k = torch.empty(sh.n_kv, a + 1, sh.head_dim, dtype=s.fused.dtype, device=dev())
        v = torch.empty_like(k)
        capi.dflash_cache_read(s.tcache, li, 0, P, a + 1, k, v)
        idx = torch.as_tensor(path, device=dev())
        assert torch.equal(k, before_k[li][:, idx]) and torch.equal(v, before_v[li][:, idx]), li
    assert torch.equal(s.hcap[:a + 1], hcap_before[torch.as_tensor(path, device=dev())])
    assert s.status() == 0
    s.close()


def test_chain_tree_decode_equals_linear_decode(setup):
    """K = 1, budget B - 1: the tree is the drafter's greedy chain, and the GPU
    decode is the linear one bit for bit (stream and accepted counts)."""
    wl, m, tg, dr = setup
    B, steps = wl.block, 6
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    cap = wl.prompt_len + (steps + 2) * B + 8
    a = Session(m, batch=1, capacity=cap, block=B, stream_cap=cap)
    a.prefill([prompt])
    acc_a = []
    for _ in range(steps):
        a.step()
        acc_a.append(a.accept_len.item())
    t = Session(m, batch=1, capacity=cap, block=B, stream_cap=cap, tree_budget=B - 1)
    t.prefill([prompt])
    acc_t = []
    for _ in range(steps):
        t.step_tree(1)
        acc_t.append(t.accept_len.item())
    assert acc_a == acc_t
    assert np.array_equal(a.emitted()[0], t.emitted()[0])
    assert a.status() == 0 and t.status() == 0
    a.close()
    t.close()


@pytest.mark.parametrize("topk,budget", [(3, 24), (2, 40)])
def test_tree_decode_matches_oracle(setup, topk, budget):
    wl, m, tg, dr = setup
    B, steps = wl.block, 6
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    cap = wl.prompt_len + (steps + 2) * (budget + 1) + 8
    s = Session(m, batch=1, capacity=cap, block=B, stream_cap=cap, tree_budget=budget)
    s.prefill([prompt])
    for _ in range(steps):
        s.step_tree(topk)
    E = s.emitted()[0]
    assert s.status() == 0
    s.close()
    # every emitted token is the oracle's greedy token after the GPU's own prefix (near-ties excepted)
    assert len(E) >= 1 + steps
    exp, gap = oracle_logits_along(tg, prompt, E, rounder(wl))
    check_tokens(E, exp, gap, wl.dtype, f"tree decode topk={topk} budget={budget}")
