"""Stage-level parity through the C ABI: fuse, inject, draft, verify (prefill
and speculative), accept/rollback and teacher forcing, each against the
oracle on identical seeded inputs."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Session, desc_of
from gpu_util import (GAP, GAP_TOL, assert_close, build_model, check_tokens, check_tokens_vs_logits, dev, rounder,
                      to_dev, to_np)
from conftest import shrink
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny-f32", "small-bf16-gqa4", "small-bf16-gqa5"]


@pytest.fixture(scope="module", params=WORKLOADS)
def setup(request):
    wl = synth.WORKLOADS[request.param]
    m, tg, dr, w = build_model(wl)
    return wl, m, tg, dr


def _rnd_in(wl, a):
    return synth.to_bf16_f32(a) if wl.dtype == "bf16" else a.astype(np.float32)


def test_fuse(setup):
    wl, m, tg, dr = setup
    H = wl.target.hidden
    rows = 16
    hcap = _rnd_in(wl, synth.gaussian((rows, 5 * H), seed=30, scale=2.0))
    s = Session(m, batch=1, capacity=256, block=16)
    fused = torch.empty(rows, H, dtype=s.fused.dtype, device=dev())
    _, drc = m.structs()
    capi.dflash_fuse_features(drc, to_dev(hcap, wl.dtype), rows, fused, s.ws)
    ref = O.fuse_features(dr, hcap, rounder(wl))
    assert_close(to_np(fused), ref, wl.dtype, "fused features")
    assert s.status() == 0
    s.close()


def _read_cache(cache, layer, seq, pos0, n, nkv, hd, dtype):
    k = torch.empty(nkv, n, hd, dtype=dtype, device=dev())
    v = torch.empty(nkv, n, hd, dtype=dtype, device=dev())
    capi.dflash_cache_read(cache, layer, seq, pos0, n, k, v)
    return to_np(k), to_np(v)


def test_inject(setup):
    wl, m, tg, dr = setup
    sh = wl.target
    batch, rps = 3, 16
    lens0 = [0, 37, 200]
    npend = [16, 1, 9]
    F = _rnd_in(wl, synth.gaussian((batch, rps, sh.hidden), seed=31))
    s = Session(m, batch=batch, capacity=320, block=16)
    capi.dflash_cache_set_lengths(s.dcache, lens0)
    s.n_pend.copy_(torch.tensor(npend, dtype=torch.int32))
    _, drc = m.structs()
    capi.dflash_inject_kv(drc, to_dev(F.reshape(batch * rps, -1), wl.dtype), batch, rps, s.n_pend, s.dcache, s.ws)
    assert s.draft_len() == [a + b for a, b in zip(lens0, npend)]
    assert s.n_pend.cpu().tolist() == [0, 0, 0]
    rnd = rounder(wl)
    for b in range(batch):
        ref = O.inject_kv(dr, F[b, :npend[b]], np.arange(lens0[b], lens0[b] + npend[b]), rnd)
        for li in range(wl.draft_layers):
            k, v = _read_cache(s.dcache, li, b, lens0[b], npend[b], sh.n_kv, sh.head_dim, s.fused.dtype)
            assert_close(np.transpose(k, (1, 0, 2)), ref[li][0], wl.dtype, f"inject K b={b} l={li}")
            assert_close(np.transpose(v, (1, 0, 2)), ref[li][1], wl.dtype, f"inject V b={b} l={li}")
    assert s.status() == 0
    s.close()


def _synthetic_cache(wl, cache, n_layers, lens, seed):
    """Fill positions 0..len-1 of every layer with seeded keys/values; returns
    the oracle KV objects (one per sequence)."""
    sh = wl.target
    kvs = []
    for b, P in enumerate(lens):
        kv = O.KV.empty(n_layers, sh.n_kv, sh.head_dim)
        for li in range(n_layers):
            if P == 0:
                continue
            k = _rnd_in(wl, synth.gaussian((sh.n_kv, P, sh.head_dim), seed=seed, stream=1000 * b + 2 * li))
            v = _rnd_in(wl, synth.gaussian((sh.n_kv, P, sh.head_dim), seed=seed, stream=1000 * b + 2 * li + 1))
            capi.dflash_cache_write(cache, li, b, 0, P, to_dev(k, wl.dtype), to_dev(v, wl.dtype))
            kv.k[li], kv.v[li] = k.astype(np.float64), v.astype(np.float64)
        kvs.append(kv)
    capi.dflash_cache_set_lengths(cache, lens)
    return kvs


def test_draft_block(setup):
    wl, m, tg, dr = setup
    B = wl.block
    lens = [40, 1, 133]
    batch = len(lens)
    s = Session(m, batch=batch, capacity=200, block=B)
    kvs = _synthetic_cache(wl, s.dcache, wl.draft_layers, lens, seed=32)
    anchors = synth.prompt_tokens(batch, wl.target.vocab, stream=33)
    s.anchor.copy_(torch.as_tensor(anchors, dtype=torch.int32))
    tgc, drc = m.structs()
    capi.dflash_draft_block(drc, tgc, s.anchor, batch, B, s.dcache, s.draft, s.ws)
    got = s.draft.cpu().numpy()
    lg = to_np(capi.dflash_workspace_logits(s.ws, batch * B, wl.target.vocab, which=1)).reshape(batch, B, -1)
    assert s.draft_len() == lens  # the block's keys/values are scratch beyond the length
    rnd = rounder(wl)
    for b in range(batch):
        ref_logits = O.draft_logits(dr, tg, int(anchors[b]), B, kvs[b], rnd)
        ref, gap = O.draft_forward(dr, tg, int(anchors[b]), B, kvs[b], rnd)
        assert got[b, 0] == anchors[b]
        check_tokens_vs_logits(got[b, 1:], ref[1:], gap, lg[b, 1:], ref_logits, wl.dtype, f"draft tokens b={b}")
        assert_close(lg[b, 1:], ref_logits, wl.dtype, f"draft logits b={b}")
    assert s.status() == 0
    s.close()


def test_verify_prefill_commit(setup):
    wl, m, tg, dr = setup
    sh = wl.target
    prompt = synth.prompt_tokens(wl.prompt_len, sh.vocab)
    s = Session(m, batch=1, capacity=wl.prompt_len + 32, block=16)
    tgc, _ = m.structs()
    n = len(prompt)
    tok = torch.as_tensor(prompt.astype(np.int32), device=dev())
    capi.target_verify(tgc, tok, 1, n, 2, s.tcache, s.argmax, s.gap, s.hcap, s.anchor, s.n_pend, s.stream,
                       s.stream_len, s.stream_cap, s.ws)
    rnd = rounder(wl)
    ref = O.target_forward(tg, prompt, O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim), rnd)
    lg = to_np(capi.dflash_workspace_logits(s.ws, n, sh.vocab))
    assert_close(lg, ref.logits, wl.dtype, "prefill logits")
    check_tokens_vs_logits(s.argmax[:n].cpu().numpy(), ref.argmax, ref.gap, lg, ref.logits, wl.dtype,
                           "prefill argmax")
    assert_close(s.gap[:n].cpu().numpy(), ref.gap, wl.dtype, "prefill top-2 gap", tol=GAP_TOL[wl.dtype])
    assert_close(to_np(s.hcap[:n]), ref.hcap, wl.dtype, "prefill captured states")
    for li in (0, sh.n_layers // 2, sh.n_layers - 1):
        k, v = _read_cache(s.tcache, li, 0, 0, n, sh.n_kv, sh.head_dim, s.fused.dtype)
        assert_close(np.transpose(k, (1, 0, 2)), ref.new_k[li], wl.dtype, f"prefill K layer {li}")
        assert_close(np.transpose(v, (1, 0, 2)), ref.new_v[li], wl.dtype, f"prefill V layer {li}")
    assert s.target_len() == [n]
    assert s.n_pend.item() == n
    assert s.anchor.item() == s.argmax[n - 1].item()
    assert s.emitted()[0].tolist() == [s.anchor.item()]
    assert s.status() == 0
    s.close()


def test_verify_block_on_context(setup):
    wl, m, tg, dr = setup
    sh, B = wl.target, wl.block
    lens = [0, 77, 260]
    batch = len(lens)
    s = Session(m, batch=batch, capacity=300, block=B)
    kvs = _synthetic_cache(wl, s.tcache, sh.n_layers, lens, seed=34)
    toks = synth.prompt_tokens(batch * B, sh.vocab, stream=35).reshape(batch, B)
    tgc, _ = m.structs()
    capi.target_verify(tgc, to_dev(toks.astype(np.int32), torch.int32), batch, B, 0, s.tcache, s.argmax, s.gap,
                       s.hcap, None, None, None, None, 0, s.ws)
    assert s.target_len() == lens  # speculative: lengths untouched
    rnd = rounder(wl)
    am = s.argmax.cpu().numpy()[:batch * B].reshape(batch, B)
    hc = to_np(s.hcap)[:batch * B].reshape(batch, B, -1)
    lg = to_np(capi.dflash_workspace_logits(s.ws, batch * B, sh.vocab)).reshape(batch, B, -1)
    for b in range(batch):
        ref = O.target_forward(tg, toks[b], kvs[b], rnd)
        assert_close(lg[b], ref.logits, wl.dtype, f"verify logits b={b}")
        check_tokens_vs_logits(am[b], ref.argmax, ref.gap, lg[b], ref.logits, wl.dtype, f"verify argmax b={b}")
        assert_close(hc[b], ref.hcap, wl.dtype, f"verify hcap b={b}")
    assert s.status() == 0
    s.close()


def test_prefill_chunked_equals_oracle(setup):
    """A prompt longer than one 128-row chunk (ragged last chunk) prefilled in
    chunks, with fusion + injection per chunk."""
    wl, m, tg, dr = setup
    sh = wl.target
    P0 = 300
    prompt = synth.prompt_tokens(P0, sh.vocab, stream=36)
    s = Session(m, batch=1, capacity=P0 + 32, block=wl.block)
    s.prefill([prompt])
    rnd = rounder(wl)
    ref = O.target_forward(tg, prompt, O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim), rnd)
    assert s.target_len() == [P0] and s.draft_len() == [P0] and s.n_pend.item() == 0
    check_tokens([s.anchor.item()], [ref.argmax[-1]], [ref.gap[-1]], wl.dtype, "first token")
    k, v = _read_cache(s.tcache, sh.n_layers - 1, 0, 0, P0, sh.n_kv, sh.head_dim, s.fused.dtype)
    assert_close(np.transpose(k, (1, 0, 2)), ref.new_k[-1], wl.dtype, "chunked prefill K")
    fused = O.fuse_features(dr, ref.hcap, rnd)
    inj = O.inject_kv(dr, fused, np.arange(P0), rnd)
    for li in range(wl.draft_layers):
        k, v = _read_cache(s.dcache, li, 0, 0, P0, sh.n_kv, sh.head_dim, s.fused.dtype)
        assert_close(np.transpose(k, (1, 0, 2)), inj[li][0], wl.dtype, f"injected K l={li}")
        assert_close(np.transpose(v, (1, 0, 2)), inj[li][1], wl.dtype, f"injected V l={li}")
    assert s.status() == 0
    s.close()


# ---------------------------------------------------------------- integer stages (no model)


@pytest.mark.parametrize("block", [2, 8, 15, 16])
def test_accept_rollback_random(block):
    rng = np.random.default_rng(block)
    batch = 8
    d = capi.ModelDesc(1, 256, 4, 4, 64, 768, 2048, 1e6, 1e-6, capi.F32)
    cache = capi.dflash_cache_alloc(d, 1, batch, 4096)
    ws = capi.dflash_workspace_alloc(d, None, 16, 4096)
    cap = 64
    try:
        i32 = dict(dtype=torch.int32, device=dev())
        stream = torch.full((batch, cap), -1, **i32)
        stream_len = torch.zeros(batch, **i32)
        anchor = torch.zeros(batch, **i32)
        npend = torch.zeros(batch, **i32)
        acc = torch.zeros(batch, **i32)
        lens = rng.integers(0, 1000, size=batch)
        capi.dflash_cache_set_lengths(cache, lens.tolist())
        host_stream = [[] for _ in range(batch)]
        host_len = lens.copy()
        for trial in range(5):
            V = 3
            g = rng.integers(0, V, size=(batch, block))
            dr = rng.integers(0, V, size=(batch, block))
            for b in range(batch):   # force long prefixes sometimes
                k = int(rng.integers(0, block))
                dr[b, 1:k + 1] = g[b, :k]
            capi.dflash_accept_rollback(to_dev(dr.astype(np.int32), torch.int32),
                                        to_dev(g.astype(np.int32), torch.int32), batch, block, cache, anchor, npend,
                                        acc, stream, stream_len, cap, ws)
            for b in range(batch):
                a = O.accept_length(dr[b], g[b])
                assert acc[b].item() == a
                assert anchor[b].item() == g[b, a] and npend[b].item() == a + 1
                host_stream[b] += list(g[b, :a + 1])
                host_len[b] += a + 1
            assert capi.dflash_cache_get_lengths(cache, batch) == host_len.tolist()
        st, sl = stream.cpu().numpy(), stream_len.cpu().numpy()
        for b in range(batch):
            assert st[b, :sl[b]].tolist() == host_stream[b]
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_cache_free(cache)
        capi.dflash_workspace_free(ws)


@pytest.mark.parametrize("block", [2, 15, 16])
def test_teacher_force(block):
    rng = np.random.default_rng(7 + block)
    batch, V, L, steps = 5, 97, 300, 6
    d = capi.ModelDesc(1, 256, 4, 4, 64, 768, 2048, 1e6, 1e-6, capi.F32)
    ws = capi.dflash_workspace_alloc(d, None, 16, 256)
    try:
        ref = rng.integers(0, V, size=(batch, L)).astype(np.int32)
        k, r = synth.acceptance_draws(steps, V, batch=batch)
        i32 = dict(dtype=torch.int32, device=dev())
        step = torch.zeros(1, **i32)
        for s in range(steps):
            e = rng.integers(1, L - block - 1, size=batch).astype(np.int32)
            drafts = rng.integers(0, V, size=(batch, block)).astype(np.int32)
            dd = to_dev(drafts, torch.int32)
            capi.dflash_teacher_force(dd, batch, block, to_dev(ref, torch.int32), L, L, to_dev(e, torch.int32),
                                      to_dev(k.astype(np.int32), torch.int32), to_dev(r.astype(np.int32), torch.int32),
                                      steps, step, V, ws)
            got = dd.cpu().numpy()
            for b in range(batch):
                exp = O.teacher_force(drafts[b], ref[b], int(e[b]), k[s, b], r[s, b], V)
                assert got[b].tolist() == exp.tolist()
                assert O.accept_length(got[b], ref[b, e[b]:e[b] + block]) == min(int(k[s, b]), block - 1)
        assert step.item() == steps
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_workspace_free(ws)
