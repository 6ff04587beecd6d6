"""The drafter's cross-context window on the GPU against the oracle: the
attention kernel with a window (keys below len - W dropped, chunk boundaries
unchanged), the windowed drafter block, and a windowed speculative decode
whose stream is still the greedy autoregressive one."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Session
from gpu_util import assert_close, build_model, check_tokens, dev, rounder, to_dev, to_np
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt,nq,nkv,hd", [("bf16", 32, 8, 128), ("bf16", 40, 8, 128), ("f32", 4, 4, 64)])
@pytest.mark.parametrize("W", [1, 100, 256, 300, 700, 5000])
def test_attention_window_matches_masked_softmax(dt, nq, nkv, hd, W):
    P, n = 700, 16
    d = capi.ModelDesc(1, nq * hd, nq, nkv, hd, 256, 256, 1e6, 1e-6, capi.BF16 if dt == "bf16" else capi.F32)
    cache = capi.dflash_cache_alloc(d, 1, 1, P + n + 40)
    ws = capi.dflash_workspace_alloc(d, None, n, P + n + 40)
    try:
        rnd = synth.to_bf16_f32 if dt == "bf16" else (lambda a: a.astype(np.float32))
        k = rnd(synth.gaussian((nkv, P + n, hd), seed=80, stream=W))
        v = rnd(synth.gaussian((nkv, P + n, hd), seed=81, stream=W))
        capi.dflash_cache_write(cache, 0, 0, 0, P + n, to_dev(k, dt), to_dev(v, dt))
        capi.dflash_cache_set_lengths(cache, [P])
        q = rnd(synth.gaussian((1, n, nq, hd), seed=82, scale=1.5))
        out = torch.empty(1, n, nq * hd, dtype=torch.bfloat16 if dt == "bf16" else torch.float32, device=dev())
        capi.dflash_attention(d, to_dev(q, dt), 1, n, 0, cache, 0, out, ws, window=W)
        got = to_np(out).reshape(n, nq, hd)
        allowed = np.ones((n, P + n), bool)
        allowed[:, :O.cross_window(P, W)] = False
        G = nq // nkv
        for h in range(0, nq, max(1, nq // 5)):
            ref = O.attention(q[0, :, h], k[h // G], v[h // G], allowed)
            assert_close(got[:, h], ref, dt, f"window {W} head {h}")
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_workspace_free(ws)
        capi.dflash_cache_free(cache)


@pytest.fixture(scope="module", params=["tiny-f32", "small-bf16-gqa4"])
def setup(request):
    wl = synth.WORKLOADS[request.param]
    m, tg, dr, _ = build_model(wl)
    return wl, m, tg, dr


@pytest.mark.parametrize("W", [64, 300])
def test_draft_block_with_window(setup, W):
    wl, m, tg, dr = setup
    sh, B = wl.target, wl.block
    lens = [40, 600, 333]
    batch = len(lens)
    s = Session(m, batch=batch, capacity=640, block=B)
    kvs = []
    for b, P in enumerate(lens):
        kv = O.KV.empty(wl.draft_layers, sh.n_kv, sh.head_dim)
        for li in range(wl.draft_layers):
            mk = synth.to_bf16_f32 if wl.dtype == "bf16" else (lambda a: a.astype(np.float32))
            k = mk(synth.gaussian((sh.n_kv, P, sh.head_dim), seed=83, stream=1000 * b + 2 * li))
            v = mk(synth.gaussian((sh.n_kv, P, sh.head_dim), seed=83, stream=1000 * b + 2 * li + 1))
            capi.dflash_cache_write(s.dcache, li, b, 0, P, to_dev(k, wl.dtype), to_dev(v, wl.dtype))
            kv.k[li], kv.v[li] = k.astype(np.float64), v.astype(np.float64)
        kvs.append(kv)
    capi.dflash_cache_set_lengths(s.dcache, lens)
    anchors = synth.prompt_tokens(batch, sh.vocab, stream=84)
    s.anchor.copy_(torch.as_tensor(anchors, dtype=torch.int32))
    m.set_cross_ctx(W)
    try:
        tgc, drc = m.structs()
        capi.dflash_draft_block(drc, tgc, s.anchor, batch, B, s.dcache, s.draft, s.ws)
    finally:
        m.set_cross_ctx(0)
    got = s.draft.cpu().numpy()
    lg = to_np(capi.dflash_workspace_logits(s.ws, batch * B, sh.vocab, which=1)).reshape(batch, B, -1)
    rnd = rounder(wl)
    for b in range(batch):
        ref_logits = O.draft_logits(dr, tg, int(anchors[b]), B, kvs[b], rnd, window=W)
        ref_tok, gap = O.argmax_top2(ref_logits)
        assert got[b, 0] == anchors[b]
        check_tokens(got[b, 1:], ref_tok, gap, wl.dtype, f"windowed draft b={b}")
        assert_close(lg[b, 1:], ref_logits, wl.dtype, f"windowed draft logits b={b}")
    assert s.status() == 0
    s.close()


def test_windowed_decode_is_lossless(setup):
    """Speculative decoding with a 32-position window: the GPU's emitted
    stream equals its greedy autoregressive stream bit for bit."""
    wl, m, tg, dr = setup
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    steps, B = 8, wl.block
    cap = wl.prompt_len + (steps + 2) * B + 16
    ar = Session(m, batch=1, capacity=cap, block=B, with_draft=False, stream_cap=cap)
    ar.prefill([prompt], inject=False)
    for _ in range((steps + 1) * B):
        ar.ar_step()
    G = ar.emitted()[0]
    ar.close()
    m.set_cross_ctx(32)
    try:
        s = Session(m, batch=1, capacity=cap, block=B, stream_cap=cap)
        s.prefill([prompt])
        for _ in range(steps):
            s.step()
        E = s.emitted()[0]
        assert s.status() == 0
        s.close()
    finally:
        m.set_cross_ctx(0)
    assert len(E) > steps and np.array_equal(E, G[:len(E)])
