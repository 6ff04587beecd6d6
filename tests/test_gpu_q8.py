"""The 8-bit K/V cache on the GPU against the oracle's reading: the quantiser
(codes and scales bit for bit on identical inputs), attention over 8-bit
keys/values with a half-precision query, the target forward that writes its
own rows quantised, and whole decodes (speculative equal to the GPU's own
greedy decode bit for bit, and to the oracle's greedy stream)."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Session
from gpu_util import (assert_close, assert_close_rounded, build_model, check_tokens, check_tokens_vs_logits, dev,
                      oracle_logits_along, rounder, to_dev, to_np)
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


def _desc(nq, nkv, L=1, H=None, F=256, V=256):
    return capi.ModelDesc(L, H or nq * 128, nq, nkv, 128, F, V, 1e6, 1e-6, capi.BF16)


@pytest.fixture(scope="module")
def ws():
    h = capi.dflash_workspace_alloc(_desc(40, 8, H=5120, F=25600, V=151936), None, 128, 8192 + 128)
    yield h
    capi.dflash_workspace_free(h)


def _read_q8(cache, layer, seq, pos0, n, nkv):
    kc = torch.empty(nkv, n, 128, dtype=torch.uint8, device=dev())
    vc = torch.empty_like(kc)
    ks = torch.empty(nkv, n, dtype=torch.float32, device=dev())
    vs = torch.empty_like(ks)
    capi.dflash_cache_read_q8(cache, layer, seq, pos0, n, kc, vc, ks, vs)
    code = lambda t: (t.cpu().numpy().astype(np.int16) - 128).astype(np.int8)
    return code(kc), ks.cpu().numpy(), code(vc), vs.cpu().numpy()


def _bf16_rows(shape, seed, stream):
    """Seeded rows with row magnitudes spread over six decades (bf16 values)."""
    x = synth.gaussian(shape, seed=seed, stream=stream)
    mag = 10.0 ** synth.gaussian(shape[:-1] + (1,), seed=seed, stream=stream + 100)
    return synth.to_bf16_f32(x * mag)


def test_q8_cache_write_matches_oracle_quantizer():
    nkv, n = 3, 50
    d = _desc(nkv, nkv, L=2)
    cache = capi.dflash_cache_alloc_ex(d, 2, 2, 203, capi.KV_Q8)  # capacity rounds up to 208
    try:
        assert capi.dflash_cache_kv_format(cache) == capi.KV_Q8
        k = _bf16_rows((nkv, n, 128), 90, 0)
        v = _bf16_rows((nkv, n, 128), 90, 1)
        k[0, 3] = 0.0                                   # a zero row: s = 0, codes 0
        k[1, 4] = 0.0
        k[1, 4, :7] = [127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 3.0]  # ties at the half steps
        v[2, 5] = 0.0
        v[2, 5, 9] = -1e-3                              # a single entry
        k, v = synth.to_bf16_f32(k), synth.to_bf16_f32(v)  # both sides quantise the same bf16 values
        capi.dflash_cache_write(cache, 1, 1, 37, n, to_dev(k, "bf16"), to_dev(v, "bf16"))
        capi.dflash_cache_write(cache, 0, 0, 158, 50, to_dev(k, "bf16"), to_dev(v, "bf16"))  # up to 208
        kq, ks, vq, vs = _read_q8(cache, 1, 1, 37, n, nkv)
        rq, rs = O.quantize_q8(k.astype(np.float32))
        assert np.array_equal(kq, rq) and np.array_equal(ks, rs)
        rq, rs = O.quantize_q8(v.astype(np.float32))
        assert np.array_equal(vq, rq) and np.array_equal(vs, rs)
        assert kq[1, 4, :7].tolist() == [127, 0, 2, 2, 0, -2, 3] and ks[1, 4] == 1.0
        # the neighbours keep the initial zeros (codes 0, scale 0)
        for pos in (36, 37 + n):
            a, s_, b, t = _read_q8(cache, 1, 1, pos, 1, nkv)
            assert not a.any() and not b.any() and not s_.any() and not t.any()
        with pytest.raises(capi.DFlashError):  # the codes are read with dflash_cache_read_q8
            capi.dflash_cache_read(cache, 1, 1, 37, n, torch.empty(nkv, n, 128, dtype=torch.bfloat16, device=dev()),
                                   torch.empty(nkv, n, 128, dtype=torch.bfloat16, device=dev()))
    finally:
        capi.dflash_cache_free(cache)


Q8_CASES = [
    # nq, nkv, lengths, n, window
    (32, 8, [4096], 16, 0),           # GQA 4, several key groups
    (40, 8, [1000], 15, 0),           # GQA 5
    (4, 1, [200, 513], 37, 0),        # two sequences, three 16-row blocks, ragged tails
    (8, 4, [300, 17], 1, 0),          # GQA 2, one row
    (8, 8, [3000], 16, 0),            # GQA 1
    (32, 8, [700], 16, 256),          # cross-context window
    # four tiles per unit: the 3-stage byte ring wraps (GQA 4: converter warps convert the values;
    # GQA 5: the softmax warps do)
    (32, 8, [8000], 16, 0),
    (40, 8, [8000], 15, 0),
]


@pytest.mark.parametrize("nq,nkv,lens,n,window", Q8_CASES)
@pytest.mark.parametrize("causal", [1, 0])
def test_q8_attention_matches_oracle(ws, nq, nkv, lens, n, window, causal):
    batch = len(lens)
    cap = max(lens) + n + 64
    d = _desc(nq, nkv)
    cache = capi.dflash_cache_alloc_ex(d, 1, batch, cap, capi.KV_Q8)
    try:
        ks, vs = [], []
        for b, P in enumerate(lens):
            k = synth.to_bf16_f32(synth.gaussian((nkv, P + n, 128), seed=91, stream=b))
            v = synth.to_bf16_f32(synth.gaussian((nkv, P + n, 128), seed=92, stream=b))
            capi.dflash_cache_write(cache, 0, b, 0, P + n, to_dev(k, "bf16"), to_dev(v, "bf16"))
            ks.append(O.kv_q8_store(k))
            vs.append(O.kv_q8_store(v))
        capi.dflash_cache_set_lengths(cache, lens)
        q = O.round_f16(synth.gaussian((batch, n, nq, 128), seed=93, scale=1.5))
        out = torch.empty(batch, n, nq * 128, dtype=torch.bfloat16, device=dev())
        capi.dflash_attention(d, to_dev(q, torch.float16), batch, n, causal, cache, 0, out, ws, window=window)
        got = to_np(out).reshape(batch, n, nq, 128)
        G = nq // nkv
        for b, P in enumerate(lens):
            allowed = np.ones((n, P + n), bool)
            if causal:
                allowed[:, P:] = np.tril(np.ones((n, n), bool))
            if window:
                allowed[:, :max(0, P - window)] = False
            for h in range(nq):
                ref = O.attention(q[b, :, h], ks[b][h // G], vs[b][h // G], allowed)
                assert_close_rounded(got[b, :, h], ref, f"q8 attention b={b} h={h} P={P} n={n} causal={causal}")
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_cache_free(cache)


@pytest.fixture(scope="module", params=["small-bf16-gqa4", "small-bf16-gqa5"])
def setup(request):
    wl = synth.WORKLOADS[request.param]
    m, tg, dr, _ = build_model(wl)
    return wl, m, dataclasses.replace(tg, kv_format="q8"), dr


def test_q8_verify_block_on_context(setup):
    wl, m, tg, dr = setup
    sh, B = wl.target, wl.block
    lens = [0, 77, 260]
    batch = len(lens)
    s = Session(m, batch=batch, capacity=300, block=B, kv_format="q8")
    kvs = []
    for b, P in enumerate(lens):
        kv = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
        for li in range(sh.n_layers):
            if P == 0:
                continue
            k = synth.to_bf16_f32(synth.gaussian((sh.n_kv, P, sh.head_dim), seed=94, stream=1000 * b + 2 * li))
            v = synth.to_bf16_f32(synth.gaussian((sh.n_kv, P, sh.head_dim), seed=94, stream=1000 * b + 2 * li + 1))
            capi.dflash_cache_write(s.tcache, li, b, 0, P, to_dev(k, "bf16"), to_dev(v, "bf16"))
            kv.k[li], kv.v[li] = O.kv_q8_store(k), O.kv_q8_store(v)
        kvs.append(kv)
    capi.dflash_cache_set_lengths(s.tcache, lens)
    toks = synth.prompt_tokens(batch * B, sh.vocab, stream=95).reshape(batch, B)
    tgc, _ = m.structs()
    capi.target_verify(tgc, to_dev(toks.astype(np.int32), torch.int32), batch, B, 0, s.tcache, s.argmax, s.gap,
                       s.hcap, None, None, None, None, 0, s.ws)
    rnd = rounder(wl)
    am = s.argmax.cpu().numpy()[:batch * B].reshape(batch, B)
    lg = to_np(capi.dflash_workspace_logits(s.ws, batch * B, sh.vocab)).reshape(batch, B, -1)
    for b, P in enumerate(lens):
        ref = O.target_forward(tg, toks[b], kvs[b], rnd)
        assert_close(lg[b], ref.logits, wl.dtype, f"q8 verify logits b={b}")
        check_tokens_vs_logits(am[b], ref.argmax, ref.gap, lg[b], ref.logits, wl.dtype, f"q8 verify argmax b={b}")
        # the block's own rows as stored: codes times scales, within one quantisation step of the oracle's
        for li in (0, sh.n_layers - 1):
            kq, kss, vq, vss = _read_q8(s.tcache, li, b, P, B, sh.n_kv)
            for codes, sc, refv, what in ((kq, kss, ref.new_k[li], "K"), (vq, vss, ref.new_v[li], "V")):
                got = codes.astype(np.float64) * sc.astype(np.float64)[..., None]        # [n_kv][B][d]
                want = np.transpose(refv, (1, 0, 2))
                step = np.maximum(sc, np.max(np.abs(want), axis=-1) / 127.0)[..., None]
                assert np.all(np.abs(got - want) <= 1.01 * step + 1e-2), f"q8 block {what} b={b} layer {li}"
                assert np.all(np.abs(codes).max(axis=-1) == 127), f"q8 block {what} codes span b={b} layer {li}"
    assert s.status() == 0
    s.close()


def test_q8_decode_lossless_and_matches_oracle(setup):
    wl, m, tg, dr = setup
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    B, steps = wl.block, 8
    n_ref = 1 + steps * B + B
    cap = wl.prompt_len + n_ref + 16
    ar = Session(m, batch=1, capacity=cap, block=B, with_draft=False, stream_cap=n_ref + 8, kv_format="q8")
    ar.prefill([prompt], inject=False)
    for _ in range(n_ref - 1):
        ar.ar_step()
    G = ar.emitted()[0]
    assert ar.status() == 0
    ar.close()
    rnd = rounder(wl)
    ref_tok, ref_gap = oracle_logits_along(tg, prompt, G, rnd)
    check_tokens(G, ref_tok, ref_gap, wl.dtype, f"{wl.name} q8 AR stream")
    k, r = synth.acceptance_draws(steps, wl.target.vocab)
    s = Session(m, batch=1, capacity=cap, block=B, stream_cap=n_ref + 8, kv_format="q8")
    s.prefill([prompt])
    s.set_teacher(G[None, :], k, r)
    acc = []
    for _ in range(steps):
        s.step(teacher=True)
        acc.append(s.accept_len.item())
    out = s.emitted()[0]
    assert s.status() == 0
    s.close()
    assert acc == np.minimum(k[:, 0], B - 1).tolist()
    assert np.array_equal(out, G[:len(out)])


def test_q8_unsupported_paths(setup):
    wl, m, tg, dr = setup
    sh = wl.target
    s = Session(m, batch=1, capacity=64, block=wl.block, tree_budget=8, kv_format="q8")
    n = 9
    i32 = dict(dtype=torch.int32, device=dev())
    tt, td = torch.zeros(1, n, **i32), torch.zeros(1, n, **i32)
    tm = torch.zeros(1, n, dtype=torch.int64, device=dev())
    tgc, drc = m.structs()
    with pytest.raises(capi.DFlashError) as e:
        capi.target_verify_tree(tgc, tt, td, tm, 1, n, s.tcache, s.argmax, s.gap, s.hcap, s.ws)
    assert e.value.code == capi.ERR_UNSUPPORTED_SHAPE
    dq = capi.dflash_cache_alloc_ex(s.ddesc, wl.draft_layers, 1, 64, capi.KV_Q8)
    try:
        with pytest.raises(capi.DFlashError) as e:
            capi.dflash_inject_kv(drc, s.fused, 1, wl.block, s.n_pend, dq, s.ws)
        assert e.value.code == capi.ERR_UNSUPPORTED_SHAPE
    finally:
        capi.dflash_cache_free(dq)
    assert s.status() == 0
    s.close()
