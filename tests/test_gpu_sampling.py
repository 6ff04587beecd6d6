"""Sampling mode (temperature T > 0) on the GPU against the oracle: inverse-CDF
draws, the drafter's sampled block, speculative-sampling verification with
rollback, and a whole sampling-mode decode of the fp32 model.

A draw is a discrete decision taken from float32 sums on the GPU and float64
sums in the oracle.  Where the uniform number falls within EPS of a boundary
of the oracle's cumulative distribution (or of an acceptance threshold) both
answers are correct; the tests check that the GPU's answer is then one of the
valid ones, and require equality everywhere else."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Session
from gpu_util import build_model, dev, rounder, to_dev
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

EPS = 1e-4  # relative margin of a float32 decision against the float64 one


def _cdf(p):
    c = np.cumsum(np.asarray(p, np.float64))
    return c / c[-1]


def _draw_ok(weights, v, got):
    """got is a valid draw for v: v within EPS of its cumulative interval."""
    c = _cdf(weights)
    lo = c[got - 1] if got > 0 else 0.0
    return weights[got] > 0 and lo - EPS <= v <= c[got] + EPS


def _ambiguous(weights, v):
    c = _cdf(weights)
    return bool(np.min(np.abs(c - v)) < EPS)


@pytest.fixture(scope="module")
def ws():
    d = capi.ModelDesc(1, 256, 4, 4, 64, 768, 151936, 1e6, 1e-6, capi.F32)
    h = capi.dflash_workspace_alloc(d, None, 128, 256)
    yield h
    capi.dflash_workspace_free(h)


@pytest.mark.parametrize("V", [2048, 151936])
@pytest.mark.parametrize("T", [0.6, 1.0, 1.7])
def test_sample_rows_inverse_cdf(ws, V, T):
    rows = 40
    z = synth.gaussian((rows, V), seed=100, stream=V, scale=3.0)
    v = np.random.default_rng(int(T * 10) + V).random(rows).astype(np.float32)
    out = torch.empty(rows, dtype=torch.int32, device=dev())
    capi.dflash_sample(to_dev(z, "f32"), rows, V, T, to_dev(v, "f32"), out, ws)
    got = out.cpu().numpy()
    p = O.softmax_t(z.astype(np.float64), T)
    for r in range(rows):
        exp = O.sample_inverse_cdf(p[r], float(v[r]))
        if not _ambiguous(p[r], float(v[r])):
            assert got[r] == exp, (r, got[r], exp)
        assert _draw_ok(p[r], float(v[r]), int(got[r])), r
    assert capi.dflash_status(ws) == 0


def _block_case(batch, B, V, seed):
    """Target logits of the verify rows and drafter logits of the block: the
    drafter's slot j is the target's row j - 1 plus noise, so that some drafts
    are accepted and some are not."""
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((batch, B, V)) * 2.0).astype(np.float32)
    zd = np.empty_like(zt)
    zd[:, 0] = rng.standard_normal((batch, V)).astype(np.float32)
    zd[:, 1:] = zt[:, :-1] + (rng.standard_normal((batch, B - 1, V)) * 0.5).astype(np.float32)
    return zt, zd


@pytest.mark.parametrize("B,batch", [(16, 3), (2, 2), (15, 1)])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_draft_sample_and_accept_sample(ws, B, batch, T):
    V = 4096
    zt, zd = _block_case(batch, B, V, seed=B * 10 + batch)
    rng = np.random.default_rng(B + batch)
    w = rng.random((batch, B - 1)).astype(np.float32)
    u = rng.random((batch, B - 1)).astype(np.float32)
    v = rng.random(batch).astype(np.float32)
    rows = batch * B
    capi.dflash_workspace_logits(ws, rows, V, which=0).copy_(to_dev(zt.reshape(rows, V), "f32"))
    capi.dflash_workspace_logits(ws, rows, V, which=1).copy_(to_dev(zd.reshape(rows, V), "f32"))
    i32 = dict(dtype=torch.int32, device=dev())
    anchors = rng.integers(0, V, batch)
    draft = torch.zeros(batch, B, **i32)
    draft[:, 0] = torch.as_tensor(anchors, **i32)
    capi.dflash_draft_sample(batch, B, V, T, to_dev(w, "f32"), draft, ws)
    d = draft.cpu().numpy()
    assert d[:, 0].tolist() == anchors.tolist()
    q = O.softmax_t(zd.astype(np.float64), T)
    p = O.softmax_t(zt.astype(np.float64), T)
    for b in range(batch):
        for j in range(1, B):
            if not _ambiguous(q[b, j], float(w[b, j - 1])):
                assert d[b, j] == O.sample_inverse_cdf(q[b, j], float(w[b, j - 1])), (b, j)
            assert _draw_ok(q[b, j], float(w[b, j - 1]), int(d[b, j]))
    # verification + rollback from known lengths and stream positions
    d_model = capi.ModelDesc(1, 256, 4, 4, 64, 768, V, 1e6, 1e-6, capi.F32)
    cache = capi.dflash_cache_alloc(d_model, 1, batch, 4096)
    try:
        lens = rng.integers(10, 1000, batch)
        capi.dflash_cache_set_lengths(cache, lens.tolist())
        cap = 64
        stream = torch.full((batch, cap), -1, **i32)
        stream_len = torch.as_tensor(rng.integers(1, 20, batch).astype(np.int32), device=dev())
        sl0 = stream_len.cpu().numpy().copy()
        anchor = torch.zeros(batch, **i32)
        npend = torch.zeros(batch, **i32)
        acc = torch.zeros(batch, **i32)
        capi.dflash_accept_sample(draft, batch, B, V, T, to_dev(u, "f32"), to_dev(v, "f32"), cache, anchor, npend, acc,
                                  stream, stream_len, cap, ws)
        got_a = acc.cpu().numpy()
        st = stream.cpu().numpy()
        for b in range(batch):
            a, em = O.accept_sampling(d[b], p[b], q[b, 1:], u[b].astype(np.float64), float(v[b]))
            # acceptance decisions away from their thresholds must agree
            margins = [abs(float(u[b, i]) * q[b, i + 1, d[b, i + 1]] - p[b, i, d[b, i + 1]]) /
                       max(p[b, i, d[b, i + 1]], 1e-30) for i in range(min(a + 1, B - 1))]
            if min(margins) < EPS:
                continue
            assert got_a[b] == a, (b, got_a[b], a)
            out = st[b, sl0[b]:sl0[b] + a + 1]
            assert out[:a].tolist() == em[:a].tolist()
            if a < B - 1:
                resid = np.maximum(p[b, a] - q[b, a + 1], 0.0)
            else:
                resid = p[b, B - 1]
            if not _ambiguous(resid, float(v[b])):
                assert out[a] == em[a], (b, out[a], em[a])
            assert _draw_ok(resid, float(v[b]), int(out[a]))
            assert anchor[b].item() == out[a] and npend[b].item() == a + 1
        assert capi.dflash_cache_get_lengths(cache, batch) == (lens + got_a + 1).tolist()
        assert stream_len.cpu().numpy().tolist() == (sl0 + got_a + 1).tolist()
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_cache_free(cache)


def test_sampling_decode_matches_oracle():
    """A whole sampling-mode decode of the fp32 model (T = 1): the GPU's
    stream and accepted counts equal the oracle's driven by the same uniform
    numbers (the fp32 model agrees with the oracle to ~1e-5, far from the
    decisions' thresholds for these draws)."""
    wl = synth.WORKLOADS["tiny-f32"]
    m, tg, dr, _ = build_model(wl)
    B, T, steps = wl.block, 1.0, 8
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    rng = np.random.default_rng(21)
    v0 = float(rng.random())
    w_all = rng.random((steps, B - 1))
    u_all = rng.random((steps, B - 1))
    v_all = rng.random(steps)
    s = Session(m, batch=1, capacity=wl.prompt_len + (steps + 2) * B, block=B)
    s.prefill([prompt])
    s.resample_first(T, [v0])
    acc = []
    for i in range(steps):
        f = lambda a: torch.as_tensor(np.asarray(a, np.float32), device=dev())
        s.step_sampling(T, f(w_all[i][None, :]), f(u_all[i][None, :]), f([v_all[i]]))
        acc.append(int(s.accept_len[0].item()))
    E = s.emitted()[0]
    assert s.status() == 0
    s.close()
    n = len(E)
    ref, ref_acc = O.spec_decode_sampling(tg, dr, prompt, n, B, T, (v0, w_all, u_all, v_all), rounder(wl))
    assert acc == ref_acc[:steps], (acc, ref_acc)
    assert np.array_equal(E, ref[:n])
