"""Failure detection on the GPU without a fault: each device-side condition the
library reports in its status word is made to happen on purpose, with inputs
the kernels' own checks turn into a status bit, and the test checks the bit,
that nothing was written where it must not be, and that the next normal call
is correct and leaves the status clear.

  CAPACITY  a verify or an injection whose rows run past the cache's capacity
  BOUNDS    teacher forcing past its draws, a stream past its capacity, a
            token id outside the vocabulary
  TIMEOUT   the weight product's main-loop waits given a limit of 0 (the
            kernel gives up at once, drains what it started and returns)
"""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from block_diffusion_speculative_target_gb300.engine import Session
from gpu_util import assert_close, build_model, dev, to_dev, to_np
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["tiny-f32", "small-bf16-gqa4"])
def model(request):
    wl = synth.WORKLOADS[request.param]
    m, tg, dr, _ = build_model(wl)
    return wl, m, tg, dr


def _cache_snapshot(s, cache, n_layers, batch):
    sh = s.m.shape
    tdt = s.fused.dtype
    out = []
    for li in range(n_layers):
        for b in range(batch):
            k = torch.empty(sh.n_kv, s.capacity, sh.head_dim, dtype=tdt, device=dev())
            v = torch.empty_like(k)
            capi.dflash_cache_read(cache, li, b, 0, s.capacity, k, v)
            out.append((k.clone(), v.clone()))
    return out


def test_capacity_verify_skips_writes_past_capacity(model):
    wl, m, tg, dr = model
    sh, B = wl.target, 16
    cap, P = 40, 30
    s = Session(m, batch=2, capacity=cap, block=B)
    g = torch.Generator(device=dev()).manual_seed(5)
    for li in range(sh.n_layers):
        for b in range(2):
            k = torch.randn(sh.n_kv, cap, sh.head_dim, generator=g, device=dev()).to(s.fused.dtype)
            capi.dflash_cache_write(s.tcache, li, b, 0, cap, k, k)
    capi.dflash_cache_set_lengths(s.tcache, [P, P])
    before = _cache_snapshot(s, s.tcache, sh.n_layers, 2)
    tgc, _ = m.structs()
    toks = torch.as_tensor(synth.prompt_tokens(B, sh.vocab, stream=90).astype(np.int32), device=dev())
    # sequence 0 only: rows P..P+15 reach positions 40..45, past the capacity of 40
    capi.target_verify(tgc, toks, 1, B, 0, s.tcache, s.argmax, s.gap, None, None, None, None, None, 0, s.ws)
    assert s.status() & capi.STATUS_CAPACITY
    after = _cache_snapshot(s, s.tcache, sh.n_layers, 2)
    for li in range(sh.n_layers):
        for b in range(2):
            kb, vb = before[li * 2 + b]
            ka, va = after[li * 2 + b]
            if b == 1:  # the other sequence is untouched
                assert torch.equal(kb, ka) and torch.equal(vb, va), (li, b)
            else:  # committed positions and the other heads are untouched; 30..39 are scratch rows of the block
                assert torch.equal(kb[:, :P], ka[:, :P]) and torch.equal(vb[:, :P], va[:, :P]), (li, b)
    assert s.target_len() == [P, P]
    # a call within capacity afterwards is correct and clean
    capi.dflash_cache_set_lengths(s.tcache, [P - B, P])
    capi.target_verify(tgc, toks, 1, B, 0, s.tcache, s.argmax, s.gap, None, None, None, None, None, 0, s.ws)
    assert s.status() == 0
    s.close()


def test_capacity_inject_skips_rows_past_capacity(model):
    wl, m, tg, dr = model
    sh = wl.target
    cap, L0, npend = 40, 35, 16
    s = Session(m, batch=1, capacity=cap, block=16)
    rows = synth.gaussian((16, sh.hidden), seed=91)
    if wl.dtype == "bf16":
        rows = synth.to_bf16_f32(rows)
    fused = to_dev(rows, wl.dtype)
    capi.dflash_cache_set_lengths(s.dcache, [L0])
    s.n_pend.fill_(npend)
    _, drc = m.structs()
    capi.dflash_inject_kv(drc, fused, 1, 16, s.n_pend, s.dcache, s.ws)
    assert s.status() & capi.STATUS_CAPACITY
    # the rows that fit were written correctly
    rnd = O.Rounder("bf16" if wl.dtype == "bf16" else "none")
    ref = O.inject_kv(dr, rows[:cap - L0].astype(np.float64), np.arange(L0, cap), rnd)
    for li in range(wl.draft_layers):
        k = torch.empty(sh.n_kv, cap - L0, sh.head_dim, dtype=s.fused.dtype, device=dev())
        v = torch.empty_like(k)
        capi.dflash_cache_read(s.dcache, li, 0, L0, cap - L0, k, v)
        assert_close(np.transpose(to_np(k), (1, 0, 2)), ref[li][0], wl.dtype, f"inject K l={li}")
        assert_close(np.transpose(to_np(v), (1, 0, 2)), ref[li][1], wl.dtype, f"inject V l={li}")
    s.close()


def test_bounds_teacher_force_past_draws_and_stream_cap(model):
    wl, m, tg, dr = model
    V, B = wl.target.vocab, 16
    s = Session(m, batch=1, capacity=64, block=B, stream_cap=20)
    ref = np.arange(64, dtype=np.int32)[None, :] % (V - 1)
    k_draw = np.full((3, 1), 5, np.int64)
    r_draw = np.zeros((3, 1), np.int64)
    s.set_teacher(ref, k_draw, r_draw)
    s.stream_len.fill_(4)
    s.step_ctr.fill_(3)  # every draw used
    draft0 = s.draft.clone()
    capi.dflash_teacher_force(s.draft, 1, B, s.ref, s.ref.shape[1], s.ref.shape[1], s.stream_len, s.k_draw, s.r_draw,
                              3, s.step_ctr, V, s.ws)
    assert s.status() & capi.STATUS_BOUNDS
    assert torch.equal(s.draft, draft0)
    # accept with every draft matching: a = 15, but only 2 stream slots are left
    s.stream_len.fill_(18)
    s.stream.fill_(-1)
    s.argmax[:B].copy_(torch.arange(100, 100 + B, dtype=torch.int32))
    s.draft[0, 1:].copy_(torch.arange(100, 100 + B - 1, dtype=torch.int32))
    capi.dflash_cache_set_lengths(s.tcache, [10])
    capi.dflash_accept_rollback(s.draft, s.argmax, 1, B, s.tcache, s.anchor, s.n_pend, s.accept_len, s.stream,
                                s.stream_len, s.stream_cap, s.ws)
    assert s.status() & capi.STATUS_BOUNDS
    assert s.accept_len.item() == B - 1 and s.stream_len.item() == 20
    assert s.stream[0, 18:].cpu().tolist() == [100, 101]
    assert s.target_len() == [10 + B]
    # a normal teacher-forced call afterwards is clean
    s.step_ctr.zero_()
    s.stream_len.fill_(4)
    capi.dflash_teacher_force(s.draft, 1, B, s.ref, s.ref.shape[1], s.ref.shape[1], s.stream_len, s.k_draw, s.r_draw,
                              3, s.step_ctr, V, s.ws)
    assert s.status() == 0
    got = s.draft[0].cpu().numpy()
    assert got[1:6].tolist() == ref[0, 4:9].tolist() and got[6] == (ref[0, 9] + 1) % V
    s.close()


def test_bounds_token_outside_vocabulary(model):
    wl, m, tg, dr = model
    sh = wl.target
    s = Session(m, batch=1, capacity=64, block=16)
    tgc, _ = m.structs()
    toks = torch.tensor([3, sh.vocab + 7, 5], dtype=torch.int32, device=dev())
    capi.target_verify(tgc, toks, 1, 3, 0, s.tcache, s.argmax, s.gap, None, None, None, None, None, 0, s.ws)
    assert s.status() & capi.STATUS_BOUNDS
    toks[1] = 4
    capi.target_verify(tgc, toks, 1, 3, 0, s.tcache, s.argmax, s.gap, None, None, None, None, None, 0, s.ws)
    assert s.status() == 0
    s.close()


def test_timeout_weight_product_gives_up_and_recovers():
    M, K, rows = 1024, 4096, 16
    d = capi.ModelDesc(1, K, 1, 1, 128, 128, 256, 1e6, 1e-6, capi.BF16)
    ws = capi.dflash_workspace_alloc(d, None, rows, 256)
    x = synth.to_bf16_f32(synth.gaussian((rows, K), seed=92))
    w = synth.to_bf16_f32(synth.gaussian((M, K), seed=93, scale=0.02))
    xd, wd = to_dev(x, "bf16"), to_dev(w, "bf16")
    y = torch.full((rows, M), 7.0, dtype=torch.float32, device=dev())
    try:
        capi.dflash_debug_set_wait_limit(0)
        capi.dflash_linear(capi.BF16, xd, wd, y, rows, M, K, ws)
        st = capi.dflash_status(ws)
    finally:
        capi.dflash_debug_set_wait_limit(-1)
    assert st & capi.STATUS_TIMEOUT
    # the kernel wrote no result
    assert torch.all(y == 7.0)
    # the next call with the default limit is correct and clean
    capi.dflash_linear(capi.BF16, xd, wd, y, rows, M, K, ws)
    assert capi.dflash_status(ws) == 0
    ref = O.linear(x.astype(np.float64), w.astype(np.float64))
    assert_close(to_np(y), ref, "f32", "linear after a time-out", tol=1e-4 * max(1.0, np.abs(ref).max()))
    capi.dflash_workspace_free(ws)
