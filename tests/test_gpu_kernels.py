"""Kernel-level parity: each building block of libdflash.so against the
oracle on seeded inputs, at sizes spanning several tiles plus ragged tails."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_speculative_target_gb300 import capi
from gpu_util import TOL, assert_close, dev, to_dev, to_np
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


def _desc(H=256, nq=4, nkv=4, hd=64, F=768, V=2048, dt=capi.F32, L=1):
    return capi.ModelDesc(L, H, nq, nkv, hd, F, V, 1e6, 1e-6, dt)


@pytest.fixture(scope="module")
def ws():
    d = _desc(H=5120, nq=40, nkv=8, hd=128, F=25600, V=151936, dt=capi.BF16)
    h = capi.dflash_workspace_alloc(d, None, 128, 20480)
    yield h
    capi.dflash_workspace_free(h)


# ---------------------------------------------------------------- linear

@pytest.mark.parametrize("rows", [1, 7, 16, 33, 128])
@pytest.mark.parametrize("M,K", [(64, 96), (200, 1280), (768, 256), (2048, 256), (130, 33)])
def test_linear_f32(ws, rows, M, K):
    x = synth.gaussian((rows, K), seed=10, stream=rows)
    w = synth.gaussian((M, K), seed=11, stream=M, scale=0.05)
    y = torch.empty(rows, M, dtype=torch.float32, device=dev())
    capi.dflash_linear(capi.F32, to_dev(x, "f32"), to_dev(w, "f32"), y, rows, M, K, ws)
    assert_close(to_np(y), O.linear(x, w), "f32", f"linear f32 {rows}x{M}x{K}")


@pytest.mark.parametrize("rows", [1, 15, 16, 17, 31, 64, 100, 128])
@pytest.mark.parametrize("M,K", [(128, 64), (256, 512), (768, 512), (1024, 4096), (4096, 4096), (384, 20480)])
def test_linear_bf16_tcgen05(ws, rows, M, K):
    x = synth.to_bf16_f32(synth.gaussian((rows, K), seed=12, stream=rows))
    w = synth.to_bf16_f32(synth.gaussian((M, K), seed=13, stream=M + K, scale=0.02))
    y = torch.empty(rows, M, dtype=torch.float32, device=dev())
    capi.dflash_linear(capi.BF16, to_dev(x, "bf16"), to_dev(w, "bf16"), y, rows, M, K, ws)
    ref = O.linear(x, w)
    # fp32 accumulation of exact bf16 products: relative error well below 1e-4
    assert_close(to_np(y), ref, "bf16", f"linear bf16 {rows}x{M}x{K}", tol=1e-4 * max(1.0, np.abs(ref).max()))
    assert capi.dflash_status(ws) == 0


def test_linear_bf16_deterministic_and_row_invariant(ws):
    """A row's result is bit-identical whether computed alone or in a block
    (fixed split count per weight shape, fixed reduction order)."""
    M, K = 4096, 12288
    x = synth.to_bf16_f32(synth.gaussian((128, K), seed=14))
    w = synth.to_bf16_f32(synth.gaussian((M, K), seed=15, scale=0.02))
    xd, wd = to_dev(x, "bf16"), to_dev(w, "bf16")
    outs = {}
    for rows in (1, 16, 128):
        y = torch.empty(rows, M, dtype=torch.float32, device=dev())
        capi.dflash_linear(capi.BF16, xd, wd, y, rows, M, K, ws)
        outs[rows] = y.cpu().numpy()
    y2 = torch.empty(16, M, dtype=torch.float32, device=dev())
    capi.dflash_linear(capi.BF16, xd, wd, y2, 16, M, K, ws)
    assert np.array_equal(outs[16], y2.cpu().numpy())
    assert np.array_equal(outs[1][0], outs[16][0])
    assert np.array_equal(outs[16], outs[128][:16])


@pytest.mark.parametrize("M,K", [(1024, 4096), (24576, 512)])
@pytest.mark.parametrize("rows", [5, 16, 128])
def test_linear_bf16_unaligned_output_equals_aligned(ws, M, K, rows):
    """An output that is not 16-byte aligned (a valid float array one element
    into a buffer) takes the per-column epilogue, split (M = 1024) or not
    (M = 24576); it holds the same values, bit for bit, as the aligned
    output's four-column or staged path."""
    x = synth.to_bf16_f32(synth.gaussian((rows, K), seed=16, stream=rows))
    w = synth.to_bf16_f32(synth.gaussian((M, K), seed=17, stream=M, scale=0.02))
    xd, wd = to_dev(x, "bf16"), to_dev(w, "bf16")
    y = torch.empty(rows, M, dtype=torch.float32, device=dev())
    buf = torch.zeros(rows * M + 4, dtype=torch.float32, device=dev())
    yu = buf[1:1 + rows * M].view(rows, M)
    assert y.data_ptr() % 16 == 0 and yu.data_ptr() % 16 == 4
    capi.dflash_linear(capi.BF16, xd, wd, y, rows, M, K, ws)
    capi.dflash_linear(capi.BF16, xd, wd, yu, rows, M, K, ws)
    assert capi.dflash_status(ws) == 0
    assert np.array_equal(y.cpu().numpy(), yu.cpu().numpy())
    assert float(buf[0]) == 0.0 and float(buf[-3]) == 0.0  # nothing written outside the view
    ref = O.linear(x, w)
    assert_close(to_np(y), ref, "bf16", f"linear bf16 {rows}x{M}x{K}", tol=1e-4 * max(1.0, np.abs(ref).max()))


# ---------------------------------------------------------------- rmsnorm

@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("rows,H", [(1, 256), (16, 4096), (37, 5120), (128, 512)])
def test_rmsnorm(dt, rows, H):
    x = synth.gaussian((rows, H), seed=16, stream=H, scale=3.0)
    g = synth.gaussian((H,), seed=17, stream=H, scale=0.5) + 1.0
    if dt == "bf16":
        g = synth.to_bf16_f32(g)
    y = torch.empty(rows, H, dtype=torch.float32 if dt == "f32" else torch.bfloat16, device=dev())
    capi.dflash_rmsnorm(capi.F32 if dt == "f32" else capi.BF16, to_dev(x, torch.float32), to_dev(g, dt), y, rows, H,
                        1e-6)
    ref = O.rmsnorm(x, g, 1e-6)
    if dt == "bf16":
        ref = O.round_bf16(ref)
        # GPU and oracle may round a value lying near a bf16 boundary differently: one ulp
        assert np.all(np.abs(to_np(y) - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    else:
        assert_close(to_np(y), ref, "f32", "rmsnorm f32", tol=1e-5)


# ---------------------------------------------------------------- argmax

@pytest.mark.parametrize("V", [2048, 1000, 1001, 20001, 151936])
def test_argmax_ties_gap(ws, V):
    rows = 20
    lg = synth.gaussian((rows, V), seed=18, stream=V, scale=2.0)
    lg[3, 10] = lg[3, V - 5] = lg[3].max() + 1.0    # tie: lowest index wins, gap 0
    lg[5, :] = 0.0                                    # all equal
    lg[7, V - 1] = 50.0                               # maximum in the ragged tail
    am = torch.empty(rows, dtype=torch.int32, device=dev())
    gp = torch.empty(rows, dtype=torch.float32, device=dev())
    capi.dflash_argmax(to_dev(lg, torch.float32), rows, V, am, gp, ws)
    ref_i, ref_g = O.argmax_top2(lg)
    assert np.array_equal(am.cpu().numpy(), ref_i)
    assert np.allclose(gp.cpu().numpy(), ref_g, rtol=1e-6, atol=1e-6)
    assert am[3].item() == 10 and gp[3].item() == 0.0 and am[5].item() == 0 and am[7].item() == V - 1
    assert capi.dflash_status(ws) == 0


def test_argmax_nonfinite_sets_status(ws):
    lg = synth.gaussian((4, 4096), seed=19)
    lg[2, 77] = np.nan
    am = torch.empty(4, dtype=torch.int32, device=dev())
    capi.dflash_argmax(to_dev(lg, torch.float32), 4, 4096, am, None, ws)
    assert capi.dflash_status(ws) & capi.STATUS_NONFINITE
    assert capi.dflash_status(ws) == 0  # cleared by the read


# ---------------------------------------------------------------- attention

ATT_CASES = [
    # dtype, nq, nkv, hd, lengths per sequence, n
    ("f32", 4, 4, 64, [0], 16),
    ("f32", 4, 4, 64, [128, 300], 16),
    ("f32", 4, 2, 64, [255, 1], 5),
    ("bf16", 4, 1, 128, [0], 16),
    ("bf16", 4, 1, 128, [96], 16),
    ("bf16", 32, 8, 128, [4096], 16),
    ("bf16", 32, 8, 128, [255, 257], 16),
    ("bf16", 40, 8, 128, [1000], 15),
    ("bf16", 8, 2, 128, [300, 17], 1),
    ("bf16", 4, 1, 128, [200, 513], 37),
    ("bf16", 8, 4, 128, [1024], 128),
    # G = 8: no padding rows, the copy/PV issuing lane sits in a live warp
    ("bf16", 64, 8, 128, [700], 16),
    # G = 1, 16 key groups of 4 tiles per sequence
    ("bf16", 8, 8, 128, [8000, 3000], 16),
    # many key groups (36 and 79): the combine merges more than 32 partials per row
    ("bf16", 4, 1, 128, [9000], 16),
    ("bf16", 8, 2, 128, [20000, 611], 16),
]


@pytest.mark.parametrize("dt,nq,nkv,hd,lens,n", ATT_CASES)
@pytest.mark.parametrize("causal", [1, 0])
def test_attention(ws, dt, nq, nkv, hd, lens, n, causal):
    batch = len(lens)
    cap = max(lens) + n + 64
    d = _desc(H=nq * hd, nq=nq, nkv=nkv, hd=hd, F=256, V=256, dt=capi.F32 if dt == "f32" else capi.BF16)
    cache = capi.dflash_cache_alloc(d, 1, batch, cap)
    try:
        rnd = (lambda a: synth.to_bf16_f32(a)) if dt == "bf16" else (lambda a: a)
        ks, vs = [], []
        for b, P in enumerate(lens):
            k = rnd(synth.gaussian((nkv, P + n, hd), seed=20, stream=b))
            v = rnd(synth.gaussian((nkv, P + n, hd), seed=21, stream=b))
            capi.dflash_cache_write(cache, 0, b, 0, P + n, to_dev(k, dt), to_dev(v, dt))
            ks.append(k)
            vs.append(v)
        capi.dflash_cache_set_lengths(cache, lens)
        q = rnd(synth.gaussian((batch, n, nq, hd), seed=22, scale=1.5))
        out = torch.empty(batch, n, nq * hd, dtype=torch.float32 if dt == "f32" else torch.bfloat16, device=dev())
        capi.dflash_attention(d, to_dev(q, dt), batch, n, causal, cache, 0, out, ws)
        got = to_np(out).reshape(batch, n, nq, hd)
        G = nq // nkv
        for b, P in enumerate(lens):
            allowed = np.ones((n, P + n), bool)
            if causal:
                allowed[:, P:] = np.tril(np.ones((n, n), bool))
            for h in range(nq):
                ref = O.attention(q[b, :, h], ks[b][h // G], vs[b][h // G], allowed)
                assert_close(got[b, :, h], ref, dt, f"attention b={b} h={h} P={P} n={n} causal={causal}")
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_cache_free(cache)


def test_attention_rejects_misaligned_query(ws):
    """The bf16 path reads the query by TMA: a query pointer off a 16-byte
    boundary is an argument error, reported before any launch."""
    d = _desc(H=4 * 128, nq=4, nkv=1, hd=128, F=256, V=256, dt=capi.BF16)
    cache = capi.dflash_cache_alloc(d, 1, 1, 256)
    try:
        capi.dflash_cache_set_lengths(cache, [16])
        buf = torch.zeros(16 * 4 * 128 + 8, dtype=torch.bfloat16, device=dev())
        q = buf[1:1 + 16 * 4 * 128]  # 2 bytes past an aligned base
        out = torch.empty(1, 16, 4 * 128, dtype=torch.bfloat16, device=dev())
        with pytest.raises(capi.DFlashError) as e:
            capi.dflash_attention(d, q, 1, 16, 1, cache, 0, out, ws)
        assert e.value.code == capi.ERR_INVALID_ARG
        assert capi.dflash_status(ws) == 0
    finally:
        capi.dflash_cache_free(cache)


def _window_case(ws, nq, nkv, lens, n, causal, window):
    """dflash_attention over a 1-layer cache; returns (output, oracle outputs,
    launches enqueued by the call)."""
    batch = len(lens)
    cap = max(lens) + n + 64
    d = _desc(H=nq * 128, nq=nq, nkv=nkv, hd=128, F=256, V=256, dt=capi.BF16)
    cache = capi.dflash_cache_alloc(d, 1, batch, cap)
    try:
        ks, vs = [], []
        for b, P in enumerate(lens):
            k = synth.to_bf16_f32(synth.gaussian((nkv, P + n, 128), seed=30, stream=b))
            v = synth.to_bf16_f32(synth.gaussian((nkv, P + n, 128), seed=31, stream=b))
            capi.dflash_cache_write(cache, 0, b, 0, P + n, to_dev(k, "bf16"), to_dev(v, "bf16"))
            ks.append(k)
            vs.append(v)
        capi.dflash_cache_set_lengths(cache, lens)
        q = synth.to_bf16_f32(synth.gaussian((batch, n, nq, 128), seed=32, scale=1.5))
        out = torch.empty(batch, n, nq * 128, dtype=torch.bfloat16, device=dev())
        torch.cuda.synchronize()
        l0 = capi.dflash_launch_count()
        capi.dflash_attention(d, to_dev(q, "bf16"), batch, n, causal, cache, 0, out, ws, window=window)
        launches = capi.dflash_launch_count() - l0
        got = to_np(out).reshape(batch, n, nq, 128)
        G = nq // nkv
        refs = []
        for b, P in enumerate(lens):
            allowed = np.ones((n, P + n), bool)
            if causal:
                allowed[:, P:] = np.tril(np.ones((n, n), bool))
            if window > 0:
                allowed[:, :max(0, P - window)] = False
            refs.append([O.attention(q[b, :, h], ks[b][h // G], vs[b][h // G], allowed) for h in range(nq)])
        assert capi.dflash_status(ws) == 0
        return got, refs, launches
    finally:
        capi.dflash_cache_free(cache)


@pytest.mark.parametrize("lens,nkv", [([700, 64], 8), ([9000, 2500], 1)])
@pytest.mark.parametrize("causal,window", [(0, 0), (0, 512), (1, 1000)])
def test_attention_window_groups(ws, lens, nkv, causal, window):
    """A few key groups (700 positions, 8 KV heads) and many (9000, one KV
    head: 36 groups of two tiles), with and without a cross-context window
    (keys below P - window not visible): every row against the oracle."""
    nq = 4 * nkv
    got, refs, launches = _window_case(ws, nq, nkv, lens, 16, causal, window)
    assert launches == 2  # the group kernel and the combine
    for b, P in enumerate(lens):
        for h in range(nq):
            assert_close(got[b, :, h], refs[b][h], "bf16", f"b={b} h={h} P={P} window={window}")
