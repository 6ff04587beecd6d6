"""Pins of the CPU oracle against facts that do not come from the oracle itself:
values the pages print, closed forms, invariants, library routines on special
cases, and brute force on tiny inputs.  No GPU."""
import itertools
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import dflash_oracle as O
from conftest import oracle_models, shrink

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NONE = O.Rounder("none")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- rounding


def test_round_bf16_ties_and_library():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.round_bf16(one) == one
    assert O.round_bf16(one + ulp / 2) == one                     # tie -> even (down)
    assert O.round_bf16(one + 3 * ulp / 2) == one + 2 * ulp       # tie -> even (up)
    assert O.round_bf16(one + ulp / 2 + 2.0 ** -30) == one + ulp  # just above the tie
    assert O.round_bf16(-(one + 3 * ulp / 2)) == -(one + 2 * ulp)
    assert O.round_bf16(0.0) == 0.0
    assert np.isinf(O.round_bf16(3.5e38))
    # float32-representable values: the library conversion must agree
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(20000).astype(np.float32) * 3.0
    x = np.concatenate([x, np.float32([1e-39, -3e-40, 6e37, 2.0 ** -130])])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_bf16(x.astype(np.float64)), ref)


# ---------------------------------------------------------------- layer selection


def test_layer_indices_golden():
    g = golden("pages_figures.json")["layer_selection"]
    assert O.layer_indices(g["n_layers"]) == g["layers"]


@pytest.mark.parametrize("L", [8, 12, 13, 36, 48, 64, 80])
def test_layer_indices_closed_form(L):
    s = O.layer_indices(L)
    assert len(s) == 5 and s[0] == 2 and s[-1] == L - 3
    assert all(a <= b for a, b in zip(s, s[1:]))
    # evenly spaced points between 2 and L-3, each within half a layer
    pts = np.linspace(2, L - 3, 5)
    assert np.all(np.abs(np.array(s) - pts) <= 0.5)


def test_layer_indices_named_targets():
    assert O.layer_indices(36) == [2, 10, 18, 25, 33]
    assert O.layer_indices(64) == [2, 17, 32, 46, 61]


# ---------------------------------------------------------------- building blocks


def test_rmsnorm_closed_forms():
    H = 64
    for c in (3.0, -0.25, 1e3):
        y = O.rmsnorm(np.full((1, H), c), np.ones(H), 0.0)
        assert np.allclose(y, np.sign(c))
    x = np.random.default_rng(1).standard_normal((5, H))
    y = O.rmsnorm(x, np.ones(H), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0)
    assert np.allclose(O.rmsnorm(7.5 * x, np.ones(H), 0.0), y)             # scale invariance
    g = np.arange(H, dtype=np.float64)
    assert np.allclose(O.rmsnorm(x, g, 0.0), y * g)                       # gain multiplies
    assert np.all(O.rmsnorm(np.zeros((1, H)), np.ones(H), 1e-6) == 0.0)   # eps keeps 0 finite
    # eps enters under the root: x = 1-vector, eps = 3 -> 1/sqrt(1 + 3) = 0.5
    assert np.allclose(O.rmsnorm(np.ones((1, 4)), np.ones(4), 3.0), 0.5)


def test_norm_linear_rounding_point():
    """The normed products: without rounding they are rmsnorm then linear; with
    bf16 rounding the stored operand is bf16(x * gain) and the row's 1/rms
    scales the results."""
    rng = np.random.default_rng(7)
    H, M, eps = 64, 24, 1e-6
    none, bf = O.Rounder("none"), O.Rounder("bf16")
    x = rng.standard_normal((3, H)) * 3
    g = 1 + 0.1 * rng.standard_normal(H)
    W = rng.standard_normal((M, H)) * 0.1
    assert np.allclose(O.norm_linear(x, g, eps, (W,), none)[0], O.linear(O.rmsnorm(x, g, eps), W),
                       rtol=1e-13, atol=1e-13)
    # x * g exactly representable in bf16 (small integers times powers of two): the bf16 reading
    # then rounds nothing and equals the exact normed product -- it would not if the normed row
    # (x * g / rms) were the rounded quantity
    xi = rng.integers(-40, 41, (3, H)).astype(np.float64)
    gp = 2.0 ** rng.integers(-2, 3, H)
    exact = O.linear(O.rmsnorm(xi, gp, eps), W)
    assert np.allclose(O.norm_linear(xi, gp, eps, (W,), bf)[0], exact, rtol=1e-12, atol=1e-12)
    assert not np.array_equal(O.round_bf16(O.rmsnorm(xi, gp, eps)), O.rmsnorm(xi, gp, eps))
    # otherwise the operand is rounded: with the identity matrix, result / (1/rms) is bf16(x * g)
    y = O.norm_linear(x, g, eps, (np.eye(H),), bf)[0]
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    assert np.allclose(y * rms, O.round_bf16(x * g), rtol=1e-14, atol=0)
    assert not np.allclose(y * rms, x * g, rtol=1e-6, atol=0)
    # several matrices share the operand and the scale
    W2 = rng.standard_normal((5, H))
    a, b = O.norm_linear(x, g, eps, (W, W2), bf)
    assert np.array_equal(a, O.norm_linear(x, g, eps, (W,), bf)[0])
    assert np.allclose(b, O.linear(y, W2), rtol=1e-12, atol=1e-12)


def test_linear_hand_values():
    x = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[1.0, 0.0, -1.0], [2.0, 1.0, 0.5]])    # [out=2, in=3]
    assert np.array_equal(O.linear(x, w), [[1 - 3, 2 + 2 + 1.5]])


def test_silu_values():
    assert O.silu(0.0) == 0.0
    assert math.isclose(O.silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    x = np.linspace(-20, 20, 101)
    assert np.allclose(O.silu(x) - O.silu(-x), x)          # x*s(x) + x*s(-x) = x
    assert abs(O.silu(40.0) - 40.0) < 1e-12 and abs(O.silu(-40.0)) < 1e-12


def test_rope_closed_form_d4():
    theta = 100.0
    x = np.zeros((1, 1, 4))
    x[0, 0, 0] = 1.0
    p = 3.0
    y = O.rope(x, [p], theta)
    # rotate-half: dims (0, 2) rotate by p * theta^0, dims (1, 3) by p * theta^(-1/2)
    assert np.allclose(y[0, 0], [math.cos(p), 0.0, math.sin(p), 0.0])
    x = np.zeros((1, 1, 4))
    x[0, 0, 3] = 1.0
    y = O.rope(x, [p], theta)
    a = p * theta ** -0.5
    assert np.allclose(y[0, 0], [0.0, -math.sin(a), 0.0, math.cos(a)])


def test_rope_invariants():
    rng = np.random.default_rng(2)
    d = 64
    q = rng.standard_normal((1, 3, d))
    k = rng.standard_normal((1, 3, d))
    assert np.allclose(O.rope(q, [0], 1e6), q)                                   # position 0
    for p in (1, 17, 4099, 98304):
        y = O.rope(q, [p], 1e6)
        assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(q, axis=-1))
        # composition: rotating by a then by b equals rotating by a + b
        assert np.allclose(O.rope(O.rope(q, [p], 1e6), [5], 1e6), O.rope(q, [p + 5], 1e6))
    # relative position: <rope(q, m), rope(k, n)> depends on m - n only
    for m, n, s in ((5, 2, 100), (0, 7, 4096), (36000, 35990, -35000)):
        a = np.sum(O.rope(q, [m], 1e6) * O.rope(k, [n], 1e6), axis=-1)
        b = np.sum(O.rope(q, [m + s], 1e6) * O.rope(k, [n + s], 1e6), axis=-1)
        assert np.allclose(a, b)


def test_attention_special_cases():
    rng = np.random.default_rng(3)
    d = 16
    q = rng.standard_normal((4, d))
    k = rng.standard_normal((6, d))
    v = rng.standard_normal((6, d))
    all_ = np.ones((4, 6), bool)
    one = np.zeros((4, 6), bool)
    one[:, 2] = True
    assert np.allclose(O.attention(q, k, v, one), np.broadcast_to(v[2], (4, d)))   # single key
    kk = np.broadcast_to(k[0], (6, d))
    assert np.allclose(O.attention(q, kk, v, all_), np.broadcast_to(v.mean(0), (4, d)))  # equal keys
    assert np.allclose(O.attention(np.zeros((4, d)), k, v, all_), np.broadcast_to(v.mean(0), (4, d)))
    # adding the same vector to every key shifts a row's scores by a constant
    u = rng.standard_normal(d)
    assert np.allclose(O.attention(q, k + u, v, all_), O.attention(q, k, v, all_))
    # a dominant key takes all the weight
    kd = k.copy()
    kd[4] = q[0] * 1e3
    assert np.allclose(O.attention(q[:1], kd, v, all_[:1]), v[4])
    # masked keys have no influence
    tri = np.tril(np.ones((4, 6), bool), 2)
    k2 = k.copy()
    k2[5] += 100.0
    v2 = v.copy()
    v2[5] -= 50.0
    assert np.allclose(O.attention(q[:3], k2, v2, tri[:3]), O.attention(q[:3], k, v, tri[:3]))
    # explicit two-key softmax
    q1 = np.array([[1.0, 0.0]])
    k1 = np.array([[2.0, 0.0], [0.0, 0.0]])
    v1 = np.array([[1.0, 0.0], [0.0, 1.0]])
    w0 = 1.0 / (1.0 + math.exp(-2.0 / math.sqrt(2.0)))
    assert np.allclose(O.attention(q1, k1, v1, np.ones((1, 2), bool)), [[w0, 1.0 - w0]])


def test_argmax_ties_and_gap():
    am, gap = O.argmax_top2(np.array([[1.0, 3.0, 3.0, 2.0], [0.5, -1.0, 0.25, 0.0]]))
    assert list(am) == [1, 0]
    assert gap[0] == 0.0 and gap[1] == 0.25


# ---------------------------------------------------------------- accept / teacher forcing


def test_accept_golden_linear_verification():
    g = golden("linear_verify_example.json")
    a = O.accept_length(g["draft"], g["target_argmax"])
    assert a == g["accept"]
    assert list(g["target_argmax"][: a + 1]) == g["emitted"]


def _accept_brute(draft, target):
    """Independent definition: the length of the longest k such that the
    drafted continuation draft[1..k] equals the target continuation
    target[0..k-1]."""
    B = len(draft)
    best = 0
    for k in range(B):
        if tuple(draft[1:k + 1]) == tuple(target[:k]):
            best = k
    return best


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5])
def test_accept_brute_force_all_inputs(B):
    V = 3
    for draft in itertools.product(range(V), repeat=B):
        for tgt in itertools.product(range(V), repeat=B):
            assert O.accept_length(draft, tgt) == _accept_brute(draft, tgt)


def test_teacher_force_gives_exact_accept():
    rng = np.random.default_rng(4)
    V = 11
    for B in (2, 5, 15, 16):
        for _ in range(200):
            ref = rng.integers(0, V, size=64)
            e = int(rng.integers(1, 30))
            d = rng.integers(0, V, size=B)
            d[0] = ref[e - 1]
            k = int(rng.geometric(1 / 8) - 1)
            r = int(rng.integers(0, V - 1))
            d2 = O.teacher_force(d, ref, e, k, r, V)
            assert O.accept_length(d2, ref[e:e + B]) == min(k, B - 1)


def test_tau_and_speedup_arithmetic():
    g = golden("pages_figures.json")
    t = g["tau"]
    assert round(O.tau(t["tokens"], t["steps"]), 2) == t["tau"]
    assert round(100 * O.tau(t["tokens"], t["steps"]) / t["block"], 1) == t["acceptance_pct"]
    assert round(t["tokens"] / t["seconds"], 1) == round(t["tok_per_s"], 1)
    for base, new, ratio in g["speedups"]["pairs"]:
        assert round(new / base, 2) == ratio


# ---------------------------------------------------------------- composed forward


def _tiny_models(tiny, **kw):
    wl, w = tiny
    if kw:
        wl = shrink(wl, **kw)
        w = synth.host_weights(wl.target, wl.draft_layers, wl.dtype)
    return (wl,) + oracle_models(wl, w)


def test_cache_equals_recompute(tiny):
    wl, tg, _ = _tiny_models(tiny)
    prompt = synth.prompt_tokens(24, wl.target.vocab)
    a, _ = O.greedy_ar(tg, prompt, 6, NONE)
    b = O.greedy_ar_recompute(tg, prompt, 6, NONE)
    assert np.array_equal(a, b)


def test_block_forward_equals_row_by_row(tiny):
    """A causal forward of n rows at once equals n one-row forwards with the
    cache growing between them (rows see exactly their prefix)."""
    wl, tg, _ = _tiny_models(tiny)
    toks = synth.prompt_tokens(20, wl.target.vocab)
    sh = tg.shape
    c1 = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    o1 = O.target_forward(tg, toks, c1, NONE)
    c2 = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    rows = []
    for t in toks:
        o = O.target_forward(tg, [t], c2, NONE)
        O.commit(c2, o, 1)
        rows.append(o.logits[0])
    assert np.allclose(o1.logits, np.array(rows), atol=1e-10)


def test_capture_order(tiny):
    """Block s of the captured state is the residual stream after layer S[s]."""
    wl, tg, _ = _tiny_models(tiny)
    toks = synth.prompt_tokens(9, wl.target.vocab)
    sh = tg.shape
    H = sh.hidden
    full = O.target_forward(tg, toks, O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim), NONE)
    for s, li in enumerate(tg.capture):
        cut = O.Target(O.Shape(li + 1, *list(vars(sh).values())[1:]), tg.embed, tg.layers[:li + 1],
                       tg.final_norm, tg.lm_head, (li,) * 5)
        part = O.target_forward(cut, toks, O.KV.empty(li + 1, sh.n_kv, sh.head_dim), NONE)
        assert np.array_equal(full.hcap[:, s * H:(s + 1) * H], part.hcap[:, :H])


def test_fuse_selects_and_normalises(tiny):
    wl, tg, dr = _tiny_models(tiny)
    H = wl.target.hidden
    rng = np.random.default_rng(5)
    hcap = rng.standard_normal((3, 5 * H))
    import dataclasses
    for s in range(5):
        sel = np.zeros((H, 5 * H))
        sel[:, s * H:(s + 1) * H] = np.eye(H)
        d2 = dataclasses.replace(dr, w_fc=sel)
        f = O.fuse_features(d2, hcap, NONE)
        blk = hcap[:, s * H:(s + 1) * H]
        assert np.allclose(f, blk / np.sqrt(np.mean(blk ** 2, axis=-1, keepdims=True) + 1e-6))


def test_draft_is_translation_invariant(tiny):
    """Context keys carry RoPE at their own positions and block queries at
    P..P+B-1: shifting every position by the same amount changes nothing."""
    wl, tg, dr = _tiny_models(tiny)
    H = wl.target.hidden
    rng = np.random.default_rng(6)
    fused = rng.standard_normal((10, H))
    outs = []
    for shift in (0, 1000):
        dc = O.KV.empty(dr.shape.n_layers, dr.shape.n_kv, dr.shape.head_dim)
        # place the 10 context rows at positions shift .. shift+9 by padding the cache
        for li, (k, v) in enumerate(O.inject_kv(dr, fused, np.arange(shift, shift + 10), NONE)):
            dc.k[li] = np.transpose(k, (1, 0, 2))
            dc.v[li] = np.transpose(v, (1, 0, 2))
        # draft_forward takes P from the cache length; emulate a cache that starts at `shift`
        # by calling the layer directly with pos0 = shift + 10.
        x = np.asarray(tg.embed, dtype=np.float64)[[5] + [dr.mask_id] * 15]
        for li, lw in enumerate(dr.layers):
            x, _, _ = O.decoder_layer(x, lw, dr.shape, dc.k[li], dc.v[li], shift + 10, False, NONE)
        outs.append(x)
    assert np.allclose(outs[0], outs[1], atol=1e-9)


def test_draft_noncausal_block_sees_all_rows(tiny):
    """Every block row sees every other row: changing the last slot's token
    changes row 0's output in the drafter, never in the causal target."""
    wl, tg, dr = _tiny_models(tiny)
    sh = dr.shape
    x = np.asarray(tg.embed, dtype=np.float64)[[3, 4, 5]]
    x2 = np.asarray(tg.embed, dtype=np.float64)[[3, 4, 6]]
    e = np.zeros((sh.n_kv, 0, sh.head_dim))
    a, _, _ = O.decoder_layer(x, dr.layers[0], sh, e, e, 0, False, NONE)
    b, _, _ = O.decoder_layer(x2, dr.layers[0], sh, e, e, 0, False, NONE)
    assert not np.allclose(a[0], b[0])
    a, _, _ = O.decoder_layer(x, dr.layers[0], sh, e, e, 0, True, NONE)
    b, _, _ = O.decoder_layer(x2, dr.layers[0], sh, e, e, 0, True, NONE)
    assert np.array_equal(a[:2], b[:2])


# ---------------------------------------------------------------- cross-context window


def _injected_cache(dr, fused, positions):
    dc = O.KV.empty(dr.shape.n_layers, dr.shape.n_kv, dr.shape.head_dim)
    for li, (k, v) in enumerate(O.inject_kv(dr, fused, positions, NONE)):
        dc.append(li, k, v)
    return dc


def test_cross_window_bounds():
    assert O.cross_window(100, 0) == 0          # no window: whole context
    assert O.cross_window(100, 30) == 70        # the 30 most recent positions 70..99
    assert O.cross_window(100, 100) == 0
    assert O.cross_window(20, 1024) == 0        # short context: all of it


def test_window_covering_the_context_equals_the_full_drafter(tiny):
    wl, tg, dr = _tiny_models(tiny)
    fused = np.random.default_rng(8).standard_normal((40, wl.target.hidden))
    dc = _injected_cache(dr, fused, np.arange(40))
    full = O.draft_logits(dr, tg, 7, 16, dc, NONE)
    for W in (40, 41, 1024):
        assert np.array_equal(O.draft_logits(dr, tg, 7, 16, dc, NONE, window=W), full)


def test_window_edge_is_exactly_w_positions(tiny):
    """Keys before P-W do not matter at all; the key at P-W does."""
    wl, tg, dr = _tiny_models(tiny)
    P, W = 50, 12
    fused = np.random.default_rng(9).standard_normal((P, wl.target.hidden))
    base = O.draft_logits(dr, tg, 3, 16, _injected_cache(dr, fused, np.arange(P)), NONE, window=W)
    outside = fused.copy()
    outside[: P - W] = np.random.default_rng(10).standard_normal((P - W, wl.target.hidden))
    got = O.draft_logits(dr, tg, 3, 16, _injected_cache(dr, outside, np.arange(P)), NONE, window=W)
    assert np.array_equal(got, base)
    edge = fused.copy()
    edge[P - W] += 1.0
    got = O.draft_logits(dr, tg, 3, 16, _injected_cache(dr, edge, np.arange(P)), NONE, window=W)
    assert not np.allclose(got, base, atol=1e-6)


def test_window_equals_full_drafter_on_the_last_w_rows(tiny):
    """With window W the drafter at P sees the W most recent context rows at
    positions P-W..P-1 and the block at P..; by RoPE's relative-position
    invariance that is the full drafter over a context of just those W rows
    placed at positions 0..W-1 (block at W..)."""
    wl, tg, dr = _tiny_models(tiny)
    P, W = 70, 20
    fused = np.random.default_rng(11).standard_normal((P, wl.target.hidden))
    win = O.draft_logits(dr, tg, 9, 16, _injected_cache(dr, fused, np.arange(P)), NONE, window=W)
    short = O.draft_logits(dr, tg, 9, 16, _injected_cache(dr, fused[P - W:], np.arange(W)), NONE)
    assert np.allclose(win, short, atol=1e-9, rtol=0)
    full = O.draft_logits(dr, tg, 9, 16, _injected_cache(dr, fused, np.arange(P)), NONE)
    assert not np.allclose(win, full, atol=1e-6)


def test_lossless_with_cross_window(tiny):
    """The window only changes what the drafter proposes: the emitted stream
    is still the greedy autoregressive one."""
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n = 24
    ref, _ = O.greedy_ar(tg, prompt, n, NONE)
    out, _ = O.spec_decode(tg, dr, prompt, n, 16, NONE, window=32)
    assert np.array_equal(out, ref)


# ---------------------------------------------------------------- tree verification


def _prefix_of(tree, i):
    out = []
    while i > 0:
        out.append(int(tree.tokens[i]))
        i = int(tree.parent[i])
    return tuple(reversed(out))


@pytest.mark.parametrize("D,K,budget,seed", [(3, 3, 10, 0), (4, 2, 7, 1), (2, 4, 8, 2), (3, 3, 39, 3), (5, 1, 4, 4)])
def test_tree_is_the_best_prefixes_by_brute_force(D, K, budget, seed):
    """Enumerate every prefix of the candidate lattice, score it, and take the
    `budget` best: exactly the tree's nodes."""
    rng = np.random.default_rng(seed)
    lp = np.sort(np.log(rng.dirichlet(np.ones(K + 3), size=D)[:, :K]), axis=1)[:, ::-1]
    toks = rng.permutation(100)[: D * K].reshape(D, K)
    tree = O.build_tree(99, toks, lp, budget)
    prefixes = []
    for d in range(1, D + 1):
        for ranks in itertools.product(range(K), repeat=d):
            prefixes.append((sum(lp[j, r] for j, r in enumerate(ranks)), tuple(toks[j, r] for j, r in enumerate(ranks))))
    prefixes.sort(key=lambda e: -e[0])
    want = {p for _, p in prefixes[: min(budget, len(prefixes))]}
    got = {_prefix_of(tree, i) for i in range(1, len(tree.tokens))}
    assert got == want
    # a tree: parents come first, depths step by one, scores never increase in creation order
    for i in range(1, len(tree.tokens)):
        assert tree.parent[i] < i and tree.depth[i] == tree.depth[tree.parent[i]] + 1
    assert np.all(np.diff(tree.score[1:]) <= 1e-12)


def test_tree_attention_sees_ancestors_only(tiny):
    wl, tg, dr = _tiny_models(tiny)
    sh = tg.shape
    ct = np.array([[10, 11], [12, 13], [14, 15]])
    cl = np.log(np.array([[0.5, 0.4], [0.6, 0.3], [0.7, 0.2]]))
    tree = O.build_tree(3, ct, cl, 8)
    cache = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    base = O.target_forward(tg, synth.prompt_tokens(20, sh.vocab), cache, NONE)
    O.commit(cache, base, 20)
    a = O.target_forward_tree(tg, tree, cache, NONE)
    anc = O.tree_ancestors(tree)
    for j in range(1, len(tree.tokens)):
        t2 = O.Tree(tree.tokens.copy(), tree.parent, tree.depth, tree.score)
        t2.tokens[j] = (t2.tokens[j] + 7) % sh.vocab
        b = O.target_forward_tree(tg, t2, cache, NONE)
        for i in range(len(tree.tokens)):
            same = np.allclose(a.logits[i], b.logits[i], atol=1e-12)
            assert same == (not anc[i, j]), (i, j)
    # a node's row equals the causal forward of its own path
    for i in range(len(tree.tokens)):
        path = [3] + list(_prefix_of(tree, i))
        ref = O.target_forward(tg, path, cache, NONE)
        assert np.allclose(a.logits[i], ref.logits[-1], atol=1e-9)


def test_accept_tree_walks_matching_children():
    tree = O.Tree(np.array([9, 1, 2, 3, 4, 5]), np.array([-1, 0, 0, 1, 3, 2]), np.array([0, 1, 1, 2, 3, 2]),
                  np.zeros(6))
    # root -> 2 (node 2) -> 5 (node 5), then node 5's greedy token 8 has no child
    am = np.array([2, 0, 5, 0, 0, 8])
    path, em = O.accept_tree(tree, am)
    assert path.tolist() == [0, 2, 5] and em.tolist() == [2, 5, 8]
    am = np.array([1, 3, 0, 4, 6, 0])
    path, em = O.accept_tree(tree, am)
    assert path.tolist() == [0, 1, 3, 4] and em.tolist() == [1, 3, 4, 6]
    path, em = O.accept_tree(tree, np.array([7, 0, 0, 0, 0, 0]))
    assert path.tolist() == [0] and em.tolist() == [7]


def test_chain_tree_is_linear_verification(tiny):
    """K = 1 and a budget of B - 1: the tree is the drafter's greedy chain and
    the loop is the linear one, step for step."""
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n, B = 30, 6
    got, acc = O.spec_decode_tree(tg, dr, prompt, n, B, 1, B - 1, NONE)
    ref, steps = O.spec_decode(tg, dr, prompt, n, B, NONE)
    assert np.array_equal(got, ref)
    assert acc == [st.accept for st in steps][: len(acc)]


@pytest.mark.parametrize("topk,budget", [(3, 20), (2, 9)])
def test_lossless_tree_verification(tiny, topk, budget):
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n = 24
    ref, _ = O.greedy_ar(tg, prompt, n, NONE)
    got, _ = O.spec_decode_tree(tg, dr, prompt, n, 16, topk, budget, NONE)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- sampling mode


def test_inverse_cdf_hand_cases():
    w = [0.0, 0.25, 0.0, 0.5, 0.25]
    assert O.sample_inverse_cdf(w, 0.0) == 1           # zero-weight entries are never drawn
    assert O.sample_inverse_cdf(w, 0.2499) == 1
    assert O.sample_inverse_cdf(w, 0.25) == 3          # right-open intervals: [0.25, 0.75) -> 3
    assert O.sample_inverse_cdf(w, 0.7499) == 3
    assert O.sample_inverse_cdf(w, 0.75) == 4
    assert O.sample_inverse_cdf(w, 0.999999) == 4
    assert O.sample_inverse_cdf([3.0, 1.0], 0.74) == 0  # unnormalised weights
    assert O.sample_inverse_cdf([3.0, 1.0], 0.76) == 1


def test_softmax_t_closed_forms():
    z = np.array([[1.0, 2.0, 4.0]])
    assert np.allclose(O.softmax_t(z, 1.0), np.exp(z) / np.exp(z).sum())
    assert np.allclose(O.softmax_t(z, 2.0), np.exp(z / 2) / np.exp(z / 2).sum())
    assert np.allclose(O.softmax_t(z + 100.0, 0.7), O.softmax_t(z, 0.7))
    assert O.softmax_t(z, 1e-3)[0, 2] == 1.0                       # T -> 0: the argmax


def _emit_distribution(p0, q1, p1, n=4000, rule=None):
    """Exact-by-quadrature distribution of the first emitted token of a
    two-slot block (one drafted token d ~ q1): acceptance depends on u alone,
    the residual on v alone, so each is integrated over its own midpoint grid."""
    rule = rule or O.accept_sampling
    V = len(p0)
    grid = (np.arange(n) + 0.5) / n
    out = np.zeros(V)
    p_rows, q_rows = np.stack([p0, p1]), q1[None, :]
    for d in range(V):
        draft = [0, d]
        acc = np.mean([rule(draft, p_rows, q_rows, [u], 0.5)[0] == 1 for u in grid])
        out[d] += q1[d] * acc
        if acc < 1.0:
            firsts = [rule(draft, p_rows, q_rows, [1.0 - 1e-12], v)[1][0] for v in grid]
            out += q1[d] * (1.0 - acc) * np.bincount(firsts, minlength=V) / n
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_accept_sampling_emits_the_target_distribution(seed):
    """Speculative sampling is lossless: whatever the drafter's q, the first
    emitted token is distributed exactly as the target's p."""
    rng = np.random.default_rng(seed)
    V = 5
    p0, p1 = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    q1 = rng.dirichlet(np.ones(V) * 0.5)
    dist = _emit_distribution(p0, q1, p1)
    assert np.allclose(dist, p0, atol=1e-3), (dist, p0)
    # planted mistake: with the roles of p and q swapped in the verification
    # (accept with min(1, q/p), residual max(0, q - p)) the output is not p
    def swapped(d, p, q, u, v):
        return O.accept_sampling(d, np.stack([q[0], p[1]]), p[:1], u, v)
    wrong = _emit_distribution(p0, q1, p1, n=1000, rule=swapped)
    assert np.max(np.abs(wrong - p0)) > 2e-2


def test_accept_sampling_bonus_and_residual_structure():
    V = 4
    p = np.array([[0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25], [0.7, 0.1, 0.1, 0.1]])
    q = np.array([[0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]])
    # q == p: always accepted, the bonus comes from the last target row
    a, em = O.accept_sampling([9, 3, 1], p, q, [0.99, 0.99], 0.05)
    assert a == 2 and em.tolist() == [3, 1, 0]
    # q puts all its mass on a token the target gives 0.1: accepted only for u < 0.1
    q2 = np.array([[0.0, 1.0, 0.0, 0.0], [0.25, 0.25, 0.25, 0.25]])
    p2 = np.array([[0.4, 0.1, 0.1, 0.4], [0.25, 0.25, 0.25, 0.25], [1.0, 0.0, 0.0, 0.0]])
    assert O.accept_sampling([9, 1, 2], p2, q2, [0.09, 0.5], 0.0)[0] == 2
    a, em = O.accept_sampling([9, 1, 2], p2, q2, [0.11, 0.5], 0.6)
    # residual max(0, p - q) = [0.4, 0, 0.1, 0.4]: v = 0.6 -> 0.54 falls in [0.5, 0.9) -> token 3
    assert a == 0 and em.tolist() == [3]
    assert O.accept_sampling([9, 1, 2], p2, q2, [0.11, 0.5], 0.5)[1].tolist() == [2]


def test_sampling_at_vanishing_temperature_is_greedy(tiny):
    """As T -> 0 every distribution collapses onto its argmax: drafting
    becomes the drafter's argmax, acceptance becomes equality with the
    target's argmax, the residual and the bonus become the target's argmax --
    the greedy loop, token for token."""
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n, B = 24, 8
    rng = np.random.default_rng(12)
    steps = n
    draws = (rng.random(), rng.random((steps, B - 1)), rng.random((steps, B - 1)), rng.random(steps))
    got, accepts = O.spec_decode_sampling(tg, dr, prompt, n, B, 1e-9, draws, NONE)
    ref, _ = O.spec_decode(tg, dr, prompt, n, B, NONE)
    assert np.array_equal(got, ref)
    greedy, _ = O.greedy_ar(tg, prompt, n, NONE)
    assert np.array_equal(O.sample_ar(tg, prompt, n, 1e-9, rng.random(n), NONE), greedy)


def test_sampling_loop_is_consistent_with_its_draws(tiny):
    """At T = 1 the loop's accepted counts and emitted tokens follow from its
    own verification of each step (re-derived from the recorded draws)."""
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n, B = 40, 16
    rng = np.random.default_rng(13)
    draws = (rng.random(), rng.random((n, B - 1)), rng.random((n, B - 1)), rng.random(n))
    got, accepts = O.spec_decode_sampling(tg, dr, prompt, n, B, 1.0, draws, NONE)
    assert len(got) == n and sum(a + 1 for a in accepts) + 1 >= n
    assert all(0 <= a <= B - 1 for a in accepts)


# ---------------------------------------------------------------- losslessness


@pytest.mark.parametrize("block", [16, 2, 5])
def test_lossless_natural_drafting(tiny, block):
    """Greedy speculative decoding emits exactly the greedy autoregressive
    stream (the target checks every drafted token)."""
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n = 24
    ref, _ = O.greedy_ar(tg, prompt, n, NONE)
    out, steps = O.spec_decode(tg, dr, prompt, n, block, NONE)
    assert np.array_equal(out, ref)
    for st in steps:
        assert st.accept == O.accept_length(st.draft, st.argmax)


@pytest.mark.parametrize("block", [16, 15, 8])
def test_lossless_teacher_forced(tiny, block):
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(wl.prompt_len, wl.target.vocab)
    n = 48
    ref, _ = O.greedy_ar(tg, prompt, n + block, NONE)
    k, r = synth.acceptance_draws(64, wl.target.vocab)
    out, steps = O.spec_decode(tg, dr, prompt, n, block, NONE, forcing=(k[:, 0], r[:, 0]), ref=ref)
    assert np.array_equal(out, ref[:n])
    for s, st in enumerate(steps):
        assert st.accept == min(int(k[s, 0]), block - 1)
    assert len(steps) < n  # forcing accepted more than one token per step on average


def test_lossless_bf16_rounding():
    wl = shrink(synth.WORKLOADS["small-bf16-gqa4"], n_layers=4, vocab=1024)
    w = synth.host_weights(wl.target, wl.draft_layers, wl.dtype)
    tg, dr = oracle_models(wl, w)
    rnd = O.Rounder("bf16")
    prompt = synth.prompt_tokens(40, wl.target.vocab)
    n = 20
    ref, _ = O.greedy_ar(tg, prompt, n + wl.block, rnd)
    k, r = synth.acceptance_draws(32, wl.target.vocab)
    out, steps = O.spec_decode(tg, dr, prompt, n, wl.block, rnd, forcing=(k[:, 0], r[:, 0]), ref=ref)
    assert np.array_equal(out, ref[:n])


# ---------------------------------------------------------------- planted mistakes


def test_planted_accept_off_by_one_breaks_losslessness(tiny, monkeypatch):
    """A plausible slip in acceptance (one token too many) is caught by the
    losslessness pin."""
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(32, wl.target.vocab)
    ref, _ = O.greedy_ar(tg, prompt, 30, NONE)
    good = O.accept_length
    monkeypatch.setattr(O, "accept_length", lambda d, g: min(good(d, g) + 1, len(d) - 1))
    out, _ = O.spec_decode(tg, dr, prompt, 12, 16, NONE)
    assert not np.array_equal(out, ref[:12])


def test_planted_rollback_slip_breaks_losslessness(tiny, monkeypatch):
    wl, tg, dr = _tiny_models(tiny)
    prompt = synth.prompt_tokens(32, wl.target.vocab)
    ref, _ = O.greedy_ar(tg, prompt, 12, NONE)
    good = O.commit
    # keeping one stale row of the rejected tail
    monkeypatch.setattr(O, "commit", lambda c, o, rows: good(c, o, min(rows + 1, len(o.argmax))))
    out, _ = O.spec_decode(tg, dr, prompt, 12, 16, NONE)
    assert not np.array_equal(out, ref)


def test_planted_rope_sign_breaks_rotation():
    q = np.random.default_rng(7).standard_normal((1, 2, 8))

    def bad(x, positions, theta):
        x = np.asarray(x, dtype=np.float64)
        half = x.shape[-1] // 2
        inv = theta ** (-np.arange(half) * 2.0 / x.shape[-1])
        ang = np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        a, b = x[..., :half], x[..., half:]
        return np.concatenate([a * c + b * s, b * c + a * s], axis=-1)

    y = bad(q, [3], 1e6)
    assert not np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(q, axis=-1))


# ---------------------------------------------------------------- 8-bit K/V cache


def test_round_f16_hand_cases():
    one = 1.0
    assert O.round_f16(one + 2.0 ** -11) == one                      # tie -> even
    assert O.round_f16(one + 3 * 2.0 ** -11) == one + 2.0 ** -9      # tie -> even (upwards)
    assert O.round_f16(one + 2.0 ** -11 + 2.0 ** -20) == one + 2.0 ** -10
    assert O.round_f16(65504.0) == 65504.0 and np.isinf(O.round_f16(65520.0))
    assert O.round_f16(-0.1) == -O.round_f16(0.1)


def test_q8_quantizer_pins():
    d = 128
    # a row whose largest entry is 127: s = 1 and the codes are the entries rounded half to even
    x = np.zeros(d)
    x[:7] = [127.0, 1.0, -0.5, 0.5, 1.5, -2.5, -126.6]
    q, s = O.quantize_q8(x)
    assert s == 1.0 and q[:7].tolist() == [127, 1, 0, 0, 2, -2, -127]
    # a row of zeros keeps s = 0 and codes 0
    q0, s0 = O.quantize_q8(np.zeros((2, d)))
    assert np.all(q0 == 0) and np.all(s0 == 0)
    rng = np.random.default_rng(11)
    x = rng.standard_normal((50, d)) * rng.uniform(0.01, 100.0, (50, 1))
    q, s = O.quantize_q8(x)
    assert q.dtype == np.int8 and s.dtype == np.float32 and s.shape == (50,)
    # the largest magnitude of a row maps to +-127; every entry within half a step of its float32 value
    assert np.all(np.max(np.abs(q.astype(int)), axis=1) == 127)
    x32 = x.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(O.dequantize_q8(q, s) - x32) <= s[:, None].astype(np.float64) * (0.5 + 1e-6))
    # scaling a row by a power of two scales s and keeps the codes
    q2, s2 = O.quantize_q8(x * 8.0)
    assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(8))
    # rows that are already integers times a power of two round-trip exactly
    qi = rng.integers(-127, 128, (5, d))
    qi[:, 3] = -127
    si = 2.0 ** -rng.integers(0, 10, 5).astype(float)
    q3, s3 = O.quantize_q8(qi * si[:, None])
    assert np.array_equal(q3, qi) and np.array_equal(s3, si)
    # ... and attention reads them back exactly (codes of 7 bits times powers of two are half values)
    assert np.array_equal(O.kv_q8_store(qi * si[:, None]), qi * si[:, None])
    # reading rounds the scale and the product to half precision: s = 0.1 (float32) is read as
    # 0.0999755859375, and 127 * that (12.6968994140625) as 12.6953125 (half spacing 2^-7 there)
    assert O.kv_q8_read(np.array([[127, 1]]), np.array([np.float32(0.1)]))[0].tolist() == [12.6953125,
                                                                                             0.0999755859375]


def _q8_small():
    wl = shrink(synth.WORKLOADS["small-bf16-gqa4"], n_layers=4, vocab=1024)
    w = synth.host_weights(wl.target, wl.draft_layers, wl.dtype)
    tg, dr = oracle_models(wl, w)
    import dataclasses
    return wl, dataclasses.replace(tg, kv_format="q8"), dr


def test_q8_block_forward_equals_row_by_row():
    """The block's own keys and values go through the 8-bit cache before
    attention reads them: a causal forward of n rows equals n one-row
    forwards that each read the earlier rows back from the cache."""
    wl, tg, _ = _q8_small()
    rnd = O.Rounder("bf16")
    toks = synth.prompt_tokens(12, wl.target.vocab)
    sh = tg.shape
    c1 = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    o1 = O.target_forward(tg, toks, c1, rnd)
    c2 = O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    rows = []
    for t in toks:
        o = O.target_forward(tg, [t], c2, rnd)
        O.commit(c2, o, 1)
        rows.append(o.logits[0])
    assert np.allclose(o1.logits, np.array(rows), rtol=0, atol=1e-9)
    # the cached entries are half-precision values ...
    assert np.array_equal(O.round_f16(c2.k[1]), c2.k[1]) and np.array_equal(O.round_f16(c2.v[2]), c2.v[2])
    # ... within one quantisation step of the bf16 configuration's layer-0 keys (same layer input), and
    # not equal to them (the quantisation is not a no-op)
    import dataclasses
    ob = O.target_forward(dataclasses.replace(tg, kv_format="bf16"), toks, O.KV.empty(sh.n_layers, sh.n_kv, sh.head_dim),
                          rnd)
    step = np.max(np.abs(ob.new_k[0]), axis=-1, keepdims=True) / 127.0
    assert np.all(np.abs(o1.new_k[0] - ob.new_k[0]) <= step)
    assert not np.allclose(ob.new_k[0], o1.new_k[0], atol=1e-6)


def test_lossless_q8_cache():
    wl, tg, dr = _q8_small()
    rnd = O.Rounder("bf16")
    prompt = synth.prompt_tokens(40, wl.target.vocab)
    n = 20
    ref, _ = O.greedy_ar(tg, prompt, n + wl.block, rnd)
    k, r = synth.acceptance_draws(32, wl.target.vocab)
    out, steps = O.spec_decode(tg, dr, prompt, n, wl.block, rnd, forcing=(k[:, 0], r[:, 0]), ref=ref)
    assert np.array_equal(out, ref[:n])
