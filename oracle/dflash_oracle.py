"""Plain CPU oracle for one DFlash speculative-decoding step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: it is used by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It
shares no code with the CUDA library and does not import it.

Everything is float64 NumPy.  The matrix product (``@``) and ``np.exp`` /
``np.cos`` / ``np.sin`` are the only library primitives; every step of the
method is written out in the order the pages state it, with no blocking,
fusion or reordering.

Sources (page titles as printed on the pages):

* [DD]  "DFlash 深度解析：块扩散模型如何让 LLM 推理加速 6 倍——2026 投机解码完全指南"
        (chenxutan.com) -- §1.1 autoregressive pseudocode, §1.2 speculative
        decoding, §2.2 architecture (feature_fusion, kv_injection,
        draft_inference), §3.3 shared embedding / LM head, §5.1 draft
        generation, §5.2 feature injection, §8.2 linear verification.
* [LC]  "从 ICML 论文到你的显卡：llama.cpp 吞下 DFlash，本地推理进入 2 倍速时代"
        (arex-research.com) -- "投机解码的瓶颈从来不是验证，而是 draft" (accept
        the matching prefix, cut at the first error) and "KV Injection".
* [RD]  "我在llama.cpp中测试了最新合并的DFlash在Qwen 3.6 27B本地AI上的表现"
        (bittide.aicompass.dev) -- greedy verification is lossless; 15-token
        block limit.

Precision.  ``rounding="none"`` keeps every intermediate in float64 (used for
the fp32 configuration).  ``rounding="bf16"`` rounds to bfloat16 (round to
nearest even) exactly at the storage points the bf16 configuration defines:
every matrix-product input that is an activation (the gain-weighted hidden
state entering a normed product -- see ``norm_linear`` --, attention output,
SwiGLU output, captured hidden states, fused feature), the query/key/value
entries that attention consumes (after RoPE), and nothing else; residual
stream and logits stay float64.

Parity pins: every function here is pinned by a test under ``tests/`` against
values the pages print, closed forms, invariants or brute force.  The one
composition that no page fixes beyond its pseudocode -- the order of the
drafter's sub-layers (pre-norm attention then SwiGLU) -- is marked
"parity unpinned" in ``draft_forward``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# Shapes and weights
# ---------------------------------------------------------------------------


@dataclass
class Shape:
    """Dimensions of one decoder (target or drafter)."""

    n_layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float = 1.0e6
    eps: float = 1.0e-6


@dataclass
class Layer:
    """One pre-norm decoder layer, stored as plain ``nn.Linear`` matrices [out, in]."""

    attn_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    ffn_norm: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray


@dataclass
class Target:
    shape: Shape
    embed: np.ndarray
    layers: list
    final_norm: np.ndarray
    lm_head: np.ndarray
    capture: tuple
    kv_format: str = "bf16"   # the target's K/V cache: "bf16" or "q8" (``kv_q8_store``)


@dataclass
class Draft:
    """Block-diffusion drafter.  Its token embedding and LM head are the
    target's ([DD] §3.3: shared and frozen), so only these are its own."""

    shape: Shape
    w_fc: np.ndarray          # [H, 5H]  fusion Linear
    fc_norm: np.ndarray       # [H]      fusion RMSNorm gain
    layers: list
    final_norm: np.ndarray
    mask_id: int


def f64(a):
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Rounding
# ---------------------------------------------------------------------------


def round_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even).

    bfloat16 keeps 8 significant bits and float32's exponent range.  Written
    from that definition: x = m * 2**e with 0.5 <= |m| < 1, so the quantum is
    2**(e-8) for normal numbers and 2**-133 below 2**-126 (subnormals)."""
    x = f64(x)
    _, e = np.frexp(x)
    q = np.maximum(e.astype(np.int64) - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(x, -q)), q)
    big = np.abs(y) > 3.3895313892515355e38
    return np.where(big, np.copysign(np.inf, x), y)


class Rounder:
    def __init__(self, mode: str):
        if mode not in ("none", "bf16"):
            raise ValueError(mode)
        self.mode = mode

    def __call__(self, x):
        return round_bf16(x) if self.mode == "bf16" else f64(x)


def round_f16(x):
    """Round to IEEE half precision, nearest even (NumPy's float16 conversion:
    11 significant bits, largest finite 65504)."""
    with np.errstate(over="ignore"):
        return f64(np.asarray(x, dtype=np.float64).astype(np.float16))


# ---------------------------------------------------------------------------
# 8-bit K/V cache
# ---------------------------------------------------------------------------
# The pages run the target's cache quantised ([DD] §8.3 "显存优化" 方案3, a
# 3-bit KV cache; the tutorial's llama.cpp runs, §5 and §7, with 5-bit keys
# and 4-bit values) but print no format.  Reading: "q8" keeps each cached
# key or value row of head_dim entries as 8-bit integers q in [-127, 127]
# with one float32 scale s per row (per position and KV head), the entry
# being q * s.  A row is quantised from its float32 value (the key after
# RoPE): s = max|x| / 127 and q = round-half-even(x / s), both in float32
# arithmetic; a row of zeros keeps s = 0.  Every row the target writes --
# the block's own rows included -- is stored this way before attention reads
# it.  Attention computes in IEEE half precision: the query enters rounded to
# half, and each cached entry is read as the half-precision product of its
# code and its scale rounded to half, round_f16(q * round_f16(s)).


def quantize_q8(x):
    """Quantise rows (last axis) to (q int8, s float32) as stated above."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1, keepdims=True)
    s = amax / np.float32(127.0)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    t = np.where(s > 0, x32 / safe, np.float32(0.0)).astype(np.float32)
    q = np.clip(np.rint(t), -127, 127).astype(np.int8)
    return q, s[..., 0].astype(np.float32)


def dequantize_q8(q, s):
    """The stored entries q * s (float64, exact)."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float64)[..., None]


def kv_q8_read(q, s):
    """The entries as attention reads them: round_f16(q * round_f16(s)) (the
    product of an 8-bit code and an 11-bit scale is exact in float64)."""
    return round_f16(np.asarray(q, dtype=np.float64) * round_f16(np.asarray(s, dtype=np.float64))[..., None])


def kv_q8_store(x):
    """What attention reads from a q8 cache that was given the rows x."""
    return kv_q8_read(*quantize_q8(x))


# ---------------------------------------------------------------------------
# Building blocks
# ---------------------------------------------------------------------------


def layer_indices(n_layers: int) -> list:
    """The 5 captured target layers: spread uniformly from layer 2 to the
    third-from-last layer ([DD] §2.2 feature_fusion: ``[2, mid1, mid2, mid3,
    len-3]``).  0-based decoder-layer indices, the three middle ones at the
    evenly spaced points rounded half up."""
    lo, hi = 2, n_layers - 3
    out = []
    for i in range(5):
        t = lo + (hi - lo) * i / 4.0
        out.append(int(math.floor(t + 0.5)))
    return out


def rmsnorm(x, gain, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gain ([DD] §2.2)."""
    x = f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * f64(gain)


def linear(x, w):
    """nn.Linear without bias: y = x W^T, W stored [out, in]."""
    return f64(x) @ f64(w).T


def norm_linear(x, gain, eps, ws, rnd):
    """The products of RMSNorm(x) * gain with each matrix of ``ws`` (the
    pre-norm sub-layers and the LM head, [DD] §2.2).

    Exactly, RMSNorm(x) * gain = r * (x * gain) with the row scale
    r = 1 / sqrt(mean(x^2) + eps), so each product equals r * ((x * gain) W^T).
    With bf16 rounding the operand that is stored and enters the products is
    x * gain rounded to bf16, and r (from the unrounded x) scales the
    products' results; without rounding the normed rows are formed first and
    the arithmetic is plain ``rmsnorm`` then ``linear``."""
    if rnd.mode == "none":
        h = rmsnorm(x, gain, eps)
        return [linear(h, w) for w in ws]
    x = f64(x)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    hg = rnd(x * f64(gain))
    return [linear(hg, w) * r for w in ws]


def silu(x):
    x = f64(x)
    return x / (1.0 + np.exp(-x))


def rope(x, positions, theta):
    """Rotary position embedding, rotate-half pairing.

    x: [n, heads, d]; positions: [n].  Pair (i, i+d/2) of a head vector is
    rotated by the angle pos * theta**(-2i/d)."""
    x = f64(x)
    n, _, d = x.shape
    half = d // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention(q, k, v, allowed):
    """Scaled dot-product attention for one head.

    q [nq, d], k [nk, d], v [nk, d], allowed [nq, nk] boolean.
    softmax(q k^T / sqrt(d)) v with disallowed keys removed."""
    q, k, v = f64(q), f64(k), f64(v)
    s = q @ k.T / math.sqrt(q.shape[-1])
    s = np.where(allowed, s, -np.inf)
    s = s - np.max(s, axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / np.sum(p, axis=-1, keepdims=True)
    return p @ v


def argmax_top2(logits):
    """Greedy token (lowest index among equal maxima) and the gap between the
    two largest logits, per row."""
    logits = f64(logits)
    idx = np.argmax(logits, axis=-1)
    top2 = np.sort(logits, axis=-1)[..., -2:]
    return idx.astype(np.int64), top2[..., 1] - top2[..., 0]


# ---------------------------------------------------------------------------
# KV cache (plain per-layer arrays)
# ---------------------------------------------------------------------------


@dataclass
class KV:
    """Keys/values per layer: lists of [n_kv, P, d] float64 arrays."""

    k: list = field(default_factory=list)
    v: list = field(default_factory=list)

    @staticmethod
    def empty(n_layers, n_kv, d):
        return KV([np.zeros((n_kv, 0, d)) for _ in range(n_layers)],
                  [np.zeros((n_kv, 0, d)) for _ in range(n_layers)])

    def length(self):
        return self.k[0].shape[1] if self.k else 0

    def append(self, layer, k_rows, v_rows):
        """k_rows/v_rows: [n, n_kv, d] at the next positions."""
        self.k[layer] = np.concatenate([self.k[layer], np.transpose(k_rows, (1, 0, 2))], axis=1)
        self.v[layer] = np.concatenate([self.v[layer], np.transpose(v_rows, (1, 0, 2))], axis=1)

    def truncate(self, length):
        for i in range(len(self.k)):
            self.k[i] = self.k[i][:, :length]
            self.v[i] = self.v[i][:, :length]

    def copy(self):
        return KV([a.copy() for a in self.k], [a.copy() for a in self.v])


# ---------------------------------------------------------------------------
# One decoder layer
# ---------------------------------------------------------------------------


def store_qkv(q, k, v, rnd, kv_format):
    """The query, keys and values as attention consumes them: rounded at the
    bf16 storage points, or (``kv_format`` "q8") keys and values through the
    8-bit cache and the query in half precision."""
    if kv_format == "q8":
        if rnd.mode != "bf16":
            raise ValueError("the 8-bit cache belongs to the bf16 configuration")
        return round_f16(q), kv_q8_store(k), kv_q8_store(v)
    return rnd(q), rnd(k), rnd(v)


def decoder_layer(x, lw: Layer, shape: Shape, ctx_k, ctx_v, pos0, causal, rnd, kv_format="bf16"):
    """Pre-norm decoder layer on the rows x [n, H] at positions pos0..pos0+n-1.

    Keys/values attended: the context ctx_k/ctx_v [n_kv, P, d] (positions
    0..P-1) followed by the rows' own keys/values.  ``causal``: row j sees the
    context and rows 0..j (target verification, [DD] §1.2).  Otherwise every
    row sees the context and every row (the drafter's in-block bidirectional
    attention, [DD] §2.2 "块内双向注意力").

    ``kv_format`` "q8" (bf16 rounding only): the rows' keys and values are
    stored in the 8-bit cache (``kv_q8_store``) and read back from it, and
    the query enters attention in half precision.

    Returns the new residual rows and the rows' (rounded) keys/values
    [n, n_kv, d] that a cache would append."""
    n = x.shape[0]
    d, nq, nkv = shape.head_dim, shape.n_q, shape.n_kv
    pos = pos0 + np.arange(n)
    yq, yk, yv = norm_linear(x, lw.attn_norm, shape.eps, (lw.wq, lw.wk, lw.wv), rnd)
    q = rope(yq.reshape(n, nq, d), pos, shape.rope_theta)
    k = rope(yk.reshape(n, nkv, d), pos, shape.rope_theta)
    v = yv.reshape(n, nkv, d)
    q, k, v = store_qkv(q, k, v, rnd, kv_format)
    P = ctx_k.shape[1]
    allowed = np.ones((n, P + n), dtype=bool)
    if causal:
        allowed[:, P:] = np.tril(np.ones((n, n), dtype=bool))
    group = nq // nkv
    o = np.zeros((n, nq, d))
    for hq in range(nq):
        hk = hq // group
        keys = np.concatenate([ctx_k[hk], k[:, hk]], axis=0)
        vals = np.concatenate([ctx_v[hk], v[:, hk]], axis=0)
        o[:, hq] = attention(q[:, hq], keys, vals, allowed)
    o = rnd(o.reshape(n, nq * d))
    x = f64(x) + linear(o, lw.wo)
    yg, yu = norm_linear(x, lw.ffn_norm, shape.eps, (lw.w_gate, lw.w_up), rnd)
    a = rnd(silu(yg) * yu)
    x = x + linear(a, lw.w_down)
    return x, k, v


# ---------------------------------------------------------------------------
# Target forward (prefill / verification / autoregressive step)
# ---------------------------------------------------------------------------


@dataclass
class TargetOut:
    argmax: np.ndarray        # [n]
    gap: np.ndarray           # [n] top-2 logit gap
    logits: np.ndarray        # [n, V]
    hcap: np.ndarray          # [n, 5H] captured hidden states (rounded)
    new_k: list               # per layer [n, n_kv, d]
    new_v: list


def target_forward(tg: Target, tokens, cache: KV, rnd, keep_logits=True):
    """Causal target forward of ``tokens`` at positions P..P+n-1 where P is the
    cache length.  The cache is NOT modified; the caller appends new_k/new_v
    for the rows it commits.  Captures the residual stream after each layer
    of ``tg.capture`` ([DD] §2.2 feature_fusion: hidden states of 5 layers)."""
    sh = tg.shape
    tokens = np.asarray(tokens, dtype=np.int64)
    P = cache.length()
    x = f64(tg.embed)[tokens]
    caps = {}
    new_k, new_v = [], []
    for li, lw in enumerate(tg.layers):
        x, k, v = decoder_layer(x, lw, sh, cache.k[li], cache.v[li], P, True, rnd, tg.kv_format)
        new_k.append(k)
        new_v.append(v)
        if li in tg.capture:
            caps[li] = rnd(x)
    hcap = np.concatenate([caps[i] for i in tg.capture], axis=-1)
    logits = norm_linear(x, tg.final_norm, sh.eps, (tg.lm_head,), rnd)[0]
    am, gap = argmax_top2(logits)
    return TargetOut(am, gap, logits if keep_logits else None, hcap, new_k, new_v)


def commit(cache: KV, out: TargetOut, rows: int):
    """Append the first ``rows`` rows of a forward's keys/values to the cache."""
    for li in range(len(cache.k)):
        cache.append(li, out.new_k[li][:rows], out.new_v[li][:rows])


# ---------------------------------------------------------------------------
# DFlash stages
# ---------------------------------------------------------------------------


def fuse_features(dr: Draft, hcap, rnd):
    """Feature fusion ([DD] §2.2 feature_fusion): the 5 captured hidden states
    are concatenated (already, in hcap [m, 5H]) -> Linear -> RMSNorm."""
    return rnd(rmsnorm(linear(hcap, dr.w_fc), dr.fc_norm, dr.shape.eps))


def inject_kv(dr: Draft, fused, positions, rnd):
    """KV injection ([DD] §2.2 kv_injection, §5.2; [LC] "KV Injection"): every
    drafter layer projects the fused context feature with its own K and V
    projections; the keys carry RoPE at the context position.  Returns per
    layer ([m, n_kv, d] keys, values) to append to that layer's cache."""
    sh = dr.shape
    m = fused.shape[0]
    out = []
    for lw in dr.layers:
        k = rope(linear(fused, lw.wk).reshape(m, sh.n_kv, sh.head_dim), positions, sh.rope_theta)
        v = linear(fused, lw.wv).reshape(m, sh.n_kv, sh.head_dim)
        out.append((rnd(k), rnd(v)))
    return out


def cross_window(P: int, window: int) -> int:
    """First injected context position the drafter attends to.  The tutorial
    page ("如何使用 DFlash 试探式解码加速本地 LLM", §7) runs the drafter with
    ``--spec-dflash-cross-ctx 1024`` and says nothing more; the reading taken
    here: with a cross-context window W > 0 the drafter's attention keeps only
    the W most recent injected positions P-W..P-1 (all of them when P <= W),
    and always the block's own B rows.  W = 0 keeps the whole context."""
    return max(0, P - window) if window > 0 else 0


def draft_logits(dr: Draft, tg: Target, anchor: int, block: int, dcache: KV, rnd, window: int = 0):
    """One non-causal drafter forward over the block [anchor, MASK x (B-1)] at
    positions P..P+B-1 (P = drafter cache length): [DD] §5.1 "given [T1] +
    target_model_context -> single forward pass -> [T2,...]", §2.2
    draft_inference.  Tokens are embedded with the target's embedding and
    decoded with the target's LM head ([DD] §3.3).  ``window``: the
    cross-context window (``cross_window``); the kept keys carry their
    absolute positions, so only which keys are attended changes.

    parity unpinned: the sub-layer order of the drafter (pre-norm attention,
    then pre-norm SwiGLU, then a final RMSNorm) is not printed on any page.

    Returns the logits [B-1, V] of slots 1..B-1 (slot 0 holds the anchor,
    whose logits are not used)."""
    sh = dr.shape
    P = dcache.length()
    lo = cross_window(P, window)
    toks = np.array([anchor] + [dr.mask_id] * (block - 1), dtype=np.int64)
    x = f64(tg.embed)[toks]
    for li, lw in enumerate(dr.layers):
        x, _, _ = decoder_layer(x, lw, sh, dcache.k[li][:, lo:], dcache.v[li][:, lo:], P, False, rnd)
    return norm_linear(x[1:], dr.final_norm, sh.eps, (tg.lm_head,), rnd)[0]


def draft_forward(dr: Draft, tg: Target, anchor: int, block: int, dcache: KV, rnd, window: int = 0):
    """The drafter's greedy block: argmax of each slot's logits
    (``draft_logits``).  Returns the B drafted tokens, slot 0 holding the
    anchor itself, and the top-2 gaps of slots 1..B-1."""
    am, gap = argmax_top2(draft_logits(dr, tg, anchor, block, dcache, rnd, window))
    return np.concatenate([[anchor], am]).astype(np.int64), gap


def accept_length(draft_tokens, target_argmax):
    """Longest accepted prefix ([DD] §1.2, §8.2 linear verification; [LC]:
    keep the matching prefix, cut at the first error).  Slot i >= 1 of the
    block is accepted when it equals the target's greedy choice after slot
    i-1; the count stops at the first mismatch.  Returns a in [0, B-1]; the
    step emits target_argmax[0..a] (a drafted tokens plus one target token)."""
    B = len(draft_tokens)
    a = 0
    while a < B - 1 and int(draft_tokens[a + 1]) == int(target_argmax[a]):
        a += 1
    return a


def teacher_force(draft_tokens, ref, emitted, k, r, vocab):
    """Overwrite drafted slots so that exactly min(k, B-1) are accepted.

    Slots 1..min(k, B-1) take the reference greedy tokens ref[emitted + j - 1];
    when k + 1 <= B - 1, slot k+1 takes (ref[emitted + k] + 1 + r) mod V with
    r in [0, V-2], which differs from the reference token.  k and r are drawn
    by the caller."""
    d = np.array(draft_tokens, dtype=np.int64).copy()
    B = len(d)
    kk = min(int(k), B - 1)
    for j in range(1, kk + 1):
        d[j] = ref[emitted + j - 1]
    if kk + 1 <= B - 1:
        d[kk + 1] = (int(ref[emitted + kk]) + 1 + int(r)) % vocab
    return d


# ---------------------------------------------------------------------------
# Whole decodes
# ---------------------------------------------------------------------------


def greedy_ar(tg: Target, prompt, n_tokens, rnd):
    """Plain greedy autoregressive decoding ([DD] §1.1): forward, take the
    argmax of the last row, append, repeat.  Returns tokens and top-2 gaps."""
    sh = tg.shape
    cache = KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    out = target_forward(tg, prompt, cache, rnd, keep_logits=False)
    commit(cache, out, len(prompt))
    toks, gaps = [int(out.argmax[-1])], [float(out.gap[-1])]
    while len(toks) < n_tokens:
        out = target_forward(tg, [toks[-1]], cache, rnd, keep_logits=False)
        commit(cache, out, 1)
        toks.append(int(out.argmax[0]))
        gaps.append(float(out.gap[0]))
    return np.array(toks, dtype=np.int64), np.array(gaps)


def greedy_ar_recompute(tg: Target, prompt, n_tokens, rnd):
    """Greedy decoding with no cache at all: every token re-runs the whole
    sequence from position 0 (the literal form of [DD] §1.1)."""
    sh = tg.shape
    seq = list(int(t) for t in prompt)
    toks = []
    while len(toks) < n_tokens:
        out = target_forward(tg, seq, KV.empty(sh.n_layers, sh.n_kv, sh.head_dim), rnd,
                             keep_logits=False)
        toks.append(int(out.argmax[-1]))
        seq.append(toks[-1])
    return np.array(toks, dtype=np.int64)


@dataclass
class StepRecord:
    P: int                    # committed target length at step start
    anchor: int
    draft: np.ndarray         # B tokens, slot 0 = anchor
    argmax: np.ndarray        # B target greedy tokens
    gap: np.ndarray           # B target top-2 gaps
    accept: int               # a
    emitted: np.ndarray       # a + 1 tokens


def spec_decode(tg: Target, dr: Draft, prompt, n_tokens, block, rnd, forcing=None, ref=None,
                max_steps=None, window=0):
    """DFlash speculative decoding, greedy ([DD] §1.2, §2.2, §5.1; [LC]).

    prefill : target forward over the prompt, cache its keys/values, capture
              its hidden states, emit the greedy token (the first anchor).
    per step: fuse the pending captured rows, inject them into every drafter
              layer's cache, draft one block, verify it with one causal target
              forward, accept the matching prefix plus one target token, and
              roll back: keep only the accepted rows' target keys/values and
              leave those rows' captured states pending for the next step.

    forcing: optional (k[steps], r[steps]) teacher-forcing draws; ``ref`` is
    the reference greedy stream they index (length >= n_tokens + block).
    window: the drafter's cross-context window (``cross_window``)."""
    sh, dsh = tg.shape, dr.shape
    tcache = KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    dcache = KV.empty(dsh.n_layers, dsh.n_kv, dsh.head_dim)
    prompt = np.asarray(prompt, dtype=np.int64)
    out = target_forward(tg, prompt, tcache, rnd, keep_logits=False)
    commit(tcache, out, len(prompt))
    pending = out.hcap
    emitted = [int(out.argmax[-1])]
    anchor = emitted[0]
    steps = []
    while len(emitted) < n_tokens:
        if max_steps is not None and len(steps) >= max_steps:
            break
        P = tcache.length()
        # fuse + inject the pending rows (positions P - m .. P - 1)
        m = pending.shape[0]
        fused = fuse_features(dr, pending, rnd)
        for li, (k, v) in enumerate(inject_kv(dr, fused, np.arange(P - m, P), rnd)):
            dcache.append(li, k, v)
        # draft
        d, _ = draft_forward(dr, tg, anchor, block, dcache, rnd, window)
        if forcing is not None:
            ks, rs = forcing
            s = len(steps)
            d = teacher_force(d, ref, len(emitted), ks[s], rs[s], sh.vocab)
        # verify
        out = target_forward(tg, d, tcache, rnd, keep_logits=False)
        a = accept_length(d, out.argmax)
        em = out.argmax[: a + 1].copy()
        steps.append(StepRecord(P, anchor, d, out.argmax.copy(), out.gap.copy(), a, em))
        emitted.extend(int(t) for t in em)
        # rollback: keep rows 0..a
        commit(tcache, out, a + 1)
        pending = out.hcap[: a + 1]
        anchor = int(em[-1])
    return np.array(emitted[:n_tokens], dtype=np.int64), steps


# ---------------------------------------------------------------------------
# Tree verification (DDTree)
# ---------------------------------------------------------------------------
#
# "DFlash 深度解析" §8.2: one target forward explores several branches of the
# drafter's guesses within a node budget, instead of a single chain; the page
# sketches the idea and prints no algorithm.  The reading taken here:
#   * candidates: for each drafted slot j = 1..B-1, the drafter's top-K tokens
#     by log-probability log q_j (softmax of the slot's logits), ranks 0..K-1
#     (ties to the lower token id);
#   * the tree: the `budget` highest-scoring token prefixes (c_1..c_d) under the
#     score sum_j log q_j(c_j) (the drafter predicts its slots in one pass, so
#     a prefix's probability under it is the product of the slots'
#     marginals), found best-first; every prefix's parent prefix scores at
#     least as high, so the set is a tree rooted at the anchor.  Ties between
#     equal scores go to the smaller depth, then to the smaller rank at that
#     depth, then to the earlier parent;
#   * verification: one causal target forward over [anchor, nodes in creation
#     order] in which node i sits at position P + depth(i) and attends to the
#     context and to its ancestors (itself included) only;
#   * acceptance: from the root, move to the child whose token equals the
#     target's greedy token after the current node, while there is one; the
#     step emits the tokens of the accepted path and the target's greedy token
#     after its last node (the bonus), exactly as linear verification does on
#     a chain.  With K = 1 and budget B-1 the tree is the drafter's greedy chain
#     and the step is linear verification.


@dataclass
class Tree:
    tokens: np.ndarray   # [N+1] node 0 = anchor
    parent: np.ndarray   # [N+1] parent index (-1 for the root)
    depth: np.ndarray    # [N+1] 0 for the root
    score: np.ndarray    # [N+1] sum of log q along the path (0 for the root)


def log_softmax(logits):
    z = f64(logits)
    z = z - np.max(z, axis=-1, keepdims=True)
    return z - np.log(np.sum(np.exp(z), axis=-1, keepdims=True))


def topk_candidates(draft_logits_rows, k):
    """Per slot row: the k highest log-probabilities and their tokens (ties
    to the lower token id)."""
    lp = log_softmax(draft_logits_rows)
    toks = np.argsort(-lp, axis=-1, kind="stable")[:, :k]
    return toks.astype(np.int64), np.take_along_axis(lp, toks, axis=-1)


def build_tree(anchor, cand_tok, cand_lp, budget):
    """The `budget` best prefixes, best-first.  cand_tok/cand_lp [B-1, K]
    sorted by rank.  A frontier entry (score, depth, rank, parent) stands for
    the prefix parent + candidate `rank` of slot `depth`; taking one adds its
    next sibling (rank + 1) and its first child (depth + 1, rank 0)."""
    D, K = cand_tok.shape
    tokens, parent, depth, score = [int(anchor)], [-1], [0], [0.0]
    frontier = [(float(cand_lp[0, 0]), 1, 0, 0)] if D >= 1 and K >= 1 else []
    while frontier and len(tokens) - 1 < budget:
        best = min(frontier, key=lambda e: (-e[0], e[1], e[2], e[3]))
        frontier.remove(best)
        sc, d, r, par = best
        node = len(tokens)
        tokens.append(int(cand_tok[d - 1, r]))
        parent.append(par)
        depth.append(d)
        score.append(sc)
        if r + 1 < K:
            frontier.append((score[par] + float(cand_lp[d - 1, r + 1]), d, r + 1, par))
        if d + 1 <= D:
            frontier.append((sc + float(cand_lp[d, 0]), d + 1, 0, node))
    return Tree(np.array(tokens, np.int64), np.array(parent, np.int64), np.array(depth, np.int64),
                np.array(score, np.float64))


def tree_ancestors(tree: Tree):
    """allowed[i, j]: node j is node i or one of its ancestors."""
    n = len(tree.tokens)
    allowed = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        while j >= 0:
            allowed[i, j] = True
            j = int(tree.parent[j])
    return allowed


def target_forward_tree(tg: Target, tree: Tree, cache: KV, rnd):
    """Target forward of the tree's nodes (see above).  Returns argmax, gap,
    hcap, new keys/values per node row, like ``target_forward``."""
    sh = tg.shape
    P = cache.length()
    tokens = tree.tokens
    n = len(tokens)
    allowed_block = tree_ancestors(tree)
    d, nq, nkv = sh.head_dim, sh.n_q, sh.n_kv
    pos = P + tree.depth
    x = f64(tg.embed)[tokens]
    caps, new_k, new_v = {}, [], []
    for li, lw in enumerate(tg.layers):
        yq, yk, yv = norm_linear(x, lw.attn_norm, sh.eps, (lw.wq, lw.wk, lw.wv), rnd)
        q, k, v = store_qkv(rope(yq.reshape(n, nq, d), pos, sh.rope_theta),
                            rope(yk.reshape(n, nkv, d), pos, sh.rope_theta), yv.reshape(n, nkv, d), rnd, tg.kv_format)
        allowed = np.concatenate([np.ones((n, P), dtype=bool), allowed_block], axis=1)
        group = nq // nkv
        o = np.zeros((n, nq, d))
        for hq in range(nq):
            hk = hq // group
            keys = np.concatenate([cache.k[li][hk], k[:, hk]], axis=0)
            vals = np.concatenate([cache.v[li][hk], v[:, hk]], axis=0)
            o[:, hq] = attention(q[:, hq], keys, vals, allowed)
        o = rnd(o.reshape(n, nq * d))
        x = x + linear(o, lw.wo)
        yg, yu = norm_linear(x, lw.ffn_norm, sh.eps, (lw.w_gate, lw.w_up), rnd)
        a = rnd(silu(yg) * yu)
        x = x + linear(a, lw.w_down)
        new_k.append(k)
        new_v.append(v)
        if li in tg.capture:
            caps[li] = rnd(x)
    hcap = np.concatenate([caps[i] for i in tg.capture], axis=-1)
    logits = norm_linear(x, tg.final_norm, sh.eps, (tg.lm_head,), rnd)[0]
    am, gap = argmax_top2(logits)
    return TargetOut(am, gap, logits, hcap, new_k, new_v)


def accept_tree(tree: Tree, target_argmax):
    """Walk from the root along the children that match the target's greedy
    token.  Returns (path node indices, emitted tokens): a = len(path) - 1
    drafted tokens plus the bonus."""
    path = [0]
    while True:
        x = path[-1]
        g = int(target_argmax[x])
        nxt = [c for c in range(len(tree.tokens)) if tree.parent[c] == x and int(tree.tokens[c]) == g]
        if not nxt:
            break
        path.append(nxt[0])
    emitted = [int(tree.tokens[c]) for c in path[1:]] + [int(target_argmax[path[-1]])]
    return np.array(path, np.int64), np.array(emitted, np.int64)


def spec_decode_tree(tg: Target, dr: Draft, prompt, n_tokens, block, topk, budget, rnd, window=0):
    """DFlash speculative decoding with tree verification (greedy): per step
    fuse + inject the pending rows, one drafter forward, the tree of its top-k
    candidates, one tree-masked target forward, the walk, and the rollback:
    the accepted path's keys/values are committed at positions P..P+a and its
    captured rows become the pending rows.  Returns the emitted tokens and the
    per-step accepted counts."""
    sh, dsh = tg.shape, dr.shape
    tcache = KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    dcache = KV.empty(dsh.n_layers, dsh.n_kv, dsh.head_dim)
    prompt = np.asarray(prompt, dtype=np.int64)
    out = target_forward(tg, prompt, tcache, rnd, keep_logits=False)
    commit(tcache, out, len(prompt))
    pending = out.hcap
    emitted = [int(out.argmax[-1])]
    anchor = emitted[0]
    accepts = []
    while len(emitted) < n_tokens:
        P = tcache.length()
        m = pending.shape[0]
        fused = fuse_features(dr, pending, rnd)
        for li, (k, v) in enumerate(inject_kv(dr, fused, np.arange(P - m, P), rnd)):
            dcache.append(li, k, v)
        ct, cl = topk_candidates(draft_logits(dr, tg, anchor, block, dcache, rnd, window), topk)
        tree = build_tree(anchor, ct, cl, budget)
        out = target_forward_tree(tg, tree, tcache, rnd)
        path, em = accept_tree(tree, out.argmax)
        accepts.append(len(path) - 1)
        emitted.extend(int(t) for t in em)
        for li in range(len(tcache.k)):
            tcache.append(li, out.new_k[li][path], out.new_v[li][path])
        pending = out.hcap[path]
        anchor = int(em[-1])
    return np.array(emitted[:n_tokens], dtype=np.int64), accepts


# ---------------------------------------------------------------------------
# Sampling mode (temperature T > 0)
# ---------------------------------------------------------------------------
#
# "DFlash 深度解析" §4.2 reports the speed-up at temperature 1 with the
# losslessness kept, and prints no rule.  The reading taken here is the
# standard speculative-sampling rule, which keeps the emitted stream
# distributed exactly as sampling the target alone:
#   * the drafter samples slot j >= 1 from q_j = softmax(z_draft_j / T);
#   * drafted token d_i (i = 1..B-1) is accepted when u_i * q_i(d_i) < p_{i-1}(d_i),
#     p_{i-1} = softmax(z_target_{i-1} / T) being the target's distribution
#     after slot i-1 (probability min(1, p/q));
#   * at the first rejection (slot a+1) the step emits one token drawn from the
#     residual max(0, p_a - q_{a+1}) (renormalised), and stops;
#   * when every drafted token is accepted it emits a bonus token drawn from
#     p_{B-1}.
# A draw from a distribution w with a uniform v in [0, 1) is the inverse CDF:
# the smallest t with w_0 + ... + w_t > v * (w_0 + ... + w_{V-1}).  Uniform
# numbers are inputs (drawn by the caller).


def softmax_t(logits, T):
    """softmax(z / T) over the last axis, float64."""
    z = f64(logits) / float(T)
    z = z - np.max(z, axis=-1, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-1, keepdims=True)


def sample_inverse_cdf(weights, v):
    """Index drawn from the non-negative weights with uniform v in [0, 1)."""
    w = f64(weights)
    c = np.cumsum(w)
    return int(np.searchsorted(c, v * c[-1], side="right"))


def draft_sample(draft_logits_rows, T, w_draws):
    """Slots 1..B-1 sampled from q_j (rows of draft_logits_rows) with the
    uniform draws w_draws[j-1]."""
    q = softmax_t(draft_logits_rows, T)
    return np.array([sample_inverse_cdf(q[j], w_draws[j]) for j in range(q.shape[0])], dtype=np.int64)


def accept_sampling(draft_tokens, p_rows, q_rows, u, v):
    """Speculative-sampling verification of one block (see above).

    draft_tokens [B] (slot 0 = anchor); p_rows [B, V] target distributions
    (row i: after slot i); q_rows [B-1, V] drafter distributions of slots
    1..B-1; u [B-1] acceptance draws; v the draw of the residual / bonus
    token.  Returns (a, emitted): a accepted drafts and the a + 1 emitted
    tokens d_1..d_a, t."""
    B = len(draft_tokens)
    a = 0
    while a < B - 1:
        d = int(draft_tokens[a + 1])
        p, q = p_rows[a], q_rows[a]
        if u[a] * q[d] < p[d]:
            a += 1
            continue
        resid = np.maximum(p - q, 0.0)
        if not np.sum(resid) > 0.0:  # p == q: nothing left to correct, sample the target
            resid = p
        t = sample_inverse_cdf(resid, v)
        return a, np.array([int(x) for x in draft_tokens[1:a + 1]] + [t], dtype=np.int64)
    t = sample_inverse_cdf(p_rows[B - 1], v)
    return a, np.array([int(x) for x in draft_tokens[1:B]] + [t], dtype=np.int64)


def sample_ar(tg: Target, prompt, n_tokens, T, v_draws, rnd):
    """Autoregressive sampling of the target at temperature T ([DD] §1.1 with
    the argmax replaced by a draw): token k is drawn from softmax(z / T) of the
    last row with the uniform v_draws[k]."""
    sh = tg.shape
    cache = KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    out = target_forward(tg, prompt, cache, rnd)
    commit(cache, out, len(prompt))
    toks = [sample_inverse_cdf(softmax_t(out.logits[-1], T), v_draws[0])]
    while len(toks) < n_tokens:
        out = target_forward(tg, [toks[-1]], cache, rnd)
        commit(cache, out, 1)
        toks.append(sample_inverse_cdf(softmax_t(out.logits[0], T), v_draws[len(toks)]))
    return np.array(toks, dtype=np.int64)


def spec_decode_sampling(tg: Target, dr: Draft, prompt, n_tokens, block, T, draws, rnd, window=0):
    """DFlash speculative decoding in sampling mode: the loop of
    ``spec_decode`` with the drafter sampling its block and the target
    verifying by ``accept_sampling``.  draws = (v0, w[steps, B-1], u[steps,
    B-1], v[steps]): v0 draws the prefill's first token, then each step uses
    one row of w (drafting), u (acceptance) and v (residual or bonus).
    Returns the emitted tokens and the per-step accepted counts."""
    v0, w_all, u_all, v_all = draws
    sh, dsh = tg.shape, dr.shape
    tcache = KV.empty(sh.n_layers, sh.n_kv, sh.head_dim)
    dcache = KV.empty(dsh.n_layers, dsh.n_kv, dsh.head_dim)
    prompt = np.asarray(prompt, dtype=np.int64)
    out = target_forward(tg, prompt, tcache, rnd)
    commit(tcache, out, len(prompt))
    pending = out.hcap
    emitted = [sample_inverse_cdf(softmax_t(out.logits[-1], T), v0)]
    anchor = emitted[0]
    accepts = []
    while len(emitted) < n_tokens:
        s = len(accepts)
        P = tcache.length()
        m = pending.shape[0]
        fused = fuse_features(dr, pending, rnd)
        for li, (k, v) in enumerate(inject_kv(dr, fused, np.arange(P - m, P), rnd)):
            dcache.append(li, k, v)
        zq = draft_logits(dr, tg, anchor, block, dcache, rnd, window)
        d = np.concatenate([[anchor], draft_sample(zq, T, w_all[s])]).astype(np.int64)
        out = target_forward(tg, d, tcache, rnd)
        a, em = accept_sampling(d, softmax_t(out.logits, T), softmax_t(zq, T), u_all[s], v_all[s])
        accepts.append(a)
        emitted.extend(int(t) for t in em)
        commit(tcache, out, a + 1)
        pending = out.hcap[: a + 1]
        anchor = int(em[-1])
    return np.array(emitted[:n_tokens], dtype=np.int64), accepts


def tau(n_emitted_tokens, n_steps):
    """Mean tokens emitted per verification step."""
    return n_emitted_tokens / n_steps
