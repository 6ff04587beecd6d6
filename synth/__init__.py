"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no arithmetic of the method.  It only draws numbers:
random-init weights (N(0, 0.02) matrices, unit RMSNorm gains), uniform random
prompts, and the teacher-forcing draws (geometric accepted counts with mean 7,
uniform corruption offsets).  Seeds: weights 0, prompts 1, acceptance draws 2,
batch prompt lengths 3.

Weights are addressed by canonical name (``layers.3.wq``, ``draft.w_fc`` ...)
and every named tensor has its own generator, so a value never depends on
where a consumer stores it.  Small models are drawn on the host with NumPy's
PCG64; large ones on the GPU with torch's Philox generator (``fill_torch``).
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import numpy as np

WEIGHT_SEED = 0
PROMPT_SEED = 1
ACCEPT_SEED = 2
LENGTH_SEED = 3
INIT_STD = 0.02


@dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float = 1.0e6
    eps: float = 1.0e-6

    def asdict(self):
        return asdict(self)


@dataclass(frozen=True)
class Workload:
    """One named workload: target and drafter shapes plus the run recipe."""

    name: str
    target: ModelShape
    draft_layers: int
    dtype: str            # "f32" or "bf16"
    block: int
    prompt_len: int
    gen_tokens: int
    teacher_forced: bool
    batch: int = 1
    final_gain: float = 1.0   # initial value of the final RMSNorm gains (test workloads widen logit gaps)
    kv: str = "bf16"          # the target's K/V cache: "bf16" or "q8" (8-bit codes, a scale per row)

    @property
    def draft(self) -> ModelShape:
        t = self.target
        return ModelShape(self.draft_layers, t.hidden, t.n_q, t.n_kv, t.head_dim, t.ffn, t.vocab,
                          t.rope_theta, t.eps)


def _qwen3_8b_shape():
    return ModelShape(36, 4096, 32, 8, 128, 12288, 151936)


def _dense27b_shape():
    return ModelShape(64, 5120, 40, 8, 128, 25600, 151936)


WORKLOADS = {
    # tiny fp32 correctness case: 12 layers, hidden 256, 4 heads x 64, SwiGLU 768, vocab 2048
    "tiny-f32": Workload("tiny-f32", ModelShape(12, 256, 4, 4, 64, 768, 2048), 1, "f32", 16, 128, 64,
                         False),
    # small bf16 cases with the production head layout (d=128, GQA 4 and GQA 5)
    "small-bf16-gqa4": Workload("small-bf16-gqa4", ModelShape(6, 512, 4, 1, 128, 1024, 4096), 2, "bf16",
                                16, 96, 48, False),
    "small-bf16-gqa5": Workload("small-bf16-gqa5", ModelShape(6, 640, 5, 1, 128, 1280, 4096), 2, "bf16",
                                15, 80, 40, False),
    # Qwen3-8B-shaped target, 5-layer drafter, block 16, 4K prompt, teacher forced
    "qwen3-8b-4k": Workload("qwen3-8b-4k", _qwen3_8b_shape(), 5, "bf16", 16, 4096, 2048, True),
    # 27B-class dense target, block 15, 36K prompt, 1500 tokens, teacher forced
    "dense27b-36k": Workload("dense27b-36k", _dense27b_shape(), 5, "bf16", 15, 36864, 1500, True),
    # the same with the target's cache in 8 bits
    "dense27b-36k-q8": Workload("dense27b-36k-q8", _dense27b_shape(), 5, "bf16", 15, 36864, 1500, True, kv="q8"),
    # Qwen3-8B shapes, 8 sequences with prompt lengths uniform on 2048..6144
    # (batch_prompt_lengths; prompt_len is the upper end), block 16
    "qwen3-8b-batch8": Workload("qwen3-8b-batch8", _qwen3_8b_shape(), 5, "bf16", 16, 6144, 512, True, batch=8),
}


def prompt_lengths(wl: Workload):
    """Per-sequence prompt lengths of a workload."""
    if wl.batch == 1:
        return [wl.prompt_len]
    return [int(x) for x in batch_prompt_lengths(wl.batch, hi=wl.prompt_len)]


# ---------------------------------------------------------------------------
# Weight specs
# ---------------------------------------------------------------------------

LAYER_PARTS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def _layer_specs(prefix, s: ModelShape):
    H, d = s.hidden, s.head_dim
    return [
        (f"{prefix}attn_norm", (H,), "ones"),
        (f"{prefix}wq", (s.n_q * d, H), "normal"),
        (f"{prefix}wk", (s.n_kv * d, H), "normal"),
        (f"{prefix}wv", (s.n_kv * d, H), "normal"),
        (f"{prefix}wo", (H, s.n_q * d), "normal"),
        (f"{prefix}ffn_norm", (H,), "ones"),
        (f"{prefix}w_gate", (s.ffn, H), "normal"),
        (f"{prefix}w_up", (s.ffn, H), "normal"),
        (f"{prefix}w_down", (H, s.ffn), "normal"),
    ]


def weight_specs(target: ModelShape, draft_layers: int):
    """Ordered (name, shape, kind) of every weight; kind is "normal"
    (N(0, 0.02)) or "ones" (RMSNorm gain)."""
    H, V = target.hidden, target.vocab
    specs = [("embed", (V, H), "normal")]
    for i in range(target.n_layers):
        specs += _layer_specs(f"layers.{i}.", target)
    specs += [("final_norm", (H,), "ones"), ("lm_head", (V, H), "normal")]
    specs += [("draft.w_fc", (H, 5 * H), "normal"), ("draft.fc_norm", (H,), "ones")]
    for i in range(draft_layers):
        specs += _layer_specs(f"draft.layers.{i}.", target)
    specs += [("draft.final_norm", (H,), "ones")]
    return specs


def spec_index(specs):
    return {name: i for i, (name, _, _) in enumerate(specs)}


# ---------------------------------------------------------------------------
# Host generation (NumPy)
# ---------------------------------------------------------------------------


def to_bf16_f32(a):
    """Round float32 values to bfloat16 (ties to even), returned as float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def host_tensor(name_index: int, shape, kind, dtype, seed=WEIGHT_SEED):
    if kind == "ones":
        return np.ones(shape, dtype=np.float32)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, name_index])))
    w = (rng.standard_normal(shape, dtype=np.float32) * np.float32(INIT_STD)).astype(np.float32)
    return to_bf16_f32(w) if dtype == "bf16" else w


def host_weights(target: ModelShape, draft_layers: int, dtype: str, seed=WEIGHT_SEED, final_gain=1.0):
    """All weights as float32 NumPy arrays (bf16-representable for "bf16")."""
    out = {}
    for i, (name, shape, kind) in enumerate(weight_specs(target, draft_layers)):
        out[name] = host_tensor(i, shape, kind, dtype, seed)
        if name in ("final_norm", "draft.final_norm"):
            out[name] = out[name] * np.float32(final_gain)
    return out


def workload_weights(wl: Workload, seed=WEIGHT_SEED):
    return host_weights(wl.target, wl.draft_layers, wl.dtype, seed, wl.final_gain)


# ---------------------------------------------------------------------------
# Device generation (torch), for models too large to draw on the host
# ---------------------------------------------------------------------------


def fill_torch(t, name_index: int, kind: str, seed=WEIGHT_SEED):
    """Fill a torch tensor (any device/dtype, possibly a strided view) in place."""
    import torch

    if kind == "ones":
        t.fill_(1.0)
        return t
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed) * 1_000_003 + int(name_index) + 17)
    tmp = torch.empty(t.shape, dtype=torch.float32, device=t.device)
    tmp.normal_(0.0, INIT_STD, generator=g)
    t.copy_(tmp)
    return t


# ---------------------------------------------------------------------------
# Prompts and acceptance draws
# ---------------------------------------------------------------------------


def prompt_tokens(n: int, vocab: int, seed=PROMPT_SEED, stream=0):
    """Uniform random ids on [0, V-2] (V-1 is the mask token)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return rng.integers(0, vocab - 1, size=n, dtype=np.int64)


def acceptance_draws(steps: int, vocab: int, batch=1, seed=ACCEPT_SEED, mean=7.0):
    """Teacher-forcing draws per (step, sequence): k ~ Geometric on {0,1,...}
    with mean ``mean`` (success probability 1/(mean+1)), r uniform on
    [0, V-2]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed])))
    p = 1.0 / (mean + 1.0)
    k = rng.geometric(p, size=(steps, batch)).astype(np.int64) - 1
    r = rng.integers(0, vocab - 1, size=(steps, batch), dtype=np.int64)
    return k, r


def batch_prompt_lengths(batch: int, lo=2048, hi=6144, seed=LENGTH_SEED):
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed])))
    return rng.integers(lo, hi + 1, size=batch, dtype=np.int64)


def gaussian(shape, seed, stream=0, scale=1.0, dtype=np.float32):
    """Generic N(0, scale^2) test tensor."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return (rng.standard_normal(shape) * scale).astype(dtype)
