"""Device-resident DFlash models and decoding sessions over the C ABI.

``Model`` owns the target's and the drafter's weights in the library's packed
layouts (q|k|v rows in one matrix, gate/up rows interleaved, the drafter's
k|v rows of every layer gathered for one injection product) and exposes each
canonical matrix as a view for loading.  ``Session`` owns the KV caches, the
workspace and the per-sequence device state, and sequences the stages:

    prefill (chunks of <= 128 rows): target_verify(commit) -> fuse -> inject
    step: fuse -> inject -> draft -> [teacher force] -> verify -> accept/rollback

Every stage is one call into libdflash.so; nothing here computes.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import capi

_DT = {"f32": (capi.F32, torch.float32), "bf16": (capi.BF16, torch.bfloat16)}
LAYER_PARTS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def desc_of(shape, dtype: str, n_layers=None) -> capi.ModelDesc:
    return capi.ModelDesc(n_layers if n_layers is not None else shape.n_layers, shape.hidden, shape.n_q, shape.n_kv,
                          shape.head_dim, shape.ffn, shape.vocab, shape.rope_theta, shape.eps, _DT[dtype][0])


class Model:
    """Target + drafter weights on the GPU.  ``shape`` has the fields n_layers,
    hidden, n_q, n_kv, head_dim, ffn, vocab, rope_theta, eps; the drafter has
    the target's width and ``draft_layers`` layers."""

    def __init__(self, shape, draft_layers: int, dtype: str, device="cuda", cross_ctx: int = 0):
        self.shape, self.draft_layers, self.dtype = shape, draft_layers, dtype
        self.cross_ctx = cross_ctx  # the drafter's cross-context window (0: whole context)
        self.device = torch.device(device)
        tdt = _DT[dtype][1]
        s = shape
        H, d, F, V = s.hidden, s.head_dim, s.ffn, s.vocab

        def alloc(*sh):
            return torch.empty(sh, dtype=tdt, device=self.device)

        def layer():
            return {"attn_norm": alloc(H), "wqkv": alloc((s.n_q + 2 * s.n_kv) * d, H), "wo": alloc(H, s.n_q * d),
                    "ffn_norm": alloc(H), "w_gate_up": alloc(2 * F, H), "w_down": alloc(H, F)}

        self.embed, self.final_norm, self.lm_head = alloc(V, H), alloc(H), alloc(V, H)
        self.layers = [layer() for _ in range(s.n_layers)]
        self.w_fc, self.fc_norm, self.d_final_norm = alloc(H, 5 * H), alloc(H), alloc(H)
        self.dlayers = [layer() for _ in range(draft_layers)]
        self.w_kv_all = alloc(draft_layers * 2 * s.n_kv * d, H)
        self.capture = capi.dflash_capture_layers(s.n_layers)
        self.mask_id = V - 1
        self._structs = None

    # -------------------------------------------------------------- loading
    def _layer_views(self, lw):
        s, d = self.shape, self.shape.head_dim
        q, kv = s.n_q * d, s.n_kv * d
        return {"attn_norm": lw["attn_norm"], "wq": lw["wqkv"][:q], "wk": lw["wqkv"][q:q + kv],
                "wv": lw["wqkv"][q + kv:], "wo": lw["wo"], "ffn_norm": lw["ffn_norm"],
                "w_gate": lw["w_gate_up"][0::2], "w_up": lw["w_gate_up"][1::2], "w_down": lw["w_down"]}

    def views(self):
        """Canonical name -> view of the packed storage."""
        out = {"embed": self.embed, "final_norm": self.final_norm, "lm_head": self.lm_head,
               "draft.w_fc": self.w_fc, "draft.fc_norm": self.fc_norm, "draft.final_norm": self.d_final_norm}
        for i, lw in enumerate(self.layers):
            for k, v in self._layer_views(lw).items():
                out[f"layers.{i}.{k}"] = v
        for i, lw in enumerate(self.dlayers):
            for k, v in self._layer_views(lw).items():
                out[f"draft.layers.{i}.{k}"] = v
        return out

    def load(self, weights: dict):
        """Copy host arrays (canonical names) into the packed device storage."""
        views = self.views()
        for name, arr in weights.items():
            v = views[name]
            t = torch.from_numpy(np.ascontiguousarray(arr)).to(dtype=v.dtype)
            v.copy_(t.reshape(v.shape))
        self.finalize()

    def set_cross_ctx(self, window: int):
        """Set the drafter's cross-context window (0: whole context)."""
        self.cross_ctx = int(window)
        self._structs = None

    def finalize(self):
        """Gather the drafter's k/v rows for the injection product and build
        the C structs.  Call after every change of the weights."""
        s, d = self.shape, self.shape.head_dim
        q, kv = s.n_q * d, s.n_kv * d
        for i, lw in enumerate(self.dlayers):
            self.w_kv_all[i * 2 * kv:(i + 1) * 2 * kv].copy_(lw["wqkv"][q:q + 2 * kv])
        self._structs = None

    def weight_bytes(self):
        t = sum(x.numel() * x.element_size() for x in (self.embed, self.final_norm, self.lm_head))
        t += sum(x.numel() * x.element_size() for lw in self.layers for x in lw.values())
        dr = sum(x.numel() * x.element_size() for lw in self.dlayers for x in lw.values())
        dr += sum(x.numel() * x.element_size() for x in (self.w_fc, self.fc_norm, self.d_final_norm, self.w_kv_all))
        return t, dr

    # -------------------------------------------------------------- C structs
    def _layer_array(self, layers):
        arr = (capi.LayerW * len(layers))()
        for i, lw in enumerate(layers):
            arr[i] = capi.LayerW(*(lw[k].data_ptr() for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate_up",
                                                              "w_down")))
        return arr

    def structs(self):
        if self._structs is None:
            tl = self._layer_array(self.layers)
            dl = self._layer_array(self.dlayers)
            tgt = capi.TargetC(desc_of(self.shape, self.dtype), self.embed.data_ptr(), self.final_norm.data_ptr(),
                               self.lm_head.data_ptr(), ctypes.cast(tl, ctypes.POINTER(capi.LayerW)),
                               (ctypes.c_int32 * 5)(*self.capture))
            dr = capi.DraftC(desc_of(self.shape, self.dtype, self.draft_layers), self.w_fc.data_ptr(),
                             self.fc_norm.data_ptr(), self.d_final_norm.data_ptr(),
                             ctypes.cast(dl, ctypes.POINTER(capi.LayerW)), self.w_kv_all.data_ptr(), self.mask_id,
                             self.cross_ctx)
            self._structs = (tgt, dr, tl, dl)  # keep the layer arrays alive
        return self._structs[0], self._structs[1]


class Session:
    """Caches, workspace and device state for ``batch`` sequences."""

    def __init__(self, model: Model, batch=1, capacity=1024, block=16, prefill_chunk=128, stream_cap=None,
                 with_draft=True, tree_budget=0, kv_format="bf16"):
        tree_n = tree_budget + 1 if tree_budget else 0
        if batch * max(block, tree_n) > 128 or prefill_chunk > 128 or tree_n > 64:
            raise ValueError("at most 128 rows per call and 64 tree nodes")
        if kv_format not in ("bf16", "q8"):
            raise ValueError(kv_format)
        self.kv_format = kv_format
        if kv_format == "q8":
            capacity = (capacity + 7) // 8 * 8  # the 8-bit cache's capacity granularity
        self.m, self.batch, self.block, self.capacity = model, batch, block, capacity
        self.chunk = prefill_chunk
        self.stream_cap = stream_cap or capacity
        s = model.shape
        self.tdesc = desc_of(s, model.dtype)
        self.ddesc = desc_of(s, model.dtype, model.draft_layers)
        dev = model.device
        tdt = _DT[model.dtype][1]
        self.tcache = capi.dflash_cache_alloc_ex(self.tdesc, s.n_layers, batch, capacity,
                                                 capi.KV_Q8 if kv_format == "q8" else capi.KV_MODEL)
        self.dcache = capi.dflash_cache_alloc(self.ddesc, model.draft_layers, batch, capacity) if with_draft else None
        self.max_rows = max(batch * block, batch * tree_n, prefill_chunk)
        self.ws = capi.dflash_workspace_alloc(self.tdesc, self.ddesc if with_draft else None, self.max_rows, capacity)
        i32 = dict(dtype=torch.int32, device=dev)
        self.anchor = torch.zeros(batch, **i32)
        self.n_pend = torch.zeros(batch, **i32)
        self.accept_len = torch.zeros(batch, **i32)
        self.draft = torch.zeros(batch, block, **i32)
        self.argmax = torch.zeros(self.max_rows, **i32)
        self.gap = torch.zeros(self.max_rows, dtype=torch.float32, device=dev)
        self.hcap = torch.zeros(self.max_rows, 5 * s.hidden, dtype=tdt, device=dev)
        self.fused = torch.zeros(self.max_rows, s.hidden, dtype=tdt, device=dev)
        self.stream = torch.full((batch, self.stream_cap), -1, **i32)
        self.stream_len = torch.zeros(batch, **i32)
        self.step_ctr = torch.zeros(1, **i32)
        self.ref = self.k_draw = self.r_draw = None
        self.steps_done = 0
        self.rps = block  # rows per sequence of the last verification (the layout of hcap)
        if tree_n:
            self.tree_budget, self.tree_n = tree_budget, tree_n
            self.tree_tokens = torch.zeros(batch, tree_n, **i32)
            self.tree_parent = torch.zeros(batch, tree_n, **i32)
            self.tree_depth = torch.zeros(batch, tree_n, **i32)
            self.tree_mask = torch.zeros(batch, tree_n, dtype=torch.int64, device=dev)  # uint64 bit masks

    def close(self):
        for h, f in ((self.tcache, capi.dflash_cache_free), (self.dcache, capi.dflash_cache_free),
                     (self.ws, capi.dflash_workspace_free)):
            if h:
                f(h)
        self.tcache = self.dcache = self.ws = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -------------------------------------------------------------- state
    def target_len(self):
        return capi.dflash_cache_get_lengths(self.tcache, self.batch)

    def draft_len(self):
        return capi.dflash_cache_get_lengths(self.dcache, self.batch)

    def emitted(self):
        torch.cuda.synchronize()
        lens = self.stream_len.cpu().numpy()
        st = self.stream.cpu().numpy()
        return [st[b, :lens[b]].copy() for b in range(self.batch)]

    def status(self):
        return capi.dflash_status(self.ws)

    # -------------------------------------------------------------- prefill
    def prefill(self, prompts, inject=True):
        """Run the target over each sequence's prompt (chunks of <= 128 rows),
        cache its keys/values, emit the first greedy token, and inject every
        prompt row into the drafter cache."""
        tgt, dr = self.m.structs()
        dev = self.m.device
        for b, p in enumerate(prompts):
            toks = torch.as_tensor(np.asarray(p, dtype=np.int32), device=dev)
            tv = capi.dflash_cache_view(self.tcache, b, 1)
            dv = capi.dflash_cache_view(self.dcache, b, 1) if (inject and self.dcache) else None
            try:
                for c0 in range(0, len(p), self.chunk):
                    n = min(self.chunk, len(p) - c0)
                    last = c0 + n == len(p)
                    if last:
                        self._last_chunk_rows = n
                    capi.target_verify(tgt, toks[c0:c0 + n], 1, n, 2 if last else 1, tv, self.argmax, self.gap,
                                       self.hcap if dv else None, self.anchor[b:], self.n_pend[b:],
                                       self.stream[b], self.stream_len[b:], self.stream_cap, self.ws)
                    if dv:
                        capi.dflash_fuse_features(dr, self.hcap, n, self.fused, self.ws)
                        capi.dflash_inject_kv(dr, self.fused, 1, n, self.n_pend[b:], dv, self.ws)
            finally:
                capi.dflash_cache_free(tv)
                if dv:
                    capi.dflash_cache_free(dv)

    def copy_target_from(self, other: "Session"):
        """Take over another session's committed target state (keys/values of
        positions 0..len-1 of every layer, lengths, anchors and emitted
        streams) instead of prefilling the same prompts again."""
        if (other.capacity, other.batch, other.kv_format) == (self.capacity, self.batch, self.kv_format):
            capi.dflash_cache_copy(self.tcache, other.tcache)  # the whole cache in a few copies
        else:
            if self.kv_format != "bf16" or other.kv_format != "bf16":
                raise ValueError("8-bit caches are copied whole, between sessions of the same geometry")
            s = self.m.shape
            lens = other.target_len()
            tdt = _DT[self.m.dtype][1]
            for b, n in enumerate(lens):
                if n == 0:
                    continue
                k = torch.empty(s.n_kv, n, s.head_dim, dtype=tdt, device=self.m.device)
                v = torch.empty_like(k)
                for li in range(s.n_layers):
                    capi.dflash_cache_read(other.tcache, li, b, 0, n, k, v)
                    capi.dflash_cache_write(self.tcache, li, b, 0, n, k, v)
            capi.dflash_cache_set_lengths(self.tcache, lens)
        self.anchor.copy_(other.anchor)
        w = min(self.stream_cap, other.stream_cap)
        self.stream[:, :w].copy_(other.stream[:, :w])
        self.stream_len.copy_(other.stream_len)
        torch.cuda.synchronize()

    # -------------------------------------------------------------- decoding
    def set_teacher(self, ref, k_draw, r_draw):
        """Teacher-forcing inputs: ref [batch][L] greedy streams, draws [steps][batch]."""
        dev = self.m.device
        self.ref = torch.as_tensor(np.ascontiguousarray(ref, dtype=np.int32), device=dev)
        self.k_draw = torch.as_tensor(np.ascontiguousarray(k_draw, dtype=np.int32), device=dev)
        self.r_draw = torch.as_tensor(np.ascontiguousarray(r_draw, dtype=np.int32), device=dev)
        self.step_ctr.zero_()

    def step(self, teacher=False):
        """One DFlash step for every sequence (asynchronous)."""
        tgt, dr = self.m.structs()
        B = self.block
        capi.dflash_fuse_features(dr, self.hcap, self.batch * self.rps, self.fused, self.ws)
        capi.dflash_inject_kv(dr, self.fused, self.batch, self.rps, self.n_pend, self.dcache, self.ws)
        capi.dflash_draft_block(dr, tgt, self.anchor, self.batch, B, self.dcache, self.draft, self.ws)
        self.rps = B
        if teacher:
            capi.dflash_teacher_force(self.draft, self.batch, B, self.ref, self.ref.shape[1], self.ref.shape[1],
                                      self.stream_len, self.k_draw, self.r_draw, self.k_draw.shape[0], self.step_ctr,
                                      self.m.shape.vocab, self.ws)
        capi.target_verify(tgt, self.draft, self.batch, B, 0, self.tcache, self.argmax, self.gap, self.hcap, None,
                           None, None, None, 0, self.ws)
        capi.dflash_accept_rollback(self.draft, self.argmax, self.batch, B, self.tcache, self.anchor, self.n_pend,
                                    self.accept_len, self.stream, self.stream_len, self.stream_cap, self.ws)
        self.steps_done += 1

    def resample_first(self, temperature, v):
        """Sampling mode after prefill: replace each sequence's first emitted
        token (the greedy one) by a draw at `temperature` from the last
        prompt row's logits with the uniform v[batch].  Needs the prefill's
        last chunk to be its only call with that sequence's last row, i.e. a
        single sequence (batch 1)."""
        if self.batch != 1:
            raise ValueError("resample_first draws from the last prefill call's logits: batch 1 only")
        n_last = int(self._last_chunk_rows)
        logits = capi.dflash_workspace_logits(self.ws, n_last, self.m.shape.vocab)[n_last - 1:]
        vv = torch.as_tensor(np.asarray(v, dtype=np.float32).reshape(1), device=self.m.device)
        capi.dflash_sample(logits, 1, self.m.shape.vocab, temperature, vv, self.anchor, self.ws)
        self.stream[:, 0].copy_(self.anchor)

    def step_sampling(self, temperature, w, u, v):
        """One DFlash step in sampling mode (asynchronous): the drafter samples
        its block with w [batch][B-1], the target verifies it by speculative
        sampling with u [batch][B-1] and v [batch] (device float32 uniforms)."""
        tgt, dr = self.m.structs()
        B, V = self.block, self.m.shape.vocab
        capi.dflash_fuse_features(dr, self.hcap, self.batch * self.rps, self.fused, self.ws)
        capi.dflash_inject_kv(dr, self.fused, self.batch, self.rps, self.n_pend, self.dcache, self.ws)
        capi.dflash_draft_block(dr, tgt, self.anchor, self.batch, B, self.dcache, self.draft, self.ws)
        self.rps = B
        capi.dflash_draft_sample(self.batch, B, V, temperature, w, self.draft, self.ws)
        capi.target_verify(tgt, self.draft, self.batch, B, 0, self.tcache, self.argmax, self.gap, self.hcap, None,
                           None, None, None, 0, self.ws)
        capi.dflash_accept_sample(self.draft, self.batch, B, V, temperature, u, v, self.tcache, self.anchor,
                                  self.n_pend, self.accept_len, self.stream, self.stream_len, self.stream_cap, self.ws)
        self.steps_done += 1

    def step_tree(self, topk):
        """One DFlash step with tree verification (asynchronous): the drafter's
        block, the tree of its top-k candidates within the session's budget,
        one ancestor-masked target forward over the tree, the walk and the
        compaction of the accepted path."""
        tgt, dr = self.m.structs()
        B, V, n = self.block, self.m.shape.vocab, self.tree_n
        capi.dflash_fuse_features(dr, self.hcap, self.batch * self.rps, self.fused, self.ws)
        capi.dflash_inject_kv(dr, self.fused, self.batch, self.rps, self.n_pend, self.dcache, self.ws)
        capi.dflash_draft_block(dr, tgt, self.anchor, self.batch, B, self.dcache, self.draft, self.ws)
        capi.dflash_draft_tree(self.anchor, self.batch, B, V, topk, self.tree_budget, self.tree_tokens,
                               self.tree_parent, self.tree_depth, self.tree_mask, self.ws)
        capi.target_verify_tree(tgt, self.tree_tokens, self.tree_depth, self.tree_mask, self.batch, n, self.tcache,
                                self.argmax, self.gap, self.hcap, self.ws)
        capi.dflash_accept_tree(tgt, self.tree_tokens, self.tree_parent, self.argmax, self.batch, n, self.tcache,
                                self.hcap, self.anchor, self.n_pend, self.accept_len, self.stream, self.stream_len,
                                self.stream_cap, self.ws)
        self.rps = n
        self.steps_done += 1

    def ar_step(self):
        """One greedy autoregressive token per sequence: the target forward of
        the anchor, committed."""
        tgt, _ = self.m.structs()
        capi.target_verify(tgt, self.anchor, self.batch, 1, 2, self.tcache, self.argmax, self.gap, None, self.anchor,
                           self.n_pend, self.stream, self.stream_len, self.stream_cap, self.ws)

    def capture_graph(self, fn):
        """Capture ``fn()`` (a step) into a CUDA graph; replay with g.replay()."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        return g

