"""ctypes binding of libdflash.so with the C ABI's names.

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and a negative return code raises
DFlashError.  Every computation runs in the library's CUDA kernels; if the
library cannot be loaded, importing the entry points raises -- there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_void_p

from . import build as _build

F32 = 0
BF16 = 1

ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_SHAPE = -2
ERR_TOO_LARGE = -5
ARGMAX_NOALLOC_MAX_ROWS = 128

STATUS_CAPACITY = 1
STATUS_NONFINITE = 2
STATUS_TIMEOUT = 4
STATUS_BOUNDS = 8


class DFlashError(RuntimeError):
    def __init__(self, msg, code=None):
        super().__init__(msg)
        self.code = code


class ModelDesc(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("hidden", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("ffn", c_int32), ("vocab", c_int32), ("rope_theta", c_float),
                ("rms_eps", c_float), ("dtype", c_int32)]


class LayerW(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate_up", "w_down")]


class TargetC(ctypes.Structure):
    _fields_ = [("d", ModelDesc), ("embed", c_void_p), ("final_norm", c_void_p), ("lm_head", c_void_p),
                ("layers", POINTER(LayerW)), ("capture", c_int32 * 5)]


class DraftC(ctypes.Structure):
    _fields_ = [("d", ModelDesc), ("w_fc", c_void_p), ("fc_norm", c_void_p), ("final_norm", c_void_p),
                ("layers", POINTER(LayerW)), ("w_kv_all", c_void_p), ("mask_id", c_int32), ("cross_ctx", c_int32)]


_P = c_void_p
_I = c_int32
_SIGS = {
    "dflash_strerror": (ctypes.c_char_p, [_I]),
    "dflash_capture_layers": (_I, [_I, POINTER(c_int32)]),
    "dflash_cache_alloc": (_I, [POINTER(ModelDesc), _I, _I, _I, POINTER(c_void_p)]),
    "dflash_cache_alloc_ex": (_I, [POINTER(ModelDesc), _I, _I, _I, _I, POINTER(c_void_p)]),
    "dflash_cache_kv_format": (_I, [_P]),
    "dflash_cache_read_q8": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "dflash_cache_copy": (_I, [_P, _P, _P]),
    "dflash_cache_free": (_I, [_P]),
    "dflash_cache_view": (_I, [_P, _I, _I, POINTER(c_void_p)]),
    "dflash_cache_lengths": (c_void_p, [_P]),
    "dflash_cache_reset": (_I, [_P, _P]),
    "dflash_cache_get_lengths": (_I, [_P, POINTER(c_int32), _I, _P]),
    "dflash_cache_write": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "dflash_cache_read": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "dflash_cache_set_lengths": (_I, [_P, POINTER(c_int32), _I, _P]),
    "dflash_workspace_alloc": (_I, [POINTER(ModelDesc), POINTER(ModelDesc), _I, _I, POINTER(c_void_p)]),
    "dflash_workspace_free": (_I, [_P]),
    "dflash_status": (_I, [_P, _P, POINTER(c_int32)]),
    "dflash_workspace_logits": (c_void_p, [_P, _I]),
    "dflash_draft_sample": (_I, [_I, _I, _I, c_float, _P, _P, _P, _P]),
    "dflash_accept_sample": (_I, [_P, _I, _I, _I, c_float, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "dflash_sample": (_I, [_P, _I, _I, c_float, _P, _P, _P, _P]),
    "dflash_draft_tree": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "target_verify_tree": (_I, [POINTER(TargetC), _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P]),
    "dflash_accept_tree": (_I, [POINTER(TargetC), _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "dflash_debug_set_wait_limit": (_I, [ctypes.c_int64]),
    "dflash_fuse_features": (_I, [POINTER(DraftC), _P, _I, _P, _P, _P]),
    "dflash_inject_kv": (_I, [POINTER(DraftC), _P, _I, _I, _P, _P, _P, _P]),
    "dflash_draft_block": (_I, [POINTER(DraftC), POINTER(TargetC), _P, _I, _I, _P, _P, _P, _P]),
    "target_verify": (_I, [POINTER(TargetC), _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "dflash_accept_rollback": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "dflash_teacher_force": (_I, [_P, _I, _I, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P]),
    "dflash_linear": (_I, [_I, _P, _P, _P, _I, _I, _I, _P, _P]),
    "dflash_rmsnorm": (_I, [_I, _P, _P, _P, _I, _I, c_float, _P]),
    "dflash_argmax": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "dflash_argmax_noalloc": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "dflash_attention": (_I, [POINTER(ModelDesc), _P, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "dflash_profile_begin": (_I, [_I]),
    "dflash_launch_count": (ctypes.c_longlong, []),
    "dflash_profile_end": (_I, [POINTER(c_float), POINTER(c_int32), _I, POINTER(c_int32)]),
}

_lib = None


def lib_path():
    return _build.LIB


def load(build_if_missing=True):
    """Load libdflash.so (building it first if absent).  Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB) or not _build.up_to_date():
        if not build_if_missing:
            raise DFlashError(f"{_build.LIB} is missing: build it with block_diffusion_speculative_target_gb300.build")
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    return list(_SIGS)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch

    return torch.cuda.current_stream().cuda_stream


def _check(rc, what):
    if rc != 0:
        raise DFlashError(f"{what}: {load().dflash_strerror(rc).decode()} ({rc})", rc)


# ---------------------------------------------------------------- caches / workspace


def dflash_capture_layers(n_layers):
    out = (c_int32 * 5)()
    _check(load().dflash_capture_layers(n_layers, out), "dflash_capture_layers")
    return list(out)


def dflash_cache_alloc(desc: ModelDesc, n_layers, batch, capacity):
    h = c_void_p()
    _check(load().dflash_cache_alloc(ctypes.byref(desc), n_layers, batch, capacity, ctypes.byref(h)),
           "dflash_cache_alloc")
    return h.value


KV_MODEL, KV_Q8 = 0, 1


def dflash_cache_alloc_ex(desc: ModelDesc, n_layers, batch, capacity, kv_format):
    h = c_void_p()
    _check(load().dflash_cache_alloc_ex(ctypes.byref(desc), n_layers, batch, capacity, kv_format, ctypes.byref(h)),
           "dflash_cache_alloc_ex")
    return h.value


def dflash_cache_kv_format(cache):
    return load().dflash_cache_kv_format(cache)


def dflash_cache_read_q8(cache, layer, seq, pos0, n, k_codes, v_codes, k_scales, v_scales, stream=None):
    _check(load().dflash_cache_read_q8(cache, layer, seq, pos0, n, _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                                       _ptr(v_scales), _stream(stream)), "dflash_cache_read_q8")


def dflash_cache_copy(dst, src, stream=None):
    _check(load().dflash_cache_copy(dst, src, _stream(stream)), "dflash_cache_copy")


def dflash_cache_free(cache):
    _check(load().dflash_cache_free(cache), "dflash_cache_free")


def dflash_cache_view(cache, seq_begin, seq_count):
    h = c_void_p()
    _check(load().dflash_cache_view(cache, seq_begin, seq_count, ctypes.byref(h)), "dflash_cache_view")
    return h.value


def dflash_cache_lengths(cache):
    return load().dflash_cache_lengths(cache)


def dflash_cache_get_lengths(cache, batch, stream=None):
    out = (c_int32 * batch)()
    _check(load().dflash_cache_get_lengths(cache, out, batch, _stream(stream)), "dflash_cache_get_lengths")
    return list(out)


def dflash_cache_write(cache, layer, seq, pos0, n, k, v, stream=None):
    _check(load().dflash_cache_write(cache, layer, seq, pos0, n, _ptr(k), _ptr(v), _stream(stream)),
           "dflash_cache_write")


def dflash_cache_read(cache, layer, seq, pos0, n, k, v, stream=None):
    _check(load().dflash_cache_read(cache, layer, seq, pos0, n, _ptr(k), _ptr(v), _stream(stream)),
           "dflash_cache_read")


def dflash_cache_set_lengths(cache, lengths, stream=None):
    arr = (c_int32 * len(lengths))(*[int(x) for x in lengths])
    _check(load().dflash_cache_set_lengths(cache, arr, len(lengths), _stream(stream)), "dflash_cache_set_lengths")


def dflash_cache_reset(cache, stream=None):
    _check(load().dflash_cache_reset(cache, _stream(stream)), "dflash_cache_reset")


def dflash_workspace_alloc(target: ModelDesc, draft: ModelDesc | None, max_rows, max_ctx):
    h = c_void_p()
    _check(load().dflash_workspace_alloc(ctypes.byref(target), ctypes.byref(draft) if draft is not None else None,
                                         max_rows, max_ctx, ctypes.byref(h)), "dflash_workspace_alloc")
    return h.value


def dflash_workspace_free(ws):
    _check(load().dflash_workspace_free(ws), "dflash_workspace_free")


def dflash_status(ws, stream=None):
    v = c_int32()
    _check(load().dflash_status(ws, _stream(stream), ctypes.byref(v)), "dflash_status")
    return v.value


def dflash_workspace_logits(ws, rows, vocab, which=0):
    """The workspace's float32 logits [rows][vocab] as a torch tensor view
    (which = 0: the target's, 1: the drafter's; device memory owned by the
    workspace, valid until the next call that writes it)."""
    import torch

    p = load().dflash_workspace_logits(ws, which)
    if not p:
        raise DFlashError("dflash_workspace_logits: no workspace")
    return _device_view(p, rows * vocab, torch.float32).view(rows, vocab)


def _device_view(ptr, numel, dtype):
    """A torch tensor over `numel` elements of library-owned device memory."""
    import torch

    class _Mem:
        def __init__(self, p, n, dt):
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": {torch.float32: "<f4", torch.int32: "<i4"}[dt],
                                             "data": (p, False), "version": 3}

    return torch.as_tensor(_Mem(ptr, numel, dtype), device="cuda")


def dflash_debug_set_wait_limit(ns):
    _check(load().dflash_debug_set_wait_limit(int(ns)), "dflash_debug_set_wait_limit")


# ---------------------------------------------------------------- stages


def dflash_fuse_features(draft: DraftC, hcap, rows, fused, ws, stream=None):
    _check(load().dflash_fuse_features(ctypes.byref(draft), _ptr(hcap), rows, _ptr(fused), ws, _stream(stream)),
           "dflash_fuse_features")


def dflash_inject_kv(draft: DraftC, fused, batch, rows_per_seq, n_pend, draft_cache, ws, stream=None):
    _check(load().dflash_inject_kv(ctypes.byref(draft), _ptr(fused), batch, rows_per_seq, _ptr(n_pend), draft_cache,
                                   ws, _stream(stream)), "dflash_inject_kv")


def dflash_draft_block(draft: DraftC, target: TargetC, anchor, batch, block, draft_cache, draft_tokens, ws,
                       stream=None):
    _check(load().dflash_draft_block(ctypes.byref(draft), ctypes.byref(target), _ptr(anchor), batch, block,
                                     draft_cache, _ptr(draft_tokens), ws, _stream(stream)), "dflash_draft_block")


def target_verify(target: TargetC, tokens, batch, n, commit, target_cache, argmax, top2_gap, hcap, anchor, n_pend,
                  stream_buf, stream_len, stream_cap, ws, stream=None):
    _check(load().target_verify(ctypes.byref(target), _ptr(tokens), batch, n, commit, target_cache, _ptr(argmax),
                                _ptr(top2_gap), _ptr(hcap), _ptr(anchor), _ptr(n_pend), _ptr(stream_buf),
                                _ptr(stream_len), stream_cap, ws, _stream(stream)), "target_verify")


def dflash_accept_rollback(draft_tokens, argmax, batch, block, target_cache, anchor, n_pend, accept_len, stream_buf,
                           stream_len, stream_cap, ws, stream=None):
    _check(load().dflash_accept_rollback(_ptr(draft_tokens), _ptr(argmax), batch, block, target_cache, _ptr(anchor),
                                         _ptr(n_pend), _ptr(accept_len), _ptr(stream_buf), _ptr(stream_len),
                                         stream_cap, ws, _stream(stream)), "dflash_accept_rollback")


def dflash_teacher_force(draft_tokens, batch, block, ref, ref_stride, ref_len, stream_len, k_draw, r_draw, max_steps,
                         step, vocab, ws, stream=None):
    _check(load().dflash_teacher_force(_ptr(draft_tokens), batch, block, _ptr(ref), ref_stride, ref_len,
                                       _ptr(stream_len), _ptr(k_draw), _ptr(r_draw), max_steps, _ptr(step), vocab, ws,
                                       _stream(stream)), "dflash_teacher_force")


# ---------------------------------------------------------------- tree verification


def dflash_draft_tree(anchor, batch, block, vocab, topk, budget, tree_tokens, tree_parent, tree_depth, tree_mask, ws,
                      stream=None):
    _check(load().dflash_draft_tree(_ptr(anchor), batch, block, vocab, topk, budget, _ptr(tree_tokens),
                                    _ptr(tree_parent), _ptr(tree_depth), _ptr(tree_mask), ws, _stream(stream)),
           "dflash_draft_tree")


def target_verify_tree(target: TargetC, tree_tokens, tree_depth, tree_mask, batch, n, target_cache, argmax, top2_gap,
                       hcap, ws, stream=None):
    _check(load().target_verify_tree(ctypes.byref(target), _ptr(tree_tokens), _ptr(tree_depth), _ptr(tree_mask),
                                     batch, n, target_cache, _ptr(argmax), _ptr(top2_gap), _ptr(hcap), ws,
                                     _stream(stream)), "target_verify_tree")


def dflash_accept_tree(target: TargetC, tree_tokens, tree_parent, argmax, batch, n, target_cache, hcap, anchor, n_pend,
                       accept_len, stream_buf, stream_len, stream_cap, ws, stream=None):
    _check(load().dflash_accept_tree(ctypes.byref(target), _ptr(tree_tokens), _ptr(tree_parent), _ptr(argmax), batch,
                                     n, target_cache, _ptr(hcap), _ptr(anchor), _ptr(n_pend), _ptr(accept_len),
                                     _ptr(stream_buf), _ptr(stream_len), stream_cap, ws, _stream(stream)),
           "dflash_accept_tree")


# ---------------------------------------------------------------- sampling mode


def dflash_draft_sample(batch, block, vocab, temperature, w, draft_tokens, ws, stream=None):
    _check(load().dflash_draft_sample(batch, block, vocab, float(temperature), _ptr(w), _ptr(draft_tokens), ws,
                                      _stream(stream)), "dflash_draft_sample")


def dflash_accept_sample(draft_tokens, batch, block, vocab, temperature, u, v, target_cache, anchor, n_pend,
                         accept_len, stream_buf, stream_len, stream_cap, ws, stream=None):
    _check(load().dflash_accept_sample(_ptr(draft_tokens), batch, block, vocab, float(temperature), _ptr(u), _ptr(v),
                                       target_cache, _ptr(anchor), _ptr(n_pend), _ptr(accept_len), _ptr(stream_buf),
                                       _ptr(stream_len), stream_cap, ws, _stream(stream)), "dflash_accept_sample")


def dflash_sample(logits, rows, vocab, temperature, v, out, ws, stream=None):
    _check(load().dflash_sample(_ptr(logits), rows, vocab, float(temperature), _ptr(v), _ptr(out), ws,
                                _stream(stream)), "dflash_sample")


# ---------------------------------------------------------------- building blocks


def dflash_linear(dtype, x, w, y, rows, M, K, ws, stream=None):
    _check(load().dflash_linear(dtype, _ptr(x), _ptr(w), _ptr(y), rows, M, K, ws, _stream(stream)), "dflash_linear")


def dflash_rmsnorm(dtype, x, gain, y, rows, H, eps, stream=None):
    _check(load().dflash_rmsnorm(dtype, _ptr(x), _ptr(gain), _ptr(y), rows, H, eps, _stream(stream)),
           "dflash_rmsnorm")


def dflash_argmax(logits, rows, V, argmax, gap, ws, stream=None):
    _check(load().dflash_argmax(_ptr(logits), rows, V, _ptr(argmax), _ptr(gap), ws, _stream(stream)),
           "dflash_argmax")


def dflash_argmax_noalloc(logits, rows, V, argmax, gap, status=None, stream=None):
    _check(load().dflash_argmax_noalloc(_ptr(logits), rows, V, _ptr(argmax), _ptr(gap), _ptr(status),
                                        _stream(stream)), "dflash_argmax_noalloc")


def dflash_attention(desc: ModelDesc, q, batch, n, causal, cache, layer, out, ws, stream=None, window=0):
    _check(load().dflash_attention(ctypes.byref(desc), _ptr(q), batch, n, causal, window, cache, layer, _ptr(out), ws,
                                   _stream(stream)), "dflash_attention")


# ---------------------------------------------------------------- kernel timing


def dflash_profile_begin(max_records):
    _check(load().dflash_profile_begin(max_records), "dflash_profile_begin")


def dflash_profile_end(max_records):
    """Returns [(ms, M, K, rows), ...] for the recorded GEMM launches."""
    ms = (c_float * max_records)()
    tags = (c_int32 * (3 * max_records))()
    n = c_int32()
    _check(load().dflash_profile_end(ms, tags, max_records, ctypes.byref(n)), "dflash_profile_end")
    return [(ms[i], tags[3 * i], tags[3 * i + 1], tags[3 * i + 2]) for i in range(n.value)]


def dflash_launch_count():
    return int(load().dflash_launch_count())
