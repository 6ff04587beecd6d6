"""Time single kernels of libdflash.so at production shapes (small device
footprint, suitable for Nsight Compute captures).

    python -m block_diffusion_speculative_target_gb300.kernel_bench gemm --M 24576 --K 4096 --rows 16
    python -m block_diffusion_speculative_target_gb300.kernel_bench attention --P 4096 --nq 32 --nkv 8 --n 16
    python -m block_diffusion_speculative_target_gb300.kernel_bench rmsnorm --rows 16 --H 4096
    python -m block_diffusion_speculative_target_gb300.kernel_bench argmax --rows 16 --V 151936

Weights rotate over enough copies that every launch streams from HBM, not L2.
The timed launches are captured in a CUDA graph, so host launch overhead is
excluded: time per launch = graph time / launches (back-to-back kernels).
Prints one JSON line per kernel with the time per launch and the achieved
algorithmic bandwidth.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import capi

L2_BYTES = 129 * 2 ** 20


def _graph_time(fn, launches, replays=5):
    """Capture fn() (issuing `launches` kernels' worth of work) in a CUDA graph
    and return the median milliseconds per launch over several replays."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / launches)
    times.sort()
    return times[len(times) // 2]


def bench_gemm(M, K, rows, iters, warmup, copies=None):
    dev = torch.device("cuda")
    wbytes = 2 * M * K
    copies = copies or max(2, -(-3 * L2_BYTES // wbytes))
    g = torch.Generator(device=dev).manual_seed(0)
    ws_desc = capi.ModelDesc(1, K, 1, 1, 128, 128, 256, 1e6, 1e-6, capi.BF16)
    ws = capi.dflash_workspace_alloc(ws_desc, None, 128, 256)
    W = [torch.empty(M, K, dtype=torch.bfloat16, device=dev).normal_(0, 0.02, generator=g) for _ in range(copies)]
    x = torch.empty(rows, K, dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
    y = torch.empty(rows, M, dtype=torch.float32, device=dev)
    for i in range(warmup):
        capi.dflash_linear(capi.BF16, x, W[i % copies], y, rows, M, K, ws)
    avg = _graph_time(lambda: [capi.dflash_linear(capi.BF16, x, W[i % copies], y, rows, M, K, ws)
                               for i in range(iters)], iters)
    assert capi.dflash_status(ws) == 0
    capi.dflash_workspace_free(ws)
    byt = wbytes + 2 * rows * K + 4 * rows * M
    return {"kernel": "gemm_cl_kernel", "M": M, "K": K, "rows": rows, "ms": avg, "bytes": byt,
            "GBps": byt / (avg / 1e3) / 1e9, "splits_copies": copies}


def bench_attention(P, nq, nkv, n, iters, warmup, causal=1, kv="bf16"):
    dev = torch.device("cuda")
    hd = 128
    d = capi.ModelDesc(1, nq * hd, nq, nkv, hd, 256, 256, 1e6, 1e-6, capi.BF16)
    cap = (P + n + 64 + 7) // 8 * 8
    ebytes = 1 if kv == "q8" else 2          # bytes per cached entry (q8: plus 4 per row of 128)
    copies = max(2, -(-3 * L2_BYTES // (2 * ebytes * nkv * cap * hd)))
    fmt = capi.KV_Q8 if kv == "q8" else capi.KV_MODEL
    caches = [capi.dflash_cache_alloc_ex(d, 1, 1, cap, fmt) for _ in range(copies)]
    ws = capi.dflash_workspace_alloc(d, None, max(16, n), cap)
    g = torch.Generator(device=dev).manual_seed(1)
    kvt = torch.empty(nkv, P + n, hd, dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
    for c in caches:
        capi.dflash_cache_write(c, 0, 0, 0, P + n, kvt, kvt)
        capi.dflash_cache_set_lengths(c, [P])
    q = torch.empty(n, nq, hd, dtype=torch.float16 if kv == "q8" else torch.bfloat16, device=dev).normal_(
        0, 1, generator=g)
    out = torch.empty(n, nq * hd, dtype=torch.bfloat16, device=dev)
    for i in range(warmup):
        capi.dflash_attention(d, q, 1, n, causal, caches[i % copies], 0, out, ws)
    avg = _graph_time(lambda: [capi.dflash_attention(d, q, 1, n, causal, caches[i % copies], 0, out, ws)
                               for i in range(iters)], iters)
    assert capi.dflash_status(ws) == 0
    for c in caches:
        capi.dflash_cache_free(c)
    capi.dflash_workspace_free(ws)
    byt = 2 * nkv * (P + n) * (ebytes * hd + (4 if kv == "q8" else 0))
    return {"kernel": "attn_fa_kernel+attn_combine_kernel", "kv": kv, "P": P, "nq": nq, "nkv": nkv, "n": n,
            "ms": avg, "bytes": byt, "GBps": byt / (avg / 1e3) / 1e9}


def bench_rmsnorm(rows, H, iters, warmup):
    """RMSNorm of float32 rows [rows][H] into bf16 (copies rotate so every
    launch reads from HBM)."""
    dev = torch.device("cuda")
    copies = max(2, -(-3 * L2_BYTES // (4 * rows * H)))
    g = torch.Generator(device=dev).manual_seed(2)
    xs = [torch.empty(rows, H, dtype=torch.float32, device=dev).normal_(0, 3, generator=g) for _ in range(copies)]
    gain = torch.ones(H, dtype=torch.bfloat16, device=dev)
    y = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
    for i in range(warmup):
        capi.dflash_rmsnorm(capi.BF16, xs[i % copies], gain, y, rows, H, 1e-6)
    avg = _graph_time(lambda: [capi.dflash_rmsnorm(capi.BF16, xs[i % copies], gain, y, rows, H, 1e-6)
                               for i in range(iters)], iters)
    byt = 4 * rows * H + 2 * rows * H + 2 * H
    return {"kernel": "rmsnorm_kernel", "rows": rows, "H": H, "ms": avg, "bytes": byt,
            "GBps": byt / (avg / 1e3) / 1e9}


def bench_argmax(rows, V, iters, warmup):
    """Greedy token + top-2 gap of float32 logits [rows][V]."""
    dev = torch.device("cuda")
    copies = max(2, -(-3 * L2_BYTES // (4 * rows * V)))
    g = torch.Generator(device=dev).manual_seed(3)
    zs = [torch.empty(rows, V, dtype=torch.float32, device=dev).normal_(0, 2, generator=g) for _ in range(copies)]
    d = capi.ModelDesc(1, 256, 4, 4, 64, 768, V, 1e6, 1e-6, capi.F32)
    ws = capi.dflash_workspace_alloc(d, None, max(rows, 16), 256)
    out = torch.empty(rows, dtype=torch.int32, device=dev)
    gap = torch.empty(rows, dtype=torch.float32, device=dev)
    for i in range(warmup):
        capi.dflash_argmax(zs[i % copies], rows, V, out, gap, ws)
    avg = _graph_time(lambda: [capi.dflash_argmax(zs[i % copies], rows, V, out, gap, ws) for i in range(iters)], iters)
    assert capi.dflash_status(ws) == 0
    capi.dflash_workspace_free(ws)
    byt = 4 * rows * V
    return {"kernel": "argmax_kernel", "rows": rows, "V": V, "ms": avg, "bytes": byt, "GBps": byt / (avg / 1e3) / 1e9}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["gemm", "attention", "step-gemms", "rmsnorm", "argmax"])
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--V", type=int, default=151936)
    ap.add_argument("--M", type=int, default=24576)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--rows", type=int, default=16)
    ap.add_argument("--P", type=int, default=4096)
    ap.add_argument("--nq", type=int, default=32)
    ap.add_argument("--nkv", type=int, default=8)
    ap.add_argument("--n", type=int, default=16)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--kv", choices=["bf16", "q8"], default="bf16", help="attention: the cache's storage")
    a = ap.parse_args()
    capi.load()
    if a.kernel == "gemm":
        print(json.dumps(bench_gemm(a.M, a.K, a.rows, a.iters, a.warmup)))
    elif a.kernel == "attention":
        print(json.dumps(bench_attention(a.P, a.nq, a.nkv, a.n, a.iters, a.warmup, kv=a.kv)))
    elif a.kernel == "rmsnorm":
        print(json.dumps(bench_rmsnorm(a.rows, a.H, a.iters, a.warmup)))
    elif a.kernel == "argmax":
        print(json.dumps(bench_argmax(a.rows, a.V, a.iters, a.warmup)))
    else:
        # every weight-GEMM shape of one Qwen3-8B-shaped step (4096 hidden, 32/8 x 128 heads, FFN 12288)
        for M, K in ((6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288), (151936, 4096), (4096, 20480),
                     (10240, 4096)):
            print(json.dumps(bench_gemm(M, K, a.rows, a.iters, a.warmup)))


if __name__ == "__main__":
    main()
