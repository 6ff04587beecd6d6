"""dflash_argmax_noalloc: the workspace-free argmax entry point, checked
against dflash_argmax (workspace scratch) through the C-ABI.

The file's name sorts it after the other test files, so in a full run it also
runs after every other GPU test; the subprocess test repeats the comparison in
a fresh process whose first library call is the no-allocation one."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from block_diffusion_speculative_target_gb300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _logits(rows, V, seed):
    lg = synth.gaussian((rows, V), seed=seed, stream=V, scale=2.0)
    if rows > 7:
        lg[3, 10] = lg[3, V - 5] = lg[3].max() + 1.0   # tie: lowest index wins
        lg[5, :] = 0.0                                   # all equal
        lg[7, V - 1] = 50.0                              # maximum in the ragged tail
    return lg


# ------------------------------------------------------------------ host checks

def test_noalloc_rejects_sizes_without_gpu():
    build.build()
    lib = capi.load()
    fake = ctypes.c_void_p(256)  # never dereferenced: the checks return first
    mx = capi.ARGMAX_NOALLOC_MAX_ROWS
    assert lib.dflash_argmax_noalloc(fake, mx + 1, 4096, fake, None, None, None) == capi.ERR_TOO_LARGE
    assert lib.dflash_argmax_noalloc(fake, 1 << 20, 4096, fake, None, None, None) == capi.ERR_TOO_LARGE
    assert lib.dflash_argmax_noalloc(fake, 0, 4096, fake, None, None, None) == capi.ERR_INVALID_ARG
    assert lib.dflash_argmax_noalloc(fake, 4, 0, fake, None, None, None) == capi.ERR_INVALID_ARG
    assert lib.dflash_argmax_noalloc(None, 4, 4096, fake, None, None, None) == capi.ERR_INVALID_ARG
    assert lib.dflash_argmax_noalloc(fake, 4, 4096, None, None, None, None) == capi.ERR_INVALID_ARG
    assert lib.dflash_strerror(capi.ERR_TOO_LARGE) == b"size above the entry point's fixed maximum"


# ------------------------------------------------------------------ GPU parity

# rows, V: the full vocabulary at the maximum row count, a ragged row count,
# and a vocabulary small enough for the single-slice launch
CASES = [(128, 151936, 31), (37, 151936, 32), (5, 1000, 33), (1, 151936, 34)]

COMPARE = r'''
import sys, numpy as np, torch
import synth
from block_diffusion_speculative_target_gb300 import capi

def logits(rows, V, seed):
    lg = synth.gaussian((rows, V), seed=seed, stream=V, scale=2.0)
    if rows > 7:
        lg[3, 10] = lg[3, V - 5] = lg[3].max() + 1.0
        lg[5, :] = 0.0
        lg[7, V - 1] = 50.0
    return lg

def compare(cases, ws):
    dev = torch.device("cuda:0")
    for rows, V, seed in cases:
        lg = torch.from_numpy(logits(rows, V, seed)).to(dev, torch.float32)
        am_n = torch.full((rows,), -1, dtype=torch.int32, device=dev)
        gp_n = torch.full((rows,), -1.0, dtype=torch.float32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        capi.dflash_argmax_noalloc(lg, rows, V, am_n, gp_n, st)
        am_w = torch.full((rows,), -2, dtype=torch.int32, device=dev)
        gp_w = torch.full((rows,), -2.0, dtype=torch.float32, device=dev)
        capi.dflash_argmax(lg, rows, V, am_w, gp_w, ws)
        assert np.array_equal(am_n.cpu().numpy(), am_w.cpu().numpy()), (rows, V)
        assert np.array_equal(gp_n.cpu().numpy().view(np.uint32), gp_w.cpu().numpy().view(np.uint32)), (rows, V)
        assert st.item() == 0 and capi.dflash_status(ws) == 0
        if rows > 7:
            assert am_n[3].item() == 10 and gp_n[3].item() == 0.0
            assert am_n[5].item() == 0 and am_n[7].item() == V - 1

def workspace(V):
    d = capi.ModelDesc(1, 256, 4, 4, 64, 768, V, 1e6, 1e-6, 0)
    return capi.dflash_workspace_alloc(d, None, 128, 256)
'''

FRESH = COMPARE + r'''
dev = torch.device("cuda:0")
torch.cuda.init()
lg = torch.from_numpy(logits(128, 151936, 41)).to(dev, torch.float32)
am = torch.empty(128, dtype=torch.int32, device=dev)
gp = torch.empty(128, dtype=torch.float32, device=dev)
torch.cuda.synchronize()
# the first call into the library: the one-time set-up runs here
capi.dflash_argmax_noalloc(lg, 128, 151936, am, gp)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(3):
    capi.dflash_argmax_noalloc(lg, 128, 151936, am, gp)
torch.cuda.synchronize()
assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across calls"
ws = workspace(151936)
cases = [(128, 151936, 41), (37, 151936, 42), (5, 1000, 43)]
compare(cases, ws)
compare(cases, ws)   # two calls in a row
capi.dflash_workspace_free(ws)
print("NOALLOC-OK")
'''


def _env():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    return env


@pytest.mark.gpu
def test_noalloc_matches_workspace_argmax():
    ns = {}
    exec(compile(COMPARE, "compare", "exec"), ns)
    ws = ns["workspace"](151936)
    try:
        ns["compare"](CASES, ws)
        ns["compare"](CASES, ws)   # two calls in a row reuse the same scratch
    finally:
        capi.dflash_workspace_free(ws)


@pytest.mark.gpu
def test_noalloc_nonfinite_status_and_reuse():
    import torch
    dev = torch.device("cuda:0")
    lg = _logits(4, 4096, 35)
    lg[2, 77] = np.nan
    t = torch.from_numpy(lg).to(dev, torch.float32)
    am = torch.empty(4, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    capi.dflash_argmax_noalloc(t, 4, 4096, am, None, st)
    torch.cuda.synchronize()
    assert st.item() & capi.STATUS_NONFINITE
    # the next call starts from cleared tickets and gives the plain result
    ok = _logits(4, 4096, 36)
    am2 = torch.empty(4, dtype=torch.int32, device=dev)
    capi.dflash_argmax_noalloc(torch.from_numpy(ok).to(dev, torch.float32), 4, 4096, am2, None)
    assert np.array_equal(am2.cpu().numpy(), ok.argmax(axis=1).astype(np.int32))


@pytest.mark.gpu
def test_noalloc_first_call_in_fresh_process():
    r = subprocess.run([sys.executable, "-c", FRESH], cwd=ROOT, env=_env(), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "NOALLOC-OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
