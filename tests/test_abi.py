"""The C-ABI library builds, loads, and exports every symbol its header
declares; host-only logic (argument checks, layer selection) without a GPU."""
import ctypes
import os
import re

import pytest

from block_diffusion_speculative_target_gb300 import build, capi
from oracle import dflash_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    # the binding covers the whole header
    assert set(names) <= set(capi.exported_symbols())


def test_capture_layers_match_oracle(lib):
    for L in range(6, 130):
        assert capi.dflash_capture_layers(L) == O.layer_indices(L), L


def test_argument_checks_without_gpu(lib):
    assert lib.dflash_cache_alloc(None, 1, 1, 1, None) == -1
    h = ctypes.c_void_p()
    assert lib.dflash_cache_alloc(None, 1, 1, 16, ctypes.byref(h)) == -1
    bad = capi.ModelDesc(1, 256, 4, 3, 64, 768, 2048, 1e6, 1e-6, 0)  # 4 % 3 != 0
    assert lib.dflash_cache_alloc(ctypes.byref(bad), 1, 1, 16, ctypes.byref(h)) == -1
    bad = capi.ModelDesc(1, 256, 4, 4, 96, 768, 2048, 1e6, 1e-6, 0)  # head_dim 96 unsupported
    assert lib.dflash_workspace_alloc(ctypes.byref(bad), None, 16, 16, ctypes.byref(h)) == -1
    assert lib.dflash_capture_layers(5, (ctypes.c_int32 * 5)()) == -1
    assert lib.target_verify(None, None, 1, 1, 0, None, None, None, None, None, None, None, None, 0, None,
                             None) == -1
    assert lib.dflash_accept_rollback(None, None, 1, 16, None, None, None, None, None, None, 0, None, None) == -1
    assert lib.dflash_strerror(-1) == b"invalid argument"
    assert lib.dflash_strerror(-2) == b"unsupported shape"


def test_build_flags_target_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
