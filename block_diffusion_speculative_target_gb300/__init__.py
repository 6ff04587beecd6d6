"""GB300-native DFlash speculative-decoding step: fuse -> inject -> draft ->
verify -> accept/rollback as sm_103a CUDA kernels behind a C ABI
(libdflash.so, include/dflash.h), with a thin ctypes binding."""
from . import capi  # noqa: F401
from .capi import DFlashError  # noqa: F401

__all__ = ["capi", "DFlashError"]
