"""GB300-native quantized-KV decode attention.

Hot path: libkvq.so (hand-written CUDA for sm_103a behind a C ABI, declared in
include/kvq.h).  This package only builds that library, marshals arguments to
it through ctypes and lets PyTorch own device memory and streams.
"""
from . import _lib  # noqa: F401
from ._lib import (APPEND_QUANT, APPEND_RING, APPEND_STEP, CacheDesc, KvqError, kvq_append, kvq_decode,
                   kvq_decode_workspace_size, kvq_dequant, kvq_make_decode_plan, kvq_workspace_init)

__all__ = ["APPEND_QUANT", "APPEND_RING", "APPEND_STEP", "CacheDesc", "KvqError", "kvq_append", "kvq_decode",
           "kvq_decode_workspace_size", "kvq_dequant", "kvq_make_decode_plan", "kvq_workspace_init"]
