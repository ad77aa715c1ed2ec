"""ctypes binding of libkvq.so (argument marshalling only).

Every function here forwards to the C entry point of the same name declared in
include/kvq.h; torch tensors are passed as raw device pointers and the current
torch CUDA stream is used unless one is given.  Nothing is computed here, and
there is no fallback: if the shared library is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int32, c_size_t, c_uint32, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_ALIGNMENT = 3
KVQ_ERR_WORKSPACE = 4
KVQ_ERR_CUDA = 5

KVQ_DEVERR_BLOCK_ID = 1
KVQ_DEVERR_SEQ_LEN = 2
KVQ_DEVERR_TIMEOUT = 4
KVQ_DEVERR_RANGE = 8
KVQ_DEVERR_POSITION = 16

APPEND_QUANT = 0
APPEND_RING = 1
APPEND_STEP = 2
PREFILL_TILES = -1  # kvq_prefill stream_ctas: the query-tile path
DECODE_GEOMETRY_READY = 1  # kvq_decode_ex flag: lengths and block table final before the previous kernel ends


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class CacheDesc(ctypes.Structure):
    """Mirror of kvq_cache_desc."""
    _fields_ = [
        ("num_kv_heads", c_int32), ("head_dim", c_int32), ("block_size", c_int32), ("num_blocks", c_int32),
        ("k_bits", c_int32), ("v_bits", c_int32),
        ("k_codes", c_void_p), ("v_codes", c_void_p), ("meta", c_void_p), ("asym", c_int32),
        ("k_channel_factor", c_void_p),
        ("window", c_int32), ("window_batch", c_int32),
        ("k_window", c_void_p), ("v_window", c_void_p),
        ("q_bits", c_int32), ("k_per_channel", c_int32),
    ]


class DecodePlan(ctypes.Structure):
    """Mirror of kvq_decode_plan."""
    _fields_ = [("stream_ctas", c_int32), ("window_ctas", c_int32), ("units", c_int32),
                ("partial_slots", c_int32), ("workspace_bytes", c_size_t)]


_lib = None

# Exported symbol -> (restype, argtypes)
SIGNATURES = {
    "kvq_status_string": (c_char_p, [c_int32]),
    "kvq_block_bytes": (c_int32, [c_int32, POINTER(c_size_t)]),
    "kvq_append": (c_int32, [POINTER(CacheDesc), c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32,
                             c_void_p, c_int32, c_int32, c_void_p, c_void_p]),
    "kvq_make_decode_plan": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32,
                                       POINTER(DecodePlan)]),
    "kvq_decode_device_plan": (c_int32, [POINTER(CacheDesc), c_int32, c_int32, c_int32, POINTER(DecodePlan)]),
    "kvq_decode_workspace_size": (c_int32, [POINTER(CacheDesc), c_int32, c_int32, c_int32, POINTER(c_size_t)]),
    "kvq_workspace_init": (c_int32, [c_void_p, c_size_t, c_void_p]),
    "kvq_decode": (c_int32, [POINTER(CacheDesc), c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32,
                             c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_int32, c_void_p, c_void_p]),
    "kvq_decode_ex": (c_int32, [POINTER(CacheDesc), c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32,
                                c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_int32, c_uint32, c_void_p,
                                c_void_p]),
    "kvq_dequant": (c_int32, [POINTER(CacheDesc), c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
    "kvq_prefill": (c_int32, [POINTER(CacheDesc), c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_int32,
                              c_void_p, c_void_p]),
    "kvq_prefill_workspace_size": (c_int32, [POINTER(CacheDesc), c_int32, c_int32, c_int32, POINTER(c_size_t)]),
    "kvq_decode_static_scratch": (c_int32, [POINTER(CacheDesc), c_void_p, c_int32, c_int32, c_void_p, c_void_p,
                                            c_int32, c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_void_p]),
}

STATIC_SCRATCH_BYTES = 8 << 20


def load() -> ctypes.CDLL:
    """Load libkvq.so (built in-tree by build.py); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkvq.so not built ({LIB_PATH}); run quantized_kv_cache_07_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().kvq_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != KVQ_OK:
        raise KvqError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def block_bytes(bits: int) -> int:
    out = c_size_t(0)
    _check(load().kvq_block_bytes(bits, ctypes.byref(out)), "kvq_block_bytes")
    return out.value


def kvq_append(desc: CacheDesc, k_new, v_new, seq_idx, pos, mode: int, block_table, batch: int,
               max_blocks_per_seq: int, err_word=None, stream=None, n: int | None = None):
    n = int(seq_idx.shape[0]) if n is None else n
    _check(load().kvq_append(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), n, _ptr(seq_idx), _ptr(pos), mode,
                             _ptr(block_table), batch, max_blocks_per_seq, _ptr(err_word),
                             _stream(stream) if n else None), "kvq_append")


def kvq_make_decode_plan(batch: int, q_heads: int, kv_heads: int, window: int, num_sms: int, ctas_per_sm: int,
                         stream_ctas: int = 0) -> DecodePlan:
    plan = DecodePlan()
    _check(load().kvq_make_decode_plan(batch, q_heads, kv_heads, window, num_sms, ctas_per_sm, stream_ctas,
                                       ctypes.byref(plan)), "kvq_make_decode_plan")
    return plan


def kvq_decode_device_plan(desc: CacheDesc, batch: int, q_heads: int, stream_ctas: int = 0) -> DecodePlan:
    plan = DecodePlan()
    _check(load().kvq_decode_device_plan(ctypes.byref(desc), batch, q_heads, stream_ctas, ctypes.byref(plan)),
           "kvq_decode_device_plan")
    return plan


def kvq_decode_workspace_size(desc: CacheDesc, batch: int, q_heads: int, stream_ctas: int = 0) -> int:
    out = c_size_t(0)
    _check(load().kvq_decode_workspace_size(ctypes.byref(desc), batch, q_heads, stream_ctas, ctypes.byref(out)),
           "kvq_decode_workspace_size")
    return out.value


def kvq_workspace_init(workspace, nbytes: int, stream=None):
    _check(load().kvq_workspace_init(_ptr(workspace), nbytes, _stream(stream)), "kvq_workspace_init")


def kvq_decode(desc: CacheDesc, q, batch: int, q_heads: int, seq_lens, block_table, max_blocks_per_seq: int, out,
               lse=None, workspace=None, workspace_bytes: int = 0, stream_ctas: int = 0, err_word=None,
               stream=None, out_fp32: bool | None = None, flags: int = 0):
    """kvq_decode (flags 0) or kvq_decode_ex with flags (DECODE_GEOMETRY_READY)."""
    if out_fp32 is None:
        import torch
        out_fp32 = out.dtype == torch.float32
    if flags:
        _check(load().kvq_decode_ex(ctypes.byref(desc), _ptr(q), batch, q_heads, _ptr(seq_lens), _ptr(block_table),
                                    max_blocks_per_seq, _ptr(out), int(bool(out_fp32)), _ptr(lse), _ptr(workspace),
                                    workspace_bytes, stream_ctas, flags, _ptr(err_word), _stream(stream)),
               "kvq_decode_ex")
        return
    _check(load().kvq_decode(ctypes.byref(desc), _ptr(q), batch, q_heads, _ptr(seq_lens), _ptr(block_table),
                             max_blocks_per_seq, _ptr(out), int(bool(out_fp32)), _ptr(lse), _ptr(workspace),
                             workspace_bytes, stream_ctas, _ptr(err_word), _stream(stream)), "kvq_decode")


def kvq_prefill_workspace_size(desc: CacheDesc, n: int, q_heads: int, stream_ctas: int = 0) -> int:
    out = c_size_t(0)
    _check(load().kvq_prefill_workspace_size(ctypes.byref(desc), n, q_heads, stream_ctas, ctypes.byref(out)),
           "kvq_prefill_workspace_size")
    return out.value


def kvq_prefill(desc: CacheDesc, q, q_heads: int, seq_idx, pos, block_table, batch: int, max_blocks_per_seq: int,
                out, k_new=None, v_new=None, lse=None, workspace=None, workspace_bytes: int = 0, stream_ctas: int = 0,
                err_word=None, stream=None, out_fp32: bool | None = None, n: int | None = None):
    n = int(seq_idx.shape[0]) if n is None else n
    if out_fp32 is None:
        import torch
        out_fp32 = out.dtype == torch.float32
    _check(load().kvq_prefill(ctypes.byref(desc), _ptr(q), n, q_heads, _ptr(seq_idx), _ptr(pos), _ptr(k_new),
                              _ptr(v_new), _ptr(block_table), batch, max_blocks_per_seq, _ptr(out),
                              int(bool(out_fp32)), _ptr(lse), _ptr(workspace), workspace_bytes, stream_ctas,
                              _ptr(err_word), _stream(stream)), "kvq_prefill")


def kvq_dequant(desc: CacheDesc, slots, k_out, v_out, stream=None, n: int | None = None):
    n = int(slots.shape[0]) if n is None else n
    _check(load().kvq_dequant(ctypes.byref(desc), _ptr(slots), n, _ptr(k_out), _ptr(v_out), _stream(stream)),
           "kvq_dequant")


def kvq_decode_static_scratch(desc: CacheDesc, q, batch: int, q_heads: int, seq_lens, block_table,
                              max_blocks_per_seq: int, out, lse=None, stream_ctas: int = 0, err_word=None,
                              stream=None, out_fp32: bool | None = None):
    """kvq_decode without a caller workspace (fixed device scratch inside the
    library; see include/kvq.h for the size limit and the sharing rules)."""
    if out_fp32 is None:
        import torch
        out_fp32 = out.dtype == torch.float32
    _check(load().kvq_decode_static_scratch(ctypes.byref(desc), _ptr(q), batch, q_heads, _ptr(seq_lens),
                                            _ptr(block_table), max_blocks_per_seq, _ptr(out), int(bool(out_fp32)),
                                            _ptr(lse), stream_ctas, _ptr(err_word), _stream(stream)),
           "kvq_decode_static_scratch")
