"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/kvq.h declares; host-only planning and validation paths
return the documented statuses without touching a GPU; the test-side layout
reader covers every byte of a block exactly once."""
import ctypes
import os
import re

import numpy as np
import pytest

from layout_ref import offsets_are_a_permutation

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.build import build
    build()
    return _lib


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kvq_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_hot_path_entry_points():
    names = declared_functions()
    for n in ("kvq_append", "kvq_decode", "kvq_dequant", "kvq_decode_workspace_size", "kvq_workspace_init"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), name
    assert set(declared_functions()) <= set(lib.SIGNATURES)


def header_constants():
    """Integer #define constants of include/kvq.h (u suffixes and shifts evaluated)."""
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    out = {}
    for name, expr in re.findall(r"^#define\s+(KVQ_\w+)\s+(.+?)\s*(?:/\*.*)?$", src, flags=re.M):
        expr = re.sub(r"(\d+)u\b", r"\1", expr)
        if re.fullmatch(r"[\d\s()<>+*-]+", expr):
            out[name] = int(eval(expr))
    return out


def test_binding_constants_match_the_header(lib):
    """The Python binding repeats a few numbers of include/kvq.h; they must not drift."""
    h = header_constants()
    assert lib.STATIC_SCRATCH_BYTES == h["KVQ_STATIC_SCRATCH_BYTES"]
    for name in ("BLOCK_ID", "SEQ_LEN", "TIMEOUT", "RANGE", "POSITION"):
        assert getattr(lib, "KVQ_DEVERR_" + name) == h["KVQ_DEVERR_" + name]
    for name in ("QUANT", "RING", "STEP"):
        assert getattr(lib, "APPEND_" + name) == h["KVQ_APPEND_" + name]
    assert lib.PREFILL_TILES == h["KVQ_PREFILL_TILES"]
    assert lib.DECODE_GEOMETRY_READY == h["KVQ_DECODE_GEOMETRY_READY"]


def test_status_strings_and_block_bytes(lib):
    assert lib.status_string(0) == "KVQ_OK"
    assert "WORKSPACE" in lib.status_string(lib.KVQ_ERR_WORKSPACE)
    assert lib.block_bytes(8) == 2048 and lib.block_bytes(4) == 1024 and lib.block_bytes(16) == 4096
    assert lib.block_bytes(2) == 512
    with pytest.raises(lib.KvqError):
        lib.block_bytes(3)


def test_decode_plan_one_wave_of_ctas(lib):
    p = lib.kvq_make_decode_plan(64, 32, 8, 0, num_sms=152, ctas_per_sm=3)
    assert p.stream_ctas == 456 and p.window_ctas == 0 and p.units == 512      # units > CTAs: no rounding
    p5 = lib.kvq_make_decode_plan(4, 64, 8, 0, num_sms=152, ctas_per_sm=3)
    assert p5.stream_ctas == 448                                               # 14 CTAs per unit
    p3 = lib.kvq_make_decode_plan(32, 32, 8, 0, num_sms=152, ctas_per_sm=3)
    assert p3.stream_ctas == 456                                               # 456 % 256 too large to drop
    # one record slot per (CTA, unit) pair a CTA's range can touch (slot c + u)
    assert p.partial_slots == 456 + 512
    slots = p.partial_slots
    G = 32 // 8                                   # records hold the GQA group's rows
    assert p.workspace_bytes >= slots * G * (128 + 2) * 4 + 512 * 4 + 8
    pw = lib.kvq_make_decode_plan(8, 32, 8, 128, num_sms=152, ctas_per_sm=3)
    # window CTAs (one per unit) run first and take their slots out of the wave
    assert pw.window_ctas == 64 and pw.stream_ctas == 384        # 456 - 64 = 392, rounded to 6 x 64 units
    assert pw.partial_slots == pw.stream_ctas + 64 + 64
    pbig = lib.kvq_make_decode_plan(64, 32, 8, 128, num_sms=152, ctas_per_sm=3)
    assert pbig.window_ctas == 512 and pbig.stream_ctas == 228        # never below half a wave
    px = lib.kvq_make_decode_plan(1, 4, 4, 0, num_sms=152, ctas_per_sm=3, stream_ctas=5)
    assert px.stream_ctas == 5
    with pytest.raises(lib.KvqError):
        lib.kvq_make_decode_plan(1, 6, 4, 0, 152, 3)        # q_heads not a multiple of kv_heads


def _fake_desc(lib, **kw):
    d = dict(num_kv_heads=8, head_dim=128, block_size=16, num_blocks=4, k_bits=8, v_bits=8,
             k_codes=0x1000, v_codes=0x2000, meta=0x3000)
    d.update(kw)
    return lib.CacheDesc(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(block_size=32), 2), (dict(k_bits=2), 2), (dict(k_bits=16, v_bits=8), 2),
    (dict(k_bits=8, v_bits=2), 2), (dict(k_bits=3, v_bits=3), 2),
    # 2-bit blocks (token-group scales): both K and V, no per-channel-only keys
    (dict(k_bits=2, v_bits=2, k_per_channel=1, k_channel_factor=0xC000), 2),
    (dict(k_codes=0x1004), 3), (dict(meta=None), 1), (dict(meta=0x3008), 3), (dict(num_kv_heads=0), 1),
    (dict(window=256), 2),
    (dict(window=16), 1), (dict(window=24), 2),
    # zero points: both or neither, 16-byte aligned, only on quantized blocks
    (dict(asym=2), 1), (dict(k_bits=16, v_bits=16, meta=None, asym=1), 2),
    # quantized query: 8 (or 0/16 for bf16), quantized blocks only, not factor + window together
    (dict(q_bits=4), 2), (dict(q_bits=24), 2), (dict(k_bits=16, v_bits=16, meta=None, q_bits=8), 2),
    (dict(q_bits=8, k_channel_factor=0xC000, window=16, window_batch=1, k_window=0xD000, v_window=0xE000), 2),
    # per-channel key scales only: needs the factor and symmetric quantized keys
    (dict(k_per_channel=1), 1), (dict(k_per_channel=2, k_channel_factor=0xC000), 1),
    (dict(k_per_channel=1, k_channel_factor=0xC000, asym=1), 2),
    (dict(k_per_channel=1, k_channel_factor=0xC000, meta=None), 1),
])
def test_host_validation_without_a_gpu(lib, kw, status):
    desc = _fake_desc(lib, **kw)
    so = lib.load()
    st = so.kvq_decode(ctypes.byref(desc), 0x5000, 1, 8, 0x6000, 0x7000, 1, 0x8000, 0, None, 0x9000, 1 << 20, 5,
                       None, None)
    assert st == status


def test_append_and_decode_reject_bad_shapes_before_any_launch(lib):
    desc = _fake_desc(lib)
    so = lib.load()
    # group of 16 query heads per KV head is beyond the supported 8
    assert so.kvq_decode(ctypes.byref(desc), 0x5000, 1, 128, 0x6000, 0x7000, 1, 0x8000, 0, None, 0x9000, 1 << 20,
                         5, None, None) == lib.KVQ_ERR_UNSUPPORTED
    assert so.kvq_append(ctypes.byref(desc), 0x5000, 0x5100, 1, 0x6000, 0x6100, 7, 0x7000, 1, 1, None,
                         None) == lib.KVQ_ERR_INVALID_ARG
    # ring mode needs a window
    assert so.kvq_append(ctypes.byref(desc), 0x5000, 0x5100, 1, 0x6000, 0x6100, lib.APPEND_RING, 0x7000, 1, 1,
                         None, None) == lib.KVQ_ERR_INVALID_ARG
    # a decode-step eviction cannot write into a 2-bit block (blocks are quantized whole)
    d2 = _fake_desc(lib, k_bits=2, v_bits=2, window=16, window_batch=1, k_window=0xD000, v_window=0xE000)
    assert so.kvq_append(ctypes.byref(d2), 0x5000, 0x5100, 1, 0x6000, 0x6100, lib.APPEND_STEP, 0x7000, 1, 1,
                         None, None) == lib.KVQ_ERR_UNSUPPORTED
    # zero tokens is a no-op
    assert so.kvq_append(ctypes.byref(desc), None, None, 0, None, None, 0, None, 1, 1, None, None) == 0
    # too-small workspace
    assert so.kvq_decode(ctypes.byref(desc), 0x5000, 4, 32, 0x6000, 0x7000, 1, 0x8000, 0, None, 0x9000, 64, 5,
                         None, None) == lib.KVQ_ERR_WORKSPACE
    # kvq_decode_ex: the same validation; flag bits other than GEOMETRY_READY are refused
    assert so.kvq_decode_ex(ctypes.byref(desc), 0x5000, 4, 32, 0x6000, 0x7000, 1, 0x8000, 0, None, 0x9000, 64, 5,
                            lib.DECODE_GEOMETRY_READY, None, None) == lib.KVQ_ERR_WORKSPACE
    assert so.kvq_decode_ex(ctypes.byref(desc), 0x5000, 4, 32, 0x6000, 0x7000, 1, 0x8000, 0, None, 0x9000, 1 << 20,
                            5, 2, None, None) == lib.KVQ_ERR_INVALID_ARG


@pytest.mark.parametrize("bits", [2, 4, 8, 16])
@pytest.mark.parametrize("is_key", [True, False])
def test_layout_reader_is_a_bijection(bits, is_key):
    assert offsets_are_a_permutation(bits, is_key)


def test_package_fails_loudly_without_the_library(tmp_path, monkeypatch):
    from quantized_kv_cache_07_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()
