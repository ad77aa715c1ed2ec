"""Torch-owned device buffers for one layer's quantized KV cache.

PyTorch only allocates device memory and provides the stream; every byte of
the cache is written by the library's kernels (kvq_append) and read by them
(kvq_decode, kvq_dequant).  See include/kvq.h for the layouts.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib

HEAD_DIM = 128
BLOCK_SIZE = 16


def _require_cuda():
    if not torch.cuda.is_available():
        raise RuntimeError("a CUDA device is required (there is no CPU fallback)")


class KVCache:
    """Block pools (+ optional bf16 window ring) of one attention layer.

    ``asym=True`` selects the asymmetric format: a per-token zero point is
    stored beside each scale in the metadata pool.  ``q_bits=8``
    makes kvq_decode quantize each query row to int8 (integer dot product).
    """

    def __init__(self, num_blocks: int, kv_heads: int, k_bits: int, v_bits: int, window: int = 0,
                 window_batch: int = 0, channel_factor=None, asym: bool = False, q_bits: int = 16,
                 k_per_channel: bool = False, device="cuda"):
        _require_cuda()
        self.num_blocks, self.kv_heads = int(num_blocks), int(kv_heads)
        self.k_bits, self.v_bits = int(k_bits), int(v_bits)
        self.window, self.window_batch = int(window), int(window_batch)
        self.device = torch.device(device)
        kbb, vbb = _lib.block_bytes(k_bits), _lib.block_bytes(v_bits)
        self.k_codes = torch.zeros(self.num_blocks * kv_heads * kbb, dtype=torch.uint8, device=device)
        self.v_codes = torch.zeros(self.num_blocks * kv_heads * vbb, dtype=torch.uint8, device=device)
        quant = k_bits != 16
        self.k_per_channel = bool(k_per_channel)
        self.asym = bool(asym)
        if self.asym and not quant:
            raise ValueError("the asymmetric format needs 8-, 4- or 2-bit blocks")
        # metadata pool: per block K scales, (K zero points,) V scales, (V zero
        # points); 2-bit blocks: one K scale, K zero point, V scale, V zero point
        self.meta_floats = 4 if k_bits == 2 else (4 if self.asym else 2) * BLOCK_SIZE
        self.meta = (torch.zeros(self.num_blocks * kv_heads * self.meta_floats, dtype=torch.float32, device=device)
                     if quant else None)
        self.channel_factor = None
        if channel_factor is not None:
            self.channel_factor = torch.as_tensor(np.ascontiguousarray(channel_factor, dtype=np.float32)
                                                  ).reshape(kv_heads, HEAD_DIM).to(device)
        self.k_window = self.v_window = None
        if window > 0:
            n_w = max(window_batch, 1) * kv_heads * window * HEAD_DIM
            self.k_window = torch.zeros(n_w, dtype=torch.bfloat16, device=device)
            self.v_window = torch.zeros(n_w, dtype=torch.bfloat16, device=device)
        self.desc = _lib.CacheDesc(
            num_kv_heads=kv_heads, head_dim=HEAD_DIM, block_size=BLOCK_SIZE, num_blocks=self.num_blocks,
            k_bits=k_bits, v_bits=v_bits,
            k_codes=self.k_codes.data_ptr(), v_codes=self.v_codes.data_ptr(),
            meta=self.meta.data_ptr() if quant else None, asym=int(self.asym),
            k_channel_factor=self.channel_factor.data_ptr() if self.channel_factor is not None else None,
            window=self.window, window_batch=max(window_batch, 1) if window > 0 else 0,
            k_window=self.k_window.data_ptr() if self.k_window is not None else None,
            v_window=self.v_window.data_ptr() if self.v_window is not None else None,
            q_bits=int(q_bits), k_per_channel=int(self.k_per_channel))

    # bytes the decode reads per cached token per KV head (codes + scales + zero
    # points); 2-bit blocks share one 16-byte record per 16 tokens
    def bytes_per_token_head(self) -> float:
        if self.k_bits == 2:
            return 2 * HEAD_DIM * 2 / 8 + 16 / BLOCK_SIZE
        meta = 8 if self.asym else 4
        kb = HEAD_DIM * self.k_bits // 8 + (0 if self.k_bits == 16 or self.k_per_channel else meta)
        vb = HEAD_DIM * self.v_bits // 8 + (0 if self.v_bits == 16 else meta)
        return kb + vb

    def allocated_bytes(self) -> int:
        ts = [self.k_codes, self.v_codes, self.meta, self.k_window, self.v_window]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)


class DecodeWorkspace:
    """Scratch for the split-attention partials and merge counters of kvq_decode."""

    def __init__(self, cache: KVCache, batch: int, q_heads: int, stream_ctas: int = 0):
        self.batch, self.q_heads, self.stream_ctas = batch, q_heads, stream_ctas
        self.nbytes = _lib.kvq_decode_workspace_size(cache.desc, batch, q_heads, stream_ctas)
        self.buf = torch.empty(max(self.nbytes, 16), dtype=torch.uint8, device=cache.device)
        _lib.kvq_workspace_init(self.buf, self.nbytes)


def _bits_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def fill_from_inputs(cache: KVCache, inp, device="cuda", chunk_tokens: int = 1 << 18, err_word=None):
    """Write every cached token of a synthetic workload into ``cache``.

    Positions older than the window are quantized into the block store
    (kvq_append QUANT); the last ``window`` positions go to the bf16 ring
    (kvq_append RING).  Calls are cut into chunks of about ``chunk_tokens``
    rows (at 16-token block boundaries for 2-bit caches, whose blocks are
    quantized whole).  Runs on the current stream; returns the device block
    table and cached lengths.
    """
    w = inp.workload
    table = torch.from_numpy(inp.block_table).to(device)
    lengths = inp.lengths.astype(np.int64)
    offs = inp.seq_offsets
    n_tok = int(offs[-1])
    row_seq = np.repeat(np.arange(w.batch, dtype=np.int32), lengths)
    row_pos = (np.arange(n_tok, dtype=np.int64) - np.repeat(offs[:-1], lengths)).astype(np.int32)
    if w.window > 0:
        lq = np.maximum(lengths - w.window, 0)
        row_ring = row_pos >= np.repeat(lq, lengths)
    else:
        row_ring = np.zeros(n_tok, dtype=bool)
    H = w.kv_heads
    r0 = 0
    while r0 < n_tok:
        r1 = min(n_tok, r0 + chunk_tokens)
        if w.k_bits == 2:
            # 2-bit blocks are quantized whole: end the chunk at a block boundary
            while r1 < n_tok and row_pos[r1] % BLOCK_SIZE != 0:
                r1 += 1
        for mode, sel in ((_lib.APPEND_QUANT, ~row_ring[r0:r1]), (_lib.APPEND_RING, row_ring[r0:r1])):
            idx = np.nonzero(sel)[0] + r0
            if idx.size == 0:
                continue
            if idx.size == r1 - r0:
                kb, vb = inp.k[r0:r1], inp.v[r0:r1]
            else:
                kb, vb = inp.k[idx], inp.v[idx]
            kt = _bits_tensor(kb.reshape(-1, H, HEAD_DIM), device)
            vt = _bits_tensor(vb.reshape(-1, H, HEAD_DIM), device)
            si = torch.from_numpy(row_seq[idx]).to(device)
            po = torch.from_numpy(row_pos[idx]).to(device)
            _lib.kvq_append(cache.desc, kt, vt, si, po, mode, table, w.batch, inp.max_blocks, err_word=err_word)
        r0 = r1
    return table, torch.from_numpy(inp.lengths.astype(np.int32)).to(device)


def cache_for_inputs(inp, device="cuda") -> KVCache:
    w = inp.workload
    return KVCache(inp.num_blocks, w.kv_heads, w.k_bits, w.v_bits, window=w.window,
                   window_batch=w.batch if w.window else 0, channel_factor=inp.channel_factor,
                   asym=getattr(w, "asym", False), q_bits=getattr(w, "q_bits", 16),
                   k_per_channel=getattr(w, "k_per_channel", False), device=device)
