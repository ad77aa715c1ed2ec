"""Shared helpers of the parity tests: run the CUDA path through the C ABI and
the float64 oracle on the same seeded bits, and compare."""
from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O
from synth import Workload, make_inputs

TOL = 2e-3


def small_workload(name, **kw) -> Workload:
    base = dict(batch=3, q_heads=8, kv_heads=2, k_bits=8, v_bits=8, len_range=(1, 300))
    base.update(kw)
    return Workload(name, **base)


def seq_kv(inp, b):
    """float64 K, V [L(+1), H, D] of sequence b (with the appended token, if any)."""
    a, e = inp.seq_offsets[b], inp.seq_offsets[b + 1]
    k = O.bf16_to_f64(inp.k[a:e])
    v = O.bf16_to_f64(inp.v[a:e])
    if inp.workload.append_one:
        k = np.concatenate([k, O.bf16_to_f64(inp.k_new[b:b + 1])], axis=0)
        v = np.concatenate([v, O.bf16_to_f64(inp.v_new[b:b + 1])], axis=0)
    return k, v


def oracle_state(inp, b):
    w = inp.workload
    k, v = seq_kv(inp, b)
    c = None if inp.channel_factor is None else inp.channel_factor.astype(np.float64)
    return O.quantize_sequence(k, v, w.k_bits, w.v_bits, window=w.window, c=c, asym=w.asym,
                               k_per_channel=w.k_per_channel)


def oracle_decode(inp, units=None, states=None):
    """Oracle outputs {(b, h): (o [G, D], lse [G])} for the requested units
    (``states``: optional {b: oracle_state(inp, b)} computed beforehand)."""
    w = inp.workload
    G = w.group
    res = {}
    bs = sorted({b for b, _ in units}) if units is not None else range(w.batch)
    for b in bs:
        st = states[b] if states is not None else oracle_state(inp, b)
        q = O.bf16_to_f64(inp.q[b])
        for h in range(w.kv_heads):
            if units is not None and (b, h) not in units:
                continue
            k_hat, v_hat = O.reconstruct_sequence(st, h)
            qh = q[h * G:(h + 1) * G]
            if w.q_bits == 8:
                qh = O.effective_query(qh, None if st["c"] is None else st["c"][h])
            res[(b, h)] = O.attention(qh, k_hat, v_hat)
    return res


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 8)


def compare_outputs(inp, out, lse, ref, out_is_bf16: bool):
    """Max violation ratio (<= 1 passes) over the units in ``ref``."""
    G = inp.workload.group
    worst = 0.0
    for (b, h), (o_ref, l_ref) in ref.items():
        o = out[b, h * G:(h + 1) * G].astype(np.float64)
        tol = TOL + (bf16_half_ulp(o_ref) if out_is_bf16 else 0.0)
        worst = max(worst, float(np.max(np.abs(o - o_ref) / tol)))
        if lse is not None:
            lg = lse[b, h * G:(h + 1) * G].astype(np.float64)
            fin = np.isfinite(l_ref)
            assert np.array_equal(np.isfinite(lg), fin)
            if fin.any():
                worst = max(worst, float(np.max(np.abs(lg[fin] - l_ref[fin]) / TOL)))
            if (~fin).any():
                assert np.all(np.isneginf(lg[~fin]))
    return worst


class DeviceRun:
    """Build the cache of ``inp`` on the GPU with kvq_append and run kvq_decode."""

    def __init__(self, inp, device="cuda"):
        import torch

        from quantized_kv_cache_07_gb300 import _lib
        from quantized_kv_cache_07_gb300.cache import cache_for_inputs, fill_from_inputs
        self.torch, self.lib = torch, _lib
        self.inp = inp
        w = inp.workload
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.cache = cache_for_inputs(inp, device)
        self.table, self.lens = fill_from_inputs(self.cache, inp, device, err_word=self.err)
        if w.append_one:
            self.append_step()
        self.q = torch.from_numpy(inp.q.view(np.int16)).to(device).view(torch.bfloat16)
        self.device = device

    def append_step(self):
        torch = self.torch
        w, inp = self.inp.workload, self.inp
        kt = torch.from_numpy(inp.k_new.view(np.int16)).cuda().view(torch.bfloat16)
        vt = torch.from_numpy(inp.v_new.view(np.int16)).cuda().view(torch.bfloat16)
        si = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        po = torch.from_numpy(inp.lengths.astype(np.int32)).cuda()
        self.lib.kvq_append(self.cache.desc, kt, vt, si, po, self.lib.APPEND_QUANT, self.table, w.batch,
                            inp.max_blocks, err_word=self.err)
        self.lens = torch.from_numpy(inp.decode_lengths.astype(np.int32)).cuda()

    def decode(self, out_fp32=True, stream_ctas=0, lens=None, flags=0, table=None):
        from quantized_kv_cache_07_gb300.cache import DecodeWorkspace
        torch = self.torch
        w = self.inp.workload
        out = torch.zeros((w.batch, w.q_heads, 128), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=self.device)
        lse = torch.zeros((w.batch, w.q_heads), dtype=torch.float32, device=self.device)
        ws = DecodeWorkspace(self.cache, w.batch, w.q_heads, stream_ctas)
        self.lib.kvq_decode(self.cache.desc, self.q, w.batch, w.q_heads, self.lens if lens is None else lens,
                            self.table if table is None else table, self.inp.max_blocks, out, lse=lse,
                            workspace=ws.buf, workspace_bytes=ws.nbytes, stream_ctas=stream_ctas, err_word=self.err,
                            flags=flags)
        torch.cuda.synchronize()
        return out.float().cpu().numpy(), lse.cpu().numpy()

    def err_bits(self) -> int:
        self.torch.cuda.synchronize()
        return int(self.err.item())

    def pools(self):
        c = self.cache
        get = lambda t: None if t is None else t.cpu().numpy()
        return dict(k_codes=get(c.k_codes), v_codes=get(c.v_codes), meta=get(c.meta),
                    k_window=None if c.k_window is None else c.k_window.view(self.torch.uint8).cpu().numpy(),
                    v_window=None if c.v_window is None else c.v_window.view(self.torch.uint8).cpu().numpy())
