"""Chunked prefill (kvq_prefill) through the C ABI against the float64 oracle.

Each sequence's prefix is written first; then a chunk of new positions is
quantized into the cache and attends causally to the stored cache in the same
call.  Stored codes of the chunk are bit-exact; every row's output matches the
oracle's causal attention over the quantized sequence within 2e-3 (fp32 out),
lse within 2e-3.
"""
import numpy as np
import pytest

from harness import TOL, compare_outputs, oracle_state, small_workload
from layout_ref import unpack_blocks
from oracle import kvq_oracle as O
from synth import make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _write(lib, cache, inp, rows_by_seq, table, err):
    """kvq_append QUANT of the given positions of each sequence (rows in order)."""
    w = inp.workload
    seq, pos, rows = [], [], []
    for b, ps in rows_by_seq.items():
        seq += [b] * len(ps)
        pos += list(ps)
        rows += list(inp.seq_offsets[b] + np.asarray(ps, dtype=np.int64))
    if not rows:
        return
    rows = np.asarray(rows)
    lib.kvq_append(cache.desc, _bits(inp.k[rows]), _bits(inp.v[rows]), torch.tensor(seq, dtype=torch.int32).cuda(),
                   torch.tensor(pos, dtype=torch.int32).cuda(), lib.APPEND_QUANT, table, w.batch, inp.max_blocks,
                   err_word=err)


def _run(fmt, chunk=24, fused=True, stream_ctas=0, seed=5):
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.cache import cache_for_inputs
    w = small_workload(f"prefill_{fmt}", batch=3, q_heads=8, kv_heads=2, len_range=(40, 300), paged=True,
                       **PREFILL_FORMATS[fmt])
    inp = make_inputs(w)
    L = inp.lengths.astype(int)
    # chunk = the last `chunk` positions of each sequence (a block boundary for 2-bit caches)
    start = {b: (L[b] - chunk) // 16 * 16 if w.k_bits == 2 else L[b] - chunk for b in range(w.batch)}
    start = {b: max(s, 0) for b, s in start.items()}
    cache = cache_for_inputs(inp)
    table = torch.from_numpy(inp.block_table).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    prefix = {b: range(0, start[b]) for b in range(w.batch)}
    chunk_pos = {b: range(start[b], L[b]) for b in range(w.batch)}
    _write(_lib, cache, inp, prefix if fused else {b: range(0, L[b]) for b in range(w.batch)}, table, err)
    seq = np.concatenate([[b] * len(chunk_pos[b]) for b in range(w.batch)]).astype(np.int32)
    pos = np.concatenate([list(chunk_pos[b]) for b in range(w.batch)]).astype(np.int32)
    rows = np.concatenate([inp.seq_offsets[b] + np.asarray(chunk_pos[b], dtype=np.int64) for b in range(w.batch)])
    n = len(seq)
    from synth import query_rows
    qbits = query_rows(n, w.q_heads, seed)
    out = torch.zeros((n, w.q_heads, 128), dtype=torch.float32, device="cuda")
    lse = torch.zeros((n, w.q_heads), dtype=torch.float32, device="cuda")
    nb = _lib.kvq_prefill_workspace_size(cache.desc, n, w.q_heads, stream_ctas)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")
    _lib.kvq_prefill(cache.desc, _bits(qbits), w.q_heads, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                     table, w.batch, inp.max_blocks, out, k_new=_bits(inp.k[rows]) if fused else None,
                     v_new=_bits(inp.v[rows]) if fused else None, lse=lse, workspace=ws, workspace_bytes=nb,
                     stream_ctas=stream_ctas, err_word=err)
    torch.cuda.synchronize()
    return inp, cache, qbits, seq, pos, out.cpu().numpy(), lse.cpu().numpy(), int(err.item())


def _oracle(inp, qbits, seq, pos):
    w = inp.workload
    G = w.group
    o_ref = np.zeros((len(seq), w.q_heads, 128))
    l_ref = np.zeros((len(seq), w.q_heads))
    for b in np.unique(seq):
        st = oracle_state(inp, int(b))          # the whole stored sequence
        sel = np.nonzero(seq == b)[0]
        q = O.bf16_to_f64(qbits[sel])
        for h in range(w.kv_heads):
            qh = q[:, h * G:(h + 1) * G]
            if w.q_bits == 8:
                qh = np.stack([O.effective_query(x, None if st["c"] is None else st["c"][h]) for x in qh])
            o, l = O.prefill_attention(qh, st, h, pos[sel])
            o_ref[sel, h * G:(h + 1) * G] = o
            l_ref[sel, h * G:(h + 1) * G] = l
    return o_ref, l_ref


PREFILL_FORMATS = {
    "int8": dict(k_bits=8, v_bits=8, outlier_channels=4),
    "int4_factor": dict(k_bits=4, v_bits=4, channel_factor=True),
    "asym_k4v8": dict(k_bits=4, v_bits=8, asym=True, k_dist="t3"),
    "int2": dict(k_bits=2, v_bits=2),
    "q32_k8v4": dict(k_bits=8, v_bits=4, q_bits=32),
    "qint8_int8": dict(k_bits=8, v_bits=8, q_bits=8),
}


@pytest.mark.parametrize("fmt", list(PREFILL_FORMATS))
def test_prefill_matches_the_oracle_causal_attention(fmt):
    inp, cache, qbits, seq, pos, out, lse, err = _run(fmt)
    assert err == 0
    o_ref, l_ref = _oracle(inp, qbits, seq, pos)
    assert np.max(np.abs(out - o_ref)) <= TOL
    assert np.max(np.abs(lse - l_ref)) <= TOL
    # the chunk's codes were written by the same call, bit for bit
    w = inp.workload
    kc = unpack_blocks(cache.k_codes.cpu().numpy(), w.k_bits, True, w.kv_heads, asym=w.asym)
    for b in range(w.batch):
        st = oracle_state(inp, b)
        ps = pos[seq == b]
        phys = inp.block_table[b, ps // 16]
        np.testing.assert_array_equal(kc[phys, :, ps % 16], st["k_codes"][ps])


def test_prefill_without_the_write_and_split_counts_agree():
    """The chunk already in the cache (k_new = v_new = NULL) gives the same
    outputs as writing it in the call; a different split of the rows agrees
    within the default mode's weight rounding."""
    a = _run("int8", fused=True)
    b = _run("int8", fused=False)
    np.testing.assert_array_equal(a[5], b[5])
    np.testing.assert_array_equal(a[6], b[6])
    c = _run("int8", fused=False, stream_ctas=7)
    vmax = float(np.abs(O.bf16_to_f64(a[0].v)).max()) * (1 + 1 / 14)
    np.testing.assert_allclose(c[5], a[5], rtol=0, atol=2.0 ** -11 * vmax + 1e-5)


def test_prefill_rejects_a_window_and_flags_bad_sequences():
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.cache import KVCache
    c = KVCache(8, 2, 8, 8, window=32, window_batch=2)
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    out = torch.zeros((1, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(_lib.KvqError) as e:
        _lib.kvq_prefill(c.desc, q, 8, one, one, table, 2, 4, out, workspace=None, workspace_bytes=0)
    assert e.value.status == _lib.KVQ_ERR_UNSUPPORTED
    c0 = KVCache(8, 2, 8, 8)
    nb = _lib.kvq_prefill_workspace_size(c0.desc, 1, 8)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    bad = torch.full((1,), 5, dtype=torch.int32, device="cuda")   # sequence 5 of a batch of 2
    _lib.kvq_prefill(c0.desc, q, 8, bad, one, table, 2, 4, out, lse=lse, workspace=ws, workspace_bytes=nb,
                     err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & _lib.KVQ_DEVERR_POSITION
    assert np.all(out.cpu().numpy() == 0) and np.all(np.isneginf(lse.cpu().numpy()))
