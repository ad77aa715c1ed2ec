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


def _run(fmt, chunk=24, fused=True, stream_ctas=0, seed=5, order="seq", heads=(8, 2), q_bias=0.0):
    """Prefix written first, then one kvq_prefill call over the last `chunk`
    positions of every sequence; rows grouped by sequence ("seq") or
    alternating between sequences ("interleaved")."""
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.cache import cache_for_inputs
    spec = PREFILL_FORMATS.get(fmt) or TILE_FORMATS[fmt]
    w = small_workload(f"prefill_{fmt}", batch=3, q_heads=heads[0], kv_heads=heads[1], len_range=(40, 300),
                       paged=True, **spec)
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
    if order == "seq":
        pairs = [(b, p) for b in range(w.batch) for p in chunk_pos[b]]
    else:
        longest = max(len(chunk_pos[b]) for b in range(w.batch))
        pairs = [(b, chunk_pos[b][c]) for c in range(longest) for b in range(w.batch) if c < len(chunk_pos[b])]
    seq = np.asarray([b for b, _ in pairs], dtype=np.int32)
    pos = np.asarray([p for _, p in pairs], dtype=np.int32)
    rows = np.asarray([inp.seq_offsets[b] + p for b, p in pairs], dtype=np.int64)
    n = len(seq)
    from synth import query_rows
    qbits = query_rows(n, w.q_heads, seed)
    if q_bias:
        from synth import f32_to_bf16_bits
        qbits = f32_to_bf16_bits((O.bf16_to_f64(qbits) + q_bias).astype(np.float32))
    out = torch.zeros((n, w.q_heads, 128), dtype=torch.float32, device="cuda")
    lse = torch.zeros((n, w.q_heads), dtype=torch.float32, device="cuda")
    nb = _lib.kvq_prefill_workspace_size(cache.desc, n, w.q_heads, stream_ctas)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
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


# formats the query-tile path takes (symmetric 8-/4-bit blocks, fp16 query)
TILE_FORMATS = {
    "k4v8_t3": dict(k_bits=4, v_bits=8, k_dist="t3"),
    "k8v4_chan": dict(k_bits=8, v_bits=4, channel_factor=True, k_per_channel=True),
    "asym_int8_factor": dict(k_bits=8, v_bits=8, asym=True, channel_factor=True),
    "asym_int2": dict(k_bits=2, v_bits=2, asym=True),
    "qint8_asym_k4v4_factor": dict(k_bits=4, v_bits=4, asym=True, channel_factor=True, q_bits=8),
    "q32_asym_int4_factor_outliers": dict(k_bits=4, v_bits=4, asym=True, channel_factor=True, outlier_channels=4,
                                          q_bits=32),
    "bf16": dict(k_bits=16, v_bits=16),
}
TILE_PATH_FORMATS = ["int8", "int4_factor", "k4v8_t3", "k8v4_chan", "asym_k4v8", "asym_int8_factor", "int2",
                     "asym_int2", "qint8_int8", "qint8_asym_k4v4_factor", "q32_k8v4", "q32_asym_int4_factor_outliers"]


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


def _check_against_oracle(res):
    inp, cache, qbits, seq, pos, out, lse, err = res
    assert err == 0
    o_ref, l_ref = _oracle(inp, qbits, seq, pos)
    assert np.max(np.abs(out - o_ref)) <= TOL
    assert np.max(np.abs(lse - l_ref)) <= TOL


@pytest.mark.parametrize("fmt", ["int8", "qint8_int8"])
@pytest.mark.parametrize("bias", [4.0, 16.0])
def test_prefill_tiles_with_biased_queries(fmt, bias):
    """Query rows with a large common component on int8 keys: the tile path's
    score accumulators start at minus 1152 times each row's sums (the int8 key
    codes enter with their offset), largest relative to the code dot here.
    Both paths: the tile kernel and split rows (the decode kernel)."""
    from quantized_kv_cache_07_gb300 import _lib
    _check_against_oracle(_run(fmt, order="interleaved", q_bias=bias, stream_ctas=_lib.PREFILL_TILES))
    _check_against_oracle(_run(fmt, order="interleaved", q_bias=bias, stream_ctas=7))


def test_prefill_auto_takes_tiles_when_they_fill_the_gpu():
    """stream_ctas = 0 takes the tile path once its (tile, KV head) CTAs number
    at least 9/16 of the SMs: its outputs then equal the tile path's bit for bit."""
    from quantized_kv_cache_07_gb300 import _lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    auto = _run("int8", chunk=64, fused=False, stream_ctas=0, heads=(32, 8))
    rows = len(auto[3])
    ctas = ((rows + 3) // 4) * 8  # 16 / G = 4 rows per tile, 8 KV heads
    if ctas * 16 < 9 * sms:
        pytest.skip(f"{ctas} tile CTAs do not reach 9/16 of {sms} SMs on this GPU")
    tiles = _run("int8", chunk=64, fused=False, stream_ctas=_lib.PREFILL_TILES, heads=(32, 8))
    np.testing.assert_array_equal(auto[5], tiles[5])
    np.testing.assert_array_equal(auto[6], tiles[6])


@pytest.mark.parametrize("fmt", TILE_PATH_FORMATS)
@pytest.mark.parametrize("order", ["seq", "interleaved"])
def test_prefill_tiles_match_the_oracle(fmt, order):
    """The query-tile path (16 query vectors per CTA): rows grouped by sequence,
    and rows alternating between sequences so that every tile holds rows of
    several sequences (taken in turn)."""
    from quantized_kv_cache_07_gb300 import _lib
    # 2-bit blocks are written whole by runs of rows in order: interleaved rows
    # attend to a chunk written beforehand
    fused = not (order == "interleaved" and "int2" in fmt)
    _check_against_oracle(_run(fmt, stream_ctas=_lib.PREFILL_TILES, order=order, fused=fused))


@pytest.mark.parametrize("heads", [(4, 4), (6, 2), (16, 2)], ids=["g1", "g3", "g8"])
@pytest.mark.parametrize("fmt", ["int8", "asym_k4v8", "int2"])
def test_prefill_tiles_group_sizes(heads, fmt):
    """16 / G rows per tile for G = 1 (16 rows), 3 (5 rows, 15 vectors) and 8 (2 rows)."""
    from quantized_kv_cache_07_gb300 import _lib
    _check_against_oracle(_run(fmt, stream_ctas=_lib.PREFILL_TILES, order="interleaved", heads=heads,
                               fused=fmt != "int2"))


def test_prefill_tiles_and_split_rows_agree_without_the_write():
    from quantized_kv_cache_07_gb300 import _lib
    a = _run("int4_factor", fused=False, stream_ctas=_lib.PREFILL_TILES)
    b = _run("int4_factor", fused=False, stream_ctas=5)
    assert a[7] == 0 and b[7] == 0
    np.testing.assert_allclose(a[5], b[5], rtol=0, atol=TOL)
    np.testing.assert_allclose(a[6], b[6], rtol=0, atol=TOL)


@pytest.mark.parametrize("fmt", ["bf16"])
def test_prefill_tiles_refuse_other_formats(fmt):
    from quantized_kv_cache_07_gb300 import _lib
    with pytest.raises(_lib.KvqError) as e:
        _run(fmt, stream_ctas=_lib.PREFILL_TILES)
    assert e.value.status == _lib.KVQ_ERR_UNSUPPORTED


def test_prefill_tiles_flag_bad_sequences_and_clamp_positions():
    """Rows with a sequence outside [0, batch): out = 0, lse = -inf and the
    POSITION bit; a position beyond the block table's capacity: the SEQ_LEN bit
    and attention over the capacity, as the split-rows path."""
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.cache import KVCache
    c0 = KVCache(8, 2, 8, 8)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    kv = torch.randn((8 * 16, 2, 128), generator=g, device="cuda").bfloat16()
    seq0 = torch.zeros(8 * 16, dtype=torch.int32, device="cuda")
    pos0 = torch.arange(8 * 16, dtype=torch.int32, device="cuda")
    table = torch.arange(8, dtype=torch.int32, device="cuda").view(2, 4)
    _lib.kvq_append(c0.desc, kv[:64], kv[64:], seq0[:64], pos0[:64], _lib.APPEND_QUANT, table, 2, 4)
    q = torch.randn((3, 8, 128), generator=g, device="cuda").bfloat16()
    seq = torch.tensor([5, 0, 0], dtype=torch.int32, device="cuda")       # sequence 5 of a batch of 2
    pos = torch.tensor([3, 10, 200], dtype=torch.int32, device="cuda")    # 200 is beyond 4 blocks
    outs = []
    for sc in (_lib.PREFILL_TILES, 3):
        nb = _lib.kvq_prefill_workspace_size(c0.desc, 3, 8, sc)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full((3, 8, 128), 7.0, dtype=torch.float32, device="cuda")
        lse = torch.zeros((3, 8), dtype=torch.float32, device="cuda")
        _lib.kvq_prefill(c0.desc, q, 8, seq, pos, table, 2, 4, out, lse=lse, workspace=ws, workspace_bytes=nb,
                         stream_ctas=sc, err_word=err)
        torch.cuda.synchronize()
        e = int(err.item())
        assert e & _lib.KVQ_DEVERR_POSITION and e & _lib.KVQ_DEVERR_SEQ_LEN
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
        assert np.all(np.isfinite(o[1:])) and np.all(np.isfinite(l[1:]))
        outs.append((o, l))
    np.testing.assert_allclose(outs[0][0], outs[1][0], rtol=0, atol=TOL)
    np.testing.assert_allclose(outs[0][1], outs[1][1], rtol=0, atol=TOL)
