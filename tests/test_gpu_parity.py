"""Parity of the CUDA path (through the C ABI) against the float64 oracle.

Stored codes and scales must match bit for bit; decode outputs must be within
2e-3 max-abs (fp32 output), 2e-3 + half a bf16 ulp (bf16 output), and lse within
2e-3.  Small cases span several 64-token stages and ragged tails; the five
named workloads run at full size on sampled (sequence, kv head) units.
"""
import numpy as np
import pytest

from harness import DeviceRun, compare_outputs, oracle_decode, oracle_state, small_workload
from layout_ref import meta_by_block, unpack_blocks
from oracle import kvq_oracle as O
from synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

SMALL = {
    "int8_g4": small_workload("int8_g4"),
    "int8_g1": small_workload("int8_g1", q_heads=4, kv_heads=4, len_range=(1, 200)),
    "int4_factor_g8": small_workload("int4_factor_g8", batch=4, q_heads=16, kv_heads=2, k_bits=4, v_bits=4,
                                     channel_factor=True),
    "k4v8_g8_t3": small_workload("k4v8_g8_t3", batch=2, q_heads=16, kv_heads=2, k_bits=4, v_bits=8,
                                 len_range=(100, 700), k_dist="t3"),
    "k8v4_g2": small_workload("k8v4_g2", batch=3, q_heads=8, kv_heads=4, k_bits=8, v_bits=4),
    "window32_int8": small_workload("window32_int8", batch=5, len_range=(1, 120), window=32,
                                    outlier_channels=4),
    "window128_int8": small_workload("window128_int8", batch=3, len_range=(100, 400), window=128),
    "paged_append": small_workload("paged_append", batch=4, len_range=(1, 250), paged=True, append_one=True),
    "bf16": small_workload("bf16", k_bits=16, v_bits=16, len_range=(1, 333)),
    "bf16_g8": small_workload("bf16_g8", batch=2, q_heads=16, kv_heads=2, k_bits=16, v_bits=16,
                              len_range=(50, 400), k_dist="t3"),
    # asymmetric format (per-token scale and zero point)
    "asym_int8_g4": small_workload("asym_int8_g4", asym=True, outlier_channels=4),
    "asym_int4_factor_g8": small_workload("asym_int4_factor_g8", batch=4, q_heads=16, kv_heads=2, k_bits=4,
                                          v_bits=4, channel_factor=True, asym=True),
    "asym_k4v8_window32_t3": small_workload("asym_k4v8_window32_t3", batch=3, q_heads=16, kv_heads=2, k_bits=4,
                                            v_bits=8, len_range=(1, 500), window=32, k_dist="t3", asym=True),
    "asym_k8v4_paged_append": small_workload("asym_k8v4_paged_append", batch=4, q_heads=4, kv_heads=4, k_bits=8,
                                             v_bits=4, len_range=(1, 250), paged=True, append_one=True,
                                             asym=True),
    # quantized query (int8 query rows, integer dot product)
    "qint8_int8_g4": small_workload("qint8_int8_g4", q_bits=8, outlier_channels=4),
    "qint8_int4_factor_g8": small_workload("qint8_int4_factor_g8", batch=4, q_heads=16, kv_heads=2, k_bits=4,
                                           v_bits=4, channel_factor=True, q_bits=8),
    "qint8_k4v8_window32_t3": small_workload("qint8_k4v8_window32_t3", batch=3, q_heads=16, kv_heads=2, k_bits=4,
                                             v_bits=8, len_range=(1, 500), window=32, k_dist="t3", q_bits=8),
    "qint8_asym_k8v4_g1": small_workload("qint8_asym_k8v4_g1", batch=3, q_heads=4, kv_heads=4, k_bits=8, v_bits=4,
                                         len_range=(1, 300), asym=True, q_bits=8),
    # keys under per-channel scales only (calibrated on the first half of the tokens: the clamp binds)
    "kchan_int8_g4": small_workload("kchan_int8_g4", channel_factor=True, k_per_channel=True, outlier_channels=4),
    # heavy-tailed keys under per-channel scales give scores near 10: the fp16
    # query's 11 bits are not enough for 2e-3, the two-part query is (q_bits 32)
    "kchan_k4v8_window32_g8": small_workload("kchan_k4v8_window32_g8", batch=3, q_heads=16, kv_heads=2, k_bits=4,
                                             v_bits=8, len_range=(1, 500), window=32, channel_factor=True,
                                             k_per_channel=True, k_dist="t3", q_bits=32),
    "kchan_qint8_int4_g8": small_workload("kchan_qint8_int4_g8", batch=4, q_heads=16, kv_heads=2, k_bits=4,
                                          v_bits=4, channel_factor=True, k_per_channel=True, q_bits=8),
    # two-part fp16 query (q_bits 32)
    "q32_int8_g4": small_workload("q32_int8_g4", q_bits=32, outlier_channels=4, window=32, len_range=(1, 200)),
    "q32_asym_int4_factor_g8": small_workload("q32_asym_int4_factor_g8", batch=4, q_heads=16, kv_heads=2, k_bits=4,
                                              v_bits=4, channel_factor=True, asym=True, q_bits=32),
    # 2-bit codes with one scale (and zero point) per 16-token block
    "int2_g4": small_workload("int2_g4", k_bits=2, v_bits=2, outlier_channels=4),
    "int2_factor_g8": small_workload("int2_factor_g8", batch=4, q_heads=16, kv_heads=2, k_bits=2, v_bits=2,
                                     channel_factor=True),
    "asym_int2_window32_t3": small_workload("asym_int2_window32_t3", batch=3, q_heads=16, kv_heads=2, k_bits=2,
                                            v_bits=2, len_range=(1, 500), window=32, k_dist="t3", asym=True),
    "q32_int2_g1": small_workload("q32_int2_g1", batch=3, q_heads=4, kv_heads=4, k_bits=2, v_bits=2,
                                  len_range=(1, 300), q_bits=32),
    "qint8_asym_int2_g8": small_workload("qint8_asym_int2_g8", batch=2, q_heads=16, kv_heads=2, k_bits=2, v_bits=2,
                                         asym=True, q_bits=8),
}


@pytest.fixture(scope="module")
def runs():
    cache = {}

    def get(name):
        if name not in cache:
            inp = make_inputs(SMALL[name])
            cache[name] = (inp, DeviceRun(inp))
        return cache[name]
    return get


def check_stored_cache(inp, run, units=None, max_positions=None, states=None):
    """Block-store codes/scales and window ring vs the oracle, bit for bit."""
    w = inp.workload
    pools = run.pools()
    kc = unpack_blocks(pools["k_codes"], w.k_bits, True, w.kv_heads, asym=w.asym)
    vc = unpack_blocks(pools["v_codes"], w.v_bits, False, w.kv_heads, asym=w.asym)
    bs = sorted({b for b, _ in units}) if units else range(w.batch)
    rng = np.random.default_rng(7)
    checked = 0
    for b in bs:
        st = states[b] if states is not None else oracle_state(inp, b)
        Lq = st["Lq"]
        pos = np.arange(Lq)
        if max_positions and Lq > max_positions:
            pos = np.unique(np.concatenate([pos[:64], pos[-64:], rng.choice(Lq, max_positions, replace=False)]))
        phys = inp.block_table[b, pos // 16]
        tok = pos % 16
        if w.k_bits == 16:
            from synth import f32_to_bf16_bits
            np.testing.assert_array_equal(kc[phys, :, tok], f32_to_bf16_bits(st["k_plain"][pos].astype(np.float32)))
            np.testing.assert_array_equal(vc[phys, :, tok], f32_to_bf16_bits(st["v_plain"][pos].astype(np.float32)))
        else:
            np.testing.assert_array_equal(kc[phys, :, tok], st["k_codes"][pos])
            np.testing.assert_array_equal(vc[phys, :, tok], st["v_codes"][pos])
            md = meta_by_block(pools["meta"], w.kv_heads, w.asym, group=w.k_bits == 2)
            vs = md["v_scale"][phys, :, tok]
            if not w.k_per_channel:
                ks = md["k_scale"][phys, :, tok]
                np.testing.assert_array_equal(ks.view(np.uint32),
                                              st["k_scale"][pos].astype(np.float32).view(np.uint32))
            np.testing.assert_array_equal(vs.view(np.uint32), st["v_scale"][pos].astype(np.float32).view(np.uint32))
            if w.asym:
                ko = md["k_offset"][phys, :, tok]
                vo = md["v_offset"][phys, :, tok]
                np.testing.assert_array_equal(ko.view(np.uint32),
                                              st["k_offset"][pos].astype(np.float32).view(np.uint32))
                np.testing.assert_array_equal(vo.view(np.uint32),
                                              st["v_offset"][pos].astype(np.float32).view(np.uint32))
        checked += len(pos)
        if w.window:
            L = Lq + st["k_window"].shape[0]
            wp = np.arange(Lq, L)
            ring_k = unpack_blocks(pools["k_window"], 16, True, 1).reshape(w.batch, w.kv_heads, w.window, 128)[b][:, wp % w.window]
            ring_v = unpack_blocks(pools["v_window"], 16, False, 1).reshape(w.batch, w.kv_heads, w.window, 128)[b][:, wp % w.window]
            from synth import f32_to_bf16_bits
            np.testing.assert_array_equal(ring_k.transpose(1, 0, 2), f32_to_bf16_bits(st["k_window"].astype(np.float32)))
            np.testing.assert_array_equal(ring_v.transpose(1, 0, 2), f32_to_bf16_bits(st["v_window"].astype(np.float32)))
    return checked


@pytest.mark.parametrize("name", list(SMALL))
def test_append_stores_bit_exact_codes_and_scales(runs, name):
    inp, run = runs(name)
    assert check_stored_cache(inp, run) > 0
    assert run.err_bits() == 0


def _exact_rn32(a, b):
    """RN32(a + b) for float64 a, b whose float64 sum is exact (checked with the
    error term of Knuth's TwoSum), so one rounding to float32 is the correctly
    rounded result."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    assert np.all(err == 0.0), "float64 sum not exact: the reference would round twice"
    return s.astype(np.float32)


@pytest.mark.parametrize("name", ["asym_int8_g4", "asym_int4_factor_g8", "asym_k4v8_window32_t3",
                                  "asym_int2_window32_t3"])
def test_dequant_asym_returns_rn32_of_code_times_scale_plus_offset(runs, name):
    inp, run = runs(name)
    w = inp.workload
    b = 0
    st = oracle_state(inp, b)
    pos = np.arange(st["Lq"])
    if pos.size == 0:
        pytest.skip("sequence 0 lies entirely in the window")
    slots = inp.block_table[b, pos // 16].astype(np.int64) * 16 + pos % 16
    st_t = torch.from_numpy(slots.astype(np.int32)).cuda()
    ko = torch.empty((len(pos), w.kv_heads, 128), dtype=torch.float32, device="cuda")
    vo = torch.empty_like(ko)
    run.lib.kvq_dequant(run.cache.desc, st_t, ko, vo)
    torch.cuda.synchronize()
    for got, tag in ((ko, "k"), (vo, "v")):
        u = st[f"{tag}_codes"][pos].astype(np.float64)
        prod = u * st[f"{tag}_scale"][pos].astype(np.float64)[..., None]          # exact: <= 32 significant bits
        ref = _exact_rn32(prod, np.broadcast_to(st[f"{tag}_offset"][pos].astype(np.float64)[..., None], prod.shape))
        np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("name", ["kchan_int8_g4", "kchan_k4v8_window32_g8"])
def test_dequant_per_channel_keys_return_rn32_of_code_times_channel_scale(runs, name):
    inp, run = runs(name)
    w = inp.workload
    st = oracle_state(inp, 0)
    pos = np.arange(st["Lq"])
    if pos.size == 0:
        pytest.skip("sequence 0 lies entirely in the window")
    slots = inp.block_table[0, pos // 16].astype(np.int64) * 16 + pos % 16
    ko = torch.empty((len(pos), w.kv_heads, 128), dtype=torch.float32, device="cuda")
    vo = torch.empty_like(ko)
    run.lib.kvq_dequant(run.cache.desc, torch.from_numpy(slots.astype(np.int32)).cuda(), ko, vo)
    torch.cuda.synchronize()
    ref_k = (st["k_codes"][pos].astype(np.float64) * inp.channel_factor.astype(np.float64)).astype(np.float32)
    np.testing.assert_array_equal(ko.cpu().numpy().view(np.uint32), ref_k.view(np.uint32))
    if w.k_bits == 8:  # calibrated on the first half of the tokens: later ones hit the clamp
        assert np.abs(st["k_codes"]).max() == 127


@pytest.mark.parametrize("name", ["int8_g4", "int4_factor_g8", "k4v8_g8_t3", "bf16", "int2_factor_g8"])
def test_dequant_returns_rn32_of_code_times_scale(runs, name):
    inp, run = runs(name)
    w = inp.workload
    b = 0
    st = oracle_state(inp, b)
    pos = np.arange(st["Lq"])
    slots = inp.block_table[b, pos // 16].astype(np.int64) * 16 + pos % 16
    st_t = torch.from_numpy(slots.astype(np.int32)).cuda()
    ko = torch.empty((len(pos), w.kv_heads, 128), dtype=torch.float32, device="cuda")
    vo = torch.empty_like(ko)
    run.lib.kvq_dequant(run.cache.desc, st_t, ko, vo)
    torch.cuda.synchronize()
    if w.k_bits == 16:
        np.testing.assert_array_equal(ko.cpu().numpy(), st["k_plain"][pos].astype(np.float32))
        return
    ref_k = O.dequantize(st["k_codes"][pos], st["k_scale"][pos]).astype(np.float32)   # exact, then RN32
    ref_v = O.dequantize(st["v_codes"][pos], st["v_scale"][pos]).astype(np.float32)
    np.testing.assert_array_equal(ko.cpu().numpy().view(np.uint32), ref_k.view(np.uint32))
    np.testing.assert_array_equal(vo.cpu().numpy().view(np.uint32), ref_v.view(np.uint32))


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("out_fp32", [True, False])
def test_decode_matches_oracle(runs, name, out_fp32):
    inp, run = runs(name)
    out, lse = run.decode(out_fp32=out_fp32)
    ref = oracle_decode(inp)
    worst = compare_outputs(inp, out, lse, ref, out_is_bf16=not out_fp32)
    assert worst <= 1.0, f"max error ratio {worst:.3f}"
    assert run.err_bits() == 0


@pytest.mark.parametrize("name", ["int8_g4", "k4v8_g8_t3", "window32_int8", "asym_k4v8_window32_t3",
                                  "qint8_k4v8_window32_t3"])
def test_decode_split_count_changes_default_weights_by_their_rounding_only(runs, name):
    """Default mode: the fp16 value weights p*s_v are rounded relative to each
    split's running maximum, so a weight moves by at most 2^-11 relative and the
    outputs of two splits differ by at most 2^-11 * max|v_hat| (+ fp32 noise).
    The two-part mode below removes this term."""
    inp, run = runs(name)
    vmax = float(np.abs(O.bf16_to_f64(inp.v)).max()) * (1 + 1 / 14)
    atol = 2.0 ** -11 * vmax + 1e-5
    base, base_lse = run.decode(out_fp32=True, stream_ctas=1)
    for p in (2, 3, 7, 64, 0):
        out, lse = run.decode(out_fp32=True, stream_ctas=p)
        np.testing.assert_allclose(out, base, rtol=0, atol=atol)
        np.testing.assert_allclose(lse, base_lse, rtol=0, atol=2e-5)


SPLIT_TWO_PART = {
    # code blocks in the two-part mode (query and value weights as fp16 hi + lo)
    "int8_g4": SMALL["int8_g4"].with_(name="split2_int8_g4", q_bits=32),
    "k4v8_g8_t3": SMALL["k4v8_g8_t3"].with_(name="split2_k4v8_g8_t3", q_bits=32),
    "window32_int8": SMALL["window32_int8"].with_(name="split2_window32_int8", q_bits=32),
    "asym_k4v8_window32_t3": SMALL["asym_k4v8_window32_t3"].with_(name="split2_asym_k4v8_window32_t3", q_bits=32),
    "int4_factor_g8": SMALL["int4_factor_g8"].with_(name="split2_int4_factor_g8", q_bits=32),
    "int2_factor_g8": SMALL["int2_factor_g8"].with_(name="split2_int2_factor_g8", q_bits=32),
    # bf16 blocks always carry two-part weights and an exact bf16 query
    "bf16": SMALL["bf16"],
    "bf16_g8": SMALL["bf16_g8"],
}


@pytest.mark.parametrize("name", list(SPLIT_TWO_PART))
def test_decode_split_count_does_not_change_result(name):
    """Any split of the token range gives the same attention up to fp32
    rounding (the log-sum-exp merge is exact algebra): splits 1 and N agree
    within 1e-5 in the two-part mode, where the weights carry about 22 bits and
    no operand is rounded to 11 bits relative to a split's running maximum.
    bf16 blocks carry their weights as two bf16 parts (about 17 bits): there
    the bound is 2^-17 * max|v_hat| + 1e-5, still below 1e-4 here."""
    inp = make_inputs(SPLIT_TWO_PART[name])
    w = inp.workload
    run = DeviceRun(inp)
    atol = 1e-5
    if w.v_bits == 16:
        atol += 2.0 ** -17 * float(np.abs(O.bf16_to_f64(inp.v)).max())
    assert atol <= 1e-4
    base, base_lse = run.decode(out_fp32=True, stream_ctas=1)
    for p in (2, 3, 7, 64, 0):
        out, lse = run.decode(out_fp32=True, stream_ctas=p)
        np.testing.assert_allclose(out, base, rtol=0, atol=atol, err_msg=f"{p} splits")
        np.testing.assert_allclose(lse, base_lse, rtol=0, atol=1e-5, err_msg=f"{p} splits")
    assert compare_outputs(inp, base, base_lse, oracle_decode(inp), out_is_bf16=False) <= 1.0
    assert run.err_bits() == 0


def test_two_part_query_removes_the_query_rounding_error():
    """On heavy-tailed keys under per-channel scales (scores near 10) the fp16
    query (q_bits 16) leaves a score error that the log-sum-exp shows directly;
    the fp16 hi + lo query (q_bits 32) cuts it at least fourfold and brings the
    whole comparison inside the tolerance."""
    base = SMALL["kchan_k4v8_window32_g8"]
    lse_err, ratio = {}, {}
    for qb in (16, 32):
        inp = make_inputs(base.with_(name=f"kchan_q{qb}", q_bits=qb))
        run = DeviceRun(inp)
        out, lse = run.decode(out_fp32=True)
        ref = oracle_decode(inp)
        G = inp.workload.group
        lse_err[qb] = max(float(np.abs(lse[b, h * G:(h + 1) * G] - l).max()) for (b, h), (_, l) in ref.items())
        ratio[qb] = compare_outputs(inp, out, lse, ref, out_is_bf16=False)
        assert run.err_bits() == 0
    assert lse_err[32] * 4 <= lse_err[16], lse_err
    assert ratio[32] <= 1.0, ratio


EDGE_FORMATS = {
    "int8": {},
    "asym_k4v8": dict(k_bits=4, v_bits=8, asym=True),
    "qint8": dict(q_bits=8),
    "kchan_int4_q32": dict(k_bits=4, v_bits=4, channel_factor=True, k_per_channel=True, q_bits=32),
    "int2": dict(k_bits=2, v_bits=2),
}


@pytest.mark.parametrize("fmt", list(EDGE_FORMATS))
@pytest.mark.parametrize("window", [0, 32])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_edge_lengths(window, group, fmt):
    lengths = np.array([0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129], dtype=np.int32)
    w = small_workload(f"edge_{window}_{group}_{fmt}", batch=len(lengths), q_heads=2 * group, kv_heads=2,
                       seq_len=1, len_range=None, window=window, **EDGE_FORMATS[fmt])
    inp = make_inputs(w)
    # replace the lengths (and the matching packed K/V rows) by the edge set
    rng = np.random.default_rng(3)
    from synth import f32_to_bf16_bits
    n = int(lengths.sum())
    inp.lengths = lengths
    inp.seq_offsets = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    inp.k = f32_to_bf16_bits(rng.standard_normal((n, 2, 128)).astype(np.float32))
    inp.v = f32_to_bf16_bits(rng.standard_normal((n, 2, 128)).astype(np.float32))
    nblk = np.maximum((lengths + 15) // 16, 1)
    table = np.full((len(lengths), int(nblk.max())), -1, np.int32)
    off = 0
    for b, nb in enumerate(nblk):
        table[b, :nb] = np.arange(off, off + nb)
        off += nb
    inp.block_table = table
    inp.num_blocks = off
    run = DeviceRun(inp)
    for out_fp32 in (True, False):
        out, lse = run.decode(out_fp32=out_fp32)
        ref = oracle_decode(inp)
        assert compare_outputs(inp, out, lse, ref, out_is_bf16=not out_fp32) <= 1.0
        assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert run.err_bits() == 0


STEP_FORMATS = {
    "int4_factor": dict(k_bits=4, v_bits=4, channel_factor=True),
    "asym_int8": dict(k_bits=8, v_bits=8, asym=True),
    "kchan_k4v8": dict(k_bits=4, v_bits=8, channel_factor=True, k_per_channel=True),
}


@pytest.mark.parametrize("fmt", list(STEP_FORMATS))
def test_step_append_equals_bulk_fill(fmt):
    """Token-by-token window steps leave the same bytes as the bulk fill."""
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.cache import cache_for_inputs
    w = small_workload(f"step_vs_bulk_{fmt}", batch=3, len_range=(1, 90), window=32, **STEP_FORMATS[fmt])
    inp = make_inputs(w)
    bulk = DeviceRun(inp)
    step_cache = cache_for_inputs(inp)
    table = bulk.table
    for p in range(int(inp.lengths.max())):
        seqs = np.nonzero(inp.lengths > p)[0]
        rows = inp.seq_offsets[seqs] + p
        kt = torch.from_numpy(inp.k[rows].view(np.int16)).cuda().view(torch.bfloat16)
        vt = torch.from_numpy(inp.v[rows].view(np.int16)).cuda().view(torch.bfloat16)
        si = torch.from_numpy(seqs.astype(np.int32)).cuda()
        po = torch.full((len(seqs),), p, dtype=torch.int32, device="cuda")
        _lib.kvq_append(step_cache.desc, kt, vt, si, po, _lib.APPEND_STEP, table, w.batch, inp.max_blocks)
    torch.cuda.synchronize()
    a = bulk.pools()
    for key in ("k_window", "v_window"):
        np.testing.assert_array_equal(getattr(step_cache, key).view(torch.uint8).cpu().numpy(), a[key])
    # block store: compare every position older than the window
    kc_s = unpack_blocks(step_cache.k_codes.cpu().numpy(), w.k_bits, True, w.kv_heads, w.asym)
    kc_b = unpack_blocks(a["k_codes"], w.k_bits, True, w.kv_heads, w.asym)
    vc_s = unpack_blocks(step_cache.v_codes.cpu().numpy(), w.v_bits, False, w.kv_heads, w.asym)
    vc_b = unpack_blocks(a["v_codes"], w.v_bits, False, w.kv_heads, w.asym)
    md_s = meta_by_block(step_cache.meta.cpu().numpy(), w.kv_heads, w.asym)
    md_b = meta_by_block(a["meta"], w.kv_heads, w.asym)
    for b in range(w.batch):
        for p in range(max(int(inp.lengths[b]) - w.window, 0)):
            ph, t = inp.block_table[b, p // 16], p % 16
            np.testing.assert_array_equal(kc_s[ph, :, t], kc_b[ph, :, t])
            np.testing.assert_array_equal(vc_s[ph, :, t], vc_b[ph, :, t])
            for key in md_b:
                if key == "k_scale" and w.k_per_channel:
                    continue  # not written under per-channel key scales
                np.testing.assert_array_equal(md_s[key][ph, :, t], md_b[key][ph, :, t])


def test_two_bit_blocks_are_written_whole():
    """A 2-bit block shares one scale over its 16 tokens, so kvq_append writes
    it from a run of rows that starts at the block's first position: a lone
    token in the middle of a block is flagged (KVQ_DEVERR_POSITION) and writes
    nothing, a run that starts mid-block likewise, and a decode-step eviction
    into a 2-bit cache is refused on the host."""
    inp = make_inputs(small_workload("int2_whole", batch=2, len_range=(40, 60), k_bits=2, v_bits=2))
    run = DeviceRun(inp)
    assert run.err_bits() == 0
    w = inp.workload
    before = run.pools()["k_codes"].copy()
    kt = torch.from_numpy(inp.k[:3].view(np.int16)).cuda().view(torch.bfloat16)
    vt = torch.from_numpy(inp.v[:3].view(np.int16)).cuda().view(torch.bfloat16)
    for si, po in (([0], [5]), ([1, 1, 1], [17, 18, 19])):
        run.err.zero_()
        n = len(si)
        run.lib.kvq_append(run.cache.desc, kt[:n], vt[:n], torch.tensor(si, dtype=torch.int32, device="cuda"),
                           torch.tensor(po, dtype=torch.int32, device="cuda"), run.lib.APPEND_QUANT, run.table,
                           w.batch, inp.max_blocks, err_word=run.err)
        assert run.err_bits() & run.lib.KVQ_DEVERR_POSITION
    np.testing.assert_array_equal(run.pools()["k_codes"], before)
    with pytest.raises(run.lib.KvqError) as e:
        from quantized_kv_cache_07_gb300.cache import KVCache
        c = KVCache(8, 2, 2, 2, window=32, window_batch=2)
        run.lib.kvq_append(c.desc, kt[:1], vt[:1], torch.zeros(1, dtype=torch.int32, device="cuda"),
                           torch.zeros(1, dtype=torch.int32, device="cuda"), run.lib.APPEND_STEP, run.table, 2,
                           inp.max_blocks)
    assert e.value.status == run.lib.KVQ_ERR_UNSUPPORTED


def test_graph_captured_steps_equal_eager_steps():
    """kvq_append + kvq_decode captured in a CUDA graph (as the benchmark times
    them) and replayed give the eager calls' results bit for bit."""
    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.cache import DecodeWorkspace
    from quantized_kv_cache_07_gb300.cache import cache_for_inputs, fill_from_inputs
    inp = make_inputs(small_workload("graph", batch=4, len_range=(30, 300), paged=True, append_one=True))
    w = inp.workload
    eager = DeviceRun(inp)                    # eager: fill, append the new token, decode
    o_e, l_e = eager.decode(out_fp32=True)
    # the same cache before the append; the append and the decode are captured
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = cache_for_inputs(inp)
    table, _ = fill_from_inputs(cache, inp, err_word=err)
    q = torch.from_numpy(inp.q.view(np.int16)).cuda().view(torch.bfloat16)
    kt = torch.from_numpy(inp.k_new.view(np.int16)).cuda().view(torch.bfloat16)
    vt = torch.from_numpy(inp.v_new.view(np.int16)).cuda().view(torch.bfloat16)
    si = torch.arange(w.batch, dtype=torch.int32, device="cuda")
    po = torch.from_numpy(inp.lengths.astype(np.int32)).cuda()
    dl = torch.from_numpy(inp.decode_lengths.astype(np.int32)).cuda()
    out = torch.zeros((w.batch, w.q_heads, 128), dtype=torch.float32, device="cuda")
    lse = torch.zeros((w.batch, w.q_heads), dtype=torch.float32, device="cuda")
    ws = DecodeWorkspace(cache, w.batch, w.q_heads)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _lib.kvq_append(cache.desc, kt, vt, si, po, _lib.APPEND_QUANT, table, w.batch, inp.max_blocks, err_word=err)
        _lib.kvq_decode(cache.desc, q, w.batch, w.q_heads, dl, table, inp.max_blocks, out, lse=lse,
                        workspace=ws.buf, workspace_bytes=ws.nbytes, err_word=err)
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), o_e)
    np.testing.assert_array_equal(lse.cpu().numpy(), l_e)
    g.replay()                      # a second replay (same appended token, same result)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), o_e)
    assert int(err.item()) == 0 and eager.err_bits() == 0


def test_unit_channel_factor_gives_the_plain_result_bit_for_bit():
    """A per-channel key factor of all ones divides and multiplies by one: the
    stored codes and the decode output equal the run without a factor exactly."""
    w = small_workload("unit_factor", batch=3, q_heads=16, kv_heads=2, k_bits=4, v_bits=8, len_range=(1, 300))
    inp = make_inputs(w)
    plain = DeviceRun(inp)
    inp1 = make_inputs(w.with_(channel_factor=True))
    inp1.channel_factor = np.ones_like(inp1.channel_factor)
    unit = DeviceRun(inp1)
    torch.cuda.synchronize()
    assert np.array_equal(plain.pools()["k_codes"], unit.pools()["k_codes"])
    o0, l0 = plain.decode(out_fp32=True)
    o1, l1 = unit.decode(out_fp32=True)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


def test_device_errors_are_flagged_not_trapped():
    inp = make_inputs(small_workload("errs", batch=2, len_range=(40, 80)))
    run = DeviceRun(inp)
    bad = run.table.clone()
    bad[1, 1] = inp.num_blocks + 5                 # block id out of range
    from quantized_kv_cache_07_gb300.cache import DecodeWorkspace
    w = inp.workload
    out = torch.zeros((w.batch, w.q_heads, 128), dtype=torch.float32, device="cuda")
    ws = DecodeWorkspace(run.cache, w.batch, w.q_heads)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run.lib.kvq_decode(run.cache.desc, run.q, w.batch, w.q_heads, run.lens, bad, inp.max_blocks, out,
                       workspace=ws.buf, workspace_bytes=ws.nbytes, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & run.lib.KVQ_DEVERR_BLOCK_ID
    # a length beyond the table's capacity is clamped and flagged
    err.zero_()
    long = run.lens.clone()
    long[0] = inp.max_blocks * 16 + 100
    run.lib.kvq_decode(run.cache.desc, run.q, w.batch, w.q_heads, long, run.table, inp.max_blocks, out,
                       workspace=ws.buf, workspace_bytes=ws.nbytes, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & run.lib.KVQ_DEVERR_SEQ_LEN
    # the workspace counters are back at zero: a normal call still matches the oracle
    o2, l2 = run.decode(out_fp32=True)
    assert compare_outputs(inp, o2, l2, oracle_decode(inp), out_is_bf16=False) <= 1.0


@pytest.mark.parametrize("name", ["int8_g4", "window32_int8", "int4_factor_g8", "asym_int4_factor_g8", "int2_g4",
                                  "bf16", "q32_int2_g1"])
def test_geometry_ready_flag_gives_identical_results(runs, name):
    """kvq_decode_ex with KVQ_DECODE_GEOMETRY_READY scans the lengths before
    the dependency wait; the arithmetic is unchanged, so outputs and lse are
    bit-identical to kvq_decode."""
    inp, run = runs(name)
    from quantized_kv_cache_07_gb300 import _lib
    for p in (0, 5):
        o0, l0 = run.decode(out_fp32=True, stream_ctas=p)
        o1, l1 = run.decode(out_fp32=True, stream_ctas=p, flags=_lib.DECODE_GEOMETRY_READY)
        np.testing.assert_array_equal(o0, o1)
        np.testing.assert_array_equal(l0, l1)
    assert run.err_bits() == 0


def test_geometry_ready_flag_reports_device_errors():
    """Lengths beyond the table's capacity (found before the dependency wait)
    and out-of-range table entries are flagged as without the flag, with the
    same outputs."""
    from quantized_kv_cache_07_gb300 import _lib
    inp = make_inputs(small_workload("ready_errs", batch=3, len_range=(40, 300)))
    run = DeviceRun(inp)
    bad = run.table.clone()
    bad[0, 0] = inp.num_blocks + 3                 # the first entry a producer reads
    bad[2, 1] = -1
    long = run.lens.clone()
    long[1] = inp.max_blocks * 16 + 50
    res = []
    for flags in (0, _lib.DECODE_GEOMETRY_READY):
        run.err.zero_()
        o, l = run.decode(out_fp32=True, lens=long, flags=flags, table=bad)
        res.append((o, l, run.err_bits()))
    assert res[0][2] == res[1][2] == (_lib.KVQ_DEVERR_BLOCK_ID | _lib.KVQ_DEVERR_SEQ_LEN)
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])


def test_workspace_counters_return_to_zero():
    """The merge counters at the head of the workspace are zero after every
    completed call: normal calls at several split counts, and a call whose
    block table holds an out-of-range entry (injected on the host; the kernel
    flags it and reads block 0 instead)."""
    from quantized_kv_cache_07_gb300.cache import DecodeWorkspace
    inp = make_inputs(small_workload("counters", batch=6, len_range=(40, 400), window=32))
    run = DeviceRun(inp)
    w = inp.workload
    units = w.batch * w.kv_heads
    out = torch.zeros((w.batch, w.q_heads, 128), dtype=torch.float32, device="cuda")
    bad = run.table.clone()
    bad[2, 1] = inp.num_blocks + 7
    for p in (0, 3, 7, 40):
        ws = DecodeWorkspace(run.cache, w.batch, w.q_heads, p)
        for table, expect in ((run.table, 0), (bad, run.lib.KVQ_DEVERR_BLOCK_ID), (run.table, 0)):
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            run.lib.kvq_decode(run.cache.desc, run.q, w.batch, w.q_heads, run.lens, table, inp.max_blocks, out,
                               workspace=ws.buf, workspace_bytes=ws.nbytes, stream_ctas=p, err_word=err)
            torch.cuda.synchronize()
            assert int(err.item()) == expect
            counters = ws.buf[: 4 * units].view(torch.int32).cpu().numpy()
            assert np.all(counters == 0), (p, counters)
        # the last call (good table) still matches the oracle
        assert compare_outputs(inp, out.cpu().numpy(), None, oracle_decode(inp), out_is_bf16=False) <= 1.0


@pytest.mark.parametrize("exp2", [18, -20])
def test_value_scales_far_from_one_decode_correctly(exp2):
    """Scaling the values by 2^18 (value scales near 10^4, far beyond what
    fp16 weights p * s_v could hold at a fixed offset) or by 2^-20 (weights
    that would fall into fp16 subnormals) scales the exact output by the same
    power of two; the kernel's weight offset follows the value scales, so the
    decode matches the oracle after undoing the factor, with nothing flagged."""
    from synth import f32_to_bf16_bits
    inp = make_inputs(small_workload(f"vscale_{exp2}", batch=3, len_range=(40, 300), k_bits=4, v_bits=8))
    ref = oracle_decode(inp)
    big = (O.bf16_to_f64(inp.v) * 2.0 ** exp2).astype(np.float32)     # exact: a power of two
    inp.v = f32_to_bf16_bits(big)
    run = DeviceRun(inp)
    out, lse = run.decode(out_fp32=True)
    assert compare_outputs(inp, out * 2.0 ** -exp2, lse, ref, out_is_bf16=False) <= 1.0
    assert run.err_bits() == 0


@pytest.mark.parametrize("q_bits", [16, 8])
@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("bias", [4.0, 16.0])
def test_biased_queries_on_int8_keys(bias, asym, q_bits):
    """Queries with a large common component (every dimension shifted by
    `bias`) against int8 keys of a few thousand tokens: the int8 key codes enter
    the score product with their offset of 1152, and each block's accumulators
    start at minus 1152 times the query's sums, which are largest relative to
    the code dot for such queries.  The bf16 query is exact in the kernel's fp16
    staging here (no per-channel factor), so the comparison sees the offset's
    fp32 rounding; int8 query codes keep every partial sum an exact integer."""
    from synth import f32_to_bf16_bits
    w = small_workload(f"qbias_{bias}_{int(asym)}_{q_bits}", batch=2, len_range=(1500, 3000), asym=asym,
                       q_bits=q_bits)
    inp = make_inputs(w)
    inp.q = f32_to_bf16_bits((O.bf16_to_f64(inp.q) + bias).astype(np.float32))
    ref = oracle_decode(inp)
    run = DeviceRun(inp)
    out, lse = run.decode(out_fp32=True)
    assert compare_outputs(inp, out, lse, ref, out_is_bf16=False) <= 1.0
    assert run.err_bits() == 0


def test_append_out_of_range_positions_are_flagged_and_skipped():
    """A sequence index outside the batch or a position beyond the block
    table's capacity sets KVQ_DEVERR_POSITION and writes nothing."""
    inp = make_inputs(small_workload("pos", batch=2, len_range=(20, 40)))
    run = DeviceRun(inp)
    w = inp.workload
    before = {k: v.copy() for k, v in run.pools().items() if v is not None}
    kt = torch.from_numpy(inp.k[:2].view(np.int16)).cuda().view(torch.bfloat16)
    vt = torch.from_numpy(inp.v[:2].view(np.int16)).cuda().view(torch.bfloat16)
    for si, po in (([w.batch, 0], [5, 5]), ([0, 1], [inp.max_blocks * 16, inp.max_blocks * 16 + 3])):
        run.err.zero_()
        run.lib.kvq_append(run.cache.desc, kt, vt, torch.tensor(si, dtype=torch.int32, device="cuda"),
                           torch.tensor(po, dtype=torch.int32, device="cuda"), run.lib.APPEND_QUANT, run.table,
                           w.batch, inp.max_blocks, err_word=run.err)
        assert run.err_bits() & run.lib.KVQ_DEVERR_POSITION
    after = run.pools()
    # the second call wrote nothing; the first wrote only sequence 0 (row 1): check sequence 1's blocks
    for key in ("k_codes", "v_codes"):
        assert after[key].shape == before[key].shape
    kc_b = unpack_blocks(before["k_codes"], w.k_bits, True, w.kv_heads)
    kc_a = unpack_blocks(after["k_codes"], w.k_bits, True, w.kv_heads)
    ph1 = inp.block_table[1, : (int(inp.lengths[1]) + 15) // 16]
    np.testing.assert_array_equal(kc_a[ph1], kc_b[ph1])


def test_host_validation_errors():
    inp = make_inputs(small_workload("val", batch=1, len_range=(10, 10)))
    run = DeviceRun(inp)
    lib = run.lib
    w = inp.workload
    out = torch.zeros((1, w.q_heads, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.KvqError) as e:
        lib.kvq_decode(run.cache.desc, run.q, 1, w.q_heads, run.lens, run.table, inp.max_blocks, out,
                       workspace=None, workspace_bytes=0)
    assert e.value.status == lib.KVQ_ERR_WORKSPACE
    with pytest.raises(lib.KvqError) as e:
        lib.kvq_decode(run.cache.desc, run.q, 1, 3, run.lens, run.table, inp.max_blocks, out)
    assert e.value.status == lib.KVQ_ERR_INVALID_ARG


# ---------------------------------------------------------------- full-size named workloads
def _sample_units(w, k, seed=11):
    rng = np.random.default_rng(seed)
    units = {(int(b), int(h)) for b, h in zip(rng.integers(0, w.batch, k), rng.integers(0, w.kv_heads, k))}
    units.add((w.batch - 1, w.kv_heads - 1))
    return units


FULL = dict(WORKLOADS)
# the asymmetric format on two of the named shapes
FULL["asym_gqa_int8_window128_b8_t4096"] = WORKLOADS["gqa_int8_window128_b8_t4096"].with_(
    name="asym_gqa_int8_window128_b8_t4096", asym=True)
FULL["asym_long_k4v8_b4_t131072"] = WORKLOADS["long_k4v8_b4_t131072"].with_(name="asym_long_k4v8_b4_t131072",
                                                                          asym=True)
# the quantized-query mode on the int4 / per-channel factor shape
FULL["qint8_int4_factor_b32_len1k_8k"] = WORKLOADS["int4_factor_b32_len1k_8k"].with_(
    name="qint8_int4_factor_b32_len1k_8k", q_bits=8)
# per-channel key scales only on the int4 / factor shape
FULL["kchan_int4_factor_b32_len1k_8k"] = WORKLOADS["int4_factor_b32_len1k_8k"].with_(
    name="kchan_int4_factor_b32_len1k_8k", k_per_channel=True)
# 2-bit codes with token-group scales on the int4 / factor shape (symmetric and asymmetric)
FULL["int2_factor_b32_len1k_8k"] = WORKLOADS["int4_factor_b32_len1k_8k"].with_(
    name="int2_factor_b32_len1k_8k", k_bits=2, v_bits=2)
FULL["asym_int2_factor_b32_len1k_8k"] = WORKLOADS["int4_factor_b32_len1k_8k"].with_(
    name="asym_int2_factor_b32_len1k_8k", k_bits=2, v_bits=2, asym=True)
# the asymmetric format on the paged append-then-decode shape
FULL["asym_paged_int8_b64_len2k_32k"] = WORKLOADS["paged_int8_b64_len2k_32k"].with_(
    name="asym_paged_int8_b64_len2k_32k", asym=True)


def _full_size_units(name, w):
    """Every (sequence, kv_head) unit of the five named workloads up to 256
    units (all of c1, c2, c3 and c5), 64 sampled units beyond that (c4), 16 for
    the format variants on the same shapes."""
    n = w.batch * w.kv_heads
    if name in WORKLOADS and n <= 256:
        return {(b, h) for b in range(w.batch) for h in range(w.kv_heads)}
    k = 64 if name in WORKLOADS else 16
    units = set()
    seed = 11
    while len(units) < min(k, n):
        units |= _sample_units(w, k - len(units), seed)
        seed += 1
    return units


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workload(name):
    w = FULL[name]
    inp = make_inputs(w)
    run = DeviceRun(inp)
    units = _full_size_units(name, w)
    every_position = w.batch * w.kv_heads <= 256 and name in WORKLOADS and w.batch <= 32
    states = {b: oracle_state(inp, b) for b in sorted({b for b, _ in units})}
    assert check_stored_cache(inp, run, units=units, max_positions=None if every_position else 8192,
                              states=states) > 0
    ref = oracle_decode(inp, units, states=states)
    del states
    # fp32 outputs: the plain 2e-3 bound; bf16 outputs: 2e-3 + half a bf16 ulp
    for out_fp32 in (True, False):
        out, lse = run.decode(out_fp32=out_fp32)
        worst = compare_outputs(inp, out, lse, ref, out_is_bf16=not out_fp32)
        assert worst <= 1.0, f"max error ratio {worst:.3f} (out_fp32={out_fp32})"
        # properties that hold for every unit: finite outputs and lse
        assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    assert run.err_bits() == 0


# ---------------------------------------------------------------- seeded random configurations
def _random_workload(i):
    """A valid small workload drawn from the whole option space (seeded)."""
    rng = np.random.default_rng(1000 + i)
    kb, vb = [(8, 8), (4, 4), (4, 8), (8, 4), (2, 2), (16, 16)][int(rng.integers(6))]
    quant = kb != 16
    G = int(rng.choice([1, 2, 4, 8]))
    H = int(rng.integers(1, 4))
    kw = dict(batch=int(rng.integers(1, 5)), q_heads=G * H, kv_heads=H, k_bits=kb, v_bits=vb,
              len_range=(1, int(rng.integers(20, 400))), paged=bool(rng.integers(2)),
              k_dist=str(rng.choice(["normal", "t3"])), outlier_channels=int(rng.choice([0, 4])))
    if quant:
        kw["asym"] = bool(rng.integers(2))
        kw["channel_factor"] = bool(rng.integers(2))
        if kw["channel_factor"] and not kw["asym"] and kb != 2 and rng.integers(3) == 0:
            kw["k_per_channel"] = True
        kw["q_bits"] = int(rng.choice([16, 32, 8]))
    kw["window"] = int(rng.choice([0, 16, 48]))
    if kw.get("q_bits") == 8 and kw.get("channel_factor") and kw["window"]:
        kw["q_bits"] = 16                    # int8 query rows, a factor and a window: refused by the library
    if kw.get("q_bits") == 16 and kw.get("channel_factor") and (
            kw["outlier_channels"] or (kw.get("k_per_channel") and kw["k_dist"] == "t3")):
        # outlier channels, or heavy tails under per-channel scales, put large
        # factors on the query: its 11-bit fp16 form alone moves the
        # log-sum-exp past 2e-3 (2.7e-3 in a float64 emulation of case 14), so
        # these caches take the two-part mode
        kw["q_bits"] = 32
    kw["append_one"] = kb != 2 and not kw["window"] and bool(rng.integers(2))
    return small_workload(f"random_{i}", **kw)


@pytest.mark.parametrize("i", range(24))
def test_random_configuration_matches_the_oracle(i):
    w = _random_workload(i)
    inp = make_inputs(w)
    run = DeviceRun(inp)
    check_stored_cache(inp, run)                 # codes, scales, zero points and ring: bit for bit
    out, lse = run.decode(out_fp32=True)
    worst = compare_outputs(inp, out, lse, oracle_decode(inp), out_is_bf16=False)
    assert worst <= 1.0, f"{w}: max error ratio {worst:.3f}"
    assert run.err_bits() == 0
