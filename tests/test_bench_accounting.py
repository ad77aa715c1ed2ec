"""The bench's algorithmic bytes per step agree with the oracle's byte
accounting (which is pinned to the metadata fractions and the cache-size
formula the pages print), for every named workload and format variant."""
import numpy as np
import pytest

import bench
from oracle import kvq_oracle as O
from synth import WORKLOADS, make_inputs

VARIANTS = [dict(), dict(asym=True), dict(k_bits=16, v_bits=16, window=0, channel_factor=False),
            dict(k_bits=2, v_bits=2), dict(k_bits=2, v_bits=2, asym=True)]


def expected_bytes(inp) -> int:
    w = inp.workload
    per_q = O.cache_bytes_per_token_head(w.head_dim, w.k_bits, w.v_bits, asym=w.asym,
                                         k_per_channel=w.k_per_channel)
    total = 0
    for L in inp.decode_lengths.astype(int):
        lq = O.window_split(int(L), w.window)
        if w.k_bits == 2:
            # codes per token, plus the 16-byte record of each started 16-token group
            per_code = per_q - 16 / O.GROUP_TOKENS
            total += int(per_code * lq) + 16 * -(-lq // O.GROUP_TOKENS) + 2 * w.head_dim * 2 * (int(L) - lq)
            continue
        total += per_q * lq + 2 * w.head_dim * 2 * (int(L) - lq)      # bf16 window tokens: K and V
    return w.kv_heads * total


@pytest.mark.parametrize("name", ["int8_b1_h4_t256", "gqa_int8_window128_b8_t4096"])
@pytest.mark.parametrize("variant", range(len(VARIANTS)))
def test_bench_bytes_match_oracle_accounting(name, variant):
    w = WORKLOADS[name].with_(**VARIANTS[variant])
    inp = make_inputs(w)
    assert bench.cache_bytes_per_step(inp) == expected_bytes(inp)


def test_bench_bytes_per_channel_keys_drop_the_key_scales():
    w = WORKLOADS["int4_factor_b32_len1k_8k"].with_(k_per_channel=True)
    inp = make_inputs(w)
    base = make_inputs(WORKLOADS["int4_factor_b32_len1k_8k"])
    tokens = int(np.sum(inp.decode_lengths)) * w.kv_heads
    assert bench.cache_bytes_per_step(base) - bench.cache_bytes_per_step(inp) == 4 * tokens
    assert bench.cache_bytes_per_step(inp) == expected_bytes(inp)


@pytest.mark.parametrize("bits", [(8, 8), (4, 4), (4, 8)])
def test_token_head_bytes_match_oracle_accounting(bits):
    assert bench.token_head_bytes(*bits) == O.cache_bytes_per_token_head(128, *bits)


def test_prefill_row_bytes_count_every_row_prefix():
    """Each row at position p reads positions 0..p of its sequence: brute force
    over the rows of a small chunked-prefill call."""
    prefix, chunk, batch, heads, per = 37, 5, 3, 2, 264
    rows = [(b, p) for b in range(batch) for p in range(prefix, prefix + chunk)]
    total = sum(len(range(0, p + 1)) * per * heads for _, p in rows)
    assert bench.prefill_row_bytes(prefix, chunk, batch, heads, per) == total
