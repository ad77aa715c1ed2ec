"""Seeded synthetic workloads (input generation only, no method arithmetic).

The five named workloads mirror the decode configurations the method is
measured on: head dimension 128, 16-token cache blocks, int8 / int4 / bf16
cache formats, an optional 128-token bf16 recent-token window, an optional
per-channel key factor and an optional paged (randomly permuted) block table.

Draw order is fixed so every consumer sees the same bits for a given seed:
lengths -> block permutation -> outlier channel ids -> q -> K -> V -> new K/V.
Floats are drawn in float32, outlier channels are multiplied by their factor
in float32, then every value is rounded to bf16 (round to nearest even) and
carried as raw uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128
BLOCK_SIZE = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits.

    Inputs are finite by construction (no NaN handling is needed here).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """Shape and structure of one decode workload."""
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    k_bits: int                      # 4, 8 or 16 (16 = plain bf16 cache)
    v_bits: int
    seq_len: int | None = None       # fixed cached length, or None for a range
    len_range: tuple[int, int] | None = None   # inclusive uniform integer range
    window: int = 0                  # bf16 recent-token window (tokens), 0 = none
    channel_factor: bool = False     # per-channel key factor folded onto the query
    paged: bool = False              # random permutation block table
    append_one: bool = False         # one step = append 1 token/seq, then decode
    k_dist: str = "normal"           # "normal" or "t3" (Student-t, nu = 3)
    outlier_channels: int = 0        # number of key channels scaled by outlier_mult
    outlier_mult: float = 10.0
    asym: bool = False               # asymmetric format: per-token scale and zero point
    q_bits: int = 16                 # 8: int8-quantized query rows (integer dot)
    k_per_channel: bool = False      # keys carry per-channel scales only (needs channel_factor)
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    seed: int = 0
    description: str = ""

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("int8_b1_h4_t256", batch=1, q_heads=4, kv_heads=4, k_bits=8, v_bits=8, seq_len=256,
                 description="single-layer int8 decode, batch 1, 4 q heads = 4 KV heads, T=256"),
        Workload("gqa_int8_window128_b8_t4096", batch=8, q_heads=32, kv_heads=8, k_bits=8, v_bits=8,
                 seq_len=4096, window=128, outlier_channels=4,
                 description="GQA int8 decode, batch 8, 32/8 heads, T=4096, 4 outlier key channels x10, "
                             "most recent 128 tokens kept bf16"),
        Workload("int4_factor_b32_len1k_8k", batch=32, q_heads=32, kv_heads=8, k_bits=4, v_bits=4,
                 len_range=(1024, 8192), channel_factor=True,
                 description="packed int4 K and V, batch 32, 32/8 heads, lengths U[1024,8192], "
                             "per-channel key factor folded onto q"),
        Workload("paged_int8_b64_len2k_32k", batch=64, q_heads=32, kv_heads=8, k_bits=8, v_bits=8,
                 len_range=(2048, 32768), paged=True, append_one=True,
                 description="paged int8 serving step, batch 64, 32/8 heads, lengths U[2048,32768], "
                             "16-token blocks in a random permutation, append 1 token/seq then decode"),
        Workload("long_k4v8_b4_t131072", batch=4, q_heads=64, kv_heads=8, k_bits=4, v_bits=8,
                 seq_len=131072, k_dist="t3",
                 description="long-context split-KV, batch 4, 64/8 heads, T=131072, K int4 (Student-t nu=3), "
                             "V int8"),
    ]
}


@dataclass
class Inputs:
    """All bits of one workload, generated once from the seed."""
    workload: Workload
    lengths: np.ndarray            # int32 [B]: cached tokens before the step
    seq_offsets: np.ndarray        # int64 [B+1]: row offsets of each sequence in k/v
    q: np.ndarray                  # uint16 [B, H_q, D] bf16 bits
    k: np.ndarray                  # uint16 [sum L, H_kv, D] bf16 bits (token-major, packed by seq)
    v: np.ndarray                  # uint16 [sum L, H_kv, D]
    k_new: np.ndarray | None       # uint16 [B, H_kv, D] (append_one workloads)
    v_new: np.ndarray | None
    block_table: np.ndarray        # int32 [B, max_blocks]; -1 marks unused entries
    num_blocks: int
    channel_factor: np.ndarray | None = None   # float32 [H_kv, D]
    outlier_ids: np.ndarray | None = None
    extra: dict = field(default_factory=dict)

    @property
    def decode_lengths(self) -> np.ndarray:
        """Lengths the decode step attends to (after the optional append)."""
        return self.lengths + (1 if self.workload.append_one else 0)

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _draw_f32(rng: np.random.Generator, n: int, dist: str, chunk: int = 1 << 25) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        if dist == "normal":
            out[s:e] = rng.standard_normal(e - s, dtype=np.float32)
        elif dist == "t3":
            out[s:e] = rng.standard_t(3.0, e - s).astype(np.float32)
        else:
            raise ValueError(dist)
    return out


def _bf16_tokens(rng, n_tok, h_kv, d, dist, outliers=None, mult=1.0) -> np.ndarray:
    x = _draw_f32(rng, n_tok * h_kv * d, dist).reshape(n_tok, h_kv, d)
    if outliers is not None and len(outliers):
        x[..., outliers] *= np.float32(mult)
    return f32_to_bf16_bits(x)


def make_inputs(w: Workload, seed: int | None = None) -> Inputs:
    """Generate every input of workload ``w`` from one seeded generator."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    B, D, bs = w.batch, w.head_dim, w.block_size
    # 1. lengths
    if w.seq_len is not None:
        lengths = np.full(B, w.seq_len, dtype=np.int32)
    else:
        lo, hi = w.len_range
        lengths = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    cap = lengths.astype(np.int64) + (1 if w.append_one else 0)
    nblk = (cap + bs - 1) // bs
    max_blocks = int(nblk.max()) if B else 0
    # 2. block placement
    total_blocks = int(nblk.sum())
    if w.paged:
        perm = rng.permutation(total_blocks).astype(np.int32)
    else:
        perm = np.arange(total_blocks, dtype=np.int32)
    table = np.full((B, max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, : nblk[b]] = perm[off: off + nblk[b]]
        off += int(nblk[b])
    # 3. outlier channels
    outliers = None
    if w.outlier_channels:
        outliers = np.sort(rng.choice(D, w.outlier_channels, replace=False))
    # 4. q, K, V, new tokens
    q = f32_to_bf16_bits(rng.standard_normal((B, w.q_heads, D), dtype=np.float32))
    seq_off = np.zeros(B + 1, dtype=np.int64)
    seq_off[1:] = np.cumsum(lengths.astype(np.int64))
    n_tok = int(seq_off[-1])
    k = _bf16_tokens(rng, n_tok, w.kv_heads, D, w.k_dist, outliers, w.outlier_mult)
    v = _bf16_tokens(rng, n_tok, w.kv_heads, D, "normal")
    k_new = v_new = None
    if w.append_one:
        k_new = _bf16_tokens(rng, B, w.kv_heads, D, w.k_dist, outliers, w.outlier_mult)
        v_new = _bf16_tokens(rng, B, w.kv_heads, D, "normal")
    # per-channel key factor: the per-channel absmax of the seeded keys (0 -> 1).
    # With per-channel key scales only, the caller's calibration is the
    # per-channel absmax of the first half of the cached tokens divided by the
    # code range (127 or 7): later tokens can fall outside it.
    factor = None
    if w.channel_factor and w.k_per_channel:
        kf = bf16_bits_to_f32(k[: max(n_tok // 2, 1)]) if n_tok else np.ones((1, w.kv_heads, D), np.float32)
        qmax = np.float32(127.0 if w.k_bits == 8 else 7.0)
        factor = (np.abs(kf).max(axis=0) / qmax).astype(np.float32)
        factor[factor == 0] = 1.0
        del kf
    elif w.channel_factor:
        kf = bf16_bits_to_f32(k)
        factor = np.abs(kf).max(axis=0).astype(np.float32) if n_tok else np.ones((w.kv_heads, D), np.float32)
        if k_new is not None:
            factor = np.maximum(factor, np.abs(bf16_bits_to_f32(k_new)).max(axis=0))
        factor[factor == 0] = 1.0
        del kf
    return Inputs(workload=w, lengths=lengths, seq_offsets=seq_off, q=q, k=k, v=v, k_new=k_new,
                  v_new=v_new, block_table=table, num_blocks=max(total_blocks, 1),
                  channel_factor=factor, outlier_ids=outliers)


def query_rows(n: int, q_heads: int, seed: int) -> np.ndarray:
    """Seeded query rows for a prefill chunk: N(0, 1) in float32 rounded to
    bf16, uint16 bits [n, q_heads, 128]."""
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((n, q_heads, HEAD_DIM), dtype=np.float32))


def shard_units(num_units: int, rank: int, world: int) -> range:
    """Contiguous share of ``num_units`` independent work units for one rank."""
    per, rem = divmod(num_units, world)
    start = rank * per + min(rank, rem)
    return range(start, start + per + (1 if rank < rem else 0))
