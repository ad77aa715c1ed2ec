"""Test-side reader of the cache layouts, written from the layout text in
include/kvq.h (independent of the CUDA sources): maps a stored block back to
logical codes [token, dim] so stored codes can be compared with the oracle."""
import numpy as np

BLOCK = 16
D = 128


def block_bytes(bits: int) -> int:
    return BLOCK * D * bits // 8


def key_offsets(bits: int):
    i = np.arange(BLOCK)[:, None]
    d = np.arange(D)[None, :]
    g, hi, t, e = i & 7, i >> 3, d >> 5, d & 31
    lane = 4 * g + t
    if bits == 8:
        return (2 * hi + (e >> 4)) * 512 + lane * 16 + (e & 15), np.zeros((BLOCK, D), int)
    if bits == 2:
        bit = 16 * (e & 1) + 8 * ((e >> 2) & 1) + 2 * (hi + 2 * ((e & 3) >> 1))
        return lane * 16 + (e >> 3) * 4 + bit // 8, bit % 8
    if bits == 4:
        nib = ((e & 7) >> 1) + 4 * (e & 1)
        return hi * 512 + lane * 16 + (e >> 3) * 4 + nib // 2, (nib & 1) * 4
    return (4 * hi + (e >> 3)) * 512 + lane * 16 + 2 * (e & 7), np.zeros((BLOCK, D), int)


def value_offsets(bits: int):
    i = np.arange(BLOCK)[:, None]
    d = np.arange(D)[None, :]
    mt, r = d >> 4, d & 15
    g, hi = r & 7, r >> 3
    t, j = (i & 7) >> 1, 2 * (i & 1) + (i >> 3)
    lane = 4 * g + t
    if bits == 8:
        return (mt >> 1) * 512 + lane * 16 + (2 * (mt & 1) + hi) * 4 + j, np.zeros((BLOCK, D), int)
    if bits == 2:
        bit = 16 * (j & 1) + 8 * (mt & 1) + 2 * (hi + 2 * (j >> 1))
        return lane * 16 + (mt >> 1) * 4 + bit // 8, bit % 8
    if bits == 4:
        nib = 2 * hi + (j >> 1) + 4 * (j & 1)
        return (mt >> 2) * 512 + lane * 16 + (mt & 3) * 4 + nib // 2, (nib & 1) * 4
    return mt * 512 + lane * 16 + (2 * hi + (j >> 1)) * 4 + 2 * (j & 1), np.zeros((BLOCK, D), int)


def unpack_blocks(pool: np.ndarray, bits: int, is_key: bool, heads: int, asym: bool = False) -> np.ndarray:
    """pool: uint8 [heads * num_blocks * block_bytes] (head-major) -> int32 codes
    [num_blocks, heads, 16, 128], or uint16 bf16 bits for bits == 16.  Symmetric
    codes are stored offset-binary (byte = code + 128, nibble = code + 8);
    asymmetric codes are the stored byte / nibble itself."""
    bb = block_bytes(bits)
    blocks = pool.reshape(heads, -1, bb).transpose(1, 0, 2)
    off, sh = (key_offsets if is_key else value_offsets)(bits)
    if bits == 16:
        lo = blocks[..., off].astype(np.uint16)
        hi = blocks[..., off + 1].astype(np.uint16)
        return lo | (hi << 8)
    raw = blocks[..., off].astype(np.int32)
    if bits == 8:
        return raw if asym else raw - 128
    if bits == 2:
        return ((raw >> sh) & 0x3) - (0 if asym else 2)
    return ((raw >> sh) & 0xF) - (0 if asym else 8)


def offsets_are_a_permutation(bits: int, is_key: bool) -> bool:
    off, sh = (key_offsets if is_key else value_offsets)(bits)
    if bits == 16:
        cells = np.concatenate([off.ravel(), off.ravel() + 1])
        return np.array_equal(np.sort(cells), np.arange(block_bytes(16)))
    per_byte = {2: 4, 4: 2}.get(bits, 1)
    cells = (off * per_byte + sh // (8 // per_byte)).ravel()
    n = block_bytes(bits) * per_byte
    return np.array_equal(np.sort(cells), np.arange(n))


def meta_by_block(pool: np.ndarray, heads: int, asym: bool = False, group: bool = False) -> dict:
    """Metadata pool float [heads * num_blocks * M] (head-major, M = 32, or 64
    asymmetric) -> {"k_scale", "v_scale"(, "k_offset", "v_offset")} each
    [num_blocks, heads, 16]: per block K scales, (K zero points,) V scales,
    (V zero points).  group (2-bit blocks, M = 4): one record (K scale, K zero
    point, V scale, V zero point) per block, repeated for its 16 tokens."""
    if group:
        rec = pool.reshape(heads, -1, 4).transpose(1, 0, 2)
        out = {name: np.repeat(rec[:, :, i:i + 1], BLOCK, axis=2)
               for i, name in enumerate(("k_scale", "k_offset", "v_scale", "v_offset"))}
        return out if asym else {"k_scale": out["k_scale"], "v_scale": out["v_scale"]}
    parts = ("k_scale", "k_offset", "v_scale", "v_offset") if asym else ("k_scale", "v_scale")
    rec = pool.reshape(heads, -1, len(parts), BLOCK).transpose(1, 0, 2, 3)
    return {name: rec[:, :, i] for i, name in enumerate(parts)}
