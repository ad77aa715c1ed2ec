"""Float64 CPU oracle for quantized-KV decode attention.

TEST INFRASTRUCTURE ONLY. This module is the slow, plainly written definition
the CUDA path is checked against. Only the test suite, the package smoke check
and the benchmark's CPU-baseline / reference leg may import it; the product
path never calls it and shares no code with it.

Sources (page title, then section):
  [P1] "KV Cache Quantization Perturbs Attention Through Stored Keys and Values"
  [P2] "KV Cache Quantization Reduces Cache Bytes with Separate Accuracy and Kernel Costs"
  [P3] "KV Cache Quantization and Per-Token Scale Placement"

Every step follows the plain definition; nothing is fused, blocked or
reordered beyond what the cited passage states. In particular the oracle does
NOT fold the per-token key scale after the dot product, does not move the
per-channel key factor onto the query and does not split the sequence: those
are the GPU's rewrites and are checked separately as identities.

Readings taken where the pages leave a step open:
  * rounding is round-half-to-even of the exact quotient x/s (the [P3] listing
    uses Python's round, which is half-to-even);
  * the scale is stored as float32, s = RN32(amax/qmax), and codes are computed
    from that stored scale;
  * an all-zero vector stores codes 0 with scale 1.0 ([P3] listing);
  * int8 codes clamp to [-127, 127] ([P3] listing clamps to +-qmax); int4 codes
    clamp to [-8, 7] (qmax = 7); neither bound below -qmax is reachable;
  * with a per-channel key factor c, keys are first divided by c (rounded to
    float32) and then quantized per token; the reconstruction is c * code * s;
  * with a recent-token window of W tokens, the last min(W, L) positions are
    kept as their bf16 values and only older positions are quantized;
  * the log-sum-exp is in natural-log units of the score q.k/sqrt(D).
  * asymmetric format (scale and zero point, [P1] "Quantization granularity
    defines which values share a scale": a scale and, depending on the scheme,
    a zero point or another offset convention; [P3] "Per-token scales and
    where they can live": "a scale and zero point add 6 percent"): per token
    per head the offset is the vector minimum m, s = RN32((max - min) / qmaxu)
    with qmaxu = 2^bits - 1, u = clamp(rint((x - m) / s), 0, qmaxu) with the
    difference and the quotient evaluated in float64, x_hat = u * s + m; a
    constant vector stores s = 1, u = 0 and m = its value.
  * per-channel key scales only ([P3] "The axis choice is a kernel decision":
    schemes with per-channel key scales move them onto the query; read here as
    the variant where the keys carry no per-token scale at all): code_j =
    clamp(rint(k_j / c_j)) with c_j the caller's per-channel scale (the clamp
    binds for values outside the calibrated range), k_hat_j = c_j * code_j; the
    decode multiplies the query by c once.  The default per-channel factor
    reading divides by c and then quantizes per token (quantize_keys).
  * quantized query ([P3] "Precision floors and mixed cache formats": an 8-bit
    query meets the integer key codes, the dot product accumulates in integers
    and is converted to floating point before the exponential): the query row,
    after the per-channel key factor is moved onto it, is quantized by the same
    symmetric int8 rule as the cache, s_q = RN32(max|x| / 127), q_int =
    clamp(rint(x / s_q)); the folded row q * c is formed in float32, the
    kernel's precision, because it decides integer codes.  The score is
    s_q * s_k * (q_int . k_int) / sqrt(D); against bf16 window keys the query
    is q_int * s_q / c (q_int * s_q without a factor).
  * 2-bit codes with token-group scales ([P3] "Per-token scales and where they
    can live": at 2 bits a 4-byte per-token scale is 12 percent of the entry,
    which is why 2-bit schemes group several tokens under one scale): the
    symmetric rule with qmax = 2^(2-1) - 1 = 1 (codes in [-2, 1], -2 never
    produced), applied to a group of up to 16 consecutive positions of one
    head -- one 16-token cache block -- as if the group were one vector: one
    scale from the absolute maximum over all its values.  The asymmetric rule
    (u in [0, 3]) applies to the same groups when the cache is asymmetric.  The
    last group of a sequence may be partial: it is quantized over the
    positions it holds.
Every function below is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

QMAX = {8: 127, 4: 7, 2: 1}
CLAMP = {8: (-127, 127), 4: (-8, 7), 2: (-2, 1)}


# ---------------------------------------------------------------- inputs
def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- quantizer
def quantize(x: np.ndarray, bits: int):
    """Symmetric per-vector quantization along the last axis.

    [P2] "Quantization needs a scale convention": q = clamp(round(x / s)),
    x_hat = q * s.  [P3] "Per-token scales and where they can live": one scale
    per token per head, computed from the vector at write time.  [P3] "The axis
    choice is a kernel decision" (listing quantize_kv_vector): amax = max |x|,
    zero vector -> (codes 0, scale 1.0), scale = amax / qmax.

    Returns (codes int16 [..., D], scale float32 [...]).
    """
    x = np.asarray(x, dtype=np.float64)
    qmax = QMAX[bits]
    lo, hi = CLAMP[bits]
    amax = np.max(np.abs(x), axis=-1)
    # RN32(amax / qmax): float64 quotient then one rounding to float32.  Double
    # rounding is harmless for a quotient of float32 operands (53 >= 2*24 + 2).
    s = (amax / qmax).astype(np.float32)
    s = np.where(amax == 0.0, np.float32(1.0), s).astype(np.float32)
    quotient = x / s.astype(np.float64)[..., None]
    codes = np.clip(np.rint(quotient), lo, hi).astype(np.int16)   # rint: half to even
    return codes, s


QMAXU = {8: 255, 4: 15, 2: 3}


def quantize_asym(x: np.ndarray, bits: int):
    """Asymmetric per-vector quantization along the last axis (scale and zero
    point; see the module notes for the reading).

    Returns (codes uint16 [..., D] in [0, 2^bits - 1], scale float32 [...],
    offset float32 [...]).
    """
    x = np.asarray(x, dtype=np.float64)
    qmaxu = QMAXU[bits]
    lo = np.min(x, axis=-1)
    hi = np.max(x, axis=-1)
    rng = hi - lo                                   # float64 difference of float32 values
    s = (rng / qmaxu).astype(np.float32)
    s = np.where(rng == 0.0, np.float32(1.0), s).astype(np.float32)
    quotient = (x - lo[..., None]) / s.astype(np.float64)[..., None]
    codes = np.clip(np.rint(quotient), 0, qmaxu).astype(np.uint16)
    return codes, s, lo.astype(np.float32)


def dequantize_asym(codes: np.ndarray, scale: np.ndarray, offset: np.ndarray) -> np.ndarray:
    """x_hat = u * s + m, exact in float64."""
    return (np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[..., None]
            + np.asarray(offset, np.float64)[..., None])


GROUP_TOKENS = 16


def quantize_token_groups(x: np.ndarray, bits: int, asym: bool = False, group: int = GROUP_TOKENS):
    """Quantize x [L, H, D] with one scale (and, asymmetric, one zero point) per
    group of ``group`` consecutive positions of each head (see the module notes
    on 2-bit codes).  Each group's values are quantized by the per-vector rule
    (quantize / quantize_asym) applied to the group flattened into one vector.

    Returns codes [L, H, D] and per-position scale [L, H] (and offset [L, H]),
    the group's scale repeated for each of its positions.
    """
    x = np.asarray(x, dtype=np.float64)
    L, H, D = x.shape
    codes = np.zeros((L, H, D), dtype=np.uint16 if asym else np.int16)
    scale = np.zeros((L, H), dtype=np.float32)
    offset = np.zeros((L, H), dtype=np.float32)
    for g0 in range(0, L, group):
        g1 = min(L, g0 + group)
        flat = x[g0:g1].transpose(1, 0, 2).reshape(H, (g1 - g0) * D)      # one vector per head
        if asym:
            c, s, m = quantize_asym(flat, bits)
            offset[g0:g1] = m[None, :]
        else:
            c, s = quantize(flat, bits)
        codes[g0:g1] = c.reshape(H, g1 - g0, D).transpose(1, 0, 2)
        scale[g0:g1] = s[None, :]
    return (codes, scale, offset) if asym else (codes, scale)


def dequantize(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x_hat = q * s ([P2] "Quantization needs a scale convention"), exact in float64."""
    return np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[..., None]


def quantize_query(q: np.ndarray, c: np.ndarray | None = None):
    """Integer query of the quantized-query mode (see the module notes):
    (codes int16 [..., D] in [-127, 127], scale float32 [...])."""
    x = np.asarray(q, np.float64)
    if c is not None:
        x = (x * np.asarray(c, np.float64)).astype(np.float32).astype(np.float64)
    return quantize(x, 8)


def effective_query(q: np.ndarray, c: np.ndarray | None = None) -> np.ndarray:
    """The float query whose dot product with the reconstructed keys c * k'_hat
    equals s_q * (q_int . k'_hat): q_int * s_q / c (float64)."""
    codes, s = quantize_query(q, c)
    qe = dequantize(codes, s)
    return qe if c is None else qe / np.asarray(c, np.float64)


def divide_by_channel_factor(k: np.ndarray, c: np.ndarray) -> np.ndarray:
    """k'_j = RN32(k_j / c_j): the per-channel key factor taken out before the
    per-token quantizer ([P3] "The axis choice is a kernel decision": the
    per-channel factor is moved onto the query)."""
    return (np.asarray(k, np.float64) / np.asarray(c, np.float64)).astype(np.float32).astype(np.float64)


def quantize_keys(k: np.ndarray, bits: int, c: np.ndarray | None = None):
    """Per-token key quantization, optionally after the per-channel factor."""
    x = k if c is None else divide_by_channel_factor(k, c)
    return quantize(x, bits)


def quantize_keys_per_channel(k: np.ndarray, bits: int, c: np.ndarray) -> np.ndarray:
    """Key codes under per-channel scales only: clamp(rint(k / c)) with the
    float64 quotient of float32 operands (equal to rounding the exact quotient,
    as in quantize); int16 [..., D]."""
    lo, hi = CLAMP[bits]
    x = np.asarray(k, np.float64) / np.asarray(c, np.float64)
    return np.clip(np.rint(x), lo, hi).astype(np.int16)


def reconstruct_keys(codes, scale, c=None) -> np.ndarray:
    """k_hat = c * (q * s); without a factor, k_hat = q * s."""
    kh = dequantize(codes, scale)
    return kh if c is None else kh * np.asarray(c, np.float64)


# ---------------------------------------------------------------- attention
def attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray):
    """Plain softmax attention of one or more queries over T cached tokens.

    [P1] "Key error acts before the softmax": s = q K^T / sqrt(d), a = softmax(s),
    o = a V.  [P2] "Keys and values need not have identical error sensitivity":
    score_i = q^T k_hat_i / sqrt(D), output = sum_i softmax(score)_i v_hat_i.

    q [G, D], k_hat [T, D], v_hat [T, D] -> (o [G, D], lse [G]) with
    lse = ln sum_i exp(score_i).  T == 0 gives o = 0 and lse = -inf.
    """
    q = np.atleast_2d(np.asarray(q, np.float64))
    G, D = q.shape
    T = k_hat.shape[0]
    if T == 0:
        return np.zeros((G, v_hat.shape[1] if v_hat.ndim == 2 else D)), np.full(G, -np.inf)
    scores = (q @ np.asarray(k_hat, np.float64).T) / np.sqrt(D)        # [G, T]
    m = scores.max(axis=1, keepdims=True)
    e = np.exp(scores - m)
    l = e.sum(axis=1, keepdims=True)
    a = e / l
    o = a @ np.asarray(v_hat, np.float64)
    lse = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention_weights(q: np.ndarray, k_hat: np.ndarray) -> np.ndarray:
    """a = softmax(q K^T / sqrt(d)) ([P1] "Key error acts before the softmax")."""
    q = np.atleast_2d(np.asarray(q, np.float64))
    scores = (q @ np.asarray(k_hat, np.float64).T) / np.sqrt(q.shape[1])
    e = np.exp(scores - scores.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def lse_merge(parts):
    """Combine attention over disjoint token subsets given (o_p, lse_p) each.

    A softmax over the union equals the lse-weighted mix of the per-subset
    softmaxes: o = sum_p exp(lse_p - lse) o_p with lse = ln sum_p exp(lse_p).
    Used only to pin that splitting the sequence does not change the result.
    """
    lses = np.stack([p[1] for p in parts])            # [P, G]
    M = lses.max(axis=0)
    w = np.exp(lses - M)
    tot = w.sum(axis=0)
    o = sum(w[i][:, None] * parts[i][0] for i in range(len(parts))) / tot[:, None]
    return o, M + np.log(tot)


# ---------------------------------------------------------------- one cached sequence
def window_split(length: int, window: int) -> int:
    """Number of leading positions that are quantized when the last ``window``
    positions stay in bf16 ([P1] "Cache growth changes the serving trade":
    recent tokens in higher precision, older ones quantized)."""
    if window <= 0:
        return length
    return max(length - window, 0)


def quantize_sequence(k, v, k_bits: int, v_bits: int, window: int = 0, c=None, asym: bool = False,
                      k_per_channel: bool = False):
    """Store one sequence: k, v float64 [L, H, D] (exact bf16 values).

    Returns a dict with the quantized prefix (codes/scales for K and V) and the
    bf16 window values (float64).  16-bit formats store the values unchanged.
    k_per_channel: keys carry the per-channel scales c only (no per-token scale).
    """
    L = k.shape[0]
    Lq = window_split(L, window)
    st = {"Lq": Lq, "k_bits": k_bits, "v_bits": v_bits, "c": c, "asym": asym, "k_per_channel": k_per_channel}
    if k_per_channel and (c is None or asym or k_bits == 16):
        raise ValueError("per-channel-only key scales need c, symmetric codes and 8- or 4-bit keys")
    if (k_bits == 2) != (v_bits == 2) or (k_bits == 2 and k_per_channel):
        raise ValueError("2-bit codes come as K and V together, with token-group scales")
    if k_bits == 2:
        kx = k[:Lq] if c is None else divide_by_channel_factor(k[:Lq], c)
        if asym:
            st["k_codes"], st["k_scale"], st["k_offset"] = quantize_token_groups(kx, 2, asym=True)
            st["v_codes"], st["v_scale"], st["v_offset"] = quantize_token_groups(v[:Lq], 2, asym=True)
        else:
            st["k_codes"], st["k_scale"] = quantize_token_groups(kx, 2)
            st["v_codes"], st["v_scale"] = quantize_token_groups(v[:Lq], 2)
        st["k_window"] = k[Lq:]
        st["v_window"] = v[Lq:]
        return st
    if k_bits == 16:
        st["k_plain"] = k[:Lq]
    elif k_per_channel:
        st["k_codes"] = quantize_keys_per_channel(k[:Lq], k_bits, c)
    elif asym:
        kx = k[:Lq] if c is None else divide_by_channel_factor(k[:Lq], c)
        st["k_codes"], st["k_scale"], st["k_offset"] = quantize_asym(kx, k_bits)
    else:
        st["k_codes"], st["k_scale"] = quantize_keys(k[:Lq], k_bits, c)
    if v_bits == 16:
        st["v_plain"] = v[:Lq]
    elif asym:
        st["v_codes"], st["v_scale"], st["v_offset"] = quantize_asym(v[:Lq], v_bits)
    else:
        st["v_codes"], st["v_scale"] = quantize(v[:Lq], v_bits)
    st["k_window"] = k[Lq:]
    st["v_window"] = v[Lq:]
    return st


def reconstruct_sequence(st, head: int):
    """k_hat, v_hat [L, D] of one KV head: dequantized prefix then bf16 window."""
    c = st["c"]
    if st["k_bits"] == 16:
        kq = st["k_plain"][:, head]
    elif st.get("k_per_channel"):
        kq = np.asarray(st["k_codes"][:, head], np.float64) * np.asarray(c[head], np.float64)
    elif st.get("asym"):
        kq = dequantize_asym(st["k_codes"][:, head], st["k_scale"][:, head], st["k_offset"][:, head])
        kq = kq if c is None else kq * np.asarray(c[head], np.float64)
    else:
        kq = reconstruct_keys(st["k_codes"][:, head], st["k_scale"][:, head],
                              None if c is None else c[head])
    if st["v_bits"] == 16:
        vq = st["v_plain"][:, head]
    elif st.get("asym"):
        vq = dequantize_asym(st["v_codes"][:, head], st["v_scale"][:, head], st["v_offset"][:, head])
    else:
        vq = dequantize(st["v_codes"][:, head], st["v_scale"][:, head])
    k_hat = np.concatenate([kq, st["k_window"][:, head]], axis=0)
    v_hat = np.concatenate([vq, st["v_window"][:, head]], axis=0)
    return k_hat, v_hat


def decode_sequence(q_bits, st, kv_heads: int, query_bits: int = 16):
    """One decode step of one sequence: q_bits [H_q, D] bf16 bits.

    Query head h reads KV head h // (H_q / H_kv) (grouped-query sharing; the
    pages' one-head formulas applied per head).  query_bits = 8 selects the
    quantized-query mode (effective_query).  Returns (o [H_q, D], lse [H_q]).
    """
    q = bf16_to_f64(q_bits)
    H_q, D = q.shape
    G = H_q // kv_heads
    o = np.zeros((H_q, D))
    lse = np.zeros(H_q)
    c = st["c"]
    for h in range(kv_heads):
        k_hat, v_hat = reconstruct_sequence(st, h)
        qh = q[h * G:(h + 1) * G]
        if query_bits == 8:
            qh = effective_query(qh, None if c is None else c[h])
        o[h * G:(h + 1) * G], lse[h * G:(h + 1) * G] = attention(qh, k_hat, v_hat)
    return o, lse


def prefill_attention(q_rows: np.ndarray, st, head: int, pos: np.ndarray):
    """Chunked prefill over one stored sequence: row r (query [G, D] of KV head
    ``head``) is the new position pos[r] and attends causally to the stored
    positions 0..pos[r], itself included ([P3] opening section: the cache is
    written incrementally and read repeatedly; each query reads the entries
    written before it and its own).  Returns (o [R, G, D], lse [R, G])."""
    k_hat, v_hat = reconstruct_sequence(st, head)
    outs, lses = [], []
    for r, p in enumerate(np.asarray(pos, dtype=np.int64)):
        o, lse = attention(q_rows[r], k_hat[: p + 1], v_hat[: p + 1])
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)


# ---------------------------------------------------------------- byte accounting
def kv_payload_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int, bytes_per_elem: float) -> float:
    """KV_bytes = 2 * L * H_kv * D * T * b ([P2] "Cache precision is separate from
    weight precision"): the factor 2 is keys plus values; metadata excluded."""
    return 2 * layers * kv_heads * head_dim * tokens * bytes_per_elem


def metadata_fraction(head_dim: int, bits: int, metadata_bytes: int) -> float:
    """Per-token metadata over the code bytes of one head vector ([P3] "Per-token
    scales and where they can live")."""
    return metadata_bytes / (head_dim * bits / 8)


def cache_bytes_per_token_head(head_dim: int, k_bits: int, v_bits: int, scale_bytes: int = 4,
                               asym: bool = False, k_per_channel: bool = False) -> float:
    """Bytes read per cached token per KV head: codes plus one scale (and, for
    the asymmetric format, one offset) for each of K and V (no metadata for a
    16-bit cache, none for keys under per-channel scales only).  2-bit codes
    share their scales over a 16-token group, stored as one 16-byte record
    (K scale, K offset, V scale, V offset) per group: one byte per token."""
    if k_bits == 2:
        return 2 * head_dim * 2 / 8 + 16 / GROUP_TOKENS
    meta = scale_bytes * (2 if asym else 1)
    kb = head_dim * k_bits // 8 + (0 if (k_bits == 16 or k_per_channel) else meta)
    vb = head_dim * v_bits // 8 + (0 if v_bits == 16 else meta)
    return kb + vb
