// Chunked prefill attention on query tiles (kvq_prefill, tile path).
//
// [P3] "KV Cache Quantization and Per-Token Scale Placement", opening section:
// the cache is written incrementally and read repeatedly; a chunk of new
// positions of a sequence attends to the stored cache up to each position.
// Unlike decode, where one query group meets each cached block, a chunk has
// many query rows per block, so the contraction is dense: here a CTA takes a
// tile of 16 query vectors (consecutive rows of the call x the G query heads
// of one KV head) and every converted key and value block feeds a full
// 16-row tensor-core tile.
//
// Work: CTA (tile, kv head); tile = rows [TR*tile, TR*tile + TR) of the call,
// TR = 16 / G.  Rows of one tile that belong to different sequences are taken
// in turn ("sub-passes"), one per distinct sequence.  A producer warp streams
// the sequence's blocks 0 .. ceil(max len / 16) - 1 with bulk copies into an
// mbarrier ring, four blocks per stage; consumer warp w takes block w of each
// stage for all 16 query vectors and keeps its own online-softmax state; the
// four states are merged through shared memory at the end of a sub-pass.
//
// Scores: S (16 query vectors x 16 tokens) = Q (16 x 128, fp16, each row
// scaled by a power of two) . K^T (codes converted exactly to fp16; int8 codes
// keep the conversion's offset, 1152 + c, and each block's accumulators start
// at minus 1152 times the row's sums), two m16n8k16 products per 16-dim slice;
// the per-token key scale multiplies the scalar after the dot product ([P3]
// "The axis choice is a kernel decision").
// Values: O (16 x 128) += (P * s_v) (16 x 16 tokens, fp16) . V (codes), the
// value scale folded into the weight ([P2] "Keys and values need not have
// identical error sensitivity").  Asymmetric blocks add the key zero-point
// term m'_k * sum(q) to each score and sum(p * m'_v) to each output row, as
// the decode kernel does.  In the two-part mode (q_bits 32) the query and the
// weights p * s_v are each carried as fp16 high + low parts: a second product
// per slice with the low parts, as in decode.  The cache's fragment-native block order
// (include/kvq.h) gives each lane exactly the B-operand pairs of these
// products, the same registers the decode kernel uses as A operands.
#include "kvq_decode_impl.cuh"

namespace kvq {
namespace {

constexpr int kTileQ = 16;       // query vectors per tile: one m16 row tile
constexpr int kOStride = 132;    // float row stride of the combine buffer (bank spread)
constexpr int kCombineBytes = kConsumerWarps * kTileQ * kOStride * 4;

template <int KB, int VB, bool ASYM>
struct TileFmt {
  using F = Fmt<KB, VB, ASYM>;
  static constexpr int kBlocksPerStage = kConsumerWarps;  // block w of a stage -> consumer warp w
  static constexpr int kStageBytes = kBlocksPerStage * F::kPerBlock;
  static constexpr int kStagesRaw = 65536 / kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 16 ? 16 : kStagesRaw);
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kBlocksPerStage * F::kKBB;
  static constexpr int kOffMeta = kOffV + kBlocksPerStage * F::kVBB;
  // the four warps' states merge in the ring once a sub-pass has drained it
  static_assert(kStages * kStageBytes >= kCombineBytes, "combine buffer must fit in the ring");
};

struct TileSmem {
  int qf, qlo, qs, qz, zo, qlen, cm, cl, rowseq, rowlen, bars, total;
};

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline TileSmem tile_smem(int ring_bytes, int stages) {
  TileSmem m{};
  int o = align16(ring_bytes);
  m.qf = o;  // query tile in A-operand order: [slice kk][g][t] x (rows g, g + 8) x 4 fp16
  o = align16(o + 8 * 8 * 4 * 16);
  m.qlo = o;  // two-part mode: the low fp16 parts in the same order
  o = align16(o + 8 * 8 * 4 * 16);
  m.qs = o;
  o = align16(o + kTileQ * 4);
  m.qz = o;  // asymmetric blocks: sum of each fp16 query vector as the MMA sees it
  o = align16(o + kTileQ * 4);
  m.zo = o;  // offset int8 keys: float4 per g {even g, even g + 8, odd g, odd g + 8}
  o = align16(o + kTileQ * 2 * 4);
  m.qlen = o;
  o = align16(o + kTileQ * 4);
  m.cm = o;
  o = align16(o + kConsumerWarps * kTileQ * 4);
  m.cl = o;
  o = align16(o + kConsumerWarps * kTileQ * 4);
  m.rowseq = o;
  o = align16(o + kTileQ * 4);
  m.rowlen = o;
  o = align16(o + kTileQ * 4);
  m.bars = o;
  o = align16(o + (2 * stages + 2) * 8);
  m.total = o;
  return m;
}

// A sub-pass: the rows of the tile that belong to sequence seq; nblk blocks
// cover the longest of them (maxlen tokens).
struct SubPass {
  int seq, maxlen, nblk;
};

// The sub-pass led by tile row ri (the first row of its sequence in the tile),
// or seq = -1 when row ri leads none.
__device__ __forceinline__ SubPass sub_pass_at(const int* rowseq, const int* rowlen, int nrows, int ri) {
  SubPass sp{-1, 0, 0};
  const int sb = rowseq[ri];
  if (sb < 0) return sp;
  for (int k = 0; k < ri; ++k)
    if (rowseq[k] == sb) return sp;
  int ml = 0;
  for (int k = ri; k < nrows; ++k)
    if (rowseq[k] == sb) ml = max(ml, rowlen[k]);
  sp.seq = sb;
  sp.maxlen = ml;
  sp.nblk = (ml + kBlock - 1) / kBlock;
  return sp;
}

// Int8 keys of the one-part query modes enter the score product with their
// offset (s8x4_to_f16_r_off: 1152 + c, exact) and each block's accumulators
// start at minus 1152 times the row's sum over the dims they cover (the even
// k-slices for s, the odd ones for the second chain), as in the decode kernel.
template <int KB, bool LOQ>
struct TileOffsetKeys {
  static constexpr bool kOn = !LOQ && KB == 8;
};

// Four int8 codes -> (1152 + c0, 1152 + c1), (1152 + c2, 1152 + c3); c64 as below.
__device__ __forceinline__ void s8x4_to_f16_r_off(uint32_t w, uint32_t c64, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(w, c64, 0x4140);
  hi = __byte_perm(w, c64, 0x4342);
}

// Four int8 codes -> fp16 pairs as s8x4_to_f16, with the byte constant 0x64
// of the permutes in a register (c64 = 0x64646464 from the caller) instead of
// being rebuilt before every permute.
__device__ __forceinline__ void s8x4_to_f16_r(uint32_t w, uint32_t c64, uint32_t& lo, uint32_t& hi) {
  const uint32_t a = __byte_perm(w, c64, 0x4140);
  const uint32_t b = __byte_perm(w, c64, 0x4342);
  const uint32_t bias = 0x64806480u;  // (1152, 1152) = 1024 + 128
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Online-softmax state of one consumer warp over its blocks of a sub-pass:
// each thread holds rows g and g + 8 of the tile, output dims 8 nt + 2t, +1.
struct TileState {
  float O[16][4];
  float m0, m1, l0, l1;
  float z0, z1;     // asymmetric values: sum of p * m'_v of this thread's tokens per row
  float sg, svlim;  // sigma and the largest value scale it allows (as in decode)
  __device__ __forceinline__ void reset() {
    m0 = m1 = kNegInf;
    l0 = l1 = 0.f;
    z0 = z1 = 0.f;
    sg = float(kSigma0);
    svlim = ldexpf(1.f, kWeightExp - int(kMaxSlack) - kSigma0);
#pragma unroll
    for (int i = 0; i < 16; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
  }
};

// Scores of one block: s[n][c] for n-tile n (tokens 8n..8n+7), row g (c < 2)
// or g + 8, token 8n + 2t + (c & 1).  Key slice kk covers dims 32t + 4kk + 0..3
// of every lane (the fragment-native key order); qf holds the query tile in
// the same order with rows g and g + 8 interleaved, so the A operand of slice
// kk is one 16-byte load, its four registers in operand order.
// With OFF the accumulators start at zi: {even row g, even row g + 8, odd row
// g, odd row g + 8} (TileOffsetKeys).
template <int KB, bool LOQ, bool OFF>
__device__ __forceinline__ void tile_scores(const uint8_t* kb, const uint4* qf, const uint4* qlo, float (&s)[2][4],
                                            int lane, uint32_t km, uint32_t c64, float4 zi) {
  auto qa = [&](int kk, uint32_t (&r)[4]) {
    const uint4 u = qf[kk * 32 + lane];
    r[0] = u.x;
    r[1] = u.y;
    r[2] = u.z;
    r[3] = u.w;
  };
  // one slice's product for n-tile d: the high query parts, then (two-part
  // mode) the low parts into the same accumulator
  auto mma2 = [&](float (&d)[4], int kk, const uint32_t (&q)[4], uint32_t b0, uint32_t b1) {
    mma_f16(d, q[0], q[1], q[2], q[3], b0, b1);
    if constexpr (LOQ) {
      const uint4 l = qlo[kk * 32 + lane];
      mma_f16(d, l.x, l.y, l.z, l.w, b0, b1);
    }
  };
  float e[2][4];  // odd slices: a second chain
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    s[n][0] = s[n][1] = OFF ? zi.x : 0.f;
    s[n][2] = s[n][3] = OFF ? zi.y : 0.f;
    e[n][0] = e[n][1] = OFF ? zi.z : 0.f;
    e[n][2] = e[n][3] = OFF ? zi.w : 0.f;
  }
  const uint4* p = reinterpret_cast<const uint4*>(kb) + lane;
  if constexpr (KB == 8) {
    const uint4 r0a = p[0], r0b = p[32], r1a = p[64], r1b = p[96];
    const uint32_t g0[8] = {r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
    const uint32_t g8[8] = {r1a.x, r1a.y, r1a.z, r1a.w, r1b.x, r1b.y, r1b.z, r1b.w};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a0, a1, a2, a3, q[4];
      qa(kk, q);
      if constexpr (OFF) {
        s8x4_to_f16_r_off(g0[kk], c64, a0, a2);  // tokens 0-7
        s8x4_to_f16_r_off(g8[kk], c64, a1, a3);  // tokens 8-15
      } else {
        s8x4_to_f16_r(g0[kk], c64, a0, a2);
        s8x4_to_f16_r(g8[kk], c64, a1, a3);
      }
      float(&d)[2][4] = (kk & 1) ? e : s;
      mma2(d[0], kk, q, a0, a2);
      mma2(d[1], kk, q, a1, a3);
    }
  } else if constexpr (KB == 2) {
    // one 16-byte load: word w holds slices 2w (outputs 0-3) and 2w+1 (4-7),
    // outputs (token g, token g+8) x (dims +0,+1 and +2,+3) of the slice
    const uint4 r = p[0];
    const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t o[8], q0[4], q1[4];
      s2x16_to_f16(wd[wi], km, o);
      qa(2 * wi, q0);
      qa(2 * wi + 1, q1);
      mma2(s[0], 2 * wi, q0, o[0], o[2]);
      mma2(s[1], 2 * wi, q0, o[1], o[3]);
      mma2(e[0], 2 * wi + 1, q1, o[4], o[6]);
      mma2(e[1], 2 * wi + 1, q1, o[5], o[7]);
    }
  } else {
    const uint4 r0 = p[0], r1 = p[32];
    const uint32_t g0[4] = {r0.x, r0.y, r0.z, r0.w};
    const uint32_t g8[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
      s4x8_to_f16(g0[wi], km, x0, x1, x2, x3);
      s4x8_to_f16(g8[wi], km, y0, y1, y2, y3);
      uint32_t q0[4], q1[4];
      qa(2 * wi, q0);
      qa(2 * wi + 1, q1);
      mma2(s[0], 2 * wi, q0, x0, x1);
      mma2(s[1], 2 * wi, q0, y0, y1);
      mma2(e[0], 2 * wi + 1, q1, x2, x3);
      mma2(e[1], 2 * wi + 1, q1, y2, y3);
    }
  }
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) s[n][c] += e[n][c];
}

// O += P . V for one block: P in A-operand registers (rows g / g + 8, token
// slots in the value block's order), V codes converted to the B-operand pairs
// of dims 16 mt + g (O[2 mt]) and 16 mt + 8 + g (O[2 mt + 1]).
template <int VB, bool LOW>
__device__ __forceinline__ void tile_values(const uint8_t* vb, const uint32_t (&ph)[4], const uint32_t (&pl)[4],
                                            float (&O)[16][4], int lane, uint32_t km, uint32_t c64) {
  const uint4* p = reinterpret_cast<const uint4*>(vb) + lane;
  // the high weights, then (two-part mode) the low weights into the same accumulator
  auto mma2 = [&](float (&d)[4], uint32_t b0, uint32_t b1) {
    mma_f16(d, ph[0], ph[1], ph[2], ph[3], b0, b1);
    if constexpr (LOW) mma_f16(d, pl[0], pl[1], pl[2], pl[3], b0, b1);
  };
  if constexpr (VB == 8) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 c = p[h * 32];
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};  // (mt 2h, dims lo), (2h, hi), (2h+1, lo), (2h+1, hi)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t b0, b1;
        s8x4_to_f16_r(w[k], c64, b0, b1);
        mma2(O[4 * h + k], b0, b1);
      }
    }
  } else if constexpr (VB == 2) {
    // one 16-byte load: word w holds m-tiles 2w (outputs 0-3) and 2w+1 (4-7)
    const uint4 c = p[0];
    const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t o[8];
      s2x16_to_f16(wd[wi], km, o);
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // m-tile 2 wi + h
        mma2(O[2 * (2 * wi + h)], o[4 * h], o[4 * h + 2]);
        mma2(O[2 * (2 * wi + h) + 1], o[4 * h + 1], o[4 * h + 3]);
      }
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 c = p[h * 32];
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // m-tile 4h + k
        uint32_t x0, x1, x2, x3;
        s4x8_to_f16(w[k], km, x0, x1, x2, x3);
        mma2(O[2 * (4 * h + k)], x0, x1);
        mma2(O[2 * (4 * h + k) + 1], x2, x3);
      }
    }
  }
}

// One block of one consumer warp: scores, causal mask, online softmax with the
// lazy maximum and the sigma offset of the decode kernel, value product.
template <int KB, int VB, bool ASYM, bool LOQ>
__device__ __forceinline__ void tile_block(const uint8_t* kb, const uint8_t* vb, const float* ks, const float* vs,
                                           const float* ko, const float* vo, int tok0, int maxlen, int len0,
                                           int len1, float qs0, float qs1, float qz0, float qz1, const uint4* qf,
                                           const uint4* qlo, const float4* zo, TileState& st, int lane, uint32_t km,
                                           uint32_t c64) {
  // offset-binary centre of the code conversion: c' = u - kKC (zero points: m' = m + kKC * s)
  constexpr float kKC = KB == 8 ? 128.f : (KB == 4 ? 8.f : 2.f), kVC = VB == 8 ? 128.f : (VB == 4 ? 8.f : 2.f);
  // 2-bit blocks: one scale (and zero point) for the whole block
  constexpr bool kGroup = KB == 2;
  const int t = lane & 3;
  float x[2][4];
  constexpr bool kOff = TileOffsetKeys<KB, LOQ>::kOn;
  tile_scores<KB, LOQ, kOff>(kb, qf, qlo, x, lane, km, c64, kOff ? zo[lane >> 2] : make_float4(0.f, 0.f, 0.f, 0.f));
  // this thread's tokens: 8n + 2t + j (n = 0, 1; j = 0, 1)
  const float2 k0 = kGroup ? make_float2(ks[0], ks[0]) : *reinterpret_cast<const float2*>(ks + 2 * t);
  const float2 k1 = kGroup ? make_float2(ks[0], ks[0]) : *reinterpret_cast<const float2*>(ks + 8 + 2 * t);
  const float2 v0 = kGroup ? make_float2(vs[0], vs[0]) : *reinterpret_cast<const float2*>(vs + 2 * t);
  const float2 v1 = kGroup ? make_float2(vs[0], vs[0]) : *reinterpret_cast<const float2*>(vs + 8 + 2 * t);
  const float ksc[2][2] = {{k0.x, k0.y}, {k1.x, k1.y}};
  float vsc[2][2] = {{v0.x, v0.y}, {v1.x, v1.y}};
  float mk[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, mv[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  if constexpr (ASYM) {
    const float2 a0 = kGroup ? make_float2(ko[0], ko[0]) : *reinterpret_cast<const float2*>(ko + 2 * t);
    const float2 a1 = kGroup ? make_float2(ko[0], ko[0]) : *reinterpret_cast<const float2*>(ko + 8 + 2 * t);
    const float2 b0 = kGroup ? make_float2(vo[0], vo[0]) : *reinterpret_cast<const float2*>(vo + 2 * t);
    const float2 b1 = kGroup ? make_float2(vo[0], vo[0]) : *reinterpret_cast<const float2*>(vo + 8 + 2 * t);
    mk[0][0] = fmaf(kKC, k0.x, a0.x);
    mk[0][1] = fmaf(kKC, k0.y, a0.y);
    mk[1][0] = fmaf(kKC, k1.x, a1.x);
    mk[1][1] = fmaf(kKC, k1.y, a1.y);
    mv[0][0] = fmaf(kVC, v0.x, b0.x);
    mv[0][1] = fmaf(kVC, v0.y, b0.y);
    mv[1][0] = fmaf(kVC, v1.x, b1.x);
    mv[1][1] = fmaf(kVC, v1.y, b1.y);
  }
  float svm = 0.f;
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int pos = tok0 + 8 * n + 2 * t + j;
      if constexpr (ASYM) {
        x[n][j] = pos < len0 ? fmaf(x[n][j], ksc[n][j], mk[n][j] * qz0) * qs0 : kNegInf;
        x[n][2 + j] = pos < len1 ? fmaf(x[n][2 + j], ksc[n][j], mk[n][j] * qz1) * qs1 : kNegInf;
        mv[n][j] = pos < maxlen ? mv[n][j] : 0.f;
      } else {
        x[n][j] = pos < len0 ? x[n][j] * (ksc[n][j] * qs0) : kNegInf;
        x[n][2 + j] = pos < len1 ? x[n][2 + j] * (ksc[n][j] * qs1) : kNegInf;
      }
      // scales of slots past the sub-pass's longest row are not data
      vsc[n][j] = pos < maxlen ? vsc[n][j] : 0.f;
      svm = fmaxf(svm, vsc[n][j]);
    }
  float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
  float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {  // the four lanes of a row
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
  }
  if (__any_sync(kFull, (mx0 > st.m0 + kMaxSlack) || (mx1 > st.m1 + kMaxSlack))) {
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float al0 = (mn0 == kNegInf) ? 1.f : ex2(st.m0 - mn0);
    const float al1 = (mn1 == kNegInf) ? 1.f : ex2(st.m1 - mn1);
    st.l0 *= al0;
    st.l1 *= al1;
    st.z0 *= al0;
    st.z1 *= al1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      st.O[i][0] *= al0;
      st.O[i][1] *= al0;
      st.O[i][2] *= al1;
      st.O[i][3] *= al1;
    }
    st.m0 = mn0;
    st.m1 = mn1;
  }
  if (__any_sync(kFull, svm > st.svlim)) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) svm = fmaxf(svm, __shfl_xor_sync(kFull, svm, o));
    int ex;
    frexpf(svm, &ex);  // svm < 2^ex
    const int sg_new = min(int(st.sg), kWeightExp - int(kMaxSlack) - ex);
    const float f = ldexpf(1.f, sg_new - int(st.sg));  // exact power of two
    st.l0 *= f;
    st.l1 *= f;
    st.z0 *= f;
    st.z1 *= f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      st.O[i][0] *= f;
      st.O[i][1] *= f;
      st.O[i][2] *= f;
      st.O[i][3] *= f;
    }
    st.sg = float(sg_new);
    st.svlim = ldexpf(1.f, kWeightExp - int(kMaxSlack) - sg_new);
  }
  const float base0 = (st.m0 == kNegInf) ? 0.f : st.m0 - st.sg;
  const float base1 = (st.m1 == kNegInf) ? 0.f : st.m1 - st.sg;
  float w[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float pa = ex2(x[n][j] - base0), pb = ex2(x[n][2 + j] - base1);
      st.l0 += pa;
      st.l1 += pb;
      if constexpr (ASYM) {
        st.z0 = fmaf(pa, mv[n][j], st.z0);
        st.z1 = fmaf(pb, mv[n][j], st.z1);
      }
      w[n][j] = pa * vsc[n][j];
      w[n][2 + j] = pb * vsc[n][j];
    }
  // A operand of the value product: token slot k of the value block order
  // holds tokens (2t, 2t + 8) at k = (2t, 2t + 1) and (2t + 1, 2t + 9) at
  // k = (2t + 8, 2t + 9)
  const float wr[4][2] = {{w[0][0], w[1][0]}, {w[0][2], w[1][2]}, {w[0][1], w[1][1]}, {w[0][3], w[1][3]}};
  uint32_t ph[4], pl[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // registers: row g, row g + 8, row g, row g + 8
    ph[i] = pack_half2(wr[i][0], wr[i][1]);
    if constexpr (LOQ) {  // low parts w - hi (exact in fp32)
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&ph[i]));
      pl[i] = pack_half2(wr[i][0] - hf.x, wr[i][1] - hf.y);
    }
  }
  tile_values<VB, LOQ>(vb, ph, pl, st.O, lane, km, c64);
}

template <int KB, int VB, bool ASYM, bool LOQ>
__global__ void __launch_bounds__(kThreads, 3) prefill_tile_kernel(const DecodeArgs a, int n_tiles, int TR) {
  using F = Fmt<KB, VB, ASYM>;
  using T = TileFmt<KB, VB, ASYM>;
  constexpr int S = T::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  const TileSmem mp = tile_smem(S * T::kStageBytes, S);
  uint32_t* qf = reinterpret_cast<uint32_t*>(smem + mp.qf);
  uint32_t* qlo = reinterpret_cast<uint32_t*>(smem + mp.qlo);
  float* qs_s = reinterpret_cast<float*>(smem + mp.qs);
  float* qz_s = reinterpret_cast<float*>(smem + mp.qz);
  float* zo_s = reinterpret_cast<float*>(smem + mp.zo);
  int* qlen_s = reinterpret_cast<int*>(smem + mp.qlen);
  float* cm = reinterpret_cast<float*>(smem + mp.cm);
  float* cl = reinterpret_cast<float*>(smem + mp.cl);
  float* co = reinterpret_cast<float*>(smem);  // over the ring (see cdone)
  int* rowseq = reinterpret_cast<int*>(smem + mp.rowseq);
  int* rowlen = reinterpret_cast<int*>(smem + mp.rowlen);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + mp.bars);
  uint64_t* empty = full + S;
  uint64_t* cbar = empty + S;
  uint64_t* cdone = cbar + 1;  // consumers have merged a sub-pass: the ring may be refilled

  const int G = a.G;
  const int tile = blockIdx.x % n_tiles, h = blockIdx.x / n_tiles;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = tile * TR;
  const int nrows = min(TR, a.B - r0);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(cbar, kConsumers);
    mbar_init(cdone, 1);
    fence_mbar_init();
  }
  // keys under per-channel scales only: the key-scale slots of the ring hold
  // 1.0 (the producer never copies over them; refilled after each merge)
  auto unit_key_scales = [&](int first, int stride) {
    for (int i = first; i < S * T::kBlocksPerStage * kBlock; i += stride) {
      const int st = i / (T::kBlocksPerStage * kBlock), r = i % (T::kBlocksPerStage * kBlock);
      reinterpret_cast<float*>(smem + st * T::kStageBytes + T::kOffMeta)[(r / kBlock) * F::kMF + F::kKS + r % kBlock] =
          1.f;
    }
  };
  if (a.c.k_chan) unit_key_scales(tid, kThreads);
  // programmatic dependent launch: wait for the previous kernel (the chunk's
  // quantizing write) before reading memory
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // the tile's rows: sequence and causal length (positions 0..pos), clamped to
  // the block table's capacity as kvq_decode clamps lengths; a row with an
  // invalid sequence or no position to attend to is empty (sequence -1)
  if (warp == 0 && lane < kTileQ) {
    int sb = -1, len = 0;
    if (lane < nrows) {
      sb = a.seq_of[r0 + lane];
      if (sb < 0 || sb >= a.nseq) {
        if (h == 0) flag(a.err, KVQ_DEVERR_POSITION);
        sb = -1;
      } else {
        len = a.pos[r0 + lane] + 1;
        if (len < 0 || len > a.mbps * kBlock) {
          if (h == 0) flag(a.err, KVQ_DEVERR_SEQ_LEN);
          len = len < 0 ? 0 : a.mbps * kBlock;
        }
        if (len == 0) sb = -1;
      }
    }
    rowseq[lane] = sb;
    rowlen[lane] = len;
  }
  __syncthreads();
  // empty rows: out = 0, lse = -inf (as kvq_decode for a sequence of length 0)
  if (warp < kConsumerWarps)
    for (int i = tid; i < nrows * G * kHeadDim; i += kConsumers) {
      const int rr = i / (G * kHeadDim);
      if (rowseq[rr] >= 0) continue;
      const int hj = (i / kHeadDim) % G, d = i % kHeadDim;
      const size_t row = size_t(r0 + rr) * a.Hq + h * G + hj;
      if (a.out_fp32) reinterpret_cast<float*>(a.out)[row * kHeadDim + d] = 0.f;
      else reinterpret_cast<__nv_bfloat16*>(a.out)[row * kHeadDim + d] = __float2bfloat16_rn(0.f);
      if (d == 0 && a.lse) a.lse[row] = kNegInf;
    }

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    const uint64_t pol = l2_evict_normal_policy();
    int s = 0, it = 0;
    uint32_t ph = 0;
    bool ok = true;
    const uint32_t meta_bytes = a.c.k_chan ? F::kMB / 2 : F::kMB;
    int spi = 0;  // sub-passes issued
    for (int ri = 0; ri < nrows && ok; ++ri) {
      const SubPass sp = sub_pass_at(rowseq, rowlen, nrows, ri);
      if (sp.seq < 0) continue;
      if (spi > 0) {  // the previous sub-pass's merge uses the ring
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(cdone, uint32_t(spi - 1) & 1u);
        if (!__shfl_sync(kFull, w_ok ? 1 : 0, 0)) {
          if (lane == 0) flag(a.err, KVQ_DEVERR_TIMEOUT);
          break;
        }
      }
      ++spi;
      for (int b0 = 0; b0 < sp.nblk; b0 += T::kBlocksPerStage) {
        const int nb = min(T::kBlocksPerStage, sp.nblk - b0);
        if (it >= S) {
          bool w_ok = true;
          if (lane == 0) w_ok = mbar_wait(&empty[s], ph ^ 1u);
          if (!__shfl_sync(kFull, w_ok ? 1 : 0, 0)) {
            if (lane == 0) flag(a.err, KVQ_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
        }
        int phys = 0;
        if (lane < nb) {
          phys = a.table[size_t(sp.seq) * a.mbps + b0 + lane];
          if (phys < 0 || phys >= a.c.num_blocks) {
            flag(a.err, KVQ_DEVERR_BLOCK_ID);
            phys = 0;
          }
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(nb) * (F::kKBB + F::kVBB + meta_bytes));
        __syncwarp();
        if (lane < nb) {
          uint8_t* stg = smem + s * T::kStageBytes;
          const size_t hb = size_t(h) * a.c.num_blocks + phys;  // head-major pools
          bulk_g2s(stg + T::kOffK + lane * F::kKBB, a.c.k_codes + hb * F::kKBB, F::kKBB, &full[s], pol);
          bulk_g2s(stg + T::kOffV + lane * F::kVBB, a.c.v_codes + hb * F::kVBB, F::kVBB, &full[s], pol);
          if (a.c.k_chan)
            bulk_g2s(stg + T::kOffMeta + lane * F::kMB + F::kVS * 4, a.c.meta + hb * F::kMF + F::kVS, F::kMB / 2,
                     &full[s], pol);
          else
            bulk_g2s(stg + T::kOffMeta + lane * F::kMB, a.c.meta + hb * F::kMF, F::kMB, &full[s], pol);
        }
        ++it;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // drain: the most recent use of every stage must have landed before exit
    if (lane == 0)
      for (int k = max(0, it - S); k < it; ++k)
        if (!mbar_wait(&full[k % S], (k / S) & 1)) flag(a.err, KVQ_DEVERR_TIMEOUT);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const uint32_t km = magic_f16x2(a.B);
  const uint32_t c64 = 0x64646464u | (uint32_t(a.B) >> 16);  // a.B <= 4096: the constant itself
  const int g = lane >> 2, t = lane & 3;
  const int nq = TR * G;  // query vectors of a full tile (<= 16)
  int s = 0;
  uint32_t ph = 0, cphase = 0;
  for (int ri = 0; ri < nrows; ++ri) {
    const SubPass sp = sub_pass_at(rowseq, rowlen, nrows, ri);
    if (sp.seq < 0) continue;
    // stage the sub-pass's query vectors: v = row * G + head, fp16 scaled by a
    // power of two per vector (the decode kernel's query format)
    for (int v = warp; v < kTileQ; v += kConsumerWarps) {
      const int rr = v / G, hj = v % G;
      const bool act = v < nq && rr < nrows && rowseq[rr] == sp.seq;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (act) {
        const uint2 raw = *reinterpret_cast<const uint2*>(a.q + (size_t(r0 + rr) * a.Hq + h * G + hj) * kHeadDim +
                                                          4 * lane);
        x[0] = __uint_as_float(raw.x << 16);
        x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        x[2] = __uint_as_float(raw.y << 16);
        x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
        if (a.c.factor) {
          const float4 c = *reinterpret_cast<const float4*>(a.c.factor + h * kHeadDim + 4 * lane);
          x[0] *= c.x;
          x[1] *= c.y;
          x[2] *= c.z;
          x[3] *= c.w;
        }
      }
      float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
      uint2 packed;
      float ylo[4] = {0.f, 0.f, 0.f, 0.f};  // the scaled fp32 values (two-part mode: their low parts)
      float qscale;  // score scale of the vector: log2(e) / sqrt(D) over its fp16 scaling
      if (a.c.q_bits == 8) {
        // int8 query rows: codes (exact in fp16) with the row scale s_q folded
        // into the score scale; the MMA then forms the integer dot exactly
        float cq[4];
        const float sq = quantize_int8_row(x, am, cq);
        packed.x = pack_half2(cq[0], cq[1]);
        packed.y = pack_half2(cq[2], cq[3]);
        qscale = sq * (kLog2e * kInvSqrtD);
      } else {
        int e = 0;
        if (am > 0.f) {
          int ex;
          frexpf(am, &ex);
          e = 15 - ex;  // am * 2^e in [2^14, 2^15)
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) ylo[j] = ldexpf(x[j], e);
        packed.x = pack_half2(ylo[0], ylo[1]);
        packed.y = pack_half2(ylo[2], ylo[3]);
        qscale = ldexpf(kLog2e * kInvSqrtD, -e);
      }
      if constexpr (ASYM) {  // the vector's sum exactly as the MMA sees it
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&packed.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&packed.y));
        float z = (f0.x + f0.y) + (f1.x + f1.y);
        if constexpr (LOQ) {  // plus the low parts, as the second product sees them
          const uint32_t l0 = pack_half2(ylo[0] - f0.x, ylo[1] - f0.y), l1 = pack_half2(ylo[2] - f1.x, ylo[3] - f1.y);
          const float2 g0 = __half22float2(*reinterpret_cast<const __half2*>(&l0));
          const float2 g1 = __half22float2(*reinterpret_cast<const __half2*>(&l1));
          z += (g0.x + g0.y) + (g1.x + g1.y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(kFull, z, o);
        if (lane == 0) qz_s[v] = z;
      }
      if constexpr (TileOffsetKeys<KB, LOQ>::kOn) {
        // offset terms: minus 1152 times the vector's sums over the even and
        // the odd k-slices (this lane's dims 4 lane .. +3 lie in slice lane & 7)
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&packed.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&packed.y));
        float zs = (f0.x + f0.y) + (f1.x + f1.y);
#pragma unroll
        for (int o = 16; o > 1; o >>= 1) zs += __shfl_xor_sync(kFull, zs, o);
        if (lane < 2) zo_s[(v & 7) * 4 + 2 * lane + (v >> 3)] = -kOffsetF16 * zs;
      }
      {  // dims 4 lane .. +3 = 32t + 4kk + 0..3 of vector v = row g (+ 8)
        const int at = (((lane & 7) * 8 + (v & 7)) * 4 + (lane >> 3)) * 4 + (v >> 3);
        qf[at] = packed.x;
        qf[at + 2] = packed.y;
        if constexpr (LOQ) {  // two-part query: the low parts y - hi (exact in fp32)
          const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&packed.x));
          const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&packed.y));
          qlo[at] = pack_half2(ylo[0] - h0.x, ylo[1] - h0.y);
          qlo[at + 2] = pack_half2(ylo[2] - h1.x, ylo[3] - h1.y);
        }
      }
      if (lane == 0) {
        qs_s[v] = act ? qscale : 0.f;
        qlen_s[v] = act ? rowlen[rr] : 0;
      }
    }
    if (!consumer_sync(cbar, cphase)) {
      flag(a.err, KVQ_DEVERR_TIMEOUT);
      return;
    }
    const float qs0 = qs_s[g], qs1 = qs_s[g + 8];
    const float qz0 = ASYM ? qz_s[g] : 0.f, qz1 = ASYM ? qz_s[g + 8] : 0.f;
    const int len0 = qlen_s[g], len1 = qlen_s[g + 8];
    TileState st;
    st.reset();
    for (int b0 = 0; b0 < sp.nblk; b0 += T::kBlocksPerStage) {
      if (!mbar_wait(&full[s], ph)) {
        flag(a.err, KVQ_DEVERR_TIMEOUT);
        return;
      }
      const int blk = b0 + warp;
      if (blk < sp.nblk) {
        const uint8_t* stg = smem + s * T::kStageBytes;
        const float* meta = reinterpret_cast<const float*>(stg + T::kOffMeta + warp * F::kMB);
        tile_block<KB, VB, ASYM, LOQ>(stg + T::kOffK + warp * F::kKBB, stg + T::kOffV + warp * F::kVBB,
                                      meta + F::kKS, meta + F::kVS, ASYM ? meta + F::kKO : nullptr,
                                      ASYM ? meta + F::kVO : nullptr, blk * kBlock, sp.maxlen, len0, len1, qs0, qs1,
                                      qz0, qz1, reinterpret_cast<const uint4*>(qf),
                                      reinterpret_cast<const uint4*>(qlo), reinterpret_cast<const float4*>(zo_s), st,
                                      lane, km, c64);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    // ---- merge the four warps' states through shared memory
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      st.l0 += __shfl_xor_sync(kFull, st.l0, o);
      st.l1 += __shfl_xor_sync(kFull, st.l1, o);
    }
    if constexpr (ASYM) {  // the value zero-point term is the same for every output dimension
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        st.z0 += __shfl_xor_sync(kFull, st.z0, o);
        st.z1 += __shfl_xor_sync(kFull, st.z1, o);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        st.O[i][0] += st.z0;
        st.O[i][1] += st.z0;
        st.O[i][2] += st.z1;
        st.O[i][3] += st.z1;
      }
    }
    // every warp has read its last block: the ring is free for the merge
    if (!consumer_sync(cbar, cphase)) {
      flag(a.err, KVQ_DEVERR_TIMEOUT);
      return;
    }
    if (t == 0) {
      cm[warp * kTileQ + g] = st.m0 == kNegInf ? kNegInf : st.m0 - st.sg;
      cm[warp * kTileQ + g + 8] = st.m1 == kNegInf ? kNegInf : st.m1 - st.sg;
      cl[warp * kTileQ + g] = st.l0;
      cl[warp * kTileQ + g + 8] = st.l1;
    }
    {
      float* ow = co + warp * kTileQ * kOStride;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        *reinterpret_cast<float2*>(ow + g * kOStride + 8 * nt + 2 * t) = make_float2(st.O[nt][0], st.O[nt][1]);
        *reinterpret_cast<float2*>(ow + (g + 8) * kOStride + 8 * nt + 2 * t) = make_float2(st.O[nt][2], st.O[nt][3]);
      }
    }
    if (!consumer_sync(cbar, cphase)) {
      flag(a.err, KVQ_DEVERR_TIMEOUT);
      return;
    }
    {
      const int v = tid >> 3, d0 = (tid & 7) * 16;  // 16 vectors x 8 slices of 16 dims
      if (qlen_s[v] > 0) {
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * kTileQ + v]);
        float aw[kConsumerWarps], L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = cm[w * kTileQ + v];
          aw[w] = (mw == kNegInf) ? 0.f : exp2f(mw - M);
          L += aw[w] * cl[w * kTileQ + v];
        }
        const float inv = 1.f / L;
        const int rr = v / G, hj = v % G;
        const size_t row = size_t(r0 + rr) * a.Hq + h * G + hj;
#pragma unroll
        for (int d = 0; d < 16; d += 4) {
          float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float4 c = *reinterpret_cast<const float4*>(co + (w * kTileQ + v) * kOStride + d0 + d);
            o[0] = fmaf(aw[w], c.x, o[0]);
            o[1] = fmaf(aw[w], c.y, o[1]);
            o[2] = fmaf(aw[w], c.z, o[2]);
            o[3] = fmaf(aw[w], c.w, o[3]);
          }
          const size_t idx = row * kHeadDim + d0 + d;
          if (a.out_fp32) {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx) =
                make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
          } else {
            uint2 pk;
            pk.x = pack_bf162(o[0] * inv, o[1] * inv);
            pk.y = pack_bf162(o[2] * inv, o[3] * inv);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + idx) = pk;
          }
        }
        if ((tid & 7) == 0 && a.lse) a.lse[row] = (M + log2f(L)) * kLn2;
      }
    }
    // the next sub-pass rewrites the query tile and the combine buffers; the
    // producer may refill the ring
    if (!consumer_sync(cbar, cphase)) {
      flag(a.err, KVQ_DEVERR_TIMEOUT);
      return;
    }
    if (a.c.k_chan) unit_key_scales(tid, kConsumers);  // the merge wrote over them
    if (tid == 0) mbar_arrive(cdone);
  }
}

template <int KB, int VB, bool ASYM, bool LOQ>
struct TileKernel {
  using T = TileFmt<KB, VB, ASYM>;
  static int smem_bytes() { return tile_smem(T::kStages * T::kStageBytes, T::kStages).total; }
  static cudaError_t launch(const DecodeArgs& a, cudaStream_t s) {
    static std::mutex mu;
    static std::map<int, bool> done;
    int dev = 0;
    cudaGetDevice(&dev);
    {
      std::lock_guard<std::mutex> lk(mu);
      if (!done.count(dev)) {
        cudaFuncSetAttribute(prefill_tile_kernel<KB, VB, ASYM, LOQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes());
        cudaFuncSetAttribute(prefill_tile_kernel<KB, VB, ASYM, LOQ>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        done[dev] = true;
      }
    }
    const int TR = kTileQ / a.G;
    const int n_tiles = (a.B + TR - 1) / TR;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(n_tiles * a.c.H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tile_kernel<KB, VB, ASYM, LOQ>, a, n_tiles, TR);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
};

}  // namespace

bool prefill_tiles_supported(const CacheView& c) {
  const bool bits = ((c.k_bits == 8 || c.k_bits == 4) && (c.v_bits == 8 || c.v_bits == 4)) ||
                    (c.k_bits == 2 && c.v_bits == 2);
  return bits && (c.q_bits == 0 || c.q_bits == 16 || c.q_bits == 8 || c.q_bits == 32) && c.window == 0;
}

template <bool ASYM, bool LOQ>
cudaError_t launch_tiles(const DecodeArgs& a, cudaStream_t s) {
  if (a.c.k_bits == 8 && a.c.v_bits == 8) return TileKernel<8, 8, ASYM, LOQ>::launch(a, s);
  if (a.c.k_bits == 4 && a.c.v_bits == 4) return TileKernel<4, 4, ASYM, LOQ>::launch(a, s);
  if (a.c.k_bits == 4 && a.c.v_bits == 8) return TileKernel<4, 8, ASYM, LOQ>::launch(a, s);
  if (a.c.k_bits == 8 && a.c.v_bits == 4) return TileKernel<8, 4, ASYM, LOQ>::launch(a, s);
  if (a.c.k_bits == 2 && a.c.v_bits == 2) return TileKernel<2, 2, ASYM, LOQ>::launch(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_tiles(const DecodeArgs& a, cudaStream_t s) {
  const bool loq = a.c.q_bits == 32;
  if (a.c.asym) return loq ? launch_tiles<true, true>(a, s) : launch_tiles<true, false>(a, s);
  return loq ? launch_tiles<false, true>(a, s) : launch_tiles<false, false>(a, s);
}

}  // namespace kvq
