// Fused dequantize-on-load decode attention (kvq_decode), sm_103a.
//
// What is computed, per query head of every sequence (one decode step):
//   score_i = q . k_hat_i / sqrt(D),  o = sum_i softmax(score)_i v_hat_i
//   ("KV Cache Quantization Perturbs Attention Through Stored Keys and Values",
//   section "Key error acts before the softmax"; "KV Cache Quantization Reduces
//   Cache Bytes with Separate Accuracy and Kernel Costs", section "Keys and
//   values need not have identical error sensitivity").
// How ("KV Cache Quantization and Per-Token Scale Placement"):
//   - the key dot product runs on the integer codes and the per-token key scale
//     multiplies the scalar score afterwards (section "The axis choice is a
//     kernel decision");
//   - a per-channel key factor is multiplied onto the query once (same section);
//   - codes and scales are two read streams, dequantized as they are loaded
//     (section "Per-token scales and where they can live");
//   - the value scale is folded into the attention weight, so the value loop is
//     a pure code contraction.
// Asymmetric format (scale s and zero point m per token: x_hat = u*s + m with
// unsigned codes u): the codes are read by the same offset-binary conversion as
// the symmetric ones, c' = u - c0, so x_hat = c'*s + m' with m' = m + c0*s; the
// key term m'*sum(q) is added to each score and the value term sum(p*m'_v) is
// kept per query beside O ("KV Cache Quantization Perturbs Attention Through
// Stored Keys and Values", section "Quantization granularity defines which
// values share a scale"; "KV Cache Quantization and Per-Token Scale Placement",
// section "Per-token scales and where they can live": scale plus zero point).
// The most recent W tokens may sit in a bf16 ring ("KV Cache Quantization
// Perturbs Attention ...", section "Cache growth changes the serving trade").
//
// GB300 mapping
//   * Stream-K decomposition: all (sequence, kv_head) units' 16-token blocks form
//     one global range that is cut evenly over one wave of CTAs (SMs x resident
//     CTAs).  A CTA walks its range, keeps online-softmax state per unit segment
//     and writes one partial (m, l, o) per segment; the last CTA to finish a
//     unit (atomic ticket, no spinning) merges its partials with a log-sum-exp
//     reduce.  A unit held by a single CTA is normalised in place.
//   * One producer warp streams whole 16-token blocks (codes of K and V plus
//     the block's metadata record of scales and zero points) with cp.async.bulk
//     into a ring of shared-memory stages guarded by mbarriers, one copy per run
//     of consecutive physical blocks; four consumer warps each take one block per
//     stage (two for 4-bit keys).  A CTA with a short range lets its first
//     stage land before it issues the second.
//   * Programmatic dependent launch: each CTA lets the next kernel on the stream
//     launch at once and waits for the previous one before reading memory.
//   * The GQA group (G <= 8 query heads sharing the KV head) makes the two small
//     contractions dense: S^T = Kcodes . Q^T and O^T += V^T . (p*s_v)^T run on
//     mma.sync m16n8k16 (fp16 in, fp32 accumulate), tokens/dims on M, the query
//     group on N.  Codes are converted exactly to fp16 in registers (int8 keys
//     keep the conversion's offset, cancelled by the score accumulators' start
//     value); the cache is stored in the fragment order so every lane reads 16
//     contiguous bytes.
//   * The query is scaled by an exact power of two into fp16's range; the score
//     scale s_k * 2^-e * log2(e) / sqrt(D) is applied per score in fp32.  Query
//     formats: fp16 (default), fp16 high + low parts for both the query and the
//     value weights (LOQ instantiations, one more MMA per k-slice of either
//     contraction), or int8 codes with s_q in the score scale (the MMA
//     then forms the integer dot product exactly: "KV Cache Quantization and
//     Per-Token Scale Placement", section "Precision floors and mixed cache
//     formats").
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1/sqrt(128)
#define kNegInf (-__int_as_float(0x7f800000))

template <int KB, int VB, bool ASYM>
struct Fmt {
  static constexpr bool kBf16 = (KB == 16);
  static_assert(!(kBf16 && ASYM), "bf16 blocks carry no zero point");
  // 2-bit blocks carry one scale (and zero point) per 16-token block for K and V
  static constexpr bool kGroup = (KB == 2);
  static_assert((KB == 2) == (VB == 2), "2-bit keys and values come together");
  static constexpr int kKBB = block_bytes(KB);
  static constexpr int kVBB = block_bytes(VB);
  // metadata record per block: K scales, (K zero points,) V scales, (V zero
  // points); 2-bit blocks: K scale, K zero point, V scale, V zero point
  static constexpr int kMF = kBf16 ? 0 : (kGroup ? 4 : (ASYM ? 4 : 2) * kBlock);  // floats
  static constexpr int kMB = kMF * 4;                                             // bytes
  static constexpr int kPerBlock = kKBB + kVBB + kMB;
  // 4- and 2-bit keys: each consumer warp takes two blocks per stage (two
  // independent dependency chains, one softmax reduction per 32 tokens)
  static constexpr int kBPW = (KB == 4 || KB == 2) ? 2 : 1;
  static constexpr int kBlocksPerStage = kConsumerWarps * kBPW;
  static constexpr int kStageBytes = kBlocksPerStage * kPerBlock;
  // ~52 KB ring (56 KB with zero points, which keeps three 4-bit stages): 3 CTAs per SM
  static constexpr int kStagesRaw = (ASYM ? 57344 : 53248) / kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  // stage sub-buffers
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kBlocksPerStage * kKBB;
  static constexpr int kOffMeta = kOffV + kBlocksPerStage * kVBB;
  // float offsets inside a block's record
  static constexpr int kKS = 0, kKO = kGroup ? 1 : kBlock, kVS = kGroup ? 2 : kMF / 2;
  static constexpr int kVO = kGroup ? 3 : kMF / 2 + kBlock;
};

// Shared-memory map after the stage ring (all offsets 16-byte aligned).
struct SmemMap {
  int merge_o;   // float [4 warps][4 q][128] (combine, four queries per pass)
  int merge_ml;  // float m[4][8], l[4][8]
  int qh;        // 16-bit [8][128]: B-operand rows of the current query group
  int qlo;       // fp16 [32 lanes x 16] low parts of the query fragments, in fragment order
  int qs;        // float [8] score scales, [8] sums of the fp16 query rows, [8][2] offset terms
  int qraw;      // bf16 [2][8][128]: prefetched raw query rows (double buffer)
  int fraw;      // float [2][128]: prefetched per-channel key factor row
  int hdr;       // int4 [stages]
  int bars;      // uint64 full[stages], empty[stages], cbar
  int misc;      // int [4]
  int len;       // int [B]
  int pre;       // int [B+1]
  int vpre;      // int [B+1]
  int rows;      // int [B]: sequence of each row (prefill only)
  int total;
};

__host__ __device__ inline SmemMap smem_map(int stage_bytes_total, int stages, int B, bool loq, bool rows) {
  SmemMap m;
  int o = stage_bytes_total;
  m.merge_o = o;  o += kConsumerWarps * 4 * kHeadDim * 4;
  m.merge_ml = o; o += 2 * kConsumerWarps * kMaxGroup * 4;
  m.qh = o;       o += kMaxGroup * kHeadDim * 2;
  m.qlo = o;      o += loq ? kMaxGroup * kHeadDim * 2 : 0;  // two-part query only
  m.qs = o;       o += 4 * kMaxGroup * 4;
  m.qraw = o;     o += 2 * kMaxGroup * kHeadDim * 2;
  m.fraw = o;     o += 2 * kHeadDim * 4;
  m.hdr = o;      o += stages * 16;
  m.bars = o;     o += (2 * stages + 2) * 8;
  m.misc = o;     o += 16;
  m.len = o;      o += ((B * 4 + 15) / 16) * 16;
  m.pre = o;      o += (((B + 1) * 4 + 15) / 16) * 16;
  m.vpre = o;     o += (((B + 1) * 4 + 15) / 16) * 16;
  m.rows = o;     o += rows ? ((B * 4 + 15) / 16) * 16 : 0;
  m.total = o;
  return m;
}

// ------------------------------------------------------------------ score / value contractions
// S^T of one 16-token block.  The query fragments qf hold the fp16 (or int8
// code, or bf16) query.  With LOQ (the two-part query) the low fp16 parts come
// from shared memory in the same fragment order (qlo = this lane's first
// uint4) and every k-slice runs a second MMA with them into the same fp32
// accumulator, so the score carries about 22 significant bits of the query
// instead of 11.  km holds kMagicF16x2 for the 4-bit conversion (magic_f16x2).
//
// With OFF (8-bit keys, one-part query) the codes enter the MMA with their
// offset (s8x4_to_f16_off: 1152 + c) and the accumulators start at minus 1152
// times the query's dimensions that they cover: acc the even k-slices (zi.x,
// zi.y: queries 2t, 2t + 1), acc2 the odd ones (zi.z, zi.w), so acc + acc2 is
// the code dot.  With int8 query codes every partial sum stays an integer
// below 2^24: exact.  Each block's accumulators start afresh, so the offset's
// rounding stays within the block.
template <int KB, bool LOQ, bool OFF>
__device__ __forceinline__ void score_block(const uint8_t* kb, const uint32_t (&qf)[16], const uint4* qlo,
                                            float (&acc)[4], int lane, uint32_t km, float4 zi) {
  // two accumulators halve the dependent MMA chain; summed at the end
  float acc2[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (OFF) {
    acc[0] = acc[2] = zi.x;
    acc[1] = acc[3] = zi.y;
    acc2[0] = acc2[2] = zi.z;
    acc2[1] = acc2[3] = zi.w;
  }
  const uint4* p = reinterpret_cast<const uint4*>(kb) + lane;
  if constexpr (KB == 8) {
    const uint4 r0a = p[0], r0b = p[32], r1a = p[64], r1b = p[96];
    const uint32_t g0[8] = {r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
    const uint32_t g8[8] = {r1a.x, r1a.y, r1a.z, r1a.w, r1b.x, r1b.y, r1b.z, r1b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 lo = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (LOQ) lo = qlo[i * 32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = 2 * i + h;
        uint32_t a0, a1, a2, a3;
        if constexpr (OFF) {
          s8x4_to_f16_off(g0[kk], a0, a2);
          s8x4_to_f16_off(g8[kk], a1, a3);
        } else {
          s8x4_to_f16(g0[kk], a0, a2);
          s8x4_to_f16(g8[kk], a1, a3);
        }
        float (&ac)[4] = h ? acc2 : acc;
        mma_f16(ac, a0, a1, a2, a3, qf[2 * kk], qf[2 * kk + 1]);
        if constexpr (LOQ) mma_f16(ac, a0, a1, a2, a3, h ? lo.z : lo.x, h ? lo.w : lo.y);
      }
    }
  } else if constexpr (KB == 2) {
    // one 16-byte load: word w holds k-slices 2w (outputs 0-3) and 2w+1 (4-7)
    const uint4 r = p[0];
    const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t o[8];
      s2x16_to_f16(wd[wi], km, o);
      mma_f16(acc, o[0], o[1], o[2], o[3], qf[4 * wi], qf[4 * wi + 1]);
      mma_f16(acc2, o[4], o[5], o[6], o[7], qf[4 * wi + 2], qf[4 * wi + 3]);
      if constexpr (LOQ) {
        const uint4 lo = qlo[wi * 32];
        mma_f16(acc, o[0], o[1], o[2], o[3], lo.x, lo.y);
        mma_f16(acc2, o[4], o[5], o[6], o[7], lo.z, lo.w);
      }
    }
  } else if constexpr (KB == 4) {
    const uint4 r0 = p[0], r1 = p[32];
    const uint32_t g0[4] = {r0.x, r0.y, r0.z, r0.w};
    const uint32_t g8[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
      s4x8_to_f16(g0[wi], km, x0, x1, x2, x3);
      s4x8_to_f16(g8[wi], km, y0, y1, y2, y3);
      mma_f16(acc, x0, y0, x1, y1, qf[4 * wi], qf[4 * wi + 1]);
      mma_f16(acc2, x2, y2, x3, y3, qf[4 * wi + 2], qf[4 * wi + 3]);
      if constexpr (LOQ) {
        const uint4 lo = qlo[wi * 32];
        mma_f16(acc, x0, y0, x1, y1, lo.x, lo.y);
        mma_f16(acc2, x2, y2, x3, y3, lo.z, lo.w);
      }
    }
  } else {
    uint4 c[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) c[h] = p[h * 32];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint4 lo = c[kk >> 1], hi = c[4 + (kk >> 1)];
      const uint32_t a0 = (kk & 1) ? lo.z : lo.x, a2 = (kk & 1) ? lo.w : lo.y;
      const uint32_t a1 = (kk & 1) ? hi.z : hi.x, a3 = (kk & 1) ? hi.w : hi.y;
      if (kk & 1) mma_bf16(acc2, a0, a1, a2, a3, qf[2 * kk], qf[2 * kk + 1]);
      else mma_bf16(acc, a0, a1, a2, a3, qf[2 * kk], qf[2 * kk + 1]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
}

// O^T += V^T . W^T for one 16-token block.  b0, b1 hold the fp16 (bf16 for
// bf16 blocks) weights p * s_v; with LOW (the two-part mode of code blocks, and
// always for bf16 blocks) b0lo, b1lo hold their low parts and a second MMA per
// slice adds them, so the weights carry about 22 significant bits instead of 11.
//
// The value codes are converted exactly (no offset as in score_block): the
// value accumulators run over every block of a segment, and an offset of
// about 1152 w per token would grow their fp32 rounding with the segment's
// length.
template <int VB, bool LOW>
__device__ __forceinline__ void value_block(const uint8_t* vb, uint32_t b0, uint32_t b1, uint32_t b0lo,
                                            uint32_t b1lo, float (&O)[8][4], int lane, uint32_t km) {
  const uint4* p = reinterpret_cast<const uint4*>(vb) + lane;
  if constexpr (VB == 8) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 c = p[h * 32];
      uint32_t a0, a1, a2, a3;
      s8x4_to_f16(c.x, a0, a2);
      s8x4_to_f16(c.y, a1, a3);
      mma_f16(O[2 * h], a0, a1, a2, a3, b0, b1);
      if constexpr (LOW) mma_f16(O[2 * h], a0, a1, a2, a3, b0lo, b1lo);
      s8x4_to_f16(c.z, a0, a2);
      s8x4_to_f16(c.w, a1, a3);
      mma_f16(O[2 * h + 1], a0, a1, a2, a3, b0, b1);
      if constexpr (LOW) mma_f16(O[2 * h + 1], a0, a1, a2, a3, b0lo, b1lo);
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
      for (int h = 0; h < 2; ++h) {
        mma_f16(O[2 * wi + h], o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3], b0, b1);
        if constexpr (LOW) mma_f16(O[2 * wi + h], o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3], b0lo, b1lo);
      }
    }
  } else if constexpr (VB == 4) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 c = p[h * 32];
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t x0, x1, x2, x3;
        s4x8_to_f16(w[k], km, x0, x1, x2, x3);
        mma_f16(O[4 * h + k], x0, x2, x1, x3, b0, b1);
        if constexpr (LOW) mma_f16(O[4 * h + k], x0, x2, x1, x3, b0lo, b1lo);
      }
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint4 c = p[mt * 32];
      mma_bf16(O[mt], c.x, c.z, c.y, c.w, b0, b1);
      mma_bf16(O[mt], c.x, c.z, c.y, c.w, b0lo, b1lo);
    }
  }
}

struct Params {
  DecodeArgs a;
  int P;   // stream CTAs launched (after the window CTAs)
  int Uw;  // window CTAs launched first in the grid (one per unit, 0 without a window)
};

// Geometry of the work split.  Every (sequence, kv_head) unit with data owns
// a range of "virtual blocks" in one global order: X leading virtual blocks
// that stand for the cost of starting the unit (query staging, flush of the
// previous unit, its record), then its data blocks.  The stream CTAs cut the
// virtual range evenly, so a CTA that starts more units gets fewer blocks.
struct Geo {
  const int* pre;   // [B+1] prefix sums of data blocks per sequence (one head)
  const int* vpre;  // [B+1] prefix sums of virtual blocks per sequence (one head)
  int B, H, X;
};

__device__ __forceinline__ int geo_nblk(const Geo& g, int b) { return g.pre[b + 1] - g.pre[b]; }
__device__ __forceinline__ int geo_vlen(const Geo& g, int b) { return g.vpre[b + 1] - g.vpre[b]; }
__device__ __forceinline__ long long geo_vstart(const Geo& g, int b, int h) {
  return (long long)g.H * g.vpre[b] + (long long)h * geo_vlen(g, b);
}

// Unit holding virtual block x (x < total): the largest b with H*vpre[b] <= x
// has blocks; the head follows from the offset inside that sequence's range.
__device__ __forceinline__ void locate_unit(const Geo& g, long long x, int& b, int& h) {
  int lo = 0, hi = g.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)g.H * g.vpre[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  b = lo;
  while (geo_vlen(g, b) == 0) ++b;
  h = int((x - (long long)g.H * g.vpre[b]) / geo_vlen(g, b));
}

// Base-2 exponential: the PTX ex2.approx.ftz.f32 instruction (max relative
// error about 2^-22 per the PTX ISA; ex2(-inf) = +0).  Results below 2^-126
// flush to zero: a weight that small is below fp32 resolution of the sum l,
// which holds at least one weight of 2^sigma >= 1.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Slack of the lazy running maximum (log2 units).  The softmax weights are
// p = 2^(x - m + sigma) with a warp-uniform power-of-two offset sigma (the same
// factor scales l and O, so it cancels in o = O / l), chosen so that the fp16
// value weights p * s_v <= 2^(kMaxSlack + sigma) * s_v stay at or below
// 2^kWeightExp: in fp16's normal range with room to spare, so they carry their
// full 11 (two-part: 22) significant bits instead of falling into subnormals.
// sigma starts at kSigma0, which allows value scales up to 2^-11, and steps
// down, with an exact power-of-two rescale of l and O, whenever a block brings
// a larger value scale: the first block of a segment sets it from its own
// scales, so small and large values alike keep their weights in range.  l
// stays below 2^(kSigma0 + kMaxSlack) per token, far inside fp32.
constexpr float kMaxSlack = 6.f;
constexpr int kWeightExp = 15;
constexpr int kSigma0 = 20;
// Stream CTAs with at most this many virtual blocks hold their second stage
// until the first has landed (window 4096-token workload: 36 per CTA, 20.6 ->
// 20.1 us; int4 1k-8k: ~190, 46.4 -> 45.4 us).  Longer ranges keep the deep
// initial queue (paged 2k-32k, ~1250 per CTA: 361.6 -> 365.6 us with the wait).
constexpr long long kFirstStageFirstMax = 256;

// A stream CTA owns at least this many blocks (fewer, deeper splits for tiny problems).
constexpr int kMinBlocksPerCta = 16;

// CTA-consumer barrier on an mbarrier (count = kConsumers), bounded wait.
__device__ __forceinline__ bool consumer_sync(uint64_t* bar, uint32_t& phase) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase);
  phase ^= 1u;
  return ok;
}

__device__ __forceinline__ long long cta_of(long long x, long long T, int P) {
  return ((x + 1) * (long long)P - 1) / T;
}

// Write the final normalised output of query row hq.
__device__ __forceinline__ void write_out(const DecodeArgs& a, int b, int hq, int d, float o, float l, float M) {
  const size_t idx = (size_t(b) * a.Hq + hq) * kHeadDim + d;
  const float v = o / l;
  if (a.out_fp32) reinterpret_cast<float*>(a.out)[idx] = v;
  else reinterpret_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(v);
  if (d == 0 && a.lse) a.lse[size_t(b) * a.Hq + hq] = (M + log2f(l)) * kLn2;
}

// Partial records of unit u: stream segments c0..c1 (the CTAs owning its data
// blocks, slot j + u) and, with a window, one window record (slot P + units + u).
__device__ __forceinline__ void unit_segments(const DecodeArgs& a, const int* len_s, const Geo& g, int u,
                                              long long Tv, int Pe, long long& c0, long long& c1, int& nseg,
                                              bool& has_win) {
  const int b = u / g.H, h = u % g.H;
  const int nblk = geo_nblk(g, b);
  nseg = 0;
  c0 = 0;
  c1 = -1;
  if (nblk > 0) {
    const long long d0 = geo_vstart(g, b, h) + g.X;
    c0 = cta_of(d0, Tv, Pe);
    c1 = cta_of(d0 + nblk - 1, Tv, Pe);
    nseg = int(c1 - c0 + 1);
  }
  has_win = a.c.window > 0 && len_s[b] > 0;
  nseg += has_win ? 1 : 0;
}

// Online-softmax state of one consumer warp; each thread holds queries 2t, 2t+1.
// l and O are in units of 2^(m - sg): the exponent base of the weights is
// m - sg (sg = sigma, warp-uniform), which finish_segment records.
struct WarpState {
  float O[8][4];
  float m0, m1, l0, l1;
  float z0, z1;  // asymmetric values: sum of p * m'_v of this thread's tokens
  float sg;      // sigma (an integer)
  float svlim;   // 2^(kWeightExp - kMaxSlack - sigma): the largest value scale sigma allows
  __device__ __forceinline__ void reset() {
    m0 = m1 = kNegInf;
    l0 = l1 = 0.f;
    z0 = z1 = 0.f;
    sg = float(kSigma0);
    svlim = ldexpf(1.f, kWeightExp - int(kMaxSlack) - kSigma0);  // 2^-11
#pragma unroll
    for (int i = 0; i < 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
  }
};

// Offset key codes (score_block with OFF): 8-bit keys with a one-part query.
// 4-bit keys keep the exact conversion: an offset form (every nibble moved to
// mantissa bits 4-7 by a shift) trades the fp16 subtractions for three more
// integer shifts per word and measured slower.
template <int KB, bool LOQ>
struct OffsetKeys {
  static constexpr bool kOn = !LOQ && KB == 8;
};

// NB (1 or 2) 16-token blocks of one warp: scores on the codes, per-token key
// scale after the dot product, online softmax, value scale folded into the
// weight, value MMA.  With NB = 2 the two blocks' chains interleave and share
// one lazy-maximum test and reduction.
//
// Asymmetric blocks (ASYM) add the key zero-point term m'_k * sum(q) to each
// score and accumulate the value zero-point term p * m'_v per query.
template <int KB, int VB, int NB, bool ASYM, bool LOQ>
__device__ __forceinline__ void process_blocks(const uint8_t* const (&kb)[NB], const uint8_t* const (&vb)[NB],
                                               const float* const (&ks)[NB], const float* const (&vs)[NB],
                                               const float* const (&ko)[NB], const float* const (&vo)[NB],
                                               const int (&valid)[NB], const uint32_t (&qf)[16],
                                               const uint4* qlo, const float4* qzo, float qs0, float qs1, float qz0,
                                               float qz1, WarpState& st, int lane, uint32_t km) {
  constexpr bool kBf16 = (KB == 16);
  constexpr bool kOffK = OffsetKeys<KB, LOQ>::kOn;
  // offset-binary centre of the code conversion: c' = u - kKC
  constexpr float kKC = (KB == 8) ? 128.f : (KB == 4 ? 8.f : 2.f), kVC = (VB == 8) ? 128.f : (VB == 4 ? 8.f : 2.f);
  // token g's (and g + 8's) entry of a per-token record; 2-bit blocks hold one per block
  constexpr bool kGroup = (KB == 2);
  const int g = lane >> 2, t = lane & 3;
  float x[NB][4];
  float sv[NB][2];
  float mv[NB][2];
  const float4 zi = kOffK ? qzo[t] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    score_block<KB, LOQ, kOffK>(kb[j], qf, qlo, acc, lane, km, zi);
    float sk0 = 1.f, sk1 = 1.f;
    sv[j][0] = sv[j][1] = 1.f;
    const int i0 = kGroup ? 0 : g, i1 = kGroup ? 0 : g + 8;
    if constexpr (!kBf16) {
      sk0 = ks[j][i0];  // per-channel key scales only: the ring holds 1.0 here (never copied over)
      sk1 = ks[j][i1];
      sv[j][0] = vs[j][i0];
      sv[j][1] = vs[j][i1];
    }
    if constexpr (ASYM) {
      const float mk0 = fmaf(kKC, sk0, ko[j][i0]), mk1 = fmaf(kKC, sk1, ko[j][i1]);
      mv[j][0] = fmaf(kVC, sv[j][0], vo[j][i0]);
      mv[j][1] = fmaf(kVC, sv[j][1], vo[j][i1]);
      x[j][0] = fmaf(acc[0], sk0, mk0 * qz0) * qs0;  // token g, query 2t
      x[j][1] = fmaf(acc[1], sk0, mk0 * qz1) * qs1;  // token g, query 2t+1
      x[j][2] = fmaf(acc[2], sk1, mk1 * qz0) * qs0;  // token g+8, query 2t
      x[j][3] = fmaf(acc[3], sk1, mk1 * qz1) * qs1;  // token g+8, query 2t+1
    } else {
      x[j][0] = acc[0] * (sk0 * qs0);  // token g, query 2t
      x[j][1] = acc[1] * (sk0 * qs1);  // token g, query 2t+1
      x[j][2] = acc[2] * (sk1 * qs0);  // token g+8, query 2t
      x[j][3] = acc[3] * (sk1 * qs1);  // token g+8, query 2t+1
    }
    if (valid[j] < kBlock) {  // the last block of a unit may be partial
      const bool v0 = g < valid[j], v1 = g + 8 < valid[j];
      x[j][0] = v0 ? x[j][0] : kNegInf;
      x[j][1] = v0 ? x[j][1] : kNegInf;
      x[j][2] = v1 ? x[j][2] : kNegInf;
      x[j][3] = v1 ? x[j][3] : kNegInf;
    }
  }
  // Lazy running maximum: the reference m only moves (with a full reduction
  // and a rescale of l and O) when a score exceeds it by more than
  // kMaxSlack; otherwise the weights 2^(x - m) stay below 2^kMaxSlack.
  float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
  for (int j = 1; j < NB; ++j) {
    mx0 = fmaxf(mx0, fmaxf(x[j][0], x[j][2]));
    mx1 = fmaxf(mx1, fmaxf(x[j][1], x[j][3]));
  }
  if (__any_sync(kFull, (mx0 > st.m0 + kMaxSlack) || (mx1 > st.m1 + kMaxSlack))) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
    }
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float al0 = (mn0 == kNegInf) ? 1.f : ex2(st.m0 - mn0);
    const float al1 = (mn1 == kNegInf) ? 1.f : ex2(st.m1 - mn1);
    st.l0 *= al0;
    st.l1 *= al1;
    if constexpr (ASYM) {
      st.z0 *= al0;
      st.z1 *= al1;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.O[i][0] *= al0;
      st.O[i][2] *= al0;
      st.O[i][1] *= al1;
      st.O[i][3] *= al1;
    }
    st.m0 = mn0;
    st.m1 = mn1;
  }
  if constexpr (!kBf16) {
    // the largest value scale of this call's tokens (empty slots of a partial
    // block are not data); a larger one than sigma allows lowers sigma
    float svm = 0.f;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const bool v0 = valid[j] >= kBlock || g < valid[j], v1 = valid[j] >= kBlock || g + 8 < valid[j];
      svm = fmaxf(svm, fmaxf(v0 ? sv[j][0] : 0.f, v1 ? sv[j][1] : 0.f));
    }
    if (__any_sync(kFull, svm > st.svlim)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) svm = fmaxf(svm, __shfl_xor_sync(kFull, svm, o));
      int e;
      frexpf(svm, &e);  // svm < 2^e
      const int sg_new = min(int(st.sg), kWeightExp - int(kMaxSlack) - e);
      const float f = ldexpf(1.f, sg_new - int(st.sg));  // exact power of two
      st.l0 *= f;
      st.l1 *= f;
      if constexpr (ASYM) {
        st.z0 *= f;
        st.z1 *= f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        st.O[i][0] *= f;
        st.O[i][1] *= f;
        st.O[i][2] *= f;
        st.O[i][3] *= f;
      }
      st.sg = float(sg_new);
      st.svlim = ldexpf(1.f, kWeightExp - int(kMaxSlack) - sg_new);
    }
  }
  const float base0 = (st.m0 == kNegInf) ? 0.f : st.m0 - st.sg;
  const float base1 = (st.m1 == kNegInf) ? 0.f : st.m1 - st.sg;
  const int src0 = 8 * t + (g >> 1), src1 = src0 + 4;
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const float p00 = ex2(x[j][0] - base0), p10 = ex2(x[j][2] - base0);
    const float p01 = ex2(x[j][1] - base1), p11 = ex2(x[j][3] - base1);
    st.l0 += p00 + p10;
    st.l1 += p01 + p11;
    uint32_t pk0, pk1, pk0lo = 0, pk1lo = 0;
    if constexpr (kBf16) {
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(p00, p10), h1 = __floats2bfloat162_rn(p01, p11);
      pk0 = *reinterpret_cast<const uint32_t*>(&h0);
      pk1 = *reinterpret_cast<const uint32_t*>(&h1);
      pk0lo = pack_bf162(p00 - __low2float(h0), p10 - __high2float(h0));
      pk1lo = pack_bf162(p01 - __low2float(h1), p11 - __high2float(h1));
    } else {
      // weights are at most 2^(kMaxSlack + sigma) and s_v <= svlim: p * s_v <= 2^kWeightExp
      float w00 = p00 * sv[j][0], w10 = p10 * sv[j][1], w01 = p01 * sv[j][0], w11 = p11 * sv[j][1];
      if (valid[j] < kBlock) {  // scales of empty slots of a partial block are not data
        const bool v0 = g < valid[j], v1 = g + 8 < valid[j];
        w00 = v0 ? w00 : 0.f;
        w01 = v0 ? w01 : 0.f;
        w10 = v1 ? w10 : 0.f;
        w11 = v1 ? w11 : 0.f;
        if constexpr (ASYM) {
          mv[j][0] = v0 ? mv[j][0] : 0.f;
          mv[j][1] = v1 ? mv[j][1] : 0.f;
        }
      }
      if constexpr (ASYM) {
        st.z0 = fmaf(p00, mv[j][0], fmaf(p10, mv[j][1], st.z0));
        st.z1 = fmaf(p01, mv[j][0], fmaf(p11, mv[j][1], st.z1));
      }
      pk0 = pack_half2(w00, w10);
      pk1 = pack_half2(w01, w11);
      if constexpr (LOQ) {  // two-part mode: the fp16 low parts w - hi (exact in fp32)
        const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&pk0));
        const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&pk1));
        pk0lo = pack_half2(w00 - h0.x, w10 - h0.y);
        pk1lo = pack_half2(w01 - h1.x, w11 - h1.y);
      }
    }
    // transpose the weights from the score accumulator layout (token rows,
    // query columns) into the B-operand layout of the value contraction
    const uint32_t r00 = __shfl_sync(kFull, pk0, src0), r01 = __shfl_sync(kFull, pk1, src0);
    const uint32_t r10 = __shfl_sync(kFull, pk0, src1), r11 = __shfl_sync(kFull, pk1, src1);
    const uint32_t b0 = (g & 1) ? r01 : r00, b1 = (g & 1) ? r11 : r10;
    uint32_t b0lo = 0, b1lo = 0;
    if constexpr (kBf16 || LOQ) {
      const uint32_t q00 = __shfl_sync(kFull, pk0lo, src0), q01 = __shfl_sync(kFull, pk1lo, src0);
      const uint32_t q10 = __shfl_sync(kFull, pk0lo, src1), q11 = __shfl_sync(kFull, pk1lo, src1);
      b0lo = (g & 1) ? q01 : q00;
      b1lo = (g & 1) ? q11 : q10;
    }
    value_block<VB, kBf16 || LOQ>(vb[j], b0, b1, b0lo, b1lo, st.O, lane, km);
  }
}

// Consumer warps write the query group of unit (b, h) into shared memory as
// B-operand rows: fp16 scaled by an exact power of two for code blocks (with
// the per-channel key factor applied), or the raw bf16 values for bf16 blocks.
template <bool kBf16Q>
__device__ __forceinline__ void stage_query(const DecodeArgs& a, int b, int h, uint16_t* qh, float* qs, int warp,
                                            int lane) {
  for (int q = warp; q < kMaxGroup; q += kConsumerWarps) {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (q < a.G) {
      const uint2 raw = *reinterpret_cast<const uint2*>(a.q + (size_t(b) * a.Hq + h * a.G + q) * kHeadDim + 4 * lane);
      x[0] = __uint_as_float(raw.x << 16);
      x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
      x[2] = __uint_as_float(raw.y << 16);
      x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    }
    uint2 packed;
    if constexpr (kBf16Q) {
      if (a.c.q_bits == 8) {
        // quantized query against bf16 window keys: q_int (exact in bf16) and
        // s_q in the score scale (no per-channel factor with a window here)
        float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
        float cq[4];
        const float sq = quantize_int8_row(x, am, cq);
        packed.x = pack_bf162(cq[0], cq[1]);
        packed.y = pack_bf162(cq[2], cq[3]);
        if (lane == 0) qs[q] = sq * (kLog2e * kInvSqrtD);
      } else {
        packed.x = pack_bf162(x[0], x[1]);
        packed.y = pack_bf162(x[2], x[3]);
        if (lane == 0) qs[q] = kLog2e * kInvSqrtD;
      }
    } else {
      if (a.c.factor) {
        const float4 c = *reinterpret_cast<const float4*>(a.c.factor + h * kHeadDim + 4 * lane);
        x[0] *= c.x;
        x[1] *= c.y;
        x[2] *= c.z;
        x[3] *= c.w;
      }
      float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
      int e = 0;
      if (am > 0.f) {
        int ex;
        frexpf(am, &ex);  // am = f * 2^ex, f in [0.5, 1)
        e = 15 - ex;      // am * 2^e in [2^14, 2^15)
      }
      packed.x = pack_half2(ldexpf(x[0], e), ldexpf(x[1], e));
      packed.y = pack_half2(ldexpf(x[2], e), ldexpf(x[3], e));
      if (lane == 0) qs[q] = ldexpf(kLog2e * kInvSqrtD, -e);
    }
    *reinterpret_cast<uint2*>(qh + q * kHeadDim + 4 * lane) = packed;
  }
}

__device__ __forceinline__ void load_query(const uint16_t* qh, const float* qs, uint32_t (&qf)[16], float& qs0,
                                           float& qs1, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint4* qp = reinterpret_cast<const uint4*>(qh + g * kHeadDim + 32 * t);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = qp[i];
    qf[4 * i] = v.x;
    qf[4 * i + 1] = v.y;
    qf[4 * i + 2] = v.z;
    qf[4 * i + 3] = v.w;
  }
  qs0 = qs[2 * t];
  qs1 = qs[2 * t + 1];
}

// Consumer warps start asynchronous copies of unit u's raw query rows (and of
// the per-channel key factor row) into prefetch buffer `buf`; one commit group.
__device__ __forceinline__ void prefetch_query(const DecodeArgs& a, int u, int buf, uint16_t* qraw, float* fraw,
                                               int warp, int lane) {
  const int H = a.c.H, b = u / H, h = u % H;
  uint16_t* raw = qraw + buf * kMaxGroup * kHeadDim;
  for (int q = warp; q < kMaxGroup; q += kConsumerWarps)
    if (q < a.G)
      cp_async8(raw + q * kHeadDim + 4 * lane, a.q + (size_t(b) * a.Hq + h * a.G + q) * kHeadDim + 4 * lane);
  if (a.c.factor && warp == 0) cp_async16(fraw + buf * kHeadDim + 4 * lane, a.c.factor + h * kHeadDim + 4 * lane);
  cp_async_commit();
}

// Next unit with data blocks in this CTA's virtual range [.., x1) after unit
// `cur`, or -1.
__device__ __forceinline__ int next_unit_in_range(const Geo& g, int cur, long long x1) {
  const int b = cur / g.H, h = cur % g.H;
  const long long vend = geo_vstart(g, b, h) + geo_vlen(g, b);
  if (vend >= x1) return -1;
  int b2, h2;
  locate_unit(g, vend, b2, h2);
  return (geo_vstart(g, b2, h2) + g.X < x1) ? b2 * g.H + h2 : -1;
}

// Shared scratch used by the combine and the merge.
struct Scratch {
  float* merge_o;  // [4 warps][4][128]
  float* merge_m;  // [4][8]
  float* merge_l;  // [4][8]
  int* misc;
  uint64_t* cbar;
};

// The query rows of prefetch buffer `buf` as B-operand rows in shared memory
// (fp16 scaled by a power of two, int8 codes, or raw bf16; plus the low parts
// of the two-part query and the row sums of the asymmetric format).  Out of
// line: it runs once per unit and keeps its rarely used branches out of the
// consumers' block loop.
template <bool kBf16Q, bool ASYM>
__device__ __noinline__ void write_query_rows(const DecodeArgs& a, int buf, const uint16_t* qraw, const float* fraw,
                                              uint16_t* qh, uint32_t* qlo, float* qs, int warp, int lane) {
  const uint16_t* raw = qraw + buf * kMaxGroup * kHeadDim;
  for (int q = warp; q < kMaxGroup; q += kConsumerWarps) {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (q < a.G) {
      const uint2 r = *reinterpret_cast<const uint2*>(raw + q * kHeadDim + 4 * lane);
      x[0] = __uint_as_float(r.x << 16);
      x[1] = __uint_as_float(r.x & 0xFFFF0000u);
      x[2] = __uint_as_float(r.y << 16);
      x[3] = __uint_as_float(r.y & 0xFFFF0000u);
    }
    uint2 packed;
    if constexpr (kBf16Q) {
      packed.x = pack_bf162(x[0], x[1]);
      packed.y = pack_bf162(x[2], x[3]);
      if (lane == 0) qs[q] = kLog2e * kInvSqrtD;
    } else {
      if (a.c.factor) {
        const float4 c = *reinterpret_cast<const float4*>(fraw + buf * kHeadDim + 4 * lane);
        x[0] *= c.x;
        x[1] *= c.y;
        x[2] *= c.z;
        x[3] *= c.w;
      }
      float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
      if (a.c.q_bits == 8) {
        // quantized query: int8 codes (exact in fp16) and s_q folded into the
        // score scale; the MMA then forms the integer dot exactly
        float cq[4];
        const float sq = quantize_int8_row(x, am, cq);
        packed.x = pack_half2(cq[0], cq[1]);
        packed.y = pack_half2(cq[2], cq[3]);
        if (lane == 0) qs[q] = sq * (kLog2e * kInvSqrtD);
      } else {
        int e = 0;
        if (am > 0.f) {
          int ex;
          frexpf(am, &ex);  // am = f * 2^ex, f in [0.5, 1)
          e = 15 - ex;      // am * 2^e in [2^14, 2^15)
        }
        const float y0 = ldexpf(x[0], e), y1 = ldexpf(x[1], e), y2 = ldexpf(x[2], e), y3 = ldexpf(x[3], e);
        packed.x = pack_half2(y0, y1);
        packed.y = pack_half2(y2, y3);
        if (lane == 0) qs[q] = ldexpf(kLog2e * kInvSqrtD, -e);
        if (a.c.q_bits == 32) {
          // two-part query: low parts y - hi (exact in fp32), stored in fragment
          // order: lane 4q + t holds dims 32t + 8i + 2k, +1 of row q in uint32
          // (i * 32 + lane) * 4 + k
          const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&packed.x));
          const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&packed.y));
          uint2 lo;
          lo.x = pack_half2(y0 - h0.x, y1 - h0.y);
          lo.y = pack_half2(y2 - h1.x, y3 - h1.y);
          const int ft = lane >> 3, fi = (lane & 7) >> 1, fk = 2 * (lane & 1);
          *reinterpret_cast<uint2*>(qlo + (fi * 32 + 4 * q + ft) * 4 + fk) = lo;
        }
      }
      {
        // offset terms of the key codes (score_block with OFF): minus 1152
        // times the sums of the row as the MMA sees it over the even and the
        // odd k-slices (dims with bit 2 clear or set; this lane's four dims
        // share it), stored as float4 {even 2t, even 2t+1, odd 2t, odd 2t+1}
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&packed.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&packed.y));
        float zs = (f0.x + f0.y) + (f1.x + f1.y);
#pragma unroll
        for (int o = 16; o > 1; o >>= 1) zs += __shfl_xor_sync(kFull, zs, o);
        if (lane < 2) qs[2 * kMaxGroup + (q >> 1) * 4 + 2 * lane + (q & 1)] = -kOffsetF16 * zs;
      }
      if constexpr (ASYM) {
        // sum of the fp16 row exactly as the MMA sees it (zero-point term)
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&packed.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&packed.y));
        float z = (f0.x + f0.y) + (f1.x + f1.y);
        if (a.c.q_bits == 32) {  // plus the low parts
          const uint2 lw = *reinterpret_cast<const uint2*>(
              qlo + (((lane & 7) >> 1) * 32 + 4 * q + (lane >> 3)) * 4 + 2 * (lane & 1));
          const float2 l0 = __half22float2(*reinterpret_cast<const __half2*>(&lw.x));
          const float2 l1 = __half22float2(*reinterpret_cast<const __half2*>(&lw.y));
          z += (l0.x + l0.y) + (l1.x + l1.y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(kFull, z, o);
        if (lane == 0) qs[kMaxGroup + q] = z;
      }
    }
    *reinterpret_cast<uint2*>(qh + q * kHeadDim + 4 * lane) = packed;
  }
}

// Once the copies of prefetch buffer `buf` have landed (every consumer thread
// has waited on its cp.async groups), turn the raw rows into B-operand rows
// and load this thread's fragments.
template <bool kBf16Q, bool ASYM>
__device__ __forceinline__ bool convert_query(const DecodeArgs& a, int buf, const uint16_t* qraw, const float* fraw,
                                              uint16_t* qh, uint32_t* qlo, float* qs, const Scratch& sc,
                                              uint32_t& cphase, int warp, int lane, uint32_t (&qf)[16], float& qs0,
                                              float& qs1, float& qz0, float& qz1) {
  if (!consumer_sync(sc.cbar, cphase)) return false;  // the factor row was copied by warp 0
  write_query_rows<kBf16Q, ASYM>(a, buf, qraw, fraw, qh, qlo, qs, warp, lane);
  if (!consumer_sync(sc.cbar, cphase)) return false;
  load_query(qh, qs, qf, qs0, qs1, lane);
  if constexpr (ASYM) {
    const int t = lane & 3;
    qz0 = qs[kMaxGroup + 2 * t];
    qz1 = qs[kMaxGroup + 2 * t + 1];
  }
  return true;
}

// Log-sum-exp merge of every partial record of unit u, run by the consumer
// threads of the last CTA to finish the unit.  Thread f owns float4 f of the
// G x 128 output and merges it on its own, without block synchronisation: the
// (m, l, o) of eight records are loaded at once, then folded into a running
// (M, l, o) with the usual rescaling by 2^(M_old - M_new).
__device__ __noinline__ void merge_unit(const DecodeArgs& a, int u, long long c0, long long c1, bool has_win, int P,
                                        int tid) {
  constexpr int kR = 8;  // records in flight per thread
  const int G = a.G, H = a.c.H;
  const int b = u / H, h = u % H;
  const int ns = c1 >= c0 ? int(c1 - c0 + 1) : 0;
  const int ntot = ns + (has_win ? 1 : 0);
  const size_t wslot = size_t(P) + a.lay.units + u;
  const float* pm = reinterpret_cast<const float*>(a.ws + a.lay.off_m);
  const float* pl = reinterpret_cast<const float*>(a.ws + a.lay.off_l);
  const float* po = reinterpret_cast<const float*>(a.ws + a.lay.off_o);
  const int nf = G * (kHeadDim / 4);
  for (int f = tid; f < nf; f += kConsumers) {
    const int q = f >> 5, d4 = f & 31;
    float M = kNegInf, l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < ntot; base += kR) {
      const int cnt = min(kR, ntot - base);
      float mr[kR], lr[kR];
      float4 orr[kR];
#pragma unroll
      for (int j = 0; j < kR; ++j) {
        if (j < cnt) {
          const int r = base + j;
          const size_t slot = r < ns ? size_t(c0 + r + u) : wslot;
          mr[j] = __ldcg(pm + slot * G + q);
          lr[j] = __ldcg(pl + slot * G + q);
          orr[j] = __ldcg(reinterpret_cast<const float4*>(po + (slot * G + q) * kHeadDim) + d4);
        } else {
          mr[j] = kNegInf;
          lr[j] = 0.f;
          orr[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mn = M;
#pragma unroll
      for (int j = 0; j < kR; ++j) Mn = fmaxf(Mn, mr[j]);
      const float rs = (M == kNegInf) ? 0.f : exp2f(M - Mn);
      l *= rs;
      o.x *= rs;
      o.y *= rs;
      o.z *= rs;
      o.w *= rs;
#pragma unroll
      for (int j = 0; j < kR; ++j) {
        const float w = (mr[j] == kNegInf) ? 0.f : exp2f(mr[j] - Mn);
        l = fmaf(w, lr[j], l);
        o.x = fmaf(w, orr[j].x, o.x);
        o.y = fmaf(w, orr[j].y, o.y);
        o.z = fmaf(w, orr[j].z, o.z);
        o.w = fmaf(w, orr[j].w, o.w);
      }
      M = Mn;
    }
    const float inv = 1.f / l;
    const size_t idx = (size_t(b) * a.Hq + h * G + q) * kHeadDim + 4 * d4;
    if (a.out_fp32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx) =
          make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    } else {
      uint2 pk;
      pk.x = pack_bf162(o.x * inv, o.y * inv);
      pk.y = pack_bf162(o.z * inv, o.w * inv);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + idx) = pk;
    }
    if (d4 == 0 && a.lse) a.lse[size_t(b) * a.Hq + h * G + q] = (M + log2f(l)) * kLn2;
  }
}

// Combine the four consumer warps' states of unit u and emit them: the final
// output if this is the unit's only record, else a partial record in `slot`
// followed by the arrival ticket; the last CTA to arrive merges the unit.
template <bool ASYM>
__device__ __forceinline__ bool finish_segment(const DecodeArgs& a, WarpState& st, int u, size_t slot, const int* len_s,
                                              const Geo& geo, long long Tv, int Pe, int P, const Scratch& sc,
                                              uint32_t& cphase, int warp, int lane, int tid) {
  const int g = lane >> 2, t = lane & 3;
  const int G = a.G, H = a.c.H;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    st.l0 += __shfl_xor_sync(kFull, st.l0, o);
    st.l1 += __shfl_xor_sync(kFull, st.l1, o);
  }
  if constexpr (ASYM) {
    // the value zero-point term is the same for every output dimension
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      st.z0 += __shfl_xor_sync(kFull, st.z0, o);
      st.z1 += __shfl_xor_sync(kFull, st.z1, o);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.O[i][0] += st.z0;
      st.O[i][2] += st.z0;
      st.O[i][1] += st.z1;
      st.O[i][3] += st.z1;
    }
  }
  if (g == 0) {
    // the exponent base of l and O (m - sigma; -inf stays -inf)
    sc.merge_m[warp * kMaxGroup + 2 * t] = st.m0 - st.sg;
    sc.merge_m[warp * kMaxGroup + 2 * t + 1] = st.m1 - st.sg;
    sc.merge_l[warp * kMaxGroup + 2 * t] = st.l0;
    sc.merge_l[warp * kMaxGroup + 2 * t + 1] = st.l1;
  }
  long long c0, c1;
  int nseg;
  bool has_win;
  unit_segments(a, len_s, geo, u, Tv, Pe, c0, c1, nseg, has_win);
  const int b = u / H, h = u % H;
  float* pm = reinterpret_cast<float*>(a.ws + a.lay.off_m);
  float* pl = reinterpret_cast<float*>(a.ws + a.lay.off_l);
  float* po = reinterpret_cast<float*>(a.ws + a.lay.off_o);
  const int d = tid;
  // combine the warps' O through shared memory, four queries per pass
  for (int pass = 0; pass * 4 < G; ++pass) {
    if (pass > 0 && !consumer_sync(sc.cbar, cphase)) return false;  // previous pass has read merge_o
    if ((t >> 1) == pass) {
      float* ow = sc.merge_o + warp * 4 * kHeadDim;
      const int q0 = 2 * t - 4 * pass;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        ow[q0 * kHeadDim + 16 * mt + g] = st.O[mt][0];
        ow[(q0 + 1) * kHeadDim + 16 * mt + g] = st.O[mt][1];
        ow[q0 * kHeadDim + 16 * mt + g + 8] = st.O[mt][2];
        ow[(q0 + 1) * kHeadDim + 16 * mt + g + 8] = st.O[mt][3];
      }
    }
    if (!consumer_sync(sc.cbar, cphase)) return false;
    for (int q = 4 * pass; q < min(G, 4 * pass + 4); ++q) {
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sc.merge_m[w * kMaxGroup + q]);
      float l = 0.f, o = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = sc.merge_m[w * kMaxGroup + q];
        const float al = (mw == kNegInf) ? 0.f : exp2f(mw - M);
        l += al * sc.merge_l[w * kMaxGroup + q];
        o += al * sc.merge_o[(w * 4 + (q - 4 * pass)) * kHeadDim + d];
      }
      if (nseg == 1) {
        write_out(a, b, h * G + q, d, o, l, M);
      } else {
        po[(slot * G + q) * kHeadDim + d] = o;
        if (d == 0) {
          pm[slot * G + q] = M;
          pl[slot * G + q] = l;
        }
      }
    }
  }
  if (nseg > 1) {
    // The block barrier (release/acquire at CTA scope) orders every thread's
    // record stores before thread 0; its acquire-release atomic at GPU scope
    // publishes them with the ticket and, for the last CTA to arrive, makes
    // the other CTAs' records visible; the next block barrier extends that to
    // all threads of this CTA.
    if (!consumer_sync(sc.cbar, cphase)) return false;
    if (tid == 0) {
      int* cnt = reinterpret_cast<int*>(a.ws + a.lay.off_counter);
      int tk;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(tk) : "l"(cnt + u) : "memory");
      sc.misc[0] = (tk == nseg - 1);
    }
    if (!consumer_sync(sc.cbar, cphase)) return false;
    if (sc.misc[0]) {
      merge_unit(a, u, c0, c1, has_win, P, tid);
      if (tid == 0) reinterpret_cast<int*>(a.ws + a.lay.off_counter)[u] = 0;
    }
  }
  // merge_o / misc are written again only after the next query staging sync
  return true;
}

// Clamped lengths and the two block prefix sums of every sequence, in shared
// memory (all threads; ends with a block barrier).  `load` reads a length.
// Returns (in every thread) whether a length was negative or beyond the
// table's capacity; the caller reports it.
template <typename LoadLen>
__device__ __forceinline__ bool scan_geometry(const DecodeArgs& a, int B, int W, int X, int* len_s, int* pre_s,
                                              int* vpre_s, LoadLen load, int tid, int warp, int lane) {
  const int cap = a.mbps * kBlock;
  int bad = 0;
  for (int b = tid; b < B; b += kThreads) {
    int L = load(b);
    if (L < 0) {
      bad = 1;
      L = 0;
    }
    int Lq = W > 0 ? max(L - W, 0) : L;
    if (Lq > cap) {
      bad = 1;
      Lq = cap;
      L = W > 0 ? cap + W : cap;
    }
    len_s[b] = L;
    const int nb = (Lq + kBlock - 1) / kBlock;
    pre_s[b + 1] = nb;                    // block count, scanned below
    vpre_s[b + 1] = nb > 0 ? nb + X : 0;  // virtual blocks: start cost + data
  }
  if (tid == 0) {
    pre_s[0] = 0;
    vpre_s[0] = 0;
  }
  __syncthreads();
  if (warp < 2) {  // warp 0 scans the data blocks, warp 1 the virtual blocks
    int* arr = warp == 0 ? pre_s : vpre_s;
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int i = base + lane;
      int v = i < B ? arr[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
      }
      if (i < B) arr[i + 1] = v + carry;
      carry += __shfl_sync(kFull, v, 31);
    }
  }
  return __syncthreads_or(bad) != 0;
}

// LOQ: the two-part mode (q_bits 32) of code blocks: the query and the value
// weights p * s_v each carried as fp16 high + low parts.
template <int KB, int VB, bool ASYM, bool LOQ>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(const Params prm) {
  using F = Fmt<KB, VB, ASYM>;
  constexpr int S = F::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  const DecodeArgs& a = prm.a;
  const int P = prm.P, Uw = prm.Uw;
  const int H = a.c.H, G = a.G, B = a.B;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SmemMap mp = smem_map(S * F::kStageBytes, S, B, LOQ, a.pos != nullptr);
  Scratch sc;
  sc.merge_o = reinterpret_cast<float*>(smem + mp.merge_o);
  sc.merge_m = reinterpret_cast<float*>(smem + mp.merge_ml);
  sc.merge_l = sc.merge_m + kConsumerWarps * kMaxGroup;
  uint16_t* qh = reinterpret_cast<uint16_t*>(smem + mp.qh);
  uint32_t* qlo_s = reinterpret_cast<uint32_t*>(smem + mp.qlo);
  float* qs = reinterpret_cast<float*>(smem + mp.qs);
  uint16_t* qraw = reinterpret_cast<uint16_t*>(smem + mp.qraw);
  float* fraw = reinterpret_cast<float*>(smem + mp.fraw);
  int4* hdr = reinterpret_cast<int4*>(smem + mp.hdr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + mp.bars);
  uint64_t* empty = full + S;
  sc.cbar = empty + S;
  sc.misc = reinterpret_cast<int*>(smem + mp.misc);
  int* len_s = reinterpret_cast<int*>(smem + mp.len);
  int* pre_s = reinterpret_cast<int*>(smem + mp.pre);
  int* vpre_s = reinterpret_cast<int*>(smem + mp.vpre);
  int* rows_s = reinterpret_cast<int*>(smem + mp.rows);  // prefill: each row's sequence
  const int X = a.lay.switch_blocks;

  const int W = a.c.window;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(sc.cbar, kConsumers);
    sc.misc[0] = 0;
    fence_mbar_init();
  }
  if constexpr (!F::kBf16) {
    // keys with per-channel scales only have no per-token key scale: the
    // producer never copies into the key-scale slots of the ring, which keep 1.0
    if (a.c.k_chan)
      for (int i = tid; i < S * F::kBlocksPerStage * kBlock; i += kThreads) {
        const int st = i / (F::kBlocksPerStage * kBlock), r = i % (F::kBlocksPerStage * kBlock);
        reinterpret_cast<float*>(smem + st * F::kStageBytes + F::kOffMeta)[(r / kBlock) * F::kMF + F::kKS +
                                                                           r % kBlock] = 1.f;
      }
  }
  // Programmatic dependent launch: this grid may start while the previous
  // kernel on the stream is still finishing.  Let the next kernel launch
  // early in turn, then wait until the previous kernel has completed (its
  // writes visible) before reading memory it may write.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  auto load_len = [&](int b) {
    if (!a.pos) return a.seq_lens[b];
    // prefill: row b is position pos[b] of sequence seq_of[b] and attends to 0..pos[b]
    const int sb = a.seq_of[b];
    if (sb < 0 || sb >= a.nseq) {
      if (blockIdx.x == 0) flag(a.err, KVQ_DEVERR_POSITION);
      rows_s[b] = 0;
      return 0;
    }
    rows_s[b] = sb;
    return a.pos[b] + 1;
  };
  const Geo geo{pre_s, vpre_s, B, H, X};
  // Decode whose lengths and block table the caller declares final before the
  // previous kernel ends: scan the geometry while that kernel finishes (an
  // error found here is reported after the wait).  Reading the producer's
  // first block-table entries ahead as well measured slower (register
  // pressure in the block loop), so the table is read after the wait.
  bool len_bad = false;
  if (a.ahead) len_bad = scan_geometry(a, B, W, X, len_s, pre_s, vpre_s, load_len, tid, warp, lane);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- sequence geometry: clamped lengths and block prefix sums
  if (!a.ahead) len_bad = scan_geometry(a, B, W, X, len_s, pre_s, vpre_s, load_len, tid, warp, lane);
  if (len_bad && blockIdx.x == 0 && tid == 0) flag(a.err, KVQ_DEVERR_SEQ_LEN);
  const long long T = (long long)H * vpre_s[B];  // virtual blocks in total
  const int U = B * H;
  // Effective stream split: never more CTAs than blocks / kMinBlocksPerCta, so
  // every CTA below Pe owns blocks and a unit's owners are exactly c0..c1.
  const long long cap_ctas = (T + kMinBlocksPerCta - 1) / kMinBlocksPerCta;
  const int Pe = int(cap_ctas < (long long)P ? cap_ctas : (long long)P);
  uint32_t cphase = 0;

  // ==================================================================== window CTAs
  if ((int)blockIdx.x < Uw) {
    const int u = blockIdx.x;
    const int b = u / H, h = u % H;
    const int L = len_s[b];
    if (L <= 0 || warp >= kConsumerWarps) return;  // the producer warp has no role here
    const int nw = min(L, W);
    const int nwb = (nw + kBlock - 1) / kBlock;
    stage_query<true>(a, b, h, qh, qs, warp, lane);
    if (!consumer_sync(sc.cbar, cphase)) { flag(a.err, KVQ_DEVERR_TIMEOUT); return; }
    uint32_t qf[16];
    float qs0, qs1;
    load_query(qh, qs, qf, qs0, qs1, lane);
    WarpState st;
    st.reset();
    const size_t ring0 = size_t(u) * (W / kBlock);
    for (int j = warp; j < nwb; j += kConsumerWarps) {
      const uint8_t* kb = a.c.k_win + (ring0 + j) * block_bytes(16);
      const uint8_t* vb = a.c.v_win + (ring0 + j) * block_bytes(16);
      const uint8_t* const kbs[1] = {kb};
      const uint8_t* const vbs[1] = {vb};
      const float* const nos[1] = {nullptr};
      const int val[1] = {min(kBlock, nw - j * kBlock)};
      process_blocks<16, 16, 1, false, false>(kbs, vbs, nos, nos, nos, nos, val, qf, nullptr, nullptr, qs0, qs1, 0.f, 0.f, st, lane,
                                       0u);
    }
    const size_t slot = size_t(P) + U + u;
    if (!finish_segment<false>(a, st, u, slot, len_s, geo, T, Pe, P, sc, cphase, warp, lane, tid))
      flag(a.err, KVQ_DEVERR_TIMEOUT);
    return;
  }

  // ==================================================================== stream CTAs
  const int ci = blockIdx.x - Uw;  // stream CTA index
  // units with no tokens at all: out = 0, lse = -inf
  for (int u = ci; u < U; u += P) {
    const int b = u / H, h = u % H;
    if (len_s[b] != 0) continue;
    for (int e = tid; e < G * kHeadDim; e += kThreads) {
      const int q = e / kHeadDim, d = e % kHeadDim;
      const size_t idx = (size_t(b) * a.Hq + h * G + q) * kHeadDim + d;
      if (a.out_fp32) reinterpret_cast<float*>(a.out)[idx] = 0.f;
      else reinterpret_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(0.f);
      if (d == 0 && a.lse) a.lse[size_t(b) * a.Hq + h * G + q] = kNegInf;
    }
  }
  if (ci >= Pe) return;
  const long long x0 = (long long)ci * T / Pe;
  const long long x1 = (long long)(ci + 1) * T / Pe;
  if (x0 >= x1) return;
  int b_first, h_first;
  locate_unit(geo, x0, b_first, h_first);
  const long long xs = max(x0, geo_vstart(geo, b_first, h_first) + X);  // first data block of the range
  if (xs >= x1) return;  // the range holds only unit-start cost: no data, no record

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer warp
    const uint64_t pol = l2_evict_first_policy();
    int b = b_first, h = h_first;
    int nblk = geo_nblk(geo, b);
    long long dstart = geo_vstart(geo, b, h) + X;  // virtual index of the unit's first data block
    long long x = xs;
    int it = 0, s = 0;
    uint32_t ph = 0;  // stage index and the parity of its current use
    bool ok = true;
    // 32 block-table entries of sequence tc_b, logical blocks tc_base + lane
    int tc_b = -1, tc_base = 0, tc_val = 0;
    while (x < x1) {
      if (x >= dstart + nblk) {  // next unit: skip its start cost
        ++h;
        if (h == H) {
          h = 0;
          do { ++b; } while (geo_vlen(geo, b) == 0);
          nblk = geo_nblk(geo, b);
        }
        dstart = geo_vstart(geo, b, h) + X;
        x = max(x, dstart);
        if (x >= x1) break;
      }
      const long long rem = (x1 - x) < (dstart + nblk - x) ? (x1 - x) : (dstart + nblk - x);
      const int n = int(rem < F::kBlocksPerStage ? rem : F::kBlocksPerStage);
      const int local = int(x - dstart);
      if (tc_b != b || local < tc_base || local + n > tc_base + 32) {
        tc_b = b;
        tc_base = local;
        const int idx = local + lane;
        int v = 0;
        if (idx < nblk) {
          v = a.table[size_t(a.pos ? rows_s[b] : b) * a.mbps + idx];
          if (v < 0 || v >= a.c.num_blocks) {
            flag(a.err, KVQ_DEVERR_BLOCK_ID);
            v = 0;
          }
        }
        tc_val = v;
      }
      if (it >= S) {
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(&empty[s], ph ^ 1u);
        if (!__shfl_sync(kFull, w_ok ? 1 : 0, 0)) {
          if (lane == 0) flag(a.err, KVQ_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
      }
      // physical ids of the stage's blocks on every lane; a lane whose block
      // starts a run of consecutive ids issues one copy for the whole run
      const int phys = __shfl_sync(kFull, tc_val, (local - tc_base) + min(lane, n - 1));
      const int prev = __shfl_up_sync(kFull, phys, 1);
      const bool start = lane < n && (lane == 0 || prev + 1 != phys);
      int run = 1;
      bool contig = true;
#pragma unroll
      for (int j = 1; j < F::kBlocksPerStage; ++j) {
        const int nx = __shfl_down_sync(kFull, phys, j);
        contig = contig && (lane + j < n) && (nx == phys + j);
        run += contig ? 1 : 0;
      }
      if (lane == 0) {
        hdr[s] = make_int4(b * H + h, local, n, 0);
        // per-channel key scales only: the value half of each record, not the key scales
        mbar_arrive_expect_tx(&full[s], uint32_t(n * (a.c.k_chan ? F::kPerBlock - F::kMB / 2 : F::kPerBlock)));
      }
      __syncwarp();
      if (start) {
        uint8_t* st = smem + s * F::kStageBytes;
        const size_t hb = size_t(h) * a.c.num_blocks + phys;  // head-major pools
        bulk_g2s(st + F::kOffK + lane * F::kKBB, a.c.k_codes + hb * F::kKBB, run * F::kKBB, &full[s], pol);
        bulk_g2s(st + F::kOffV + lane * F::kVBB, a.c.v_codes + hb * F::kVBB, run * F::kVBB, &full[s], pol);
        if constexpr (!F::kBf16) {
          if (!a.c.k_chan)  // the run's metadata records: one contiguous copy
            bulk_g2s(st + F::kOffMeta + lane * F::kMB, a.c.meta + hb * F::kMF, run * F::kMB, &full[s], pol);
        }
      }
      if constexpr (!F::kBf16) {
        if (a.c.k_chan && lane < n) {  // per-channel keys: each block's value half alone
          uint8_t* st = smem + s * F::kStageBytes;
          const size_t hb = size_t(h) * a.c.num_blocks + phys;
          bulk_g2s(st + F::kOffMeta + lane * F::kMB + F::kVS * 4, a.c.meta + hb * F::kMF + F::kVS, F::kMB / 2,
                   &full[s], pol);
        }
      }
      x += n;
      ++it;
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
      if (it == 1 && x < x1 && x1 - x0 <= kFirstStageFirstMax) {
        // A short range: this stage's copies land before the next ones are
        // issued, so every CTA's first stage is ahead of anyone's second in
        // the memory queues and all consumers start early (timing only).
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(&full[0], 0u);
        if (!__shfl_sync(kFull, w_ok ? 1 : 0, 0)) {
          if (lane == 0) flag(a.err, KVQ_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    if (lane != 0) return;
    if (ok) {  // terminator stage
      if (it >= S && !mbar_wait(&empty[s], ph ^ 1u)) {
        flag(a.err, KVQ_DEVERR_TIMEOUT);
      } else {
        hdr[s] = make_int4(-1, 0, 0, 0);
        mbar_arrive(&full[s]);
        ++it;
      }
    }
    // drain: the most recent use of every stage must have landed before exit
    for (int k = max(0, it - S); k < it; ++k)
      if (!mbar_wait(&full[k % S], (k / S) & 1)) flag(a.err, KVQ_DEVERR_TIMEOUT);
    return;
  }

  // -------------------------------------------------------------- consumer warps
  const uint32_t km = magic_f16x2(a.B);  // the int4 conversion's fp16 magic, in a register
  WarpState st;
  st.reset();
  uint32_t qf[16];
  float qs0 = 0.f, qs1 = 0.f, qz0 = 0.f, qz1 = 0.f;
  int cur, cur_lq, qbuf = 0, nxt;
  {
    // the first unit is known from x0: fetch its query group (and the next
    // unit's) while the first stage is still in flight
    const int b0 = b_first, h0 = h_first;
    cur = b0 * H + h0;
    cur_lq = W > 0 ? max(len_s[b0] - W, 0) : len_s[b0];
    prefetch_query(a, cur, 0, qraw, fraw, warp, lane);
    nxt = next_unit_in_range(geo, cur, x1);
    if (nxt >= 0) {
      prefetch_query(a, nxt, 1, qraw, fraw, warp, lane);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    if (!convert_query<F::kBf16, ASYM>(a, 0, qraw, fraw, qh, qlo_s, qs, sc, cphase, warp, lane, qf, qs0, qs1, qz0, qz1)) {
      flag(a.err, KVQ_DEVERR_TIMEOUT);
      return;
    }
  }
  // offset terms of the key codes (score_block with OFF), one float4 per t
  const float4* qzo = reinterpret_cast<const float4*>(qs + 2 * kMaxGroup);
  // low query parts of code blocks (only for the two-part fp16 query, q_bits = 32)
  const uint4* qlo = LOQ ? reinterpret_cast<const uint4*>(qlo_s) + lane : nullptr;
  int s = 0;
  uint32_t ph = 0;  // stage index and the parity of its current use
  for (;;) {
    if (!mbar_wait(&full[s], ph)) {
      flag(a.err, KVQ_DEVERR_TIMEOUT);
      return;
    }
    const int4 hd = hdr[s];
    if (hd.x != cur) {
      if (cur >= 0 &&
          !finish_segment<ASYM>(a, st, cur, size_t(ci) + cur, len_s, geo, T, Pe, P, sc, cphase, warp, lane, tid)) {
        flag(a.err, KVQ_DEVERR_TIMEOUT);
        return;
      }
      if (hd.x < 0) break;  // terminator
      if (hd.x != nxt) {  // not the predicted next unit: fetch its query group now
        cp_async_wait<0>();
        prefetch_query(a, hd.x, qbuf ^ 1, qraw, fraw, warp, lane);
      }
      cur = hd.x;
      qbuf ^= 1;
      const int cb = cur / H;
      cur_lq = W > 0 ? max(len_s[cb] - W, 0) : len_s[cb];
      cp_async_wait<0>();
      if (!convert_query<F::kBf16, ASYM>(a, qbuf, qraw, fraw, qh, qlo_s, qs, sc, cphase, warp, lane, qf, qs0, qs1, qz0,
                                      qz1)) {
        flag(a.err, KVQ_DEVERR_TIMEOUT);
        return;
      }
      nxt = next_unit_in_range(geo, cur, x1);
      if (nxt >= 0) prefetch_query(a, nxt, qbuf ^ 1, qraw, fraw, warp, lane);
      st.reset();
    }
    if (warp < hd.z) {
      const uint8_t* stg = smem + s * F::kStageBytes;
      auto kp = [&](int j) { return stg + F::kOffK + j * F::kKBB; };
      auto vp = [&](int j) { return stg + F::kOffV + j * F::kVBB; };
      auto meta = [&](int j) { return reinterpret_cast<const float*>(stg + F::kOffMeta + j * F::kMB); };
      auto ksp = [&](int j) { return F::kBf16 ? nullptr : meta(j) + F::kKS; };
      auto vsp = [&](int j) {
        return F::kBf16 ? nullptr : meta(j) + F::kVS;
      };
      auto kop = [&](int j) { return ASYM ? meta(j) + F::kKO : nullptr; };
      auto vop = [&](int j) { return ASYM ? meta(j) + F::kVO : nullptr; };
      auto val = [&](int j) { return min(kBlock, cur_lq - (hd.y + j) * kBlock); };
      const int j0 = warp, j1 = warp + kConsumerWarps;
      if (F::kBPW == 2 && j1 < hd.z) {
        const uint8_t* const kbs[2] = {kp(j0), kp(j1)};
        const uint8_t* const vbs[2] = {vp(j0), vp(j1)};
        const float* const kss[2] = {ksp(j0), ksp(j1)};
        const float* const vss[2] = {vsp(j0), vsp(j1)};
        const float* const kos[2] = {kop(j0), kop(j1)};
        const float* const vos[2] = {vop(j0), vop(j1)};
        const int vals[2] = {val(j0), val(j1)};
        process_blocks<KB, VB, 2, ASYM, LOQ>(kbs, vbs, kss, vss, kos, vos, vals, qf, qlo, qzo, qs0, qs1, qz0, qz1, st, lane,
                                        km);
      } else {
        const uint8_t* const kbs[1] = {kp(j0)};
        const uint8_t* const vbs[1] = {vp(j0)};
        const float* const kss[1] = {ksp(j0)};
        const float* const vss[1] = {vsp(j0)};
        const float* const kos[1] = {kop(j0)};
        const float* const vos[1] = {vop(j0)};
        const int vals[1] = {val(j0)};
        process_blocks<KB, VB, 1, ASYM, LOQ>(kbs, vbs, kss, vss, kos, vos, vals, qf, qlo, qzo, qs0, qs1, qz0, qz1, st, lane,
                                        km);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

// ------------------------------------------------------------------ host side
template <int KB, int VB, bool ASYM, bool LOQ>
struct Kernel {
  using F = Fmt<KB, VB, ASYM>;
  static int smem_bytes(int B, bool rows) {
    return smem_map(F::kStages * F::kStageBytes, F::kStages, B, LOQ, rows).total;
  }
  // Allow the largest opt-in dynamic shared memory once per device; the
  // per-launch size (which depends on the batch) then always fits.
  static void ensure_attribute(int dev) {
    static std::mutex mu;
    static std::map<int, bool> done;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return;
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncSetAttribute(decode_kernel<KB, VB, ASYM, LOQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    // Ask for the largest shared-memory carveout: the occupancy used to size
    // the single wave assumes it, and a smaller split (chosen by default)
    // would fit one CTA fewer per SM and turn the wave into 1.5 waves.
    cudaFuncSetAttribute(decode_kernel<KB, VB, ASYM, LOQ>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    done[dev] = true;
  }
  static int ctas_per_sm(int B, bool rows) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    ensure_attribute(dev);
    const int smem = smem_bytes(B, rows);
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(dev, smem);
    auto itc = cache.find(key);
    if (itc != cache.end()) return itc->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<KB, VB, ASYM, LOQ>, kThreads, smem) != cudaSuccess)
      n = 1;
    n = n < 1 ? 1 : n;
    cache[key] = n;
    return n;
  }
  static cudaError_t launch(const DecodeArgs& a, cudaStream_t s) {
    const int smem = smem_bytes(a.B, a.pos != nullptr);
    int dev = 0;
    cudaGetDevice(&dev);
    ensure_attribute(dev);
    Params p{a, a.lay.stream_ctas, a.lay.window_ctas};
    const int grid = a.lay.window_ctas + a.lay.stream_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<KB, VB, ASYM, LOQ>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
};

}  // namespace
}  // namespace kvq
