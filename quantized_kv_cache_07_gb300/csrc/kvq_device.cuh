// Device-side building blocks shared by the kvq kernels (sm_103a).
//   - fragment-native cache layout offsets (see include/kvq.h for the spec)
//   - exact integer-code -> fp16 conversions done in registers
//   - mbarrier / bulk-copy (TMA, non-tensor) wrappers with bounded waits
//   - warp-level mma.sync wrappers
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kBlock = 16;
// Wall-clock limit of any device-side wait (ns).  A decode step takes well
// under a millisecond; reaching this means the pipeline protocol broke.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__host__ __device__ constexpr int block_bytes(int bits) { return kBlock * kHeadDim * bits / 8; }

// ------------------------------------------------------------------ layout
// Byte offset (and nibble shift for 4-bit codes) of key element (token i, dim d)
// inside one 16-token block of one head.
struct Loc {
  int byte;
  int shift;  // 0 or 4 for nibbles, 0 otherwise
};

__host__ __device__ inline Loc key_loc(int bits, int i, int d) {
  const int g = i & 7, hi = i >> 3, t = d >> 5, e = d & 31, lane = 4 * g + t;
  if (bits == 8) return {(2 * hi + (e >> 4)) * 512 + lane * 16 + (e & 15), 0};
  if (bits == 2) {
    // word e >> 3 holds k-slices 2w, 2w+1 (h); field r = token half + 2 * dim pair
    const int h = (e >> 2) & 1, w = e & 3, r = hi + 2 * (w >> 1);
    const int bit = 16 * (w & 1) + 8 * h + 2 * r;
    return {lane * 16 + (e >> 3) * 4 + (bit >> 3), bit & 7};
  }
  if (bits == 4) {
    const int nib = ((e & 7) >> 1) + 4 * (e & 1);
    return {hi * 512 + lane * 16 + (e >> 3) * 4 + (nib >> 1), (nib & 1) * 4};
  }
  return {(4 * hi + (e >> 3)) * 512 + lane * 16 + 2 * (e & 7), 0};  // bf16
}

__host__ __device__ inline Loc value_loc(int bits, int i, int d) {
  const int mt = d >> 4, r = d & 15, g = r & 7, hi = r >> 3;
  const int t = (i & 7) >> 1, j = 2 * (i & 1) + (i >> 3), lane = 4 * g + t;
  if (bits == 8) return {(mt >> 1) * 512 + lane * 16 + (2 * (mt & 1) + hi) * 4 + j, 0};
  if (bits == 2) {
    // word mt >> 1 holds m-tiles 2w, 2w+1 (h); field r = dim half + 2 * token pair
    const int h = mt & 1, r = hi + 2 * (j >> 1);
    const int bit = 16 * (j & 1) + 8 * h + 2 * r;
    return {lane * 16 + (mt >> 1) * 4 + (bit >> 3), bit & 7};
  }
  if (bits == 4) {
    const int nib = 2 * hi + (j >> 1) + 4 * (j & 1);
    return {(mt >> 2) * 512 + lane * 16 + (mt & 3) * 4 + (nib >> 1), (nib & 1) * 4};
  }
  return {mt * 512 + lane * 16 + (2 * hi + (j >> 1)) * 4 + 2 * (j & 1), 0};  // bf16
}

// ------------------------------------------------------------------ error word
__device__ __forceinline__ void flag(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Round-half-even of the exact quotient x / s (s > 0, finite).  The float32
// quotient decides unless it landed exactly on a half-integer; then the sign of
// the exact residual x - q*s (computed exactly in double: q*s has at most 48
// significant bits) tells which side the true quotient lies on.
__device__ __forceinline__ float round_quotient(float x, float s) {
  const float q = __fdiv_rn(x, s);
  const float fl = floorf(q);
  if (q - fl == 0.5f) {
    const double res = double(x) - double(q) * double(s);
    if (res > 0.0) return fl + 1.0f;
    if (res < 0.0) return fl;
  }
  return rintf(q);
}

// Symmetric int8 codes of four values of a warp-wide 128-vector whose max|x| is
// amax: s = RN32(amax / 127) (1 for a zero vector), c = clamp(rint(x / s)).
__device__ __forceinline__ float quantize_int8_row(const float (&x)[4], float amax, float (&c)[4]) {
  if (amax == 0.f) {
    c[0] = c[1] = c[2] = c[3] = 0.f;
    return 1.f;
  }
  const float s = __fdiv_rn(amax, 127.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) c[j] = fminf(127.f, fmaxf(-127.f, round_quotient(x[j], s)));
  return s;
}

// ------------------------------------------------------------------ conversions
// Codes are stored offset-binary: an int8 code c is the byte c + 128, an int4
// code c is the nibble c + 8.  Placing the biased value u in the mantissa of
// 1024.0 (fp16 0x6400) gives 1024 + u exactly; one fp16 subtraction of
// 1024 + bias then yields c exactly.

// Four int8 codes (biased bytes b0..b3 of w) -> fp16 pairs lo = (c0, c1), hi = (c2, c3).
__device__ __forceinline__ void s8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x4342);
  const uint32_t bias = 0x64806480u;  // (1152, 1152) = 1024 + 128
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// The fp16 bit pattern of 1024.0 in both halves, the "magic" the int4 codes
// are placed under.  Callers pass it in a register whose value the compiler
// cannot see (magic_f16x2), so each nibble mask below is one three-input
// logic instruction (w & mask) | magic instead of two: an instruction takes
// one immediate operand, and the mask is it.
constexpr uint32_t kMagicF16x2 = 0x64006400u;

// kMagicF16x2 as a run-time value: the batch size is at most 4096 (checked on
// the host), so b >> 16 is zero, but the compiler cannot fold it.
__device__ __forceinline__ uint32_t magic_f16x2(int b) { return kMagicF16x2 | (uint32_t(b) >> 16); }

// Eight int4 codes (biased nibbles n0..n7 of w) -> fp16 pairs (c0,c4) (c1,c5) (c2,c6) (c3,c7).
// Odd nibbles land at 16 * u in the mantissa; a fused (x / 16 - 72) recovers c.
// km must hold kMagicF16x2 (see magic_f16x2).
__device__ __forceinline__ void s4x8_to_f16(uint32_t w, uint32_t km, uint32_t& p0, uint32_t& p1, uint32_t& p2,
                                            uint32_t& p3) {
  const uint32_t s = w >> 8;
  uint32_t a, b, c, d;  // lop3 table 0xEA: (x & mask) | km
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a) : "r"(w), "n"(0x000F000F), "r"(km));  // 1024 + u0, 1024 + u4
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(b) : "r"(w), "n"(0x00F000F0), "r"(km));  // 1024 + 16 u1, 1024 + 16 u5
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(c) : "r"(s), "n"(0x000F000F), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(s), "n"(0x00F000F0), "r"(km));
  const uint32_t bias = 0x64086408u;       // 1032 = 1024 + 8
  const uint32_t sixteenth = 0x2C002C00u;  // 1/16
  const uint32_t m72 = 0xD480D480u;        // -72 = -(1024/16 + 8)
  asm("sub.f16x2 %0, %1, %2;" : "=r"(p0) : "r"(a), "r"(bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(p1) : "r"(b), "r"(sixteenth), "r"(m72));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(p2) : "r"(c), "r"(bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(p3) : "r"(d), "r"(sixteenth), "r"(m72));
}

// Offset conversion of int8 codes: the byte u = c + 128 stays under the magic,
// 1024 + u = kOffsetF16 + c exactly, and the subtraction of the offset is left
// to the caller, which folds it into the key contraction once per query row
// (the accumulators of each block start at minus the offset times the
// query's sum).
constexpr float kOffsetF16 = 1152.f;

// Four int8 codes (biased bytes of w) -> (1152 + c0, 1152 + c1), (1152 + c2, 1152 + c3).
__device__ __forceinline__ void s8x4_to_f16_off(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(w, 0x64646464u, 0x4140);
  hi = __byte_perm(w, 0x64646464u, 0x4342);
}

// Sixteen 2-bit codes (biased fields u = c + 2, or the asymmetric u itself) of
// w -> eight fp16 pairs.  Output 4h + r holds the fields at bits 8h + 2r (low
// half) and 16 + 8h + 2r (high half): the field sits at 4^r * u under the
// magic, and (x / 4^r) - (1024 / 4^r + 2) recovers u - 2 exactly.  km must
// hold kMagicF16x2 (see magic_f16x2).
__device__ __forceinline__ void s2x16_to_f16(uint32_t w, uint32_t km, uint32_t (&o)[8]) {
  const uint32_t s = w >> 8;
  uint32_t a[8];
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[0]) : "r"(w), "n"(0x00030003), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[1]) : "r"(w), "n"(0x000C000C), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[2]) : "r"(w), "n"(0x00300030), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[3]) : "r"(w), "n"(0x00C000C0), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[4]) : "r"(s), "n"(0x00030003), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[5]) : "r"(s), "n"(0x000C000C), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[6]) : "r"(s), "n"(0x00300030), "r"(km));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[7]) : "r"(s), "n"(0x00C000C0), "r"(km));
  const uint32_t bias = 0x64026402u;                     // 1026 = 1024 + 2
  const uint32_t q4 = 0x34003400u, m258 = 0xDC08DC08u;   // 1/4, -258
  const uint32_t q16 = 0x2C002C00u, m66 = 0xD420D420u;   // 1/16, -66
  const uint32_t q64 = 0x24002400u, m18 = 0xCC80CC80u;   // 1/64, -18
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    asm("sub.f16x2 %0, %1, %2;" : "=r"(o[4 * h]) : "r"(a[4 * h]), "r"(bias));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[4 * h + 1]) : "r"(a[4 * h + 1]), "r"(q4), "r"(m258));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[4 * h + 2]) : "r"(a[4 * h + 2]), "r"(q16), "r"(m66));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[4 * h + 3]) : "r"(a[4 * h + 3]), "r"(q64), "r"(m18));
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ mma.sync
// D(16x8 f32) += A(16x16) * B(16x8), fp16 or bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true once the phase with `parity` has completed, false after
// kWaitLimitNs of wall-clock time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// One contiguous global -> shared bulk copy completing on `bar` (bytes: multiple
// of 16; both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Asynchronous small global -> shared copies (cp.async), grouped per commit.
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace kvq
