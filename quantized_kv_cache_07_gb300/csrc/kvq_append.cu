// Quantize-on-write (kvq_append) and read-back (kvq_dequant) kernels.
//
// Quantizer: "KV Cache Quantization and Per-Token Scale Placement", sections
// "Per-token scales and where they can live" (one scale per token per head,
// computed at write time, stored alongside the codes) and "The axis choice is a
// kernel decision" (listing: amax, zero vector -> scale 1, scale = amax/qmax,
// clamp(round(x/scale))); "KV Cache Quantization Reduces Cache Bytes with
// Separate Accuracy and Kernel Costs", section "Quantization needs a scale
// convention" (q = clamp(round(x/s)), x_hat = q*s).  Asymmetric format: "KV
// Cache Quantization Perturbs Attention Through Stored Keys and Values",
// section "Quantization granularity defines which values share a scale" (a
// scale and a zero point per group; here per token per head).
//
// 2-bit codes share one scale (and zero point) per 16-token block: "KV Cache
// Quantization and Per-Token Scale Placement", section "Per-token scales and
// where they can live" (at 2 bits, schemes group several tokens under one
// scale).  A block is quantized as one vector of up to 16 x 128 values.
//
// One warp quantizes one 128-element vector (or one 2-bit token group); lane l
// owns dims 4l..4l+3.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Warp-cooperative per-vector quantization.
__device__ __forceinline__ void quantize_warp(const float (&x)[4], int bits, int (&code)[4], float& s) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kFull, a, o));
  const int qmax = bits == 8 ? 127 : 7;
  const int lo = bits == 8 ? -127 : -8;
  if (a == 0.0f) {
    s = 1.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) code[j] = 0;
    return;
  }
  s = __fdiv_rn(a, float(qmax));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int c = int(round_quotient(x[j], s));
    code[j] = min(qmax, max(lo, c));
  }
}

// Warp-cooperative asymmetric quantization: m = min(x), s = RN32((max - min) /
// (2^bits - 1)) with the difference and the quotient in double (a constant
// vector gets s = 1), u = clamp(rint((x - m) / s), 0, 2^bits - 1) with the
// difference and the quotient in double (rint: half to even).
__device__ __forceinline__ void quantize_asym_warp(const float (&x)[4], int bits, int (&u)[4], float& s, float& m) {
  float lo = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float hi = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(kFull, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(kFull, hi, o));
  }
  const int qmaxu = bits == 8 ? 255 : 15;
  const double rng = __dsub_rn(double(hi), double(lo));
  s = rng == 0.0 ? 1.0f : __double2float_rn(__ddiv_rn(rng, double(qmaxu)));
  m = lo;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const double r = rint(__ddiv_rn(__dsub_rn(double(x[j]), double(lo)), double(s)));
    u[j] = r >= double(qmaxu) ? qmaxu : (r > 0.0 ? int(r) : 0);  // clamp before the conversion
  }
}

// Store the codes of one quantized vector (token `tok`) into its block.  The
// values given are the stored bytes / nibbles (offset-binary for symmetric
// codes, the unsigned code itself for the asymmetric format).
__device__ void store_codes(bool is_key, int bits, uint8_t* blk, int tok, const int (&code)[4], int lane) {
  if (bits == 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int d = 4 * lane + j;
      const Loc L = is_key ? key_loc(8, tok, d) : value_loc(8, tok, d);
      blk[L.byte] = uint8_t(code[j]);
    }
    return;
  }
  // 4-bit
  if (is_key) {
    // Lanes l and l^1 own the 8 nibbles of one 32-bit word of this token.
    uint32_t part = 0;
    int word_off = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int d = 4 * lane + j;
      const Loc L = key_loc(4, tok, d);
      const int nib = ((L.byte & 3) << 1) | (L.shift >> 2);
      part |= uint32_t(code[j]) << (4 * nib);
      word_off = L.byte & ~3;
    }
    const uint32_t word = part | __shfl_xor_sync(kFull, part, 1);
    if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(blk + word_off) = word;
    return;
  }
  // 4-bit values: a word mixes four tokens, so update only this token's nibbles.
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = 4 * lane + j;
    const Loc L = value_loc(4, tok, d);
    const int nib = ((L.byte & 3) << 1) | (L.shift >> 2);
    uint32_t* w = reinterpret_cast<uint32_t*>(blk + (L.byte & ~3));
    atomicAnd(w, ~(0xFu << (4 * nib)));
    atomicOr(w, uint32_t(code[j]) << (4 * nib));
  }
}

__device__ void store_bf16(bool is_key, uint8_t* blk, int tok, const uint16_t (&xb)[4], int lane) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = 4 * lane + j;
    const Loc L = is_key ? key_loc(16, tok, d) : value_loc(16, tok, d);
    *reinterpret_cast<uint16_t*>(blk + L.byte) = xb[j];
  }
}

// Quantize (or copy, for a bf16 cache) one vector into the block store at
// position p of sequence b.
__device__ void write_block_store(const AppendArgs& a, bool is_key, int b, int p, int h, const uint16_t (&xb)[4],
                                  int lane) {
  const CacheView& c = a.c;
  if (p >= a.mbps * kBlock) {
    if (lane == 0) flag(a.err, KVQ_DEVERR_POSITION);
    return;
  }
  const int phys = a.table[size_t(b) * a.mbps + p / kBlock];
  if (phys < 0 || phys >= c.num_blocks) {
    if (lane == 0) flag(a.err, KVQ_DEVERR_BLOCK_ID);
    return;
  }
  const int tok = p % kBlock;
  const int bits = is_key ? c.k_bits : c.v_bits;
  uint8_t* pool = is_key ? c.k_codes : c.v_codes;
  uint8_t* blk = pool + (size_t(h) * c.num_blocks + phys) * block_bytes(bits);
  if (bits == 16) {
    store_bf16(is_key, blk, tok, xb, lane);
    return;
  }
  float x[4];
  if (is_key && c.k_chan) {
    // per-channel scales only: code = clamp(rint(k / c)) of the exact quotient, no per-token scale
    const int lo = bits == 8 ? -127 : -8, hi = bits == 8 ? 127 : 7, bias = bits == 8 ? 128 : 8;
    int code[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float q = round_quotient(bf16_bits_to_f32(xb[j]), c.factor[h * kHeadDim + 4 * lane + j]);
      code[j] = int(fminf(float(hi), fmaxf(float(lo), q))) + bias;
    }
    store_codes(is_key, bits, blk, tok, code, lane);
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[j] = bf16_bits_to_f32(xb[j]);
    if (is_key && c.factor) x[j] = __fdiv_rn(x[j], c.factor[h * kHeadDim + 4 * lane + j]);
  }
  int code[4];
  float s, m = 0.f;
  const bool asym = c.asym != 0;
  if (asym) {
    quantize_asym_warp(x, bits, code, s, m);
  } else {
    quantize_warp(x, bits, code, s);
    const int bias = bits == 8 ? 128 : 8;  // offset binary
#pragma unroll
    for (int j = 0; j < 4; ++j) code[j] += bias;
  }
  store_codes(is_key, bits, blk, tok, code, lane);
  if (lane == 0) {
    // metadata record: K scales, (K zero points,) V scales, (V zero points)
    float* rec = c.meta + (size_t(h) * c.num_blocks + phys) * c.meta_floats;
    const int off = is_key ? 0 : c.meta_floats / 2;
    rec[off + tok] = s;
    if (asym) rec[off + kBlock + tok] = m;
  }
}

__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  // Programmatic dependent launch: wait for the previous kernel on the stream
  // (its writes visible) before touching memory; let the next one launch early.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long vec = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int H = a.c.H;
  if (vec >= (long long)a.n * 2 * H) return;
  const int r = int(vec / (2 * H));
  const int kv = int((vec / H) % 2);
  const int h = int(vec % H);
  const bool is_key = kv == 0;
  // the new vector does not depend on the destination: load it with the indices
  const uint16_t* src = (is_key ? a.k_new : a.v_new) + (size_t(r) * H + h) * kHeadDim + 4 * lane;
  const uint2 v_new = *reinterpret_cast<const uint2*>(src);
  const int b = a.seq_idx[r];
  const int p = a.pos[r];
  if (b < 0 || b >= a.batch || p < 0 ||
      (a.mode != KVQ_APPEND_QUANT && b >= a.c.window_batch)) {
    if (lane == 0) flag(a.err, KVQ_DEVERR_POSITION);
    return;
  }
  uint16_t xb[4];
  {
    const uint2 v = v_new;
    xb[0] = uint16_t(v.x & 0xFFFF);
    xb[1] = uint16_t(v.x >> 16);
    xb[2] = uint16_t(v.y & 0xFFFF);
    xb[3] = uint16_t(v.y >> 16);
  }
  if (a.mode == KVQ_APPEND_QUANT) {
    write_block_store(a, is_key, b, p, h, xb, lane);
    return;
  }
  // window ring: slot p % W is token (slot % 16) of ring block slot / 16, stored
  // in the fragment-native bf16 block layout
  const int W = a.c.window;
  const int slot = p % W;
  uint8_t* ring = (is_key ? a.c.k_win : a.c.v_win) +
                  ((size_t(b) * H + h) * (W / kBlock) + slot / kBlock) * block_bytes(16);
  const int tok = slot % kBlock;
  int off[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const Loc L = is_key ? key_loc(16, tok, 4 * lane + j) : value_loc(16, tok, 4 * lane + j);
    off[j] = L.byte;
  }
  if (a.mode == KVQ_APPEND_STEP && p >= W) {
    // the token at p - W occupies this ring slot: it leaves the window now
    uint16_t ob[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) ob[j] = *reinterpret_cast<const uint16_t*>(ring + off[j]);
    write_block_store(a, is_key, b, p - W, h, ob, lane);
    __syncwarp();
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint16_t*>(ring + off[j]) = xb[j];
}

// 2-bit blocks: one warp per (group, head, K or V).  A group is the run of rows
// of one call that fills positions 16j, 16j + 1, ... (up to 16) of one
// sequence; the row at position 16j leads it.  A row whose position is not at
// a block start and is not part of such a run is flagged and skipped: 2-bit
// blocks are written whole, in one call.
constexpr int kGroupWarps = 8;

__global__ void __launch_bounds__(kGroupWarps * 32) append_group_kernel(AppendArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ uint32_t img[kGroupWarps][kBlock * kHeadDim * 2 / 32];  // one 512-byte block per warp
  const int lane = threadIdx.x & 31, wslot = threadIdx.x >> 5;
  const long long vec = (long long)blockIdx.x * kGroupWarps + wslot;
  const int H = a.c.H;
  if (vec >= (long long)a.n * 2 * H) return;
  const int r = int(vec / (2 * H));
  const bool is_key = ((vec / H) % 2) == 0;
  const int h = int(vec % H);
  const int b = a.seq_idx[r];
  const int p = a.pos[r];
  if (b < 0 || b >= a.batch || p < 0) {
    if (lane == 0) flag(a.err, KVQ_DEVERR_POSITION);
    return;
  }
  const int j = p % kBlock;
  if (j != 0) {
    // covered by the run led by row r - j?
    bool covered = r - j >= 0;
    for (int k = 0; covered && k < j; ++k) covered = a.seq_idx[r - j + k] == b && a.pos[r - j + k] == p - j + k;
    if (!covered && lane == 0) flag(a.err, KVQ_DEVERR_POSITION);
    return;
  }
  int m = 1;
  while (m < kBlock && r + m < a.n && a.seq_idx[r + m] == b && a.pos[r + m] == p + m) ++m;
  if (p + m > a.mbps * kBlock) {
    if (lane == 0) flag(a.err, KVQ_DEVERR_POSITION);
    return;
  }
  const int phys = a.table[size_t(b) * a.mbps + p / kBlock];
  if (phys < 0 || phys >= a.c.num_blocks) {
    if (lane == 0) flag(a.err, KVQ_DEVERR_BLOCK_ID);
    return;
  }
  // the group's values, lane l holding dims 4l..4l+3 of each row
  float x[kBlock][4];
  const uint16_t* src = is_key ? a.k_new : a.v_new;
#pragma unroll
  for (int k = 0; k < kBlock; ++k) {
    if (k < m) {
      const uint2 v = *reinterpret_cast<const uint2*>(src + (size_t(r + k) * H + h) * kHeadDim + 4 * lane);
      x[k][0] = __uint_as_float(v.x << 16);
      x[k][1] = __uint_as_float(v.x & 0xFFFF0000u);
      x[k][2] = __uint_as_float(v.y << 16);
      x[k][3] = __uint_as_float(v.y & 0xFFFF0000u);
      if (is_key && a.c.factor) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[k][e] = __fdiv_rn(x[k][e], a.c.factor[h * kHeadDim + 4 * lane + e]);
      }
    } else {
      x[k][0] = x[k][1] = x[k][2] = x[k][3] = 0.f;
    }
  }
  const bool asym = a.c.asym != 0;
  float s = 1.f, zp = 0.f;
  float lo = x[0][0], hi = x[0][0], am = 0.f;
#pragma unroll
  for (int k = 0; k < kBlock; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (k < m) {
        lo = fminf(lo, x[k][e]);
        hi = fmaxf(hi, x[k][e]);
        am = fmaxf(am, fabsf(x[k][e]));
      }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(kFull, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(kFull, hi, o));
    am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
  }
  if (asym) {
    // asymmetric rule over the group: m = min, s = RN32((max - min) / 3) (1 for
    // a constant group), u = clamp(rint((x - m) / s), 0, 3), in double
    const double rng = __dsub_rn(double(hi), double(lo));
    s = rng == 0.0 ? 1.0f : __double2float_rn(__ddiv_rn(rng, 3.0));
    zp = lo;
  } else if (am > 0.f) {
    s = am;  // RN32(amax / qmax) with qmax = 1
  }
  uint32_t* im = img[wslot];
#pragma unroll
  for (int i = lane; i < kBlock * kHeadDim * 2 / 32; i += 32) im[i] = 0u;
  __syncwarp();
#pragma unroll
  for (int k = 0; k < kBlock; ++k) {
    if (k >= m) break;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int u;
      if (asym) {
        const double q = rint(__ddiv_rn(__dsub_rn(double(x[k][e]), double(lo)), double(s)));
        u = q >= 3.0 ? 3 : (q > 0.0 ? int(q) : 0);
      } else {
        const float q = am > 0.f ? round_quotient(x[k][e], s) : 0.f;
        u = int(fminf(1.f, fmaxf(-2.f, q))) + 2;  // offset binary
      }
      const Loc L = is_key ? key_loc(2, k, 4 * lane + e) : value_loc(2, k, 4 * lane + e);
      atomicOr(&im[L.byte >> 2], uint32_t(u) << (8 * (L.byte & 3) + L.shift));
    }
  }
  __syncwarp();
  uint8_t* blk = (is_key ? a.c.k_codes : a.c.v_codes) + (size_t(h) * a.c.num_blocks + phys) * block_bytes(2);
  reinterpret_cast<uint4*>(blk)[lane] = reinterpret_cast<const uint4*>(im)[lane];
  if (lane == 0) {
    float* rec = a.c.meta + (size_t(h) * a.c.num_blocks + phys) * a.c.meta_floats;
    rec[is_key ? 0 : 2] = s;
    rec[is_key ? 1 : 3] = zp;
  }
}

__global__ void __launch_bounds__(256) dequant_kernel(DequantArgs a) {
  const int lane = threadIdx.x & 31;
  const long long vec = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int H = a.c.H;
  if (vec >= (long long)a.n * 2 * H) return;
  const int r = int(vec / (2 * H));
  const bool is_key = ((vec / H) % 2) == 0;
  const int h = int(vec % H);
  const int slot = a.slots[r];
  const int phys = slot / kBlock, tok = slot % kBlock;
  float* out = (is_key ? a.k_out : a.v_out) + (size_t(r) * H + h) * kHeadDim + 4 * lane;
  if (slot < 0 || phys >= a.c.num_blocks) {
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = 0.0f;
    return;
  }
  const int bits = is_key ? a.c.k_bits : a.c.v_bits;
  const uint8_t* blk = (is_key ? a.c.k_codes : a.c.v_codes) + (size_t(h) * a.c.num_blocks + phys) * block_bytes(bits);
  float s = 1.0f, m = 0.0f;
  const bool asym = a.c.asym != 0;
  const bool chan = is_key && a.c.k_chan;  // per-channel key scale c_j instead of a per-token one
  if (bits == 2) {
    const float* rec = a.c.meta + (size_t(h) * a.c.num_blocks + phys) * a.c.meta_floats;
    s = rec[is_key ? 0 : 2];
    m = rec[is_key ? 1 : 3];
  } else if (bits != 16 && !chan) {
    const float* rec = a.c.meta + (size_t(h) * a.c.num_blocks + phys) * a.c.meta_floats;
    const int off = is_key ? 0 : a.c.meta_floats / 2;
    s = rec[off + tok];
    if (asym) m = rec[off + kBlock + tok];
  }
  const int bias = asym ? 0 : (bits == 8 ? 128 : (bits == 4 ? 8 : 2));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = 4 * lane + j;
    const Loc L = is_key ? key_loc(bits, tok, d) : value_loc(bits, tok, d);
    float v;
    if (bits == 16) {
      v = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(blk + L.byte));
    } else {
      const int raw = bits == 8 ? int(blk[L.byte]) : int((blk[L.byte] >> L.shift) & (bits == 4 ? 0xF : 0x3));
      const float sd = chan ? a.c.factor[h * kHeadDim + d] : s;
      v = asym ? __fmaf_rn(float(raw), s, m) : __fmul_rn(float(raw - bias), sd);
    }
    out[j] = v;
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  const long long vecs = (long long)a.n * 2 * a.c.H;
  if (vecs == 0) return cudaSuccess;
  const bool group = a.c.k_bits == 2 && a.mode == KVQ_APPEND_QUANT;
  const int warps = group ? kGroupWarps : 8;
  const long long grid = (vecs + warps - 1) / warps;
  // launched with programmatic stream serialisation, so the launch overlaps the
  // tail of the previous kernel (the kernel waits for it before reading memory)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = group ? cudaLaunchKernelEx(&cfg, append_group_kernel, a) : cudaLaunchKernelEx(&cfg, append_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s) {
  const long long vecs = (long long)a.n * 2 * a.c.H;
  if (vecs == 0) return cudaSuccess;
  const int warps = 8;
  const long long grid = (vecs + warps - 1) / warps;
  dequant_kernel<<<unsigned(grid), warps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
