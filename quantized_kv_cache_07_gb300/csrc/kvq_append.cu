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
// One warp quantizes one 128-element vector; lane l owns dims 4l..4l+3.
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
  if (bits != 16 && !chan) {
    const float* rec = a.c.meta + (size_t(h) * a.c.num_blocks + phys) * a.c.meta_floats;
    const int off = is_key ? 0 : a.c.meta_floats / 2;
    s = rec[off + tok];
    if (asym) m = rec[off + kBlock + tok];
  }
  const int bias = asym ? 0 : (bits == 8 ? 128 : 8);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = 4 * lane + j;
    const Loc L = is_key ? key_loc(bits, tok, d) : value_loc(bits, tok, d);
    float v;
    if (bits == 16) {
      v = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(blk + L.byte));
    } else {
      const int raw = bits == 8 ? int(blk[L.byte]) : int((blk[L.byte] >> L.shift) & 0xF);
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
  const int warps = 8;
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, append_kernel, a);
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
