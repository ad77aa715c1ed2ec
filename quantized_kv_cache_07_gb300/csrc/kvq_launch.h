// Internal host-side interface between the C ABI (kvq_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvq {

struct CacheView {
  int H;            // KV heads
  int num_blocks;
  int k_bits, v_bits;
  uint8_t* k_codes;
  uint8_t* v_codes;
  float* meta;      // [H][num_blocks][meta_floats]: K scales, (K zero points,) V scales, (V zero points)
  int asym;         // 1: scale and zero point per token (meta_floats 64), else 32
  int meta_floats;
  const float* factor;  // [H][128] or null
  int window, window_batch;
  int q_bits;      // query format: 8 int8 rows (integer dot), 16 fp16, 32 fp16 hi + lo
  int k_chan;      // 1: keys carry per-channel scales (factor) only, no per-token key scale
  uint8_t* k_win;  // bf16 ring: [window_batch][H][W/16] fragment-native bf16 blocks
  uint8_t* v_win;
};

struct AppendArgs {
  CacheView c;
  const uint16_t* k_new;
  const uint16_t* v_new;
  int n;
  const int* seq_idx;
  const int* pos;
  int mode;
  const int* table;
  int batch;
  int mbps;
  uint32_t* err;
};

struct DequantArgs {
  CacheView c;
  const int* slots;
  int n;
  float* k_out;
  float* v_out;
};

// Workspace layout of a decode call (byte offsets from the workspace base).
struct DecodeLayout {
  int stream_ctas, window_ctas, units, slots;
  int switch_blocks;  // virtual blocks charged for starting a unit (0: unit-aligned split)
  size_t off_counter;  // int [units]: merge arrival counters
  size_t off_m, off_l, off_o, total;  // partial records: m, l [slots][G], o [slots][G][128]
};

struct DecodeArgs {
  CacheView c;
  const uint16_t* q;  // bf16 [B][Hq][128]
  int B, Hq, G;
  const int* seq_lens;
  // Prefill (pos != null): row b of the call is position pos[b] of sequence
  // seq_of[b] (< nseq); it attends to positions 0..pos[b] of that sequence.
  const int* pos;
  const int* seq_of;
  int nseq;
  const int* table;
  int mbps;
  void* out;
  int out_fp32;
  float* lse;
  uint8_t* ws;
  DecodeLayout lay;
  uint32_t* err;
  // 1: seq_lens and the block table are final before the preceding kernel on
  // the stream ends (KVQ_DECODE_GEOMETRY_READY): read them before the wait
  int ahead = 0;
};

// The largest GQA group (query heads per KV head) the decode kernel takes: one
// 8-wide MMA tile of query columns.
constexpr int kMaxGroup = 8;

// Unit-start charge of the split, in blocks of the cache's format.
int switch_blocks_for(int k_bits);
// switch_cost: the unit-start charge when the split is not unit-aligned.
DecodeLayout decode_layout(int B, int Hq, int H, int window, int stream_ctas, int switch_cost);

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s);
// Resident decode CTAs per SM for this cache format and batch (occupancy
// query on the current device, cached); 0 for an unsupported format.
int decode_ctas_per_sm_for(int k_bits, int v_bits, bool asym, int q_bits, int batch, bool rows = false);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// The asymmetric instantiations (kvq_decode_asym.cu).
int decode_ctas_per_sm_asym(int k_bits, int v_bits, int batch, bool rows);
cudaError_t launch_decode_asym(const DecodeArgs& a, cudaStream_t s);
// The two-part fp16 query instantiations (kvq_decode_q32.cu).
int decode_ctas_per_sm_q32(int k_bits, int v_bits, bool asym, int batch, bool rows);
cudaError_t launch_decode_q32(const DecodeArgs& a, cudaStream_t s);
// Prefill on 16-vector query tiles (kvq_prefill_tiles.cu): quantized blocks
// (8-, 4- or 2-bit, symmetric or asymmetric), any query format, no window.
// Needs no workspace.
bool prefill_tiles_supported(const CacheView& c);
cudaError_t launch_prefill_tiles(const DecodeArgs& a, cudaStream_t s);

}  // namespace kvq
