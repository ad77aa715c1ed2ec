// C ABI of libkvq.so: argument validation, work planning and dispatch.
// Declarations and the contract of every entry point are in include/kvq.h.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kvq.h"
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace {

using kvq::kHeadDim;

constexpr int kMaxBatch = 4096;  // sequence geometry is staged in shared memory
constexpr int kMaxWindow = 128;  // window ring: at most 8 bf16 blocks per (sequence, kv head)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool format_supported(int kb, int vb) {
  return (kb == 8 && vb == 8) || (kb == 4 && vb == 4) || (kb == 4 && vb == 8) || (kb == 8 && vb == 4) ||
         (kb == 2 && vb == 2) || (kb == 16 && vb == 16);
}

kvq_status check_cache(const kvq_cache_desc* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->num_kv_heads < 1 || c->num_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->block_size != 16) return KVQ_ERR_UNSUPPORTED;
  if (!format_supported(c->k_bits, c->v_bits)) return KVQ_ERR_UNSUPPORTED;
  if (!c->k_codes || !c->v_codes) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(c->k_codes) || !aligned16(c->v_codes)) return KVQ_ERR_ALIGNMENT;
  const bool quant = c->k_bits != 16;
  if (c->asym != 0 && c->asym != 1) return KVQ_ERR_INVALID_ARG;
  if (c->k_per_channel != 0 && c->k_per_channel != 1) return KVQ_ERR_INVALID_ARG;
  if (c->asym && !quant) return KVQ_ERR_UNSUPPORTED;  // zero points only on quantized blocks
  if (c->k_per_channel && (!quant || c->asym || c->k_bits == 2)) return KVQ_ERR_UNSUPPORTED;
  if (c->k_per_channel && !c->k_channel_factor) return KVQ_ERR_INVALID_ARG;
  if (quant) {
    if (!c->meta) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(c->meta)) return KVQ_ERR_ALIGNMENT;
  }
  if (c->k_channel_factor) {
    if (!quant) return KVQ_ERR_UNSUPPORTED;
    if (!aligned16(c->k_channel_factor)) return KVQ_ERR_ALIGNMENT;
  }
  if (c->q_bits != 0 && c->q_bits != 16 && c->q_bits != 8 && c->q_bits != 32) return KVQ_ERR_UNSUPPORTED;
  if (c->q_bits == 8 && (!quant || (c->k_channel_factor && c->window > 0))) return KVQ_ERR_UNSUPPORTED;
  if (c->window < 0) return KVQ_ERR_INVALID_ARG;
  if (c->window > kMaxWindow || c->window % 16 != 0) return KVQ_ERR_UNSUPPORTED;
  if (c->window > 0) {
    if (!c->k_window || !c->v_window || c->window_batch < 1) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(c->k_window) || !aligned16(c->v_window)) return KVQ_ERR_ALIGNMENT;
  }
  return KVQ_OK;
}

kvq::CacheView view(const kvq_cache_desc* c) {
  kvq::CacheView v;
  v.H = c->num_kv_heads;
  v.num_blocks = c->num_blocks;
  v.k_bits = c->k_bits;
  v.v_bits = c->v_bits;
  v.k_codes = static_cast<uint8_t*>(c->k_codes);
  v.v_codes = static_cast<uint8_t*>(c->v_codes);
  v.meta = c->meta;
  v.asym = c->asym;
  v.meta_floats = c->k_bits == 2 ? 4 : (c->asym ? 64 : 32);
  v.factor = c->k_channel_factor;
  v.window = c->window;
  v.window_batch = c->window_batch;
  v.q_bits = c->q_bits == 0 ? 16 : c->q_bits;
  v.k_chan = c->k_per_channel;
  v.k_win = static_cast<uint8_t*>(c->k_window);
  v.v_win = static_cast<uint8_t*>(c->v_window);
  return v;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Stream CTAs for one wave of `slots` resident CTAs: the window CTAs (one per
// unit, launched first) take their slots out of the wave, down to half of it.
// When the units fit in the wave and only a few CTAs would be lost, the count
// is rounded down to a multiple of the unit count: with equal lengths every
// stream CTA then holds one segment of one unit (no unit boundary inside).
int stream_ctas_for(int slots, int window_ctas, int units) {
  int left = slots - window_ctas;
  left = left > slots / 2 ? left : (slots / 2 > 0 ? slots / 2 : 1);
  if (units > 0 && units <= left && left % units <= left / 16) left -= left % units;
  return left;
}

// Stream CTAs for the current device (0 on failure); rows: a prefill call.
int auto_stream_ctas(const kvq_cache_desc* c, int batch, bool rows = false) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  const int per = kvq::decode_ctas_per_sm_for(c->k_bits, c->v_bits, c->asym != 0, c->q_bits, batch, rows);
  return stream_ctas_for(sms * per, c->window > 0 ? batch * c->num_kv_heads : 0, batch * c->num_kv_heads);
}

kvq_status check_decode_shape(const kvq_cache_desc* c, int batch, int q_heads) {
  if (batch < 0 || q_heads < 1) return KVQ_ERR_INVALID_ARG;
  if (batch > kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  if (q_heads % c->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (q_heads / c->num_kv_heads > kvq::kMaxGroup) return KVQ_ERR_UNSUPPORTED;
  if (c->window > 0 && c->window_batch < batch) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

// CTAs of the prefill tile path: 16 / G consecutive rows x G heads per tile,
// one CTA per (tile, KV head).
long long prefill_tiles(int n, int q_heads, int kv_heads) {
  const int G = q_heads / kv_heads;
  const int TR = 16 / G;
  return (long long)((n + TR - 1) / TR) * kv_heads;
}

}  // namespace

namespace kvq {

int switch_blocks_for(int k_bits) {
  // Starting a unit (its query staging, the previous unit's record, ticket and
  // possibly merge) costs about as much time as this many blocks of the
  // format: more of the cheaper 4- and 2-bit blocks (measured optimum on
  // 32 sequences of 1k-8k tokens: 40 for 4-/2-bit keys, 32 for int8 keys,
  // 16 for a bf16 cache).
  return k_bits == 16 ? 16 : (k_bits == 8 ? 32 : 40);
}

DecodeLayout decode_layout(int B, int Hq, int H, int window, int stream_ctas, int switch_cost) {
  const int G = H > 0 ? Hq / H : 0;
  DecodeLayout L;
  L.stream_ctas = stream_ctas;
  L.units = B * H;
  L.window_ctas = window > 0 ? L.units : 0;
  L.slots = stream_ctas + L.units + L.window_ctas;
  // When the stream CTAs are a multiple of the units (equal lengths split
  // unit-aligned) every CTA starts exactly one unit: no start cost needed.
  // Otherwise starting a unit (query staging, record, ticket) is charged as
  // switch_cost blocks of work so the split balances time, not blocks.
  L.switch_blocks = (L.units > 0 && L.units <= stream_ctas && stream_ctas % L.units == 0) ? 0 : switch_cost;
  size_t o = 0;
  L.off_counter = o;
  o = round_up(o + size_t(L.units) * 4, 256);
  L.off_m = o;
  o = round_up(o + size_t(L.slots) * G * 4, 256);
  L.off_l = o;
  o = round_up(o + size_t(L.slots) * G * 4, 256);
  L.off_o = o;
  o = round_up(o + size_t(L.slots) * G * kHeadDim * 4, 256);
  L.total = o;
  return L;
}

}  // namespace kvq

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG: invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED: unsupported shape or format";
    case KVQ_ERR_ALIGNMENT: return "KVQ_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE: workspace missing or too small";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA: CUDA runtime error";
  }
  return "KVQ_UNKNOWN_STATUS";
}

kvq_status kvq_block_bytes(int32_t bits, size_t* bytes) {
  if (!bytes) return KVQ_ERR_INVALID_ARG;
  if (bits != 2 && bits != 4 && bits != 8 && bits != 16) return KVQ_ERR_UNSUPPORTED;
  *bytes = size_t(kvq::block_bytes(bits));
  return KVQ_OK;
}

kvq_status kvq_append(const kvq_cache_desc* cache, const void* k_new, const void* v_new, int32_t n,
                      const int32_t* seq_idx, const int32_t* pos, int32_t mode, const int32_t* block_table,
                      int32_t batch, int32_t max_blocks_per_seq, uint32_t* err_word, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n < 0) return KVQ_ERR_INVALID_ARG;
  if (mode != KVQ_APPEND_QUANT && mode != KVQ_APPEND_RING && mode != KVQ_APPEND_STEP) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (!k_new || !v_new || !seq_idx || !pos) return KVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) & 7u) || (reinterpret_cast<uintptr_t>(v_new) & 7u))
    return KVQ_ERR_ALIGNMENT;
  if (batch < 1) return KVQ_ERR_INVALID_ARG;
  if (mode != KVQ_APPEND_QUANT && cache->window == 0) return KVQ_ERR_INVALID_ARG;
  // 2-bit blocks are quantized whole (one scale per 16-token block): a decode
  // step cannot evict a single token into one
  if (mode == KVQ_APPEND_STEP && cache->k_bits == 2) return KVQ_ERR_UNSUPPORTED;
  if (mode != KVQ_APPEND_RING && (!block_table || max_blocks_per_seq < 1)) return KVQ_ERR_INVALID_ARG;
  if ((long long)n * 2 * cache->num_kv_heads > (1ll << 36)) return KVQ_ERR_UNSUPPORTED;
  kvq::AppendArgs a;
  a.c = view(cache);
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.n = n;
  a.seq_idx = seq_idx;
  a.pos = pos;
  a.mode = mode;
  a.table = block_table;
  a.batch = batch;
  a.mbps = max_blocks_per_seq > 0 ? max_blocks_per_seq : 1;
  a.err = err_word;
  if (kvq::launch_append(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_make_decode_plan(int32_t batch, int32_t q_heads, int32_t num_kv_heads, int32_t window,
                                int32_t num_sms, int32_t ctas_per_sm, int32_t stream_ctas,
                                kvq_decode_plan* plan) {
  if (!plan || batch < 0 || q_heads < 1 || num_kv_heads < 1 || window < 0) return KVQ_ERR_INVALID_ARG;
  if (q_heads % num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  int P = stream_ctas;
  if (P <= 0) {
    if (num_sms < 1 || ctas_per_sm < 1) return KVQ_ERR_INVALID_ARG;
    P = stream_ctas_for(num_sms * ctas_per_sm, window > 0 ? batch * num_kv_heads : 0, batch * num_kv_heads);
  }
  const kvq::DecodeLayout L = kvq::decode_layout(batch, q_heads, num_kv_heads, window, P, 16);
  plan->stream_ctas = L.stream_ctas;
  plan->window_ctas = L.window_ctas;
  plan->units = L.units;
  plan->partial_slots = L.slots;
  plan->workspace_bytes = L.total;
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_size(const kvq_cache_desc* cache, int32_t batch, int32_t q_heads,
                                     int32_t stream_ctas, size_t* bytes) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!bytes) return KVQ_ERR_INVALID_ARG;
  st = check_decode_shape(cache, batch, q_heads);
  if (st != KVQ_OK) return st;
  int P = stream_ctas > 0 ? stream_ctas : auto_stream_ctas(cache, batch);
  if (P <= 0) return KVQ_ERR_CUDA;
  *bytes = kvq::decode_layout(batch, q_heads, cache->num_kv_heads, cache->window, P,
                                                 kvq::switch_blocks_for(cache->k_bits)).total;
  return KVQ_OK;
}

kvq_status kvq_decode_device_plan(const kvq_cache_desc* cache, int32_t batch, int32_t q_heads, int32_t stream_ctas,
                                  kvq_decode_plan* plan) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!plan) return KVQ_ERR_INVALID_ARG;
  st = check_decode_shape(cache, batch, q_heads);
  if (st != KVQ_OK) return st;
  const int P = stream_ctas > 0 ? stream_ctas : auto_stream_ctas(cache, batch);
  if (P <= 0) return KVQ_ERR_CUDA;
  const kvq::DecodeLayout L = kvq::decode_layout(batch, q_heads, cache->num_kv_heads, cache->window, P,
                                                 kvq::switch_blocks_for(cache->k_bits));
  plan->stream_ctas = L.stream_ctas;
  plan->window_ctas = L.window_ctas;
  plan->units = L.units;
  plan->partial_slots = L.slots;
  plan->workspace_bytes = L.total;
  return KVQ_OK;
}

kvq_status kvq_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace && bytes) return KVQ_ERR_INVALID_ARG;
  if (!bytes) return KVQ_OK;
  if (cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_decode(const kvq_cache_desc* cache, const void* q, int32_t batch, int32_t q_heads,
                      const int32_t* seq_lens, const int32_t* block_table, int32_t max_blocks_per_seq, void* out,
                      int32_t out_fp32, float* lse, void* workspace, size_t workspace_bytes, int32_t stream_ctas,
                      uint32_t* err_word, void* stream) {
  return kvq_decode_ex(cache, q, batch, q_heads, seq_lens, block_table, max_blocks_per_seq, out, out_fp32, lse,
                       workspace, workspace_bytes, stream_ctas, 0u, err_word, stream);
}

kvq_status kvq_decode_ex(const kvq_cache_desc* cache, const void* q, int32_t batch, int32_t q_heads,
                         const int32_t* seq_lens, const int32_t* block_table, int32_t max_blocks_per_seq, void* out,
                         int32_t out_fp32, float* lse, void* workspace, size_t workspace_bytes, int32_t stream_ctas,
                         uint32_t flags, uint32_t* err_word, void* stream) {
  if (flags & ~uint32_t(KVQ_DECODE_GEOMETRY_READY)) return KVQ_ERR_INVALID_ARG;
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  st = check_decode_shape(cache, batch, q_heads);
  if (st != KVQ_OK) return st;
  if (batch == 0) return KVQ_OK;
  if (!q || !seq_lens || !block_table || !out || max_blocks_per_seq < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_ALIGNMENT;
  if (stream_ctas < 0) return KVQ_ERR_INVALID_ARG;
  const int P = stream_ctas > 0 ? stream_ctas : auto_stream_ctas(cache, batch);
  if (P <= 0) return KVQ_ERR_CUDA;
  const kvq::DecodeLayout L = kvq::decode_layout(batch, q_heads, cache->num_kv_heads, cache->window, P,
                                                 kvq::switch_blocks_for(cache->k_bits));
  if (!workspace || workspace_bytes < L.total) return KVQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVQ_ERR_ALIGNMENT;
  kvq::DecodeArgs a;
  a.c = view(cache);
  a.q = static_cast<const uint16_t*>(q);
  a.B = batch;
  a.Hq = q_heads;
  a.G = q_heads / cache->num_kv_heads;
  a.seq_lens = seq_lens;
  a.pos = nullptr;
  a.seq_of = nullptr;
  a.nseq = batch;
  a.table = block_table;
  a.mbps = max_blocks_per_seq;
  a.out = out;
  a.out_fp32 = out_fp32 ? 1 : 0;
  a.lse = lse;
  a.ws = static_cast<uint8_t*>(workspace);
  a.lay = L;
  a.err = err_word;
  a.ahead = (flags & KVQ_DECODE_GEOMETRY_READY) ? 1 : 0;
  if (kvq::launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_prefill(const kvq_cache_desc* cache, const void* q, int32_t n, int32_t q_heads,
                       const int32_t* seq_idx, const int32_t* pos, const void* k_new, const void* v_new,
                       const int32_t* block_table, int32_t batch, int32_t max_blocks_per_seq, void* out,
                       int32_t out_fp32, float* lse, void* workspace, size_t workspace_bytes, int32_t stream_ctas,
                       uint32_t* err_word, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (cache->window != 0) return KVQ_ERR_UNSUPPORTED;  // positions live in the block store only
  st = check_decode_shape(cache, n, q_heads);
  if (st != KVQ_OK) return st;
  if (n == 0) return KVQ_OK;
  if (!q || !seq_idx || !pos || !block_table || !out || max_blocks_per_seq < 1 || batch < 1)
    return KVQ_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_ALIGNMENT;
  if (stream_ctas < 0 && stream_ctas != KVQ_PREFILL_TILES) return KVQ_ERR_INVALID_ARG;
  const bool tiles_ok = kvq::prefill_tiles_supported(view(cache));
  if (stream_ctas == KVQ_PREFILL_TILES && !tiles_ok) return KVQ_ERR_UNSUPPORTED;
  bool tiles = stream_ctas == KVQ_PREFILL_TILES;
  if (stream_ctas == 0 && tiles_ok) {
    // Tiles once their CTAs fill at least 9/16 of the SMs; fewer tiles leave
    // the long prefixes to too few CTAs and split rows (every row one query
    // group of the decode split over all SMs) are faster.  Measured crossover
    // (8k-32k prefixes, int8, 32/8 heads): split rows ahead at 48 and 64 tile
    // CTAs (1.2-1.6x), tiles ahead at 96 (1.04-1.1x) and 128 (1.3x).
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      return KVQ_ERR_CUDA;
    tiles = prefill_tiles(n, q_heads, cache->num_kv_heads) * 16 >= 9ll * sms;
  }
  kvq::DecodeLayout L{};
  if (!tiles) {
    const int P = stream_ctas > 0 ? stream_ctas : auto_stream_ctas(cache, n, true);
    if (P <= 0) return KVQ_ERR_CUDA;
    L = kvq::decode_layout(n, q_heads, cache->num_kv_heads, 0, P, kvq::switch_blocks_for(cache->k_bits));
    if (!workspace || workspace_bytes < L.total) return KVQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KVQ_ERR_ALIGNMENT;
  }
  if (k_new) {  // the chunk's own keys and values first: quantize-on-write
    st = kvq_append(cache, k_new, v_new, n, seq_idx, pos, KVQ_APPEND_QUANT, block_table, batch, max_blocks_per_seq,
                    err_word, stream);
    if (st != KVQ_OK) return st;
  }
  kvq::DecodeArgs a;
  a.c = view(cache);
  a.q = static_cast<const uint16_t*>(q);
  a.B = n;
  a.Hq = q_heads;
  a.G = q_heads / cache->num_kv_heads;
  a.seq_lens = nullptr;
  a.pos = pos;
  a.seq_of = seq_idx;
  a.nseq = batch;
  a.table = block_table;
  a.mbps = max_blocks_per_seq;
  a.out = out;
  a.out_fp32 = out_fp32 ? 1 : 0;
  a.lse = lse;
  a.ws = static_cast<uint8_t*>(workspace);
  a.lay = L;
  a.err = err_word;
  const cudaError_t e = tiles ? kvq::launch_prefill_tiles(a, static_cast<cudaStream_t>(stream))
                              : kvq::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_prefill_workspace_size(const kvq_cache_desc* cache, int32_t n, int32_t q_heads, int32_t stream_ctas,
                                      size_t* bytes) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!bytes) return KVQ_ERR_INVALID_ARG;
  if (cache->window != 0) return KVQ_ERR_UNSUPPORTED;
  st = check_decode_shape(cache, n, q_heads);
  if (st != KVQ_OK) return st;
  if (stream_ctas < 0 && stream_ctas != KVQ_PREFILL_TILES) return KVQ_ERR_INVALID_ARG;
  if (stream_ctas == KVQ_PREFILL_TILES) {  // the tile path needs no workspace
    if (!kvq::prefill_tiles_supported(view(cache))) return KVQ_ERR_UNSUPPORTED;
    *bytes = 0;
    return KVQ_OK;
  }
  const int P = stream_ctas > 0 ? stream_ctas : auto_stream_ctas(cache, n, true);
  if (P <= 0) return KVQ_ERR_CUDA;
  *bytes = kvq::decode_layout(n, q_heads, cache->num_kv_heads, 0, P, kvq::switch_blocks_for(cache->k_bits)).total;
  return KVQ_OK;
}

kvq_status kvq_dequant(const kvq_cache_desc* cache, const int32_t* slots, int32_t n, float* k_out, float* v_out,
                       void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n < 0) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (!slots || !k_out || !v_out) return KVQ_ERR_INVALID_ARG;
  kvq::DequantArgs a;
  a.c = view(cache);
  a.slots = slots;
  a.n = n;
  a.k_out = k_out;
  a.v_out = v_out;
  if (kvq::launch_dequant(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

}  // extern "C"
