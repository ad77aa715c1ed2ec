// kvq_decode_static_scratch: the decode entry point for callers that cannot
// allocate device memory.  The split-attention scratch (partial records and
// merge counters) lives in one fixed file-scope device array instead of a
// caller-provided workspace; nothing here calls cudaMalloc, cudaFree or any
// allocating routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvq.h"

namespace {

constexpr size_t kStaticScratchBytes = KVQ_STATIC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// In host code g_decode_scratch names a host-side stand-in, not device memory:
// the device address is looked up at set-up, once per device, with that
// device current, and cached here together with the CUDA context it belongs
// to.  A later call under another context (after cudaDeviceReset, or once the
// primary context has been torn down and recreated) repeats the set-up, so a
// cached address never outlives the module instance it points into.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchEntry {
  CUcontext ctx;
  void* addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry-point query (no link
// against the driver library is needed); null if it cannot be resolved.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static const CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return CtxGetCurrentFn(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

kvq_status current_context(CUcontext* ctx) {
  *ctx = nullptr;
  const CtxGetCurrentFn fn = ctx_get_current();
  if (fn && fn(ctx) != CUDA_SUCCESS) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  CUcontext ctx = nullptr;
  if (current_context(&ctx) != KVQ_OK) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchEntry& e = g_scratch[dev];
  if (!e.addr || !ctx || e.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    // the lookup binds the device's primary context if none was current
    if (current_context(&ctx) != KVQ_OK) return KVQ_ERR_CUDA;
    e.ctx = ctx;
    e.addr = p;
  }
  *out = e.addr;
  return KVQ_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" kvq_status kvq_decode_static_scratch(const kvq_cache_desc* cache, const void* q, int32_t batch,
                                                int32_t q_heads, const int32_t* seq_lens, const int32_t* block_table,
                                                int32_t max_blocks_per_seq, void* out, int32_t out_fp32, float* lse,
                                                int32_t stream_ctas, uint32_t* err_word, void* stream) {
  kvq_decode_plan plan;
  kvq_status st = kvq_decode_device_plan(cache, batch, q_heads, stream_ctas, &plan);
  if (st != KVQ_OK) return st;
  if (batch == 0) return KVQ_OK;
  if (plan.workspace_bytes > kStaticScratchBytes) return KVQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  // The array keeps whatever the previous call left; the merge counters (the
  // first units * 4 bytes, padded to 256) must start every call at zero.
  const size_t counter_bytes = round_up(size_t(plan.units) * 4, 256);
  if (cudaMemsetAsync(scratch, 0, counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return kvq_decode(cache, q, batch, q_heads, seq_lens, block_table, max_blocks_per_seq, out, out_fp32, lse, scratch,
                    kStaticScratchBytes, stream_ctas, err_word, stream);
}
