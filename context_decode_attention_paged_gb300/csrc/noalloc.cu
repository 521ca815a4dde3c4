// dcp_decode_attn_noalloc: dcp_decode_attn for callers that cannot allocate
// device memory.
//
// dcp_decode_attn needs caller-provided scratch when it splits a shard's keys
// across several CTAs (small batches, long contexts).  Some callers cannot
// call cudaMalloc at that point: code running inside a memory pool owned by
// another runtime, plugins handed only input and output buffers, or a serving
// loop that forbids allocation on its decode path.  This entry point takes the
// scratch from a fixed array compiled into the library instead.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it (DCP_NOALLOC_SCRATCH_BYTES each).  All calls share it: two calls
// whose kernels overlap on the GPU (different streams, or different host
// threads) race on it and give wrong results.  Calls ordered on one stream are
// fine.  Nothing in it must start at zero: the attention kernels write every
// split slot they later read, so the previous call's contents are harmless.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dcp.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DCP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device; looked up once per
// device (the first call on a device does this set-up).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

dcp_status_t dcp_decode_attn_noalloc(const dcp_attn_desc_t* d, const void* q,
                                     const void* kv_cache, const int32_t* block_tables,
                                     const int32_t* seq_lens, int32_t dcp_size,
                                     int32_t interleave, float scale, int32_t causal_q_len,
                                     float* partial_out, float* lse, void* stream) {
  if (!d) return DCP_ERR_INVALID_ARG;
  const size_t need = dcp_decode_attn_workspace_size(d, dcp_size);
  if (need > (size_t)DCP_NOALLOC_SCRATCH_BYTES) return DCP_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (need > 0) {
    ws = scratch_address();
    if (!ws) return DCP_ERR_CUDA;
  }
  return dcp_decode_attn(d, q, kv_cache, block_tables, seq_lens, dcp_size, interleave, scale,
                         causal_q_len, partial_out, lse, ws, need, stream);
}

}  // extern "C"
