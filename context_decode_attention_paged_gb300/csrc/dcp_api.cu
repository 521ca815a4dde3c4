// C-ABI layer of libdcp: argument checks, split planning, kernel selection,
// the per-stream device status words, NVTX ranges.  Every public entry point
// is declared in include/dcp.h.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <utility>

#include "dcp_internal.h"

namespace dcp {

namespace {

// One status word per stream: the first device-side error since that
// stream's last read.  Streams get their own word in order of first use;
// once DCP_STATUS_STREAMS - 1 streams of a device have one, further streams
// share the last word.
__device__ int g_status[DCP_STATUS_STREAMS];

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
int* g_status_base[kMaxDevices] = {nullptr};
std::map<std::pair<int, cudaStream_t>, int> g_status_slot;
int g_status_used[kMaxDevices] = {0};

// Device address of the status word of `stream` on the current device (the
// first use on a device looks up the array's address).
int* status_ptr(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_base[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess || p == nullptr) return nullptr;
    g_status_base[dev] = static_cast<int*>(p);
  }
  const auto key = std::make_pair(dev, stream);
  auto it = g_status_slot.find(key);
  int slot;
  if (it != g_status_slot.end()) {
    slot = it->second;
  } else {
    slot = std::min(g_status_used[dev], DCP_STATUS_STREAMS - 1);
    if (g_status_used[dev] < DCP_STATUS_STREAMS - 1) ++g_status_used[dev];
    g_status_slot.emplace(key, slot);
  }
  return g_status_base[dev] + slot;
}

// NVTX range around a C-ABI call (no cost unless a profiler is attached)
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

dcp_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? DCP_OK : DCP_ERR_CUDA; }

// Fill AttnArgs from the public arguments; INVALID_ARG / UNSUPPORTED on bad input.
dcp_status_t make_args(const dcp_attn_desc_t* d, int32_t dcp_size, int32_t interleave,
                       float scale, int32_t causal_q_len, AttnArgs* a) {
  if (!d) return DCP_ERR_INVALID_ARG;
  if (d->kind != DCP_ATTN_GQA && d->kind != DCP_ATTN_MLA) return DCP_ERR_INVALID_ARG;
  if (d->batch < 1 || d->q_len < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1 ||
      d->head_dim_qk < 1 || d->head_dim_v < 1 || d->block_size < 1 || d->num_blocks < 1 ||
      d->max_local_blocks < 1)
    return DCP_ERR_INVALID_ARG;
  if (dcp_size < 1 || dcp_size > 32 || interleave < 1) return DCP_ERR_INVALID_ARG;
  if (causal_q_len != d->q_len) return DCP_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads) return DCP_ERR_INVALID_ARG;
  if (d->kind == DCP_ATTN_MLA && (d->num_kv_heads != 1 || d->head_dim_v > d->head_dim_qk))
    return DCP_ERR_INVALID_ARG;
  if (d->kind == DCP_ATTN_GQA && d->head_dim_v != d->head_dim_qk) return DCP_ERR_INVALID_ARG;
  if (d->head_dim_qk % 8 || d->head_dim_v % 4) return DCP_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || scale != scale) return DCP_ERR_INVALID_ARG;
  // element counts must fit the kernels' 64-bit index math and int32 grids
  if ((long long)dcp_size * d->batch > (1LL << 30)) return DCP_ERR_UNSUPPORTED;
  a->kind = d->kind;
  a->B = d->batch;
  a->Lq = d->q_len;
  a->Hq = d->num_q_heads;
  a->Hkv = d->num_kv_heads;
  a->Dqk = d->head_dim_qk;
  a->Dv = d->head_dim_v;
  a->bs = d->block_size;
  a->num_blocks = d->num_blocks;
  a->max_lb = d->max_local_blocks;
  a->N = dcp_size;
  a->I = interleave;
  a->scale = scale;
  return DCP_OK;
}

// The kernel that will run for these arguments, and its split plan.
enum class Impl { kSimt, kMlaTc, kGqaTc };

Impl select_impl(const AttnArgs& a) {
  if (mla_tc_supported(a)) return Impl::kMlaTc;
  if (gqa_tc_supported(a)) return Impl::kGqaTc;
  return Impl::kSimt;
}

SplitPlan plan_for(const AttnArgs& a, Impl impl, int sm_count) {
  switch (impl) {
    case Impl::kMlaTc:
      return plan_attn_mla_tc(a, sm_count);
    case Impl::kGqaTc:
      return plan_attn_gqa_tc(a, sm_count);
    case Impl::kSimt:
    default:
      return plan_attn_simt(a, sm_count);
  }
}

}  // namespace

namespace {
std::mutex g_hooks_mu;
TestHooks g_hooks = {2000000000ull, -1};
}  // namespace

TestHooks test_hooks() {
  std::lock_guard<std::mutex> lock(g_hooks_mu);
  return g_hooks;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 148;
  return n;
}

SplitPlan plan_splits(const AttnArgs& a, int sm_count, int tile_tokens, int units_per_split) {
  SplitPlan p;
  const long long max_local = (long long)a.max_lb * a.bs;
  const long long base_units = (long long)a.N * a.B * units_per_split;
  const long long target = 2LL * sm_count;
  long long n = 1;
  if (base_units < target && max_local > 4LL * tile_tokens) {
    // Split count by a wave model: units run in waves of sm_count CTAs and a
    // unit costs its tiles plus about kUnitStartTiles of start-up and drain,
    // so pick the count with the fewest waves x (tiles per split + start-up).
    constexpr long long kUnitStartTiles = 4;
    const long long tiles = (max_local + tile_tokens - 1) / tile_tokens;
    const long long n_hi = std::max<long long>(1, std::min<long long>(32, max_local / (4LL * tile_tokens)));
    long long best = -1;
    for (long long c = 1; c <= n_hi; ++c) {
      const long long waves = (base_units * c + sm_count - 1) / sm_count;
      const long long cost = waves * ((tiles + c - 1) / c + kUnitStartTiles);
      if (best < 0 || cost < best) {
        best = cost;
        n = c;
      }
    }
  }
  long long per = (max_local + n - 1) / n;
  per = (per + tile_tokens - 1) / tile_tokens * tile_tokens;
  if (per < tile_tokens) per = tile_tokens;
  n = (max_local + per - 1) / per;
  if (n < 1) n = 1;
  p.lpt_order = false;
  p.order_offset = 0;
  p.n_split = (int)n;
  p.split_tokens = (int)std::min<long long>(per, 1LL << 30);
  p.ws_bytes = 0;
  if (p.n_split > 1) {
    const size_t rows = (size_t)a.N * a.B * a.Lq * a.Hq;
    p.ws_bytes = align256(rows * p.n_split * a.Dv * sizeof(float)) + rows * p.n_split * sizeof(float);
  }
  return p;
}

}  // namespace dcp

using namespace dcp;

extern "C" {

const char* dcp_status_string(dcp_status_t s) {
  switch (s) {
    case DCP_OK: return "DCP_OK";
    case DCP_ERR_INVALID_ARG: return "DCP_ERR_INVALID_ARG";
    case DCP_ERR_UNSUPPORTED: return "DCP_ERR_UNSUPPORTED";
    case DCP_ERR_CUDA: return "DCP_ERR_CUDA";
    case DCP_ERR_TIMEOUT: return "DCP_ERR_TIMEOUT";
    case DCP_ERR_BOUNDS: return "DCP_ERR_BOUNDS";
  }
  return "DCP_ERR_UNKNOWN";
}

dcp_status_t dcp_build_slot_map(const int32_t* seq_lens, int32_t batch, int32_t block_size,
                                int32_t interleave, int32_t dcp_size, int32_t* local_seq_lens,
                                int32_t* local_num_blocks, int32_t* shard_of, int32_t* local_pos,
                                int32_t max_seq, void* stream) {
  NvtxRange range("dcp_build_slot_map");
  if (batch < 0 || block_size < 1 || interleave < 1 || dcp_size < 1) return DCP_ERR_INVALID_ARG;
  if (batch > 0 && (!seq_lens || !local_seq_lens || !local_num_blocks)) return DCP_ERR_INVALID_ARG;
  if ((shard_of == nullptr) != (local_pos == nullptr)) return DCP_ERR_INVALID_ARG;
  if (shard_of && max_seq < 1) return DCP_ERR_INVALID_ARG;
  if ((long long)batch * dcp_size > (1LL << 30)) return DCP_ERR_INVALID_ARG;
  // one thread per (request, token) of the optional maps: the grid must fit
  if (shard_of && (long long)batch * max_seq > (long long)INT_MAX * 256) return DCP_ERR_INVALID_ARG;
  if (batch == 0) return DCP_OK;
  int* st = status_ptr(static_cast<cudaStream_t>(stream));
  if (!st) return DCP_ERR_CUDA;
  return from_cuda(launch_slot_map(seq_lens, batch, block_size, interleave, dcp_size,
                                   local_seq_lens, local_num_blocks, shard_of, local_pos, max_seq,
                                   st, static_cast<cudaStream_t>(stream)));
}

size_t dcp_decode_attn_workspace_size(const dcp_attn_desc_t* d, int32_t dcp_size) {
  AttnArgs a{};
  if (make_args(d, dcp_size, 1, 1.0f, d ? d->q_len : 1, &a) != DCP_OK) return 0;
  return plan_for(a, select_impl(a), device_sm_count()).ws_bytes;
}

dcp_status_t dcp_decode_attn(const dcp_attn_desc_t* d, const void* q, const void* kv_cache,
                             const int32_t* block_tables, const int32_t* seq_lens,
                             int32_t dcp_size, int32_t interleave, float scale,
                             int32_t causal_q_len, float* partial_out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange range("dcp_decode_attn");
  AttnArgs a{};
  dcp_status_t st = make_args(d, dcp_size, interleave, scale, causal_q_len, &a);
  if (st != DCP_OK) return st;
  if (!q || !kv_cache || !block_tables || !seq_lens || !partial_out || !lse)
    return DCP_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(partial_out, 16) || !aligned(lse, 4))
    return DCP_ERR_INVALID_ARG;
  const Impl impl = select_impl(a);
  const SplitPlan plan = plan_for(a, impl, device_sm_count());
  if (plan.ws_bytes > 0 &&
      (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)))
    return DCP_ERR_INVALID_ARG;
  a.q = q;
  a.kv = kv_cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.partial_out = partial_out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.status = status_ptr(static_cast<cudaStream_t>(stream));
  if (!a.status) return DCP_ERR_CUDA;
  a.stream = static_cast<cudaStream_t>(stream);
  switch (impl) {
    case Impl::kMlaTc:
      return from_cuda(launch_attn_mla_tc(a, plan));
    case Impl::kGqaTc:
      return from_cuda(launch_attn_gqa_tc(a, plan));
    case Impl::kSimt:
    default:
      return from_cuda(launch_attn_simt(a, plan));
  }
}

dcp_status_t dcp_kv_cache_write(const dcp_attn_desc_t* d, const void* new_k, const void* new_v,
                                void* kv_cache, const int32_t* block_tables, const int32_t* seq_lens,
                                int32_t dcp_size, int32_t interleave, int32_t n_new, void* stream) {
  NvtxRange range("dcp_kv_cache_write");
  if (!d || !new_k || !kv_cache || !block_tables || !seq_lens) return DCP_ERR_INVALID_ARG;
  if (d->kind != DCP_ATTN_GQA && d->kind != DCP_ATTN_MLA) return DCP_ERR_INVALID_ARG;
  const bool gqa = d->kind == DCP_ATTN_GQA;
  if (gqa != (new_v != nullptr)) return DCP_ERR_INVALID_ARG;
  if (d->batch < 1 || d->num_kv_heads < 1 || d->head_dim_qk < 1 || d->block_size < 1 || d->num_blocks < 1 ||
      d->max_local_blocks < 1 || dcp_size < 1 || interleave < 1 || n_new < 1)
    return DCP_ERR_INVALID_ARG;
  if (!gqa && d->num_kv_heads != 1) return DCP_ERR_INVALID_ARG;
  const long long row_bytes = 2LL * d->head_dim_qk * (gqa ? d->num_kv_heads : 1);
  if (row_bytes % 16 || row_bytes > (1LL << 20)) return DCP_ERR_INVALID_ARG;
  if ((long long)d->batch * dcp_size * d->max_local_blocks > (1LL << 31) ||
      (long long)d->num_blocks * d->block_size > (1LL << 31))
    return DCP_ERR_INVALID_ARG;
  if (!aligned(new_k, 16) || !aligned(kv_cache, 16) || (new_v && !aligned(new_v, 16)))
    return DCP_ERR_INVALID_ARG;
  int* st = status_ptr(static_cast<cudaStream_t>(stream));
  if (!st) return DCP_ERR_CUDA;
  return from_cuda(launch_kv_write(new_k, new_v, kv_cache, block_tables, seq_lens, d->batch, n_new, dcp_size,
                                   interleave, d->block_size, d->max_local_blocks, d->num_blocks,
                                   (int)row_bytes, st, static_cast<cudaStream_t>(stream)));
}

dcp_status_t dcp_merge(const float* partial_out, const float* lse, int32_t dcp_size,
                       int32_t batch, int32_t q_len, int32_t num_q_heads, int32_t head_dim_v,
                       void* out, float* out_lse, void* stream) {
  NvtxRange range("dcp_merge");
  if (!partial_out || !lse || !out) return DCP_ERR_INVALID_ARG;
  if (dcp_size < 1 || dcp_size > 32 || batch < 1 || q_len < 1 || num_q_heads < 1 ||
      head_dim_v < 4)
    return DCP_ERR_INVALID_ARG;
  if (num_q_heads % dcp_size || head_dim_v % 4) return DCP_ERR_INVALID_ARG;
  if (!aligned(partial_out, 16) || !aligned(out, 8) || !aligned(lse, 4) ||
      (out_lse && !aligned(out_lse, 4)))
    return DCP_ERR_INVALID_ARG;
  return from_cuda(launch_merge(partial_out, lse, dcp_size, batch, q_len, num_q_heads,
                                head_dim_v, out, out_lse, static_cast<cudaStream_t>(stream)));
}

// Test-only (see TestHooks in dcp_internal.h); not declared in include/dcp.h.
DCP_API void dcp_testing_set_hooks(unsigned long long wait_ns, int32_t skip_tile) {
  std::lock_guard<std::mutex> lock(g_hooks_mu);
  g_hooks.wait_ns = wait_ns > 0 ? wait_ns : 2000000000ull;
  g_hooks.skip_tile = skip_tile;
}

dcp_status_t dcp_get_last_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* p = status_ptr(s);
  if (!p) return DCP_ERR_CUDA;
  // read and clear the word on the stream itself: later work on the stream
  // sees it cleared; no other stream is waited for
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DCP_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return DCP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DCP_ERR_CUDA;
  return static_cast<dcp_status_t>(v);
}

int32_t dcp_decode_attn_launches(const dcp_attn_desc_t* d, int32_t dcp_size) {
  AttnArgs a{};
  if (make_args(d, dcp_size, 1, 1.0f, d ? d->q_len : 1, &a) != DCP_OK) return 0;
  const SplitPlan plan = plan_for(a, select_impl(a), device_sm_count());
  return 1 + (plan.n_split > 1 ? 1 : 0) + (plan.lpt_order ? 1 : 0);
}

int32_t dcp_decode_attn_kernel_kind(const dcp_attn_desc_t* d, int32_t dcp_size) {
  AttnArgs a{};
  if (make_args(d, dcp_size, 1, 1.0f, d ? d->q_len : 1, &a) != DCP_OK) return DCP_KERNEL_NONE;
  switch (select_impl(a)) {
    case Impl::kMlaTc: return DCP_KERNEL_MLA_TC;
    case Impl::kGqaTc: return DCP_KERNEL_GQA_TC;
    case Impl::kSimt:
    default: return DCP_KERNEL_SIMT;
  }
}

}  // extern "C"
