// Storing the newest tokens of every request in the sharded cache.
//
// "Context Parallel Guide", section "Overview": DCP shards the KV cache storage
// among the ranks of the DCP group, so each new token's KV row is stored once,
// in the shard that owns its position; the owner and the shard-local index
// come from the interleave rule (section "Decode Context Parallel"; vLLM DCP
// blog, "解碼上下文並行 (DCP) 原理解析").
//
// One warp per new token: it finds the token's shard r = (t / I) % N, local
// index j = (t / (I N)) I + t % I and cache cell (block_tables[r][b][j / bs],
// slot j % bs), then copies the row with 16-byte loads and stores (GQA: the K
// row and the V row of every KV head; MLA: the 576-value latent row).  A
// decode step writes B x n_new rows, so the launch is latency-bound; the
// copies are coalesced and every byte is touched once.
#include "dcp_device.cuh"
#include "dcp_internal.h"

namespace dcp {
namespace {

constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
kv_write_kernel(const uint4* __restrict__ new_k, const uint4* __restrict__ new_v, uint4* __restrict__ pool_k,
                uint4* __restrict__ pool_v, const int32_t* __restrict__ block_tables,
                const int32_t* __restrict__ seq_lens, int B, int n_new, int N, int I, int bs, int max_lb,
                int num_blocks, int row16, int* status) {
  const long long token = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= (long long)B * n_new) return;
  const int b = (int)(token / n_new), i = (int)(token % n_new);
  const int S = seq_lens[b];
  if (S < n_new) {
    if (lane == 0) set_status(status, DCP_ERR_BOUNDS);
    return;
  }
  const long long t = (long long)S - n_new + i;
  const int r = (int)((t / I) % N);
  const long long j = (t / ((long long)I * N)) * I + t % I;
  const long long jb = j / bs;
  if (jb >= max_lb) {
    if (lane == 0) set_status(status, DCP_ERR_BOUNDS);
    return;
  }
  const int blk = block_tables[((long long)r * B + b) * max_lb + jb];
  if ((unsigned)blk >= (unsigned)num_blocks) {
    if (lane == 0) set_status(status, DCP_ERR_BOUNDS);
    return;
  }
  const long long cell = ((long long)blk * bs + j % bs) * row16;
  const long long src = token * row16;
  for (int u = lane; u < row16; u += 32) pool_k[cell + u] = new_k[src + u];
  if (new_v)
    for (int u = lane; u < row16; u += 32) pool_v[cell + u] = new_v[src + u];
}

}  // namespace

cudaError_t launch_kv_write(const void* new_k, const void* new_v, void* kv_cache, const int32_t* block_tables,
                            const int32_t* seq_lens, int B, int n_new, int N, int I, int bs, int max_lb,
                            int num_blocks, int row_bytes, int* status, cudaStream_t stream) {
  const long long tokens = (long long)B * n_new;
  if (tokens == 0) return cudaSuccess;
  const int row16 = row_bytes / 16;
  uint4* pool_k = static_cast<uint4*>(kv_cache);
  uint4* pool_v = new_v ? pool_k + (long long)num_blocks * bs * row16 : nullptr;
  const long long blocks = (tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  kv_write_kernel<<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, stream>>>(
      static_cast<const uint4*>(new_k), static_cast<const uint4*>(new_v), pool_k, pool_v, block_tables, seq_lens, B,
      n_new, N, I, bs, max_lb, num_blocks, row16, status);
  return cudaGetLastError();
}

}  // namespace dcp
