// Step a1: token -> shard slot map.
//
// vLLM DCP blog, "解碼上下文並行 (DCP) 原理解析": each rank holds a range of
// token positions of a request; the interleave flag of the vLLM Ascend Context
// Parallel Guide sets the run length.  shard(t) = (t / I) % N and the local
// index packs each shard's tokens densely in global order.  Integer only.
#include "dcp_device.cuh"
#include "dcp_internal.h"

namespace dcp {
namespace {

// One thread per (shard, request): local lengths and block counts.
__global__ void slot_map_lens_kernel(const int32_t* __restrict__ seq_lens, int B, int bs, int I,
                                     int N, int32_t* __restrict__ local_seq_lens,
                                     int32_t* __restrict__ local_num_blocks, int* status) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= N * B) return;
  const int r = idx / B, b = idx % B;
  int S = seq_lens[b];
  if (S < 0) {
    set_status(status, DCP_ERR_BOUNDS);
    S = 0;
  }
  const int n = local_len(S, r, I, N);
  local_seq_lens[idx] = n;
  local_num_blocks[idx] = (n + bs - 1) / bs;
}

// One thread per (request, token): owning shard and local index, -1 past the end.
__global__ void slot_map_tokens_kernel(const int32_t* __restrict__ seq_lens, int B, int I, int N,
                                       int max_seq, int32_t* __restrict__ shard_of,
                                       int32_t* __restrict__ local_pos) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * max_seq) return;
  const int b = (int)(idx / max_seq);
  const int t = (int)(idx % max_seq);
  if (t < seq_lens[b]) {
    shard_of[idx] = (t / I) % N;
    local_pos[idx] = (int)((long long)(t / ((long long)I * N)) * I + t % I);
  } else {
    shard_of[idx] = -1;
    local_pos[idx] = -1;
  }
}

}  // namespace

cudaError_t launch_slot_map(const int32_t* seq_lens, int B, int bs, int I, int N,
                            int32_t* local_seq_lens, int32_t* local_num_blocks,
                            int32_t* shard_of, int32_t* local_pos, int max_seq, int* status,
                            cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int threads = 256;
  const int n = N * B;
  slot_map_lens_kernel<<<(n + threads - 1) / threads, threads, 0, stream>>>(
      seq_lens, B, bs, I, N, local_seq_lens, local_num_blocks, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || shard_of == nullptr) return e;
  const long long m = (long long)B * max_seq;
  const long long blocks = (m + threads - 1) / threads;
  slot_map_tokens_kernel<<<(unsigned)blocks, threads, 0, stream>>>(seq_lens, B, I, N, max_seq,
                                                                   shard_of, local_pos);
  return cudaGetLastError();
}

}  // namespace dcp
