// Device-side helpers shared by the kernel translation units.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dcp.h"

namespace dcp {

// Record the first device-side error of a call sequence (read and cleared by
// dcp_get_last_device_status).
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Shard-local token count of a request of length S on shard r
// (closed form of the (t / I) % N rule; tokens packed in global order).
__device__ __forceinline__ int local_len(int S, int r, int I, int N) {
  const long long period = (long long)I * N;
  const long long full = (long long)(S / period) * I;
  long long rem = (long long)(S % period) - (long long)r * I;
  rem = rem < 0 ? 0 : (rem > I ? I : rem);
  return (int)(full + rem);
}

// Global position of shard r's local token j.
__device__ __forceinline__ long long global_pos(int j, int r, int I, int N) {
  return (long long)(j / I) * I * N + (long long)r * I + (j % I);
}

// Number of shard-local tokens whose global position is <= p (p >= -1).
__device__ __forceinline__ int local_count_upto(long long p, int r, int I, int N) {
  return p < 0 ? 0 : local_len((int)(p + 1), r, I, N);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace dcp
