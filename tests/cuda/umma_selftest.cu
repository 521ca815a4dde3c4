// Self-test of the tcgen05 operand forms used by the attention kernels, on one
// CTA, against torch matmuls in the test:
//   D1[128][64]  = A[128][288] . B[64][dims]^T   A from TMEM (bf16 pairs),
//                  B K-major: four 64-dim 128B-swizzled TMA boxes + one
//                  32-dim 64B-swizzled box (dims 0..255 and 512..543 of B)
//   D2[128][256] = P[128][64] . B[64][0..255]    P from TMEM, B MN-major
//                  (the same shared-memory tile read as the value operand)
// Built by the test with nvcc; not part of libdcp.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dcp_sm100.cuh"
#include "dcp_tma.h"

using namespace dcp::sm100;

namespace {

constexpr uint32_t kChunk = 64 * 128;    // one 64x64 bf16 box, 128B rows
constexpr uint32_t kRope = 64 * 64;      // one 64x32 bf16 box, 64B rows
constexpr uint32_t kTxBytes = 4 * kChunk + kRope;
constexpr uint64_t kLimitNs = 2000000000ull;

__global__ void __launch_bounds__(128, 1)
umma_probe_kernel(const __grid_constant__ CUtensorMap tm128, const __grid_constant__ CUtensorMap tm64,
                  const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ P,
                  float* __restrict__ D1, float* __restrict__ D2, int* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tile = smem;                               // 4 chunks + rope box
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 5 * kChunk);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  const uint32_t bar_tma = smem_u32(&bars[0]);
  const uint32_t bar_mma = smem_u32(&bars[1]);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (tid == 0) {
    prefetch_tmap(&tm128);
    prefetch_tmap(&tm64);
    mbar_arrive_expect_tx(bar_tma, kTxBytes);
    for (int c = 0; c < 4; ++c) tma_load_2d(smem_u32(tile + c * kChunk), &tm128, c * 64, 0, bar_tma);
    tma_load_2d(smem_u32(tile + 4 * kChunk), &tm64, 512, 0, bar_tma);
  }

  // A -> TMEM cols [0,144), P -> cols [144,176); thread tid owns row/lane tid
  const uint32_t lane_base = taddr(tbase, (uint32_t)(warp * 32), 0);
  for (int c = 0; c < 9; ++c) {
    uint32_t v[16];
    for (int k = 0; k < 16; ++k) {
      const int d = c * 32 + 2 * k;
      v[k] = pack_bf16x2(__bfloat162float(A[tid * 288 + d]), __bfloat162float(A[tid * 288 + d + 1]));
    }
    tmem_st16(lane_base + c * 16, v);
  }
  for (int c = 0; c < 2; ++c) {
    uint32_t v[16];
    for (int k = 0; k < 16; ++k) {
      const int d = c * 32 + 2 * k;
      v[k] = pack_bf16x2(__bfloat162float(P[tid * 64 + d]), __bfloat162float(P[tid * 64 + d + 1]));
    }
    tmem_st16(lane_base + 144 + c * 16, v);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (tid == 0) {
    bool ok = mbar_wait(bar_tma, 0, kLimitNs);
    if (!ok) {
      atomicExch(status, 4);
    } else {
      const uint32_t id_qk = idesc_bf16(128, 64, false);
      for (int k = 0; k < 18; ++k) {
        uint64_t bdesc;
        if (k < 16) {
          bdesc = smem_desc(smem_u32(tile + (k / 4) * kChunk + (k % 4) * 32), 16, 1024, kSw128);
        } else {
          bdesc = smem_desc(smem_u32(tile + 4 * kChunk + (k - 16) * 32), 16, 512, kSw64);
        }
        mma_ts(tbase + 192, tbase + 8 * k, bdesc, id_qk, k > 0);
      }
      const uint32_t id_pv = idesc_bf16(128, 256, true);
      for (int k = 0; k < 4; ++k) {
        const uint64_t bdesc = smem_desc(smem_u32(tile + k * 2048), kChunk, 1024, kSw128);
        mma_ts(tbase + 256, tbase + 144 + 8 * k, bdesc, id_pv, k > 0);
      }
      mma_commit(bar_mma);
    }
  }
  __syncwarp();
  const bool done = (*status == 0) ? mbar_wait(bar_mma, 0, kLimitNs) : false;
  tc_fence_after();
  if (done) {
    for (int c = 0; c < 4; ++c) {
      uint32_t r[16];
      tmem_ld16(lane_base + 192 + c * 16, r);
      tmem_wait_ld();
      for (int k = 0; k < 16; ++k) D1[tid * 64 + c * 16 + k] = __uint_as_float(r[k]);
    }
    for (int c = 0; c < 16; ++c) {
      uint32_t r[16];
      tmem_ld16(lane_base + 256 + c * 16, r);
      tmem_wait_ld();
      for (int k = 0; k < 16; ++k) D2[tid * 256 + c * 16 + k] = __uint_as_float(r[k]);
    }
  } else if (tid == 0) {
    atomicExch(status, 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace

extern "C" int umma_probe(const void* A, const void* B, const void* P, float* D1, float* D2,
                          int* status) {
  CUtensorMap tm128, tm64;
  const uint64_t dims[2] = {576, 64};
  const uint64_t strides[1] = {576 * 2};
  const uint32_t box128[2] = {64, 64};
  const uint32_t box64[2] = {32, 64};
  if (!dcp::make_tensor_map_bf16(&tm128, B, 2, dims, strides, box128, CU_TENSOR_MAP_SWIZZLE_128B))
    return -1;
  if (!dcp::make_tensor_map_bf16(&tm64, B, 2, dims, strides, box64, CU_TENSOR_MAP_SWIZZLE_64B))
    return -2;
  const int smem = 5 * kChunk + 1024 + 64;
  cudaError_t e = cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return (int)e;
  umma_probe_kernel<<<1, 128, smem>>>(tm128, tm64, static_cast<const __nv_bfloat16*>(A),
                                      static_cast<const __nv_bfloat16*>(P), D1, D2, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}
