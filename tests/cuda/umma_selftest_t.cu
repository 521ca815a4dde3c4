// Self-test of the tcgen05 operand forms of the transposed (keys-as-M) GQA
// kernel, on one CTA, against torch matmuls in the test.  For NCOL in
// {16, 32, 64}:
//   D3[128][NCOL] = K[128][128] . Q[NCOL][128]^T   A = K tile (two 64-dim
//                   128B-swizzled TMA boxes, K-major), B = Q rows stored by
//                   threads under the 128-byte swizzle (K-major)
//   D4[128][NCOL] = V[128][128]^T . P[128][NCOL]   A = V tile read MN-major,
//                   B = P rows stored by threads under the NCOL-wide swizzle
//                   (32/64/128 bytes, MN-major)
//   D5            = the same product with P loaded by TMA under that swizzle
//   D6, D7        = D3 with descriptors built once and advanced per K-step by
//                   adding the byte offset >> 4 to the start address: D6 as a
//                   64-bit add, D7 on the low 32-bit word only
// Built by the test with nvcc; not part of libdcp.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dcp_sm100.cuh"
#include "dcp_tma.h"

using namespace dcp::sm100;

namespace {

constexpr uint32_t kChunk = 128 * 128;   // 128 rows x 64 dims bf16
constexpr uint64_t kLimitNs = 2000000000ull;

// descriptor + offset on the low 32-bit word (start address field), the high
// word (strides, version, swizzle) passed through untouched
__device__ __forceinline__ uint64_t desc_add_lo(uint64_t d, uint32_t off) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"((uint32_t)d + off), "r"((uint32_t)(d >> 32)));
  return r;
}

template <int NCOL>
__device__ __forceinline__ uint32_t pchunk(uint32_t c, uint32_t k) {
  return NCOL == 16 ? (c ^ ((k >> 2) & 1u)) : NCOL == 32 ? (c ^ ((k >> 1) & 3u)) : (c ^ (k & 7u));
}

template <int NCOL>
__global__ void __launch_bounds__(128, 1)
umma_t_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_p, const __nv_bfloat16* __restrict__ Q,
              const __nv_bfloat16* __restrict__ P, float* __restrict__ D3, float* __restrict__ D4,
              float* __restrict__ D5, float* __restrict__ D6, float* __restrict__ D7, int* __restrict__ status) {
  constexpr uint32_t kPitch = NCOL * 2, kPBytes = 128 * kPitch;
  constexpr uint32_t kSwz = NCOL == 16 ? kSw32 : NCOL == 32 ? kSw64 : kSw128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ks = smem;                       // 2 chunks
  uint8_t* vs = ks + 2 * kChunk;            // 2 chunks
  uint8_t* qs = vs + 2 * kChunk;            // 2 x NCOL x 128 B
  uint8_t* pm = qs + 2 * NCOL * 128;        // P by threads
  uint8_t* pt = pm + ((kPBytes + 1023) & ~1023u);   // P by TMA
  uint64_t* bars = reinterpret_cast<uint64_t*>(pt + ((kPBytes + 1023) & ~1023u));
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
  // Q rows (K-major, 128B swizzle) and P rows (MN-major, NCOL-wide swizzle)
  for (int idx = tid; idx < NCOL * 16; idx += 128) {
    const int h = idx / 16, ch = (idx % 16) / 8, c = idx % 8;
    const uint4 v = reinterpret_cast<const uint4*>(Q + h * 128 + ch * 64)[c];
    *reinterpret_cast<uint4*>(qs + ch * NCOL * 128 + h * 128 + ((c ^ (h & 7)) << 4)) = v;
  }
  for (int c = 0; c < NCOL / 8; ++c) {
    const uint4 v = reinterpret_cast<const uint4*>(P + tid * NCOL)[c];
    *reinterpret_cast<uint4*>(pm + tid * kPitch + (pchunk<NCOL>((uint32_t)c, (uint32_t)tid) << 4)) = v;
  }
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (tid == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_p);
    mbar_arrive_expect_tx(bar_tma, 4 * kChunk + kPBytes);
    for (int c = 0; c < 2; ++c) {
      tma_load_2d(smem_u32(ks + c * kChunk), &tm_k, c * 64, 0, bar_tma);
      tma_load_2d(smem_u32(vs + c * kChunk), &tm_v, c * 64, 0, bar_tma);
    }
    tma_load_2d(smem_u32(pt), &tm_p, 0, 0, bar_tma);
    if (!mbar_wait(bar_tma, 0, kLimitNs)) {
      atomicExch(status, 4);
    } else {
      const uint32_t id_qk = idesc_bf16_ab(128, NCOL, false, false);
      const uint32_t id_pv = idesc_bf16_ab(128, NCOL, true, true);
      for (int k = 0; k < 8; ++k) {
        const uint64_t a = smem_desc(smem_u32(ks + (k >> 2) * kChunk + (k & 3) * 32), 16, 1024, kSw128);
        const uint64_t b = smem_desc(smem_u32(qs + (k >> 2) * NCOL * 128 + (k & 3) * 32), 16, 1024, kSw128);
        mma_ss(tbase, a, b, id_qk, k > 0);
      }
      // D6 / D7: base descriptors plus compile-time K-step offsets
      const uint64_t ka = smem_desc(smem_u32(ks), 16, 1024, kSw128);
      const uint64_t qb = smem_desc(smem_u32(qs), 16, 1024, kSw128);
#pragma unroll
      for (uint32_t k = 0; k < 8; ++k)
        mma_ss(tbase + 3 * NCOL, ka + (((k >> 2) * kChunk + (k & 3) * 32) >> 4),
               qb + (((k >> 2) * NCOL * 128 + (k & 3) * 32) >> 4), id_qk, k > 0);
#pragma unroll
      for (uint32_t k = 0; k < 8; ++k)
        mma_ss(tbase + 4 * NCOL, desc_add_lo(ka, ((k >> 2) * kChunk + (k & 3) * 32) >> 4),
               desc_add_lo(qb, ((k >> 2) * NCOL * 128 + (k & 3) * 32) >> 4), id_qk, k > 0);
      for (int k = 0; k < 8; ++k) {
        const uint64_t a = smem_desc(smem_u32(vs + k * 2048), kChunk, 1024, kSw128);
        const uint64_t b4 = smem_desc(smem_u32(pm + k * 16 * kPitch), kPBytes, 8 * kPitch, kSwz);
        const uint64_t b5 = smem_desc(smem_u32(pt + k * 16 * kPitch), kPBytes, 8 * kPitch, kSwz);
        mma_ss(tbase + NCOL, a, b4, id_pv, k > 0);
        mma_ss(tbase + 2 * NCOL, a, b5, id_pv, k > 0);
      }
      mma_commit(bar_mma);
    }
  }
  __syncwarp();
  const bool done = (*status == 0) ? mbar_wait(bar_mma, 0, kLimitNs) : false;
  tc_fence_after();
  const uint32_t lane_base = taddr(tbase, (uint32_t)(warp * 32), 0);
  if (__all_sync(0xffffffffu, done)) {
    float* outs[5] = {D3, D4, D5, D6, D7};
    for (int m = 0; m < 5; ++m) {
      for (int c = 0; c < NCOL / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(lane_base + m * NCOL + c * 16, r);
        tmem_wait_ld();
        for (int k = 0; k < 16; ++k) outs[m][tid * NCOL + c * 16 + k] = __uint_as_float(r[k]);
      }
    }
  } else if (tid == 0) {
    atomicExch(status, 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int NCOL>
int run(const void* K, const void* V, const void* Q, const void* P, float* D3, float* D4, float* D5, float* D6,
        float* D7, int* status) {
  CUtensorMap tm_k, tm_v, tm_p;
  const uint64_t dims[2] = {128, 128};
  const uint64_t strides[1] = {128 * 2};
  const uint32_t box[2] = {64, 128};
  if (!dcp::make_tensor_map_bf16(&tm_k, K, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return -1;
  if (!dcp::make_tensor_map_bf16(&tm_v, V, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return -2;
  const uint64_t pdims[2] = {NCOL, 128};
  const uint64_t pstrides[1] = {NCOL * 2};
  const uint32_t pbox[2] = {NCOL, 128};
  const CUtensorMapSwizzle sw = NCOL == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                : NCOL == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_128B;
  if (!dcp::make_tensor_map_bf16(&tm_p, P, 2, pdims, pstrides, pbox, sw)) return -3;
  const uint32_t pbytes = (128 * NCOL * 2 + 1023) & ~1023u;
  const int smem = 1024 + 4 * kChunk + 2 * NCOL * 128 + 2 * pbytes + 64;
  cudaError_t e = cudaFuncSetAttribute(umma_t_kernel<NCOL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return (int)e;
  umma_t_kernel<NCOL><<<1, 128, smem>>>(tm_k, tm_v, tm_p, static_cast<const __nv_bfloat16*>(Q),
                                        static_cast<const __nv_bfloat16*>(P), D3, D4, D5, D6, D7, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}

}  // namespace

extern "C" int umma_probe_t(int ncol, const void* K, const void* V, const void* Q, const void* P, float* D3,
                            float* D4, float* D5, float* D6, float* D7, int* status) {
  switch (ncol) {
    case 16: return run<16>(K, V, Q, P, D3, D4, D5, D6, D7, status);
    case 32: return run<32>(K, V, Q, P, D3, D4, D5, D6, D7, status);
    case 64: return run<64>(K, V, Q, P, D3, D4, D5, D6, D7, status);
  }
  return -9;
}
