// Step a6 (LSE merge + head-slice return) and step a5 (combine of the KV
// splits of one shard, the same rule one level down).
//
// vLLM DCP blog, "DCP 執行流程" (AllGather + ReduceScatter): partial outputs
// and their log-sum-exp values are shared, reweighted with the online-softmax
// rule and summed; each rank keeps only its slice of heads.
//   LSE = m + log sum_r exp(lse_r - m),  m = max_r lse_r
//   o   = sum_r exp(lse_r - LSE) * o_r
// HBM-bound: one warp per output row streams the N partial rows with 16-byte
// loads; the N weights come from one lse load per lane and warp shuffles.
#include "dcp_device.cuh"
#include "dcp_internal.h"

namespace dcp {
namespace {

constexpr int kWarpsPerBlock = 8;

// Weights for up to 32 sources, one per lane: returns this lane's weight and
// writes the merged LSE.  lane_lse is -inf for lanes >= n.
__device__ __forceinline__ float lse_weights(float lane_lse, float* merged_lse) {
  float m = lane_lse;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (m == -INFINITY) {
    *merged_lse = -INFINITY;
    return 0.f;
  }
  float e = (lane_lse == -INFINITY) ? 0.f : expf(lane_lse - m);
  float s = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  *merged_lse = m + logf(s);
  return e / s;
}

// out row = sum over n sources (stride src_stride floats) of w_k * src_k.
// Dv4 = Dv / 4 float4 per row.
template <bool kBf16Out>
__device__ __forceinline__ void weighted_row(const float* __restrict__ src, long long src_stride,
                                             int n, float w_lane, int Dv4, void* dst_row) {
  const int lane = threadIdx.x & 31;
  for (int c = lane; c < Dv4; c += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < n; ++k) {
      const float w = __shfl_sync(0xffffffffu, w_lane, k);
      if (w == 0.f) continue;
      const float4 v = __ldcs(reinterpret_cast<const float4*>(src + k * src_stride) + c);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (kBf16Out) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(dst_row)[c] = pk;
    } else {
      reinterpret_cast<float4*>(dst_row)[c] = acc;
    }
  }
}

// One warp per (b, i, h): merge N shard partials; write rank h / (Hq/N)'s slice.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
merge_kernel(const float* __restrict__ partial_out, const float* __restrict__ lse, int N, int B,
             int Lq, int Hq, int Dv, __nv_bfloat16* __restrict__ out, float* __restrict__ out_lse) {
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const long long rows = (long long)B * Lq * Hq;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  // row = (b * Lq + i) * Hq + h ; partial rows of shard r at r * rows + row
  const float lane_lse = lane < N ? lse[(long long)lane * rows + row] : -INFINITY;
  float merged;
  const float w = lse_weights(lane_lse, &merged);
  const int h = (int)(row % Hq);
  const long long bi = row / Hq;
  const int hs = Hq / N;
  const int r = h / hs;
  const long long dst = (((long long)r * B * Lq + bi) * hs + (h % hs));
  weighted_row<true>(partial_out + row * Dv, rows * (long long)Dv, N, w, Dv / 4, out + dst * Dv);
  if (out_lse && lane == 0) out_lse[dst] = merged;
}

// One warp per (r, b, i, h): merge n_split workspace partials into partial_out.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
split_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int n_split,
                     long long rows, int Hq, int Dv, float* __restrict__ partial_out,
                     float* __restrict__ lse) {
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  // row = ((r * B + b) * Lq + i) * Hq + h ; ws rows: (unit * n_split + s) * Hq + h
  const long long unit = row / Hq;
  const int h = (int)(row % Hq);
  const long long base = unit * n_split * Hq + h;
  const float lane_lse = lane < n_split ? ws_lse[base + (long long)lane * Hq] : -INFINITY;
  float merged;
  const float w = lse_weights(lane_lse, &merged);
  weighted_row<false>(ws_o + base * Dv, (long long)Hq * Dv, n_split, w, Dv / 4,
                      partial_out + row * Dv);
  if (lane == 0) lse[row] = merged;
}

}  // namespace

cudaError_t launch_merge(const float* partial_out, const float* lse, int N, int B, int Lq, int Hq,
                         int Dv, void* out, float* out_lse, cudaStream_t stream) {
  const long long rows = (long long)B * Lq * Hq;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  merge_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
      partial_out, lse, N, B, Lq, Hq, Dv, static_cast<__nv_bfloat16*>(out), out_lse);
  return cudaGetLastError();
}

cudaError_t launch_split_combine(const AttnArgs& a, const SplitPlan& p) {
  const long long rows = (long long)a.N * a.B * a.Lq * a.Hq;
  if (rows == 0 || p.n_split <= 1) return cudaSuccess;
  const float* ws_o = static_cast<const float*>(a.workspace);
  const size_t o_bytes = (size_t)rows * p.n_split * a.Dv * sizeof(float);
  const float* ws_lse = reinterpret_cast<const float*>(static_cast<const char*>(a.workspace) +
                                                       ((o_bytes + 255) & ~size_t(255)));
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  split_combine_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, a.stream>>>(
      ws_o, ws_lse, p.n_split, rows, a.Hq, a.Dv, a.partial_out, a.lse);
  return cudaGetLastError();
}

}  // namespace dcp
