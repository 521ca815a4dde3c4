// Steps a3/a4 for head dims the tensor-core kernels do not take: a plain SIMT
// split-KV kernel (fp32 FMA on CUDA cores).
//
// vLLM DCP blog, "DCP 執行流程", Compute: each shard attends the full query
// against its local KV slice only and emits a partial output and its LSE.
//
// One CTA = (shard r, request b, split s) x (KV head g) x (block of 16 query
// rows of that KV head).  Rows of KV head g are (query i, head h) with
// h in g's group; the causal limit of query i is a prefix of the shard-local
// keys (local tokens are in global order), so masking is a per-row count.
#include <cuda_bf16.h>

#include "dcp_device.cuh"
#include "dcp_internal.h"

namespace dcp {
namespace {

constexpr int kRows = 16;     // query rows per CTA
constexpr int kTile = 32;     // keys per smem tile
constexpr int kThreads = 128;

struct SimtParams {
  AttnArgs a;
  int n_split, split_tokens;
  float* dst_o;      // partial_out or workspace
  float* dst_lse;
};

__global__ void __launch_bounds__(kThreads) attn_simt_kernel(SimtParams P) {
  const AttnArgs& a = P.a;
  extern __shared__ float4 smem_f4[];
  float* smem = reinterpret_cast<float*>(smem_f4);
  const int gsize = a.Hq / a.Hkv;
  const int rows_total = a.Lq * gsize;
  const int row0 = blockIdx.z * kRows;
  const int g = blockIdx.y;
  const int unit = blockIdx.x;                       // ((r * B + b) * n_split + s)
  const int s = unit % P.n_split;
  const int b = (unit / P.n_split) % a.B;
  const int r = unit / (P.n_split * a.B);
  const int tid = threadIdx.x;

  float* q_s = smem;                                 // [kRows][Dqk]
  float* k_s = q_s + kRows * a.Dqk;                  // [kTile][Dqk]
  float* v_s = k_s + kTile * a.Dqk;                  // [kTile][Dv]   (GQA only)
  float* o_s = v_s + (a.kind == DCP_ATTN_GQA ? kTile * a.Dv : 0);  // [kRows][Dv]
  float* p_s = o_s + kRows * a.Dv;                   // [kRows][kTile]
  float* m_s = p_s + kRows * kTile;                  // [kRows]
  float* l_s = m_s + kRows;
  float* alpha_s = l_s + kRows;
  int* lim_s = reinterpret_cast<int*>(alpha_s + kRows);  // visible local keys per row

  const int S = a.seq_lens[b];
  const bool bad_len = S < a.Lq;
  if (bad_len && tid == 0) set_status(a.status, DCP_ERR_BOUNDS);
  int L = bad_len ? 0 : local_len(S, r, a.I, a.N);
  if ((long long)L > (long long)a.max_lb * a.bs) {   // block table too short for seq_len
    if (tid == 0) set_status(a.status, DCP_ERR_BOUNDS);
    L = a.max_lb * a.bs;
  }
  const int j_begin = min(L, s * P.split_tokens);
  int j_end = min(L, j_begin + P.split_tokens);
  {
    // a block id past the pool among the shard's keys skips the unit (every KV
    // split of it: zero partial, -inf LSE) and reports DCP_ERR_BOUNDS
    const int* btr = a.block_tables + ((long long)r * a.B + b) * a.max_lb;
    bool bad_blk = false;
    for (int jb = tid; jb < (L + a.bs - 1) / a.bs; jb += kThreads)
      bad_blk |= (unsigned)btr[jb] >= (unsigned)a.num_blocks;
    if (__syncthreads_or(bad_blk)) {
      j_end = j_begin;
      if (tid == 0) set_status(a.status, DCP_ERR_BOUNDS);
    }
  }

  // query rows -> smem (fp32), per-row visible-key limits
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  for (int idx = tid; idx < kRows * a.Dqk; idx += kThreads) {
    const int rr = idx / a.Dqk, d = idx % a.Dqk;
    const int row = row0 + rr;
    float v = 0.f;
    if (row < rows_total) {
      const int i = row / gsize, h = g * gsize + row % gsize;
      v = __bfloat162float(q[(((long long)b * a.Lq + i) * a.Hq + h) * a.Dqk + d]);
    }
    q_s[idx] = v;
  }
  for (int idx = tid; idx < kRows * a.Dv; idx += kThreads) o_s[idx] = 0.f;
  if (tid < kRows) {
    const int row = row0 + tid;
    const int i = row / gsize;
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
    lim_s[tid] = (row < rows_total && !bad_len)
                     ? min(j_end, local_count_upto((long long)S - a.Lq + i, r, a.I, a.N))
                     : j_begin;
  }
  __syncthreads();

  const __nv_bfloat16* kv = static_cast<const __nv_bfloat16*>(a.kv);
  const long long pool_elems = (long long)a.num_blocks * a.bs * a.Hkv * a.Dqk;
  const int* bt = a.block_tables + ((long long)r * a.B + b) * a.max_lb;

  for (int j0 = j_begin; j0 < j_end; j0 += kTile) {
    const int nt = min(kTile, j_end - j0);
    // stage keys (and values) of this tile
    for (int idx = tid; idx < kTile * a.Dqk; idx += kThreads) {
      const int tt = idx / a.Dqk, d = idx % a.Dqk;
      float kval = 0.f, vval = 0.f;
      if (tt < nt) {
        const int j = j0 + tt;
        const int blk = bt[j / a.bs];                 // checked against the pool above
        const long long off = (((long long)blk * a.bs + j % a.bs) * a.Hkv + g) * a.Dqk + d;
        kval = __bfloat162float(kv[off]);
        if (a.kind == DCP_ATTN_GQA && d < a.Dv) vval = __bfloat162float(kv[pool_elems + off]);
      }
      k_s[idx] = kval;
      if (a.kind == DCP_ATTN_GQA && d < a.Dv) v_s[tt * a.Dv + d] = vval;
    }
    __syncthreads();
    // scores
    for (int idx = tid; idx < kRows * kTile; idx += kThreads) {
      const int rr = idx / kTile, tt = idx % kTile;
      float sc = -INFINITY;
      if (j0 + tt < lim_s[rr]) {
        float acc = 0.f;
        const float* qr = q_s + rr * a.Dqk;
        const float* kr = k_s + tt * a.Dqk;
        for (int d = 0; d < a.Dqk; ++d) acc = fmaf(qr[d], kr[d], acc);
        sc = acc * a.scale;
      }
      p_s[idx] = sc;
    }
    __syncthreads();
    // online softmax update, one thread per row
    if (tid < kRows) {
      float mx = m_s[tid];
      for (int tt = 0; tt < kTile; ++tt) mx = fmaxf(mx, p_s[tid * kTile + tt]);
      float alpha = 1.f, sum = 0.f;
      if (mx != -INFINITY) {
        alpha = (m_s[tid] == -INFINITY) ? 0.f : expf(m_s[tid] - mx);
        for (int tt = 0; tt < kTile; ++tt) {
          const float sc = p_s[tid * kTile + tt];
          const float p = (sc == -INFINITY) ? 0.f : expf(sc - mx);
          p_s[tid * kTile + tt] = p;
          sum += p;
        }
      } else {
        for (int tt = 0; tt < kTile; ++tt) p_s[tid * kTile + tt] = 0.f;
      }
      m_s[tid] = mx;
      l_s[tid] = l_s[tid] * alpha + sum;
      alpha_s[tid] = alpha;
    }
    __syncthreads();
    // O = O * alpha + P V
    const float* vsrc = (a.kind == DCP_ATTN_GQA) ? v_s : k_s;
    const int vstride = (a.kind == DCP_ATTN_GQA) ? a.Dv : a.Dqk;
    for (int idx = tid; idx < kRows * a.Dv; idx += kThreads) {
      const int rr = idx / a.Dv, d = idx % a.Dv;
      float acc = o_s[idx] * alpha_s[rr];
      const float* pr = p_s + rr * kTile;
      for (int tt = 0; tt < nt; ++tt) acc = fmaf(pr[tt], vsrc[tt * vstride + d], acc);
      o_s[idx] = acc;
    }
    __syncthreads();
  }

  // write partial (normalised) and lse
  for (int idx = tid; idx < kRows * a.Dv; idx += kThreads) {
    const int rr = idx / a.Dv, d = idx % a.Dv;
    const int row = row0 + rr;
    if (row >= rows_total) continue;
    const int i = row / gsize, h = g * gsize + row % gsize;
    const float l = l_s[rr];
    const long long unit_row = ((((long long)r * a.B + b) * a.Lq + i) * P.n_split + s) * a.Hq + h;
    P.dst_o[unit_row * a.Dv + d] = l > 0.f ? o_s[idx] / l : 0.f;
  }
  if (tid < kRows) {
    const int row = row0 + tid;
    if (row < rows_total) {
      const int i = row / gsize, h = g * gsize + row % gsize;
      const float l = l_s[tid];
      const long long unit_row =
          ((((long long)r * a.B + b) * a.Lq + i) * P.n_split + s) * a.Hq + h;
      P.dst_lse[unit_row] = l > 0.f ? m_s[tid] + logf(l) : -INFINITY;
    }
  }
}

size_t simt_smem_bytes(const AttnArgs& a) {
  size_t f = (size_t)kRows * a.Dqk + (size_t)kTile * a.Dqk +
             (a.kind == DCP_ATTN_GQA ? (size_t)kTile * a.Dv : 0) + (size_t)kRows * a.Dv +
             (size_t)kRows * kTile + 4 * kRows;
  return f * sizeof(float);
}

}  // namespace

SplitPlan plan_attn_simt(const AttnArgs& a, int sm_count) {
  const int gsize = a.Hq / a.Hkv;
  const int row_blocks = (a.Lq * gsize + kRows - 1) / kRows;
  return plan_splits(a, sm_count, kTile, a.Hkv * row_blocks);
}

cudaError_t launch_attn_simt(const AttnArgs& a, const SplitPlan& p) {
  SimtParams P;
  P.a = a;
  P.n_split = p.n_split;
  P.split_tokens = p.split_tokens;
  if (p.n_split > 1) {
    const size_t rows = (size_t)a.N * a.B * a.Lq * a.Hq;
    const size_t o_bytes = rows * p.n_split * a.Dv * sizeof(float);
    P.dst_o = static_cast<float*>(a.workspace);
    P.dst_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) +
                                         ((o_bytes + 255) & ~size_t(255)));
  } else {
    P.dst_o = a.partial_out;
    P.dst_lse = a.lse;
  }
  const size_t smem = simt_smem_bytes(a);
  cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int gsize = a.Hq / a.Hkv;
  dim3 grid((unsigned)(a.N * a.B * p.n_split), (unsigned)a.Hkv,
            (unsigned)((a.Lq * gsize + kRows - 1) / kRows));
  attn_simt_kernel<<<grid, kThreads, smem, a.stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split <= 1) return e;
  return launch_split_combine(a, p);
}

}  // namespace dcp
