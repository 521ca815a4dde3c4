// Step a3: per-shard partial attention for GQA on tcgen05 tensor cores.
//
// vLLM DCP blog, "DCP 執行流程", Compute step (each shard attends the full
// query to its local KV slice and returns a partial output with its LSE), and
// section "Grouped-Query Attention (GQA) 後端" (query heads grouped over a few
// KV heads; query head h reads KV head h / (Hq / Hkv)).
//
// Work unit = (shard r, request b, KV head g, row tile m, KV split s), one CTA.
// The query rows of KV head g - (query i, head of the group), Lq * Hq / Hkv of
// them - are the M dimension of the MMAs, 128 per row tile (padded): the path
// moves 16 flop per cache byte, far below the tensor pipe's ridge, so the
// padding costs tensor time that is idle anyway and keeps one row per TMEM
// lane.  Long causal queries (chunked prefill) take several row tiles, each
// streaming the shard's keys.
//   S = Q K^T   (M=128, N=64 tokens, K=D; Q from TMEM, K tile K-major, 128B swizzle)
//   O += P V    (M=128, N=D, K=64; P from TMEM, V tile read MN-major)
// K and V tiles of 64 tokens stream through a TMA ring; a 3-D tensor map over
// the pool [block*block_size][Hkv][D] selects KV head g, so any block size
// that is a multiple of 8 works (small blocks take several boxes per tile).
// Softmax: one thread per query row, log2 domain, lazily rescaled reference
// max; the causal limit of query i is a prefix of the shard-local keys.
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2..5 softmax/epilogue (those holding real rows).  Every wait is
// bounded; on expiry the kernel records DCP_ERR_TIMEOUT and unwinds.
#include <cuda.h>
#include <cuda_bf16.h>

#include "dcp_device.cuh"
#include "dcp_internal.h"
#include "dcp_sm100.cuh"
#include "dcp_tma.h"

namespace dcp {
namespace {

using namespace sm100;

constexpr int kNt = 64;                        // tokens per tile
constexpr int kMaxStages = 6;
constexpr uint32_t kChunkBytes = kNt * 128;    // 64 tokens x 64 dims bf16
constexpr uint32_t kThreads = 192;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kColQ = 0;                  // D/2 columns (bf16 pairs)
constexpr uint32_t kColP = 64;                 // 32 columns
constexpr uint32_t kColS = 128;                // 64 columns fp32
constexpr uint32_t kColO = 256;                // D columns fp32
constexpr float kRescaleLog2 = 8.0f;

struct GqaParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* dst_o;
  float* dst_lse;
  int* status;
  int B, Lq, Hq, Hkv, N, I, max_lb, bs, num_blocks, n_split, split_tokens;
  int m_tiles;         // row tiles of 128 query rows per KV head
  int D;               // head dim (64 or 128)
  int stages;
  float scale_log2;
};

struct Smem {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full, s_free, p_full, pv_done, drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
gqa_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nch = p.D / 64;                               // 64-dim chunks of a row
  const uint32_t stage_bytes = 2u * nch * kChunkBytes;    // K chunks, then V chunks
  uint8_t* stages = base;
  Smem& sm = *reinterpret_cast<Smem*>(base + p.stages * stage_bytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long unit = blockIdx.x;
  const int s_idx = (int)(unit % p.n_split);
  const int mt = (int)((unit / p.n_split) % p.m_tiles);
  const long long gu = unit / ((long long)p.n_split * p.m_tiles);
  const int g = (int)(gu % p.Hkv);
  const int b = (int)((gu / p.Hkv) % p.B);
  const int r = (int)(gu / ((long long)p.Hkv * p.B));
  const int gsize = p.Hq / p.Hkv;
  const int row0 = 128 * mt;                              // first query row of this tile
  const int R = min(128, p.Lq * gsize - row0);            // real query rows of this tile
  const int n_act = (R + 31) / 32;                        // softmax warps holding real rows

  // key range: the tile's last query sees the most keys; earlier queries mask
  const int S = p.seq_lens[b];
  const bool bad_len = S < p.Lq;
  int L = bad_len ? 0 : local_len(S, r, p.I, p.N);
  const bool short_table = (long long)L > (long long)p.max_lb * p.bs;
  if (short_table) L = p.max_lb * p.bs;
  const int i_last = (row0 + R - 1) / gsize;
  const int vis = bad_len ? 0 : min(L, local_count_upto((long long)S - p.Lq + i_last, r, p.I, p.N));
  const int kb = min(vis, s_idx * p.split_tokens);
  const int ke = min(vis, kb + p.split_tokens);
  const int T = (ke - kb + kNt - 1) / kNt;
  if (tid == 0 && (bad_len || short_table)) set_status(p.status, DCP_ERR_BOUNDS);

  if (tid == 0) {
    for (int k = 0; k < p.stages; ++k) {
      mbar_init(smem_u32(&sm.kv_full[k]), 1);
      mbar_init(smem_u32(&sm.kv_empty[k]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.s_free), 32 * n_act);
    mbar_init(smem_u32(&sm.p_full), 32 * n_act);
    mbar_init(smem_u32(&sm.pv_done), 1);
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // query rows -> TMEM (row = TMEM lane; rows >= R are zero)
  if (warp >= 2) {
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = taddr(tmem, (uint32_t)((warp & 3) * 32), 0);
    const bool real = row < R && !bad_len;
    const uint4* qrow = nullptr;
    if (real) {
      const int i = (row0 + row) / gsize, head = g * gsize + (row0 + row) % gsize;
      qrow = reinterpret_cast<const uint4*>(p.q + (((long long)b * p.Lq + i) * p.Hq + head) * p.D);
    }
    for (int c = 0; c < p.D / 32; ++c) {                  // 16 columns = 32 dims per store
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 w = real ? __ldg(qrow + 4 * c + k) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k + 0] = w.x;
        v[4 * k + 1] = w.y;
        v[4 * k + 2] = w.z;
        v[4 * k + 3] = w.w;
      }
      tmem_st16(lane_addr + kColQ + 16 * c, v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  volatile int* abort_flag = &sm.abort;
  auto fail = [&](void) {
    set_status(p.status, DCP_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && T > 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const int32_t* bt = p.block_tables + ((long long)r * p.B + b) * p.max_lb;
      const int box_rows = p.bs < kNt ? p.bs : kNt;
      const int boxes = kNt / box_rows;
      int issued[kMaxStages];
      for (int k = 0; k < kMaxStages; ++k) issued[k] = 0;
      for (int t = 0; t < T; ++t) {
        const int st = t % p.stages;
        const uint32_t ph = (uint32_t)(t / p.stages) & 1u;
        if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_empty[st]), ph ^ 1u, kWaitNs)) {
          fail();
          break;
        }
        const uint32_t full = smem_u32(&sm.kv_full[st]);
        uint8_t* dst = stages + st * stage_bytes;
        mbar_arrive_expect_tx(full, stage_bytes);
        for (int k = 0; k < boxes; ++k) {
          const int j = kb + t * kNt + k * box_rows;
          // boxes past the last block of the table read block 0's slot (zeros
          // or stale rows are masked); in-range j always has a table entry
          const int jb = j / p.bs;
          const int blk = jb < p.max_lb ? bt[jb] : 0;
          if ((unsigned)blk >= (unsigned)p.num_blocks) set_status(p.status, DCP_ERR_BOUNDS);
          const int row = blk * p.bs + (j % p.bs);       // out-of-range rows read as zeros
          for (int c = 0; c < nch; ++c) {
            tma_load_3d(smem_u32(dst + c * kChunkBytes + k * box_rows * 128), &tm_k, 64 * c, g, row, full);
            tma_load_3d(smem_u32(dst + (nch + c) * kChunkBytes + k * box_rows * 128), &tm_v, 64 * c, g, row,
                        full);
          }
        }
        ++issued[st];
      }
      if (*abort_flag) {
        for (int k = 0; k < p.stages; ++k)
          if (issued[k] > 0) mbar_wait(smem_u32(&sm.kv_full[k]), (uint32_t)(issued[k] - 1) & 1u, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      const uint32_t id_qk = idesc_bf16(128, kNt, false);
      const uint32_t id_pv = idesc_bf16(128, p.D, true);
      auto issue_pv = [&](int t) -> bool {
        if (*abort_flag || !mbar_wait(smem_u32(&sm.p_full), (uint32_t)t & 1u, kWaitNs)) return false;
        tc_fence_after();
        const uint8_t* vb = stages + (t % p.stages) * stage_bytes + nch * kChunkBytes;
#pragma unroll
        for (int k = 0; k < kNt / 16; ++k) {
          const uint64_t bdesc = smem_desc(smem_u32(vb + k * 2048), kChunkBytes, 1024, kSw128);
          mma_ts(tmem + kColO, tmem + kColP + 8 * k, bdesc, id_pv, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.pv_done));
        mma_commit(smem_u32(&sm.kv_empty[t % p.stages]));
        return true;
      };
      bool ok = true;
      for (int t = 0; t < T && ok; ++t) {
        const int st = t % p.stages;
        if (*abort_flag ||
            !mbar_wait(smem_u32(&sm.kv_full[st]), (uint32_t)(t / p.stages) & 1u, kWaitNs) ||
            (t > 0 && !mbar_wait(smem_u32(&sm.s_free), (uint32_t)(t - 1) & 1u, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* kbuf = stages + st * stage_bytes;
        for (int k = 0; k < p.D / 16; ++k) {
          const uint64_t bdesc = smem_desc(smem_u32(kbuf + (k >> 2) * kChunkBytes + (k & 3) * 32), 16, 1024, kSw128);
          mma_ts(tmem + kColS, tmem + kColQ + 8 * k, bdesc, id_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.s_full));
        if (t > 0) ok = issue_pv(t - 1);
      }
      if (ok) ok = issue_pv(T - 1);
      if (!ok) fail();
      mma_commit(smem_u32(&sm.drain));
      if (!mbar_wait(smem_u32(&sm.drain), 0, kWaitNs)) fail();
    }
  } else if ((warp & 3) < n_act) {
    // ---------------- softmax / epilogue (warps holding real rows) ----------------
    const int lg = warp & 3;
    const int row = lg * 32 + lane;
    const bool real = row < R;
    const int i_q = real ? (row0 + row) / gsize : 0;
    const int head = g * gsize + (real ? (row0 + row) % gsize : 0);
    const uint32_t lane_addr = taddr(tmem, (uint32_t)(lg * 32), 0);
    // causal limit of this row's query: a prefix of the shard-local keys
    const int lim = real ? min(ke, local_count_upto((long long)S - p.Lq + i_q, r, p.I, p.N)) : kb;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
      return __all_sync(0xffffffffu, mbar_wait(bar, par, kWaitNs));
    };
    for (int t = 0; t < T; ++t) {
      if (!wwait(smem_u32(&sm.s_full), (uint32_t)t & 1u)) { ok = false; break; }
      tc_fence_after();
      float x[kNt];
      {
        uint32_t v[32];
        tmem_ld32(lane_addr + kColS, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(v[k]);
        tmem_ld32(lane_addr + kColS + 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) x[32 + k] = __uint_as_float(v[k]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_free));
      const int j0 = kb + t * kNt;
      const int valid = min(kNt, lim - j0);               // may be <= 0 for early queries
      float tmax = -INFINITY;
#pragma unroll
      for (int k = 0; k < kNt; ++k) {
        x[k] = (k < valid) ? x[k] * p.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, x[k]);
      }
      const bool grow = tmax > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - tmax);
        m_ref = tmax;
      }
      l *= alpha;
      uint32_t pk[kNt / 2];
#pragma unroll
      for (int k = 0; k < kNt; k += 2) {
        const float p0 = (k < valid) ? ex2(x[k] - m_ref) : 0.f;
        const float p1 = (k + 1 < valid) ? ex2(x[k + 1] - m_ref) : 0.f;
        l += p0 + p1;
        pk[k / 2] = pack_bf16x2(p0, p1);
      }
      if (t > 0) {
        if (!wwait(smem_u32(&sm.pv_done), (uint32_t)(t - 1) & 1u)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
          for (int c = 0; c < p.D; c += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + kColO + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(lane_addr + kColO + c, v);
          }
        }
      }
      const int tile_valid = min(kNt, ke - j0);
      if (tile_valid < kNt) {
        // ragged last tile: zero the value rows past the sequence end so that
        // 0 * (NaN/Inf) from stale cache slots cannot reach O
        uint4* vt = reinterpret_cast<uint4*>(stages + (t % p.stages) * stage_bytes + nch * kChunkBytes);
        const int n16 = (kNt - tile_valid) * 8;
        for (int idx = row; idx < nch * n16; idx += 32 * n_act) {   // row: 0 .. 32*n_act-1
          const int c = idx / n16, w = idx % n16;
          vt[(c * kChunkBytes) / 16 + tile_valid * 8 + w] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tmem_st32(lane_addr + kColP, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full));
    }
    if (!ok) fail();
    bool have = ok && T > 0;
    if (have) {
      have = wwait(smem_u32(&sm.pv_done), (uint32_t)(T - 1) & 1u);
      if (!have) fail();
    }
    tc_fence_after();
    const long long urow =
        ((((long long)r * p.B + b) * p.Lq + i_q) * p.n_split + s_idx) * p.Hq + head;
    float* orow = p.dst_o + urow * p.D;
    if (have) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      for (int c = 0; c < p.D; c += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + kColO + c, v);             // whole warp: .sync.aligned
        tmem_wait_ld();
        if (real) {
          float4* dst = reinterpret_cast<float4*>(orow + c);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                 __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
        }
      }
      if (real) p.dst_lse[urow] = l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
    } else if (real) {
      float4* dst = reinterpret_cast<float4*>(orow);
      for (int k = 0; k < p.D / 4; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.dst_lse[urow] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t gqa_smem_bytes(int D, int stages) {
  return 1024 + (size_t)stages * 2 * (D / 64) * kChunkBytes + sizeof(Smem) + 64;
}

}  // namespace

bool gqa_tc_supported(const AttnArgs& a) {
  if (a.kind != DCP_ATTN_GQA || (a.Dqk != 64 && a.Dqk != 128) || a.Dv != a.Dqk) return false;
  if ((long long)a.Lq * (a.Hq / a.Hkv) > (1LL << 20)) return false;
  if (a.bs % 8) return false;
  if (a.bs >= kNt ? (a.bs % kNt) : (kNt % a.bs)) return false;
  return (long long)a.num_blocks * a.bs < (1LL << 31);
}

static int gqa_m_tiles(const AttnArgs& a) { return (int)(((long long)a.Lq * (a.Hq / a.Hkv) + 127) / 128); }

SplitPlan plan_attn_gqa_tc(const AttnArgs& a, int sm_count) {
  return plan_splits(a, sm_count, kNt, a.Hkv * gqa_m_tiles(a));
}

cudaError_t launch_attn_gqa_tc(const AttnArgs& a, const SplitPlan& plan) {
  CUtensorMap tm_k, tm_v;
  const uint64_t rows = (uint64_t)a.num_blocks * a.bs;
  const uint64_t dims[3] = {(uint64_t)a.Dqk, (uint64_t)a.Hkv, rows};
  const uint64_t strides[2] = {(uint64_t)a.Dqk * 2, (uint64_t)a.Hkv * a.Dqk * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)(a.bs < kNt ? a.bs : kNt)};
  const char* k_pool = static_cast<const char*>(a.kv);
  const char* v_pool = k_pool + rows * a.Hkv * a.Dqk * 2;
  if (!make_tensor_map_bf16(&tm_k, k_pool, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&tm_v, v_pool, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  GqaParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.status = a.status;
  p.B = a.B;
  p.Lq = a.Lq;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N = a.N;
  p.I = a.I;
  p.max_lb = a.max_lb;
  p.bs = a.bs;
  p.num_blocks = a.num_blocks;
  p.n_split = plan.n_split;
  p.split_tokens = plan.split_tokens;
  p.m_tiles = gqa_m_tiles(a);
  p.D = a.Dqk;
  p.stages = kMaxStages;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (plan.n_split > 1) {
    const size_t nrows = (size_t)a.N * a.B * a.Lq * a.Hq;
    const size_t o_bytes = nrows * plan.n_split * a.Dv * sizeof(float);
    p.dst_o = static_cast<float*>(a.workspace);
    p.dst_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ((o_bytes + 255) & ~size_t(255)));
  } else {
    p.dst_o = a.partial_out;
    p.dst_lse = a.lse;
  }
  const size_t smem = gqa_smem_bytes(p.D, p.stages);
  cudaError_t e = cudaFuncSetAttribute(gqa_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.N * a.B * a.Hkv * p.m_tiles * plan.n_split;
  if (units == 0) return cudaSuccess;
  gqa_attn_kernel<<<(unsigned)units, kThreads, smem, a.stream>>>(tm_k, tm_v, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || plan.n_split <= 1) return e;
  return launch_split_combine(a, plan);
}

}  // namespace dcp
