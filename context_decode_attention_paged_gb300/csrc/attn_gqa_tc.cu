// Step a3: per-shard partial attention for GQA on tcgen05 tensor cores.
//
// vLLM DCP blog, "DCP 執行流程", Compute step (each shard attends the full
// query to its local KV slice and returns a partial output with its LSE), and
// section "Grouped-Query Attention (GQA) 後端" (query heads grouped over a few
// KV heads; query head h reads KV head h / (Hq / Hkv)).
//
// Work unit = (shard r, request b, KV head g, row tile m, KV split s), one CTA;
// units run longest request first (batches up to 128).
// The query rows of KV head g - (query i, head of the group), Lq * Hq / Hkv of
// them - are few (16 for one decode token of a 16-head group), so the kernel
// computes the transposed products and puts the KEYS on the 128 rows of the
// MMA, one key per TMEM lane and per softmax thread:
//   S^T = K Q^T    (M = 128 keys, N = NCOL query rows, K = D;
//                   K tile K-major and Q^T K-major, both 128B-swizzled smem)
//   O^T += V^T P^T (M = 128 value dims, N = NCOL, K = 128 keys;
//                   V tile read MN-major from the same stage, P^T MN-major smem)
// P carries two bf16 terms, P_hi = bf16(p) and P_lo = bf16(p - P_hi): p keeps
// 16 significant bits instead of 8, so a few dominant keys whose values nearly
// cancel do not leave the 2^-9 rounding of their probabilities in the output.
// The two P^T buffers of a tile sit one swizzle atom apart, so one PV MMA with
// N = 2 NCOL accumulates O_hi^T and O_lo^T side by side; the epilogue adds
// them.  The MMA count per tile stays that of one term.
// NCOL is 16, 32 or 64 (the tile's query rows, padded); longer causal queries
// (chunked prefill) take several row tiles, each streaming the shard's keys.
// K and V tiles of 128 tokens stream through a TMA ring; a 3-D tensor map over
// the pool [block*block_size][Hkv][D] selects KV head g, so any block size that
// is a multiple of 8 and divides (or is a multiple of) 128 works.
//
// Softmax: a thread owns key k of the tile and the scores of that key for a
// quarter of the query rows.  The reference max of each row is
// shared by all threads and moves lazily: one barrier per tile ORs "some score
// exceeds its row's reference by more than 2^8"; only then do the warps reduce
// the tile's row maxima, rescale O^T (after the previous PV has landed) and
// their per-thread row sums.  Row sums are reduced across the 128 key threads
// once, at the end.  Logs are base 2 with the scale folded into the exponent.
// Warp roles (608 threads): warp 0 TMA producer, warp 1 QK issuer and TMEM
// owner, warp 2 PV issuer, warps 3..18 softmax/epilogue (four per TMEM lane
// quadrant, each taking a quarter of the query-row columns).  A tcgen05.mma takes
// one issuing thread tens of cycles, so QK and PV have a thread each (PV(t)
// goes out as soon as P(t) is ready, not after the next tile's QK).
// Every wait is bounded; on expiry the
// kernel records DCP_ERR_TIMEOUT and unwinds, the softmax warps deciding
// together (barrier-reduced predicates) so that none is left at a barrier.
#include <cuda.h>
#include <cuda_bf16.h>

#include "dcp_device.cuh"
#include "dcp_internal.h"
#include "dcp_sm100.cuh"
#include "dcp_tma.h"

namespace dcp {
namespace {

using namespace sm100;

constexpr int kNt = 128;                       // keys per tile (MMA M of S^T)
constexpr int kMaxStages = 6;
constexpr uint32_t kChunkBytes = kNt * 128;    // 128 keys x 64 dims bf16
constexpr int kFirstSoftWarp = 3;             // warps 3.. : softmax
constexpr int kSoftGroups = 4;                 // softmax warps per TMEM lane quadrant
constexpr uint32_t kSoftThreads = 128 * kSoftGroups;
constexpr uint32_t kThreads = 96 + kSoftThreads;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxCols = 64;                   // query rows per row tile
constexpr size_t kSmemLimit = 232448;          // dynamic shared memory per CTA
constexpr uint32_t kBarSoftmax = 1;            // named barrier of the softmax warps
constexpr int kLptMaxBatch = 128;              // longest-first unit order up to this batch

struct GqaParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* dst_o;
  float* dst_lse;
  int* status;
  int B, Lq, Hq, Hkv, N, I, max_lb, bs, num_blocks, n_split, split_tokens;
  int m_tiles;         // row tiles of NCOL query rows per KV head
  int D;               // head dim (64 or 128)
  int stages;
  float scale_log2;
  unsigned long long wait_ns;   // limit of every bounded wait
  int skip_tile;                // test hook: the producer never loads this tile (-1: off)
};

struct Smem {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2], drain[2];
  uint32_t tmem_base;
  int abort;
  int req;                    // request of this unit
  int lim[kMaxCols];          // causal key limit of each query row of the tile
  float red[4][kMaxCols];     // per-warp row maxima / row sums
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int NCOL>
struct Cfg {
  static constexpr uint32_t kPitch = NCOL * 2;                    // bytes of one P^T row (key)
  static constexpr uint32_t kPBytes = kNt * kPitch;               // one P^T buffer
  static constexpr uint32_t kPSwz = NCOL == 16 ? kSw32 : NCOL == 32 ? kSw64 : kSw128;
  static constexpr uint32_t kTmemCols = NCOL == 16 ? 64 : NCOL == 32 ? 128 : 256;
  // 16-byte chunk c of key row k as stored under the P^T swizzle
  __device__ static __forceinline__ uint32_t pchunk(uint32_t c, uint32_t k) {
    return NCOL == 16 ? (c ^ ((k >> 2) & 1u)) : NCOL == 32 ? (c ^ ((k >> 1) & 3u)) : (c ^ (k & 7u));
  }
};

__host__ __device__ constexpr size_t gqa_fixed_bytes(int D, int ncol) {
  return 1024 + (size_t)(D / 64) * ncol * 128 + 4 * (size_t)kNt * ncol * 2 + sizeof(Smem) + 64;
}

size_t gqa_stage_bytes(int D) { return 2 * (size_t)(D / 64) * kChunkBytes; }

int gqa_stages(int D, int ncol) {
  const size_t room = kSmemLimit - gqa_fixed_bytes(D, ncol);
  const int s = (int)(room / gqa_stage_bytes(D));
  return s > kMaxStages ? kMaxStages : s;
}

size_t gqa_smem_bytes(int D, int ncol, int stages) {
  return gqa_fixed_bytes(D, ncol) + (size_t)stages * gqa_stage_bytes(D);
}

// Softmax and epilogue of the softmax warps: kSoftGroups per TMEM lane
// quadrant, each taking an equal share of the query-row columns (thread = TMEM
// lane: key k of the tile for S^T and P^T, value dim k for O^T; columns
// [h0, h0 + HC)).
template <int NCOL, typename Fail>
__device__ __forceinline__ void softmax_epilogue(const GqaParams& p, Smem& sm, uint8_t* stages,
                                                 uint32_t stage_bytes, uint8_t* ps, uint32_t tmem, int warp,
                                                 int lane, int T, int kb, int ke, int lim_min, int R, int row0,
                                                 int gsize, int g, int b, int r, int s_idx, Fail fail) {
  using C = Cfg<NCOL>;
  constexpr int HC = NCOL / kSoftGroups;                  // columns per thread
  const int nch = p.D / 64;
  const int qd = warp & 3;                                // TMEM lane quadrant of this warp
  const int h0 = ((warp - kFirstSoftWarp) >> 2) * HC;     // first column of this warp
  const int lrow = qd * 32 + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
  const uint32_t tO = lane_base + 2 * NCOL + h0;         // O_hi^T; O_lo^T is NCOL columns on
  volatile int* abort_flag = &sm.abort;
  float m[HC], l[HC];
#pragma unroll
  for (int h = 0; h < HC; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  auto ld_cols = [&](uint32_t addr, uint32_t (&v)[HC]) {
    if constexpr (HC == 4) {
      tmem_ld4(addr, v);
    } else if constexpr (HC == 8) {
      tmem_ld8(addr, v);
    } else {
#pragma unroll
      for (int c = 0; c < HC / 16; ++c) tmem_ld16(addr + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * c]));
    }
  };
  auto st_cols = [&](uint32_t addr, const uint32_t (&v)[HC]) {
    if constexpr (HC == 4) {
      tmem_st4(addr, v);
    } else if constexpr (HC == 8) {
      tmem_st8(addr, v);
    } else {
#pragma unroll
      for (int c = 0; c < HC / 16; ++c)
        tmem_st16(addr + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(&v[16 * c]));
    }
  };
  bool bad = false, broke = false;
  for (int t = 0; t < T; ++t) {
    const int bsel = t & 1;
    const bool okw = __all_sync(0xffffffffu, *abort_flag == 0 &&
                                                 mbar_wait(smem_u32(&sm.s_full[bsel]), (uint32_t)(t >> 1) & 1u, p.wait_ns));
    if (!okw) bad = true;
    float x[HC];
    {
      uint32_t v[HC];
      if (okw) {
        tc_fence_after();
        ld_cols(lane_base + bsel * NCOL + h0, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int h = 0; h < HC; ++h) v[h] = 0u;
      }
#pragma unroll
      for (int h = 0; h < HC; ++h) x[h] = __uint_as_float(v[h]);
    }
    tc_fence_before();
    mbar_arrive(smem_u32(&sm.s_free[bsel]));

    // scaled scores (log2 domain); keys a row may not see are -inf
    const int j0 = kb + t * kNt;
    const int jj = j0 + lrow;                             // this thread's shard-local key
    const bool full = j0 + kNt <= lim_min;                // every row sees every key of the tile
    float e = -INFINITY;
    if (full) {
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        x[h] *= p.scale_log2;
        e = fmaxf(e, x[h] - m[h]);
      }
    } else {
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        x[h] = jj < sm.lim[h0 + h] ? x[h] * p.scale_log2 : -INFINITY;
        e = fmaxf(e, x[h] - m[h]);
      }
    }
    // one barrier per tile: does any row's reference max have to move?
    if (bar_red_or(kBarSoftmax, kSoftThreads, e > kRescaleLog2 || bad)) {
      if (bar_red_or(kBarSoftmax, kSoftThreads, bad)) {
        broke = true;
        break;
      }
      // row maxima of the tile over its 128 keys (the four quadrant warps of a column)
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        float v = x[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) sm.red[qd][h0 + h] = v;
      }
      // O^T is rescaled below: the previous tile's PV must have landed.  Its
      // P^T buffer's barrier is at most one phase ahead of what this thread
      // last waited for there (PV(t-3)), so the parity is unambiguous.
      if (t > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_free[(t - 1) & 1]),
                                                      (uint32_t)((t - 1) >> 1) & 1u, p.wait_ns)))
        bad = true;
      if (bar_red_or(kBarSoftmax, kSoftThreads, bad)) {
        broke = true;
        break;
      }
      float alpha[HC];
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        const int hh = h0 + h;
        const float tmax = fmaxf(fmaxf(sm.red[0][hh], sm.red[1][hh]), fmaxf(sm.red[2][hh], sm.red[3][hh]));
        const float mn = fmaxf(m[h], tmax);
        alpha[h] = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
        m[h] = mn;
        l[h] *= alpha[h];
      }
      if (t > 0) {
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          uint32_t o[HC];
          ld_cols(tO + part * NCOL, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < HC; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha[k]);
          st_cols(tO + part * NCOL, o);
        }
        tmem_wait_st();
      }
    }

    // this key's probabilities for this warp's rows -> its part of the P^T
    // row, as two bf16 terms (hi, and the remainder lo)
    uint32_t pk[HC / 2], pl[HC / 2];
#pragma unroll
    for (int h = 0; h < HC; h += 2) {
      float p0, p1;
      if (full) {
        p0 = ex2(x[h] - m[h]);
        p1 = ex2(x[h + 1] - m[h + 1]);
      } else {
        p0 = x[h] == -INFINITY ? 0.f : ex2(x[h] - m[h]);
        p1 = x[h + 1] == -INFINITY ? 0.f : ex2(x[h + 1] - m[h + 1]);
      }
      l[h] += p0;
      l[h + 1] += p1;
      const uint32_t hi = pack_bf16x2(p0, p1);
      pk[h / 2] = hi;
      pl[h / 2] = pack_bf16x2(p0 - bf16_lo(hi), p1 - bf16_hi(hi));
    }
    if (t >= 2 &&
        !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_free[bsel]), (uint32_t)((t >> 1) - 1) & 1u, p.wait_ns)))
      bad = true;
    uint8_t* prow = ps + 2 * bsel * C::kPBytes + lrow * C::kPitch;
    uint8_t* lrow_p = prow + C::kPBytes;                  // the lo term's buffer, one atom on
    if constexpr (HC == 4) {
      // half of a 16-byte chunk: the swizzle moves whole chunks
      const uint32_t off = (C::pchunk((uint32_t)(h0 / 8), (uint32_t)lrow) << 4) + (h0 % 8) * 2;
      *reinterpret_cast<uint2*>(prow + off) = make_uint2(pk[0], pk[1]);
      *reinterpret_cast<uint2*>(lrow_p + off) = make_uint2(pl[0], pl[1]);
    } else {
#pragma unroll
      for (int c = 0; c < HC / 8; ++c) {
        const uint32_t off = C::pchunk((uint32_t)(h0 / 8 + c), (uint32_t)lrow) << 4;
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        *reinterpret_cast<uint4*>(lrow_p + off) = make_uint4(pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
      }
    }
    if (h0 == 0 && jj >= ke) {
      // key past the range (ragged last tile): zero its value row so that
      // 0 * (NaN/Inf) from a stale cache slot cannot reach O
      uint8_t* vt = stages + (t % p.stages) * stage_bytes + lrow * 128;
      for (int c = 0; c < nch; ++c) {
        uint4* vr = reinterpret_cast<uint4*>(vt + c * kChunkBytes);
#pragma unroll
        for (int w = 0; w < 8; ++w) vr[w] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(smem_u32(&sm.p_full[bsel]));
  }

  // the last PV (its commit also covers every earlier MMA of the issuer)
  bool have = T > 0 && !broke;
  if (have && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_free[(T - 1) & 1]),
                                                 (uint32_t)((T - 1) >> 1) & 1u, p.wait_ns)))
    bad = true;
  if (bar_red_or(kBarSoftmax, kSoftThreads, bad)) have = false;
  if (bad) fail();

  // row sums over the 128 key threads (the four quadrant warps of a column)
#pragma unroll
  for (int h = 0; h < HC; ++h) {
    float v = l[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) sm.red[qd][h0 + h] = v;
  }
  named_bar_sync(kBarSoftmax, kSoftThreads);

  // outputs: this thread holds value dim lrow of this warp's rows
  uint32_t o[HC];
#pragma unroll
  for (int h = 0; h < HC; ++h) o[h] = 0u;
  if (have) {
    tc_fence_after();
    uint32_t olo[HC];
    ld_cols(tO, o);
    ld_cols(tO + NCOL, olo);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < HC; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) + __uint_as_float(olo[h]));
  }
#pragma unroll
  for (int h = 0; h < HC; ++h) {
    const int hh = h0 + h;
    if (hh < R) {
      const float lsum = (sm.red[0][hh] + sm.red[1][hh]) + (sm.red[2][hh] + sm.red[3][hh]);
      const bool live = have && lsum > 0.f;
      const int rr = row0 + hh, i = rr / gsize, head = g * gsize + rr % gsize;
      const long long urow = ((((long long)r * p.B + b) * p.Lq + i) * p.n_split + s_idx) * p.Hq + head;
      if (lrow < p.D) p.dst_o[urow * p.D + lrow] = live ? __uint_as_float(o[h]) * (1.f / lsum) : 0.f;
      if (lrow == 0) p.dst_lse[urow] = live ? (m[h] + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

template <int NCOL>
__global__ void __launch_bounds__(kThreads, 1)
gqa_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const GqaParams p) {
  using C = Cfg<NCOL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nch = p.D / 64;                               // 64-dim chunks of a row
  const uint32_t stage_bytes = 2u * nch * kChunkBytes;    // V chunks, then K chunks
  uint8_t* stages = base;
  uint8_t* qs = stages + p.stages * stage_bytes;          // Q^T: nch chunks of NCOL rows x 128 B
  uint8_t* ps = qs + nch * NCOL * 128;                    // P^T buffers: hi 0, lo 0, hi 1, lo 1
  Smem& sm = *reinterpret_cast<Smem*>(ps + 4 * C::kPBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Units in longest-request-first order: the block scheduler starts CTAs in
  // index order, so the short units fill the tail.  Rank k of the request
  // order (length descending, index ascending) is found by counting.
  const long long unit = blockIdx.x;
  const long long per_req = (long long)p.N * p.Hkv * p.m_tiles * p.n_split;
  const int k_req = (int)(unit / per_req);
  int b = k_req;
  if (p.B <= kLptMaxBatch) {
    for (int j = tid; j < p.B; j += kThreads) {
      const int sj = p.seq_lens[j];
      int rank = 0;
      for (int i = 0; i < p.B; ++i) {
        const int si = p.seq_lens[i];
        rank += (si > sj) || (si == sj && i < j);
      }
      if (rank == k_req) sm.req = j;
    }
    __syncthreads();
    b = sm.req;
  }
  const long long rest = unit % per_req;
  const int s_idx = (int)(rest % p.n_split);
  const int mt = (int)((rest / p.n_split) % p.m_tiles);
  const int g = (int)((rest / ((long long)p.n_split * p.m_tiles)) % p.Hkv);
  const int r = (int)(rest / ((long long)p.n_split * p.m_tiles * p.Hkv));
  const int gsize = p.Hq / p.Hkv;
  const int row0 = NCOL * mt;                             // first query row of this tile
  const int R = min(NCOL, p.Lq * gsize - row0);           // real query rows of this tile

  // key range: the tile's last query sees the most keys; earlier queries mask
  const int S = p.seq_lens[b];
  const bool bad_len = S < p.Lq;
  int L = bad_len ? 0 : local_len(S, r, p.I, p.N);
  const bool short_table = (long long)L > (long long)p.max_lb * p.bs;
  if (short_table) L = p.max_lb * p.bs;
  const int i_first = row0 / gsize, i_last = (row0 + R - 1) / gsize;
  const int vis = bad_len ? 0 : min(L, local_count_upto((long long)S - p.Lq + i_last, r, p.I, p.N));
  const int kb = min(vis, s_idx * p.split_tokens);
  const int ke = min(vis, kb + p.split_tokens);
  int T = (ke - kb + kNt - 1) / kNt;
  // keys below lim_min are visible to every row of the tile
  const int lim_min = bad_len ? 0 : min(ke, local_count_upto((long long)S - p.Lq + i_first, r, p.I, p.N));
  if (tid == 0 && (bad_len || short_table)) set_status(p.status, DCP_ERR_BOUNDS);
  {
    // a block id past the pool among the tile's visible keys skips the unit
    // (every KV split of it: zero partial, -inf LSE) and reports
    // DCP_ERR_BOUNDS; table entries past the key range are never read
    const int32_t* bt = p.block_tables + ((long long)r * p.B + b) * p.max_lb;
    bool bad_blk = false;
    for (int jb = tid; jb < (vis + p.bs - 1) / p.bs; jb += (int)kThreads)
      bad_blk |= (unsigned)bt[jb] >= (unsigned)p.num_blocks;
    if (__syncthreads_or(bad_blk)) {
      T = 0;
      if (tid == 0) set_status(p.status, DCP_ERR_BOUNDS);
    }
  }

  if (tid == 0) {
    for (int k = 0; k < p.stages; ++k) {
      mbar_init(smem_u32(&sm.kv_full[k]), 1);
      mbar_init(smem_u32(&sm.kv_empty[k]), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&sm.s_full[k]), 1);
      mbar_init(smem_u32(&sm.s_free[k]), kSoftThreads);
      mbar_init(smem_u32(&sm.p_full[k]), kSoftThreads);
      mbar_init(smem_u32(&sm.p_free[k]), 1);
    }
    mbar_init(smem_u32(&sm.drain[0]), 1);
    mbar_init(smem_u32(&sm.drain[1]), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), C::kTmemCols);
  if (warp >= kFirstSoftWarp) {
    // Q^T rows -> smem, K-major with the 128-byte swizzle (rows >= R are zero),
    // and the causal key limit of every row
    const int st = tid - 32 * kFirstSoftWarp;
    const int per_row = nch * 8;                          // 16-byte chunks of a row
    for (int idx = st; idx < NCOL * per_row; idx += (int)kSoftThreads) {
      const int h = idx / per_row, ch = (idx % per_row) >> 3, c = idx & 7;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (h < R && !bad_len) {
        const int i = (row0 + h) / gsize, head = g * gsize + (row0 + h) % gsize;
        v = __ldg(reinterpret_cast<const uint4*>(p.q + (((long long)b * p.Lq + i) * p.Hq + head) * p.D + ch * 64) + c);
      }
      *reinterpret_cast<uint4*>(qs + ch * NCOL * 128 + h * 128 + ((c ^ (h & 7)) << 4)) = v;
    }
    if (st < NCOL) {
      sm.lim[st] = (st < R && !bad_len)
                       ? min(ke, local_count_upto((long long)S - p.Lq + (row0 + st) / gsize, r, p.I, p.N))
                       : ke;
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

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
        if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_empty[st]), ph ^ 1u, p.wait_ns)) {
          fail();
          break;
        }
        // test hook: this tile is never loaded, so the bounded waits on it run
        // out and the unit unwinds
        if (t == p.skip_tile) continue;
        const uint32_t full = smem_u32(&sm.kv_full[st]);
        uint8_t* dst = stages + st * stage_bytes;
        mbar_arrive_expect_tx(full, stage_bytes);
        for (int k = 0; k < boxes; ++k) {
          const int j = kb + t * kNt + k * box_rows;
          // boxes past the key range read pool row 0 (masked, values zeroed);
          // the others' block ids were checked against the pool above
          const int row = j < ke ? bt[j / p.bs] * p.bs + (j % p.bs) : 0;
          for (int c = 0; c < nch; ++c) {
            tma_load_3d(smem_u32(dst + c * kChunkBytes + k * box_rows * 128), &tm_v, 64 * c, g, row, full);
            tma_load_3d(smem_u32(dst + (nch + c) * kChunkBytes + k * box_rows * 128), &tm_k, 64 * c, g, row,
                        full);
          }
        }
        ++issued[st];
      }
      if (*abort_flag) {
        for (int k = 0; k < p.stages; ++k)
          if (issued[k] > 0) mbar_wait(smem_u32(&sm.kv_full[k]), (uint32_t)(issued[k] - 1) & 1u, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- QK issuer: S^T(t) = K(t) Q^T ----------------
    if (lane == 0 && T > 0) {
      constexpr uint32_t id_qk = idesc_bf16_ab(128, NCOL, false, false);
      // Each descriptor is built from its address at the MMA, in an unrolled
      // K-step loop.  Variants that added compile-time offsets to a run-time
      // base descriptor here (inside a swizzle row, or whole 64-dim chunks)
      // gave wrong products on the device, although the descriptor values
      // they printed were the same; the PV issuer below does add offsets (whole
      // 8-row atoms of MN-major operands), which the parity tests cover.
      const uint32_t ksteps = (uint32_t)p.D / 16;
      bool ok = true;
      for (int t = 0; t < T; ++t) {
        const int st = t % p.stages;
        if (*abort_flag ||
            !mbar_wait(smem_u32(&sm.kv_full[st]), (uint32_t)(t / p.stages) & 1u, p.wait_ns) ||
            (t >= 2 && !mbar_wait(smem_u32(&sm.s_free[t & 1]), (uint32_t)((t >> 1) - 1) & 1u, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dS = tmem + (uint32_t)(t & 1) * NCOL;
        const uint8_t* kbuf = stages + st * stage_bytes + nch * kChunkBytes;
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k) {
          if (k < ksteps)
            mma_ss(dS, smem_desc(smem_u32(kbuf + (k >> 2) * kChunkBytes + (k & 3) * 32), 16, 1024, kSw128),
                   smem_desc(smem_u32(qs + (k >> 2) * (NCOL * 128) + (k & 3) * 32), 16, 1024, kSw128), id_qk,
                   k > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.s_full[t & 1]));
      }
      if (!ok) fail();
      mma_commit(smem_u32(&sm.drain[0]));
      if (!mbar_wait(smem_u32(&sm.drain[0]), 0, p.wait_ns)) fail();
    }
  } else if (warp == 2) {
    // ---------------- PV issuer: O^T += V^T(t) P^T(t) ----------------
    if (lane == 0 && T > 0) {
      constexpr uint32_t id_pv = idesc_bf16_ab(128, 2 * NCOL, true, true);   // [P_hi | P_lo]
      const uint32_t tO = tmem + 2 * NCOL;
      // A = V^T (dims x keys) read MN-major from the value chunks; B = P^T
      bool ok = true;
      for (int t = 0; t < T; ++t) {
        if (*abort_flag || !mbar_wait(smem_u32(&sm.p_full[t & 1]), (uint32_t)(t >> 1) & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = t % p.stages;
        // base descriptors of this stage and P^T buffer; the K-steps add whole
        // 8-row swizzle atoms (2048 B of V, 8 rows of P^T) to the start address
        const uint64_t dv = smem_desc(smem_u32(stages + st * stage_bytes), kChunkBytes, 1024, kSw128);
        // the hi and lo buffers are the two N atoms of one operand (LBO = one buffer)
        const uint64_t dp = smem_desc(smem_u32(ps + 2 * (t & 1) * C::kPBytes), C::kPBytes, 8 * C::kPitch, C::kPSwz);
#pragma unroll
        for (uint32_t k = 0; k < kNt / 16; ++k)
          mma_ss(tO, dv + ((k * 2048u) >> 4), dp + ((k * 16u * C::kPitch) >> 4), id_pv, (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sm.p_free[t & 1]));
        mma_commit(smem_u32(&sm.kv_empty[st]));
      }
      if (!ok) fail();
      mma_commit(smem_u32(&sm.drain[1]));
      if (!mbar_wait(smem_u32(&sm.drain[1]), 0, p.wait_ns)) fail();
    }
  } else {
    softmax_epilogue<NCOL>(p, sm, stages, stage_bytes, ps, tmem, warp, lane, T, kb, ke, lim_min, R, row0,
                           gsize, g, b, r, s_idx, fail);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NCOL>
cudaError_t launch_ncol(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const GqaParams& p, long long units,
                        cudaStream_t stream) {
  const size_t smem = gqa_smem_bytes(p.D, NCOL, p.stages);
  cudaError_t e = cudaFuncSetAttribute(gqa_attn_kernel<NCOL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gqa_attn_kernel<NCOL><<<(unsigned)units, kThreads, smem, stream>>>(tm_k, tm_v, p);
  return cudaGetLastError();
}

}  // namespace

bool gqa_tc_supported(const AttnArgs& a) {
  if (a.kind != DCP_ATTN_GQA || (a.Dqk != 64 && a.Dqk != 128) || a.Dv != a.Dqk) return false;
  if ((long long)a.Lq * (a.Hq / a.Hkv) > (1LL << 20)) return false;
  if (a.bs % 8) return false;
  if (a.bs >= kNt ? (a.bs % kNt) : (kNt % a.bs)) return false;
  return (long long)a.num_blocks * a.bs < (1LL << 31);
}

// Query rows per row tile: the group's rows of all queries, padded to 16, 32
// or 64; more rows than 64 take several tiles.
static int gqa_ncol(const AttnArgs& a) {
  const long long rows = (long long)a.Lq * (a.Hq / a.Hkv);
  return rows <= 16 ? 16 : rows <= 32 ? 32 : kMaxCols;
}

static int gqa_m_tiles(const AttnArgs& a) {
  const long long rows = (long long)a.Lq * (a.Hq / a.Hkv);
  return (int)((rows + gqa_ncol(a) - 1) / gqa_ncol(a));
}

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
  const int ncol = gqa_ncol(a);
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
  p.stages = gqa_stages(a.Dqk, ncol);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = test_hooks().wait_ns;
  p.skip_tile = test_hooks().skip_tile;
  if (plan.n_split > 1) {
    const size_t nrows = (size_t)a.N * a.B * a.Lq * a.Hq;
    const size_t o_bytes = nrows * plan.n_split * a.Dv * sizeof(float);
    p.dst_o = static_cast<float*>(a.workspace);
    p.dst_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ((o_bytes + 255) & ~size_t(255)));
  } else {
    p.dst_o = a.partial_out;
    p.dst_lse = a.lse;
  }
  const long long units = (long long)a.N * a.B * a.Hkv * p.m_tiles * plan.n_split;
  if (units == 0) return cudaSuccess;
  cudaError_t e = ncol == 16   ? launch_ncol<16>(tm_k, tm_v, p, units, a.stream)
                  : ncol == 32 ? launch_ncol<32>(tm_k, tm_v, p, units, a.stream)
                               : launch_ncol<kMaxCols>(tm_k, tm_v, p, units, a.stream);
  if (e != cudaSuccess || plan.n_split <= 1) return e;
  return launch_split_combine(a, plan);
}

}  // namespace dcp
