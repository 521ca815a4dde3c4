// Step a4: per-shard partial attention for MLA (one shared latent KV head of
// 576 = 512 latent + 64 rope values; the value is the first 512), on tcgen05
// tensor cores.
//
// vLLM DCP blog, "DCP 執行流程", Compute step (each shard attends the full
// query to its local KV slice and returns a partial output with its LSE) and
// section "Multi-head Latent Attention (MLA) 後端" (one low-rank latent KV head
// shared by every query head).
//
// Work unit = (shard r, request b, query i, KV split s), run by a cluster of two
// CTAs that split the 512 output dims (CTA c owns dims [256c, 256c+256)).  With
// 128 query heads the fp32 output (128 x 512) would fill a whole SM's tensor
// memory, and swapping partial scores between SMs is limited by distributed
// shared memory (~15 B/clk per direction), so each CTA instead:
//   * keeps the whole query (128 x 576 bf16, 288 columns) in TMEM and computes
//     the full score tile S = Q K^T (M=128 heads, N=64 tokens, K=576; A from
//     TMEM) into one of two TMEM buffers;
//   * receives every 64-token KV tile (72 KB, nine 64-dim boxes, 128B swizzle)
//     through cluster-multicast TMA: each CTA issues part of the boxes and both
//     CTAs receive all of them, so L2 is read once per tile;
//   * runs the online softmax with two math warpgroups, each taking 32 of the 64
//     tokens of every row (one smem max exchange per tile), writes P as bf16 in
//     place over S, and
//   * computes its half of P V in eight 32-column chunks (M=128, N=32, K=64; P
//     from TMEM, V read MN-major from the latent part of the tile) through a
//     3-deep TMEM ring; the math warpgroups fold each chunk into fp32 output
//     accumulators held in registers (warpgroup w owns chunks w, w+2, w+4, w+6),
//     applying the softmax rescale there, so O never needs a TMEM round trip.
// The score MMA of tile t+2 reuses tile t's S/P buffer after tile t's PV chunks
// (in-order tensor pipe); the softmax of tile t+1 overlaps the score MMA of
// tile t+2.  QK^T is done by both CTAs (1.53x the minimum tensor work), which
// keeps the tile loop free of any cross-SM data exchange.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2..3 idle, warps 4..7 / 8..11 math warpgroups 0 / 1 (one query
// head = TMEM lane per thread); setmaxnreg moves registers to the math warps,
// which hold 128 fp32 output accumulators each.  Every wait is bounded; on expiry the kernel records
// DCP_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "dcp_device.cuh"
#include "dcp_internal.h"
#include "dcp_sm100.cuh"
#include "dcp_tma.h"

namespace dcp {
namespace {

using namespace sm100;

constexpr int kHeads = 128;
constexpr int kDqk = 576, kDv = 512;
constexpr int kNt = 64;                        // tokens per KV tile (half a 128-token block)
constexpr int kStages = 3;
constexpr int kChunks = kDqk / 64;             // 9 boxes of 64 dims per tile
constexpr uint32_t kChunkBytes = kNt * 128;    // 64 tokens x 64 dims bf16
constexpr uint32_t kStageBytes = kChunks * kChunkBytes;   // 72 KB
constexpr int kRing = 3;                       // PV chunk ring depth
constexpr int kPvChunks = 8;                   // 256 output dims / 32
constexpr uint32_t kThreads = 384;             // 3 warpgroups
// Register split (setmaxnreg): the kernel launches at kLaunchRegs per thread;
// warpgroup 0 (producer, MMA issuer, two idle warps) gives registers up, the two
// math warpgroups take them: 128 * kCtrlRegs + 256 * kMathRegs == 384 * kLaunchRegs.
constexpr int kLaunchRegs = 168, kCtrlRegs = 56, kMathRegs = 224;
static_assert(128 * kCtrlRegs + 256 * kMathRegs <= 384 * kLaunchRegs, "register split exceeds the launch");
constexpr uint64_t kWaitNs = 2000000000ull;
// TMEM columns
constexpr uint32_t kColQ = 0;                  // 288: 128 rows x 576 bf16
constexpr uint32_t kColS = 288;                // 2 x 64: scores, then P (bf16) in place
constexpr uint32_t kColRing = 416;             // 3 x 32: PV chunks
constexpr float kRescaleLog2 = 8.0f;

struct MlaParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* dst_o;        // partial_out, or the split workspace
  float* dst_lse;
  int* status;
  int B, Lq, N, I, max_lb, bs, num_blocks, n_split, split_tokens;
  float scale_log2;    // scale * log2(e)
};

struct Smem {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];   // both CTAs' MMAs are done with the stage (count 2)
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t ring_full[kRing];
  uint64_t ring_free[kRing];
  uint64_t xchg[2];             // both math warpgroups posted their partial max (count 256)
  uint64_t fin;                 // both math warpgroups posted their row sums (count 256)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float rmax[2][2][kHeads];     // [tile parity][warpgroup][head] partial row max
  float rsum[2][kHeads];        // per-warpgroup row sums, combined at the end
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* m, int32_t c0, int32_t c1,
                                               uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar), "h"(mask)
      : "memory");
}

// Arrive on `bar` in every CTA of `mask` once this thread's MMAs are done.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      :: "r"(bar), "h"(mask) : "memory");
}

// Warp-uniform bounded wait (the tcgen05 ld/st are .sync.aligned and need
// every lane); false on abort or expiry.
__device__ __forceinline__ bool warp_wait(const volatile int* abort_flag, uint32_t bar, uint32_t par) {
  if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
  return __all_sync(0xffffffffu, mbar_wait(bar, par, kWaitNs));
}

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort_flag) {
  set_status(status, DCP_ERR_TIMEOUT);
  *abort_flag = 1;
}

// Score MMAs of tile t into S buffer t & 1 (A = query in TMEM, B = K tile).
__device__ __forceinline__ bool issue_qk(int t, Smem& sm, const uint8_t* stages, uint32_t tmem, uint32_t id_qk,
                                         const volatile int* abort_flag) {
  const int st = t % kStages;
  if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_full[st]), (uint32_t)(t / kStages) & 1u, kWaitNs)) return false;
  tc_fence_after();
  const uint8_t* sb = stages + st * kStageBytes;
  const uint32_t dcol = kColS + 64u * (uint32_t)(t & 1);
#pragma unroll 4
  for (int k = 0; k < kDqk / 16; ++k) {
    const uint64_t bdesc = smem_desc(smem_u32(sb + (k >> 2) * kChunkBytes + (k & 3) * 32), 16, 1024, kSw128);
    mma_ts(tmem + dcol, tmem + kColQ + 8 * k, bdesc, id_qk, k > 0 ? 1u : 0u);
  }
  mma_commit(smem_u32(&sm.s_full[t & 1]));
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_attn_kernel(const __grid_constant__ CUtensorMap tm_kv, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;                                        // kStages x 72 KB
  Smem& sm = *reinterpret_cast<Smem*>(base + kStages * kStageBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t cta = cluster_ctarank();          // 0 or 1: output dims [256*cta, +256)
  const long long unit = blockIdx.x >> 1;
  const int s_idx = (int)(unit % p.n_split);
  const int i_q = (int)((unit / p.n_split) % p.Lq);
  const int b = (int)((unit / ((long long)p.n_split * p.Lq)) % p.B);
  const int r = (int)(unit / ((long long)p.n_split * p.Lq * p.B));

  // key range of this unit (shard-local indices [kb, ke))
  const int S = p.seq_lens[b];
  const bool bad_len = S < p.Lq;
  int L = bad_len ? 0 : local_len(S, r, p.I, p.N);
  const bool short_table = (long long)L > (long long)p.max_lb * p.bs;
  if (short_table) L = p.max_lb * p.bs;
  const int vis = bad_len ? 0 : min(L, local_count_upto((long long)S - p.Lq + i_q, r, p.I, p.N));
  const int kb = min(vis, s_idx * p.split_tokens);
  const int ke = min(vis, kb + p.split_tokens);
  const int T = (ke - kb + kNt - 1) / kNt;
  if (tid == 0 && cta == 0 && (bad_len || short_table)) set_status(p.status, DCP_ERR_BOUNDS);

  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) {
      mbar_init(smem_u32(&sm.kv_full[k]), 1);
      mbar_init(smem_u32(&sm.kv_empty[k]), 2);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&sm.s_full[k]), 1);
      mbar_init(smem_u32(&sm.p_full[k]), 256);   // all math threads
    }
    for (int k = 0; k < kRing; ++k) {
      mbar_init(smem_u32(&sm.ring_full[k]), 1);
      mbar_init(smem_u32(&sm.ring_free[k]), 128);
    }
    mbar_init(smem_u32(&sm.xchg[0]), 256);
    mbar_init(smem_u32(&sm.xchg[1]), 256);
    mbar_init(smem_u32(&sm.fin), 256);
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // the whole query -> TMEM (row = head = TMEM lane, bf16 pairs per column);
  // math warpgroup 0 stages dims [0, 288), warpgroup 1 dims [288, 576)
  if (warp >= 4) {
    const int wg = (warp - 4) >> 2;
    const int h = (warp & 3) * 32 + lane;
    const uint4* qrow = reinterpret_cast<const uint4*>(
        p.q + (((long long)b * p.Lq + i_q) * kHeads + h) * kDqk);
    const uint32_t lane_addr = taddr(tmem, (uint32_t)((warp & 3) * 32), 0);
    for (int c = 9 * wg; c < 9 * wg + 9; ++c) {      // 16 columns = 32 dims per store
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 w = __ldg(qrow + 4 * c + k);
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
  cluster_sync();            // both CTAs' barriers initialised (multicast targets), query staged
  tc_fence_after();

  volatile int* abort_flag = &sm.abort;
  const uint16_t both = 0x3;
  if (warp < 4) {
    // ---------------- warpgroup 0: control (registers given up) ----------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kCtrlRegs));
  if (warp == 0) {
    // ---------------- TMA producer: this CTA's share of each tile, multicast ----------------
    if (lane == 0 && T > 0) {
      prefetch_tmap(&tm_kv);
      const int32_t* bt = p.block_tables + ((long long)r * p.B + b) * p.max_lb;
      const int c_lo = cta == 0 ? 0 : 5, c_hi = cta == 0 ? 5 : kChunks;
      int issued[kStages];
#pragma unroll
      for (int k = 0; k < kStages; ++k) issued[k] = 0;
      int next_blk = bt[kb / 128];
      for (int t = 0; t < T; ++t) {
        const int j = kb + t * kNt;
        const int blk = next_blk;
        if (t + 1 < T) next_blk = bt[(j + kNt) / 128];
        const int st = t % kStages;
        const uint32_t ph = (uint32_t)(t / kStages) & 1u;
        // both CTAs' MMAs must be done with the stage: the multicast writes both
        if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_empty[st]), ph ^ 1u, kWaitNs)) {
          record_timeout(p.status, abort_flag);
          break;
        }
        if ((unsigned)blk >= (unsigned)p.num_blocks) set_status(p.status, DCP_ERR_BOUNDS);
        const int row = blk * 128 + (j & 127);          // out-of-range rows read as zeros
        const uint32_t full = smem_u32(&sm.kv_full[st]);
        uint8_t* dst = stages + st * kStageBytes;
        mbar_arrive_expect_tx(full, kStageBytes);       // all nine boxes land here
        for (int c = c_lo; c < c_hi; ++c)
          tma_load_2d_mc(smem_u32(dst + c * kChunkBytes), &tm_kv, 64 * c, row, full, both);
        ++issued[st];
      }
      if (*abort_flag) {
        for (int k = 0; k < kStages; ++k)
          if (issued[k] > 0) mbar_wait(smem_u32(&sm.kv_full[k]), (uint32_t)(issued[k] - 1) & 1u, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      const uint32_t id_qk = idesc_bf16(128, kNt, false);
      const uint32_t id_pv = idesc_bf16(128, 32, true);
      bool ok = issue_qk(0, sm, stages, tmem, id_qk, abort_flag);
      int rc = 0;                                       // PV chunks issued so far
      for (int t = 0; t < T && ok; ++t) {
        // the score tile of t+1 goes into the other S buffer; it was last read
        // (as P) by tile t-1's PV chunks, issued earlier on the in-order pipe
        if (t + 1 < T && !(ok = issue_qk(t + 1, sm, stages, tmem, id_qk, abort_flag))) break;
        if (*abort_flag || !mbar_wait(smem_u32(&sm.p_full[t & 1]), (uint32_t)(t >> 1) & 1u, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* vb = stages + (t % kStages) * kStageBytes;
        const uint32_t pcol = kColS + 64u * (uint32_t)(t & 1);
        for (int jc = 0; jc < kPvChunks; ++jc, ++rc) {
          const int slot = rc % kRing;
          if (rc >= kRing &&
              (*abort_flag || !mbar_wait(smem_u32(&sm.ring_free[slot]), (uint32_t)(rc / kRing - 1) & 1u, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // output dims 256*cta + 32*jc: latent box 4*cta + jc/2, 64-byte half jc%2
          const uint8_t* vchunk = vb + (4 * (int)cta + (jc >> 1)) * kChunkBytes + (jc & 1) * 64;
#pragma unroll
          for (int k = 0; k < kNt / 16; ++k) {
            const uint64_t bdesc = smem_desc(smem_u32(vchunk + k * 2048), kChunkBytes, 1024, kSw128);
            mma_ts(tmem + kColRing + 32u * slot, tmem + pcol + 8 * k, bdesc, id_pv, k > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm.ring_full[slot]));
        }
        if (!ok) break;
        mma_commit_mc(smem_u32(&sm.kv_empty[t % kStages]), both);   // this CTA is done with the stage
      }
      if (!ok) record_timeout(p.status, abort_flag);
      mma_commit(smem_u32(&sm.drain));
      if (!mbar_wait(smem_u32(&sm.drain), 0, kWaitNs)) record_timeout(p.status, abort_flag);
    }
  }
  } else {
    // ---------------- math warpgroups (warps 4..11), registers taken ----------------
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kMathRegs));
    const int wg = (warp - 4) >> 2;                // tokens [32*wg, +32) of every tile
    const int lg = warp & 3;                       // TMEM lane group
    const int h = lg * 32 + lane;                  // query head = TMEM lane
    const int mt = tid - 128;                      // 0..255 among the math threads
    const uint32_t lane_addr = taddr(tmem, (uint32_t)(lg * 32), 0);
    float o[4][32];                                // output chunks wg, wg+2, wg+4, wg+6
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int k = 0; k < 32; ++k) o[q][k] = 0.f;
    float m_ref = -INFINITY, l = 0.f;              // l: this warpgroup's tokens only
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const uint32_t scol = kColS + 64u * (uint32_t)(t & 1);
      if (!warp_wait(abort_flag, smem_u32(&sm.s_full[t & 1]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      float x[32];
      {
        uint32_t v[32];
        tmem_ld32(lane_addr + scol + 32 * wg, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(v[k]);
      }
      const int valid = min(kNt, ke - (kb + t * kNt)) - 32 * wg;   // my valid tokens (may be <= 0)
      float pmax = -INFINITY;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        x[k] = (k < valid) ? x[k] * p.scale_log2 : -INFINITY;
        pmax = fmaxf(pmax, x[k]);
      }
      // exchange the partial row max with the other warpgroup; this also orders
      // both warpgroups' score reads before either writes P over the scores
      sm.rmax[t & 1][wg][h] = pmax;
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.xchg[t & 1]));
      if (!warp_wait(abort_flag, smem_u32(&sm.xchg[t & 1]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      const float tmax = fmaxf(pmax, sm.rmax[t & 1][wg ^ 1][h]);
      const bool grow = tmax > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - tmax);
        m_ref = tmax;
      }
      l *= alpha;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float p0 = (k < valid) ? ex2(x[k] - m_ref) : 0.f;
        const float p1 = (k + 1 < valid) ? ex2(x[k + 1] - m_ref) : 0.f;
        l += p0 + p1;
        pk[k / 2] = pack_bf16x2(p0, p1);
      }
      tmem_st16(lane_addr + scol + 16 * wg, pk);   // P tokens [32wg, +32) in place
      if (valid + 32 * wg < kNt) {
        // ragged last tile: zero this CTA's value rows past the sequence end so
        // that 0 * (NaN/Inf) from stale cache slots cannot reach O
        const int tv = max(0, valid + 32 * wg);
        uint4* vt = reinterpret_cast<uint4*>(stages + (t % kStages) * kStageBytes + 4 * cta * kChunkBytes);
        const int n16 = (kNt - tv) * 8;
        for (int idx = mt; idx < 4 * n16; idx += 256) {
          const int c = idx / n16, w = idx % n16;
          vt[(c * kChunkBytes) / 16 + tv * 8 + w] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full[t & 1]));
      // fold this tile's PV chunks into the register accumulators
      // (fully unrolled, no early exit: o[][] must stay in registers)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int rc = t * kPvChunks + wg + 2 * q;
        const int slot = rc % kRing;
        const bool got = ok && warp_wait(abort_flag, smem_u32(&sm.ring_full[slot]), (uint32_t)(rc / kRing) & 1u);
        ok = got;
        if (got) {
          tc_fence_after();
          uint32_t v[32];
          tmem_ld32(lane_addr + kColRing + 32u * slot, v);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.ring_free[slot]));
#pragma unroll
          for (int k = 0; k < 32; ++k) o[q][k] = fmaf(o[q][k], alpha, __uint_as_float(v[k]));
        }
      }
      if (!ok) break;
    }
    if (!ok) record_timeout(p.status, abort_flag);
    // combine the two warpgroups' row sums, normalise, write this CTA's dims
    sm.rsum[wg][h] = l;
    mbar_arrive(smem_u32(&sm.fin));
    const bool have = ok && T > 0 && warp_wait(abort_flag, smem_u32(&sm.fin), 0u);
    const float l_tot = have ? sm.rsum[0][h] + sm.rsum[1][h] : 0.f;
    const long long urow = (((((long long)r * p.B + b) * p.Lq + i_q) * p.n_split + s_idx) * kHeads + h);
    float* orow = p.dst_o + urow * kDv + 256 * cta;
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4* dst = reinterpret_cast<float4*>(orow + 32 * (wg + 2 * q));
#pragma unroll
      for (int k = 0; k < 8; ++k)
        dst[k] = make_float4(o[q][4 * k] * inv, o[q][4 * k + 1] * inv, o[q][4 * k + 2] * inv,
                             o[q][4 * k + 3] * inv);
    }
    if (cta == 0 && wg == 0)
      p.dst_lse[urow] = l_tot > 0.f ? (m_ref + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
  }

  // teardown: the peer no longer writes into our shared memory, then free TMEM
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t mla_smem_bytes() { return 1024 + (size_t)kStages * kStageBytes + sizeof(Smem) + 64; }

}  // namespace

bool mla_tc_supported(const AttnArgs& a) {
  return a.kind == DCP_ATTN_MLA && a.Hq == kHeads && a.Hkv == 1 && a.Dqk == kDqk && a.Dv == kDv &&
         a.bs == 128 && (long long)a.num_blocks * a.bs < (1LL << 31);
}

SplitPlan plan_attn_mla_tc(const AttnArgs& a, int sm_count) {
  return plan_splits(a, sm_count, kNt, 2 * a.Lq);
}

cudaError_t launch_attn_mla_tc(const AttnArgs& a, const SplitPlan& plan) {
  CUtensorMap tm_kv;
  const uint64_t dims[2] = {(uint64_t)kDqk, (uint64_t)a.num_blocks * a.bs};
  const uint64_t strides[1] = {(uint64_t)kDqk * 2};
  const uint32_t box[2] = {64, kNt};
  if (!make_tensor_map_bf16(&tm_kv, a.kv, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  MlaParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.status = a.status;
  p.B = a.B;
  p.Lq = a.Lq;
  p.N = a.N;
  p.I = a.I;
  p.max_lb = a.max_lb;
  p.bs = a.bs;
  p.num_blocks = a.num_blocks;
  p.n_split = plan.n_split;
  p.split_tokens = plan.split_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (plan.n_split > 1) {
    const size_t rows = (size_t)a.N * a.B * a.Lq * a.Hq;
    const size_t o_bytes = rows * plan.n_split * a.Dv * sizeof(float);
    p.dst_o = static_cast<float*>(a.workspace);
    p.dst_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ((o_bytes + 255) & ~size_t(255)));
  } else {
    p.dst_o = a.partial_out;
    p.dst_lse = a.lse;
  }
  const size_t smem = mla_smem_bytes();
  // the register split assumes the compiled launch count; refuse to launch
  // otherwise (setmaxnreg.inc would wait forever for registers that do not exist)
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, mla_attn_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(mla_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.N * a.B * a.Lq * plan.n_split;
  if (units == 0) return cudaSuccess;
  mla_attn_kernel<<<(unsigned)(2 * units), kThreads, smem, a.stream>>>(tm_kv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || plan.n_split <= 1) return e;
  return launch_split_combine(a, plan);
}

}  // namespace dcp
