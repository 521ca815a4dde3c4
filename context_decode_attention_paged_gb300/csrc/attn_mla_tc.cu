// Step a4: per-shard partial attention for MLA (one shared latent KV head of
// 576 = 512 latent + 64 rope values; the value is the first 512), on tcgen05
// tensor cores.
//
// vLLM DCP blog, "DCP 執行流程", Compute step (each shard attends the full
// query to its local KV slice and returns a partial output with its LSE) and
// section "Multi-head Latent Attention (MLA) 後端" (one low-rank latent KV head
// shared by every query head).
//
// Work unit = (shard r, request b, query i, KV split s), longest request first
// for batches up to 128, run by a cluster of
// two CTAs.  With 128 query heads the fp32 output (128 x 512) fills a whole
// SM's tensor memory and the bf16 query (128 x 576) does not fit next to a KV
// ring in shared memory, so the pair splits the head dimensions:
//   CTA c holds query dims D_c = latent[256c, 256c+256) + rope[32c, 32c+32) in
//   TMEM, streams the same dims of each 64-token KV tile (TMA, 128B/64B
//   swizzle) and computes the partial score S_c = Q_c K_c^T (M=128 heads, N=64
//   tokens, K=288; A from TMEM).  The two CTAs swap S_c through distributed
//   shared memory (16-byte st.async stores counted on the receiver's mbarrier,
//   16-bit block floating point), so both hold S = S_0 + S_1 (each with the
//   peer's half quantised) and run the same online softmax.  CTA c then accumulates output dims [256c, 256c+256):
//   O_c += P V_c (M=128, N=256, K=64; P from TMEM, V read MN-major from the
//   latent part of its own KV tile).
// Every KV byte is loaded once (each CTA loads its half of the dims) and no MMA
// is repeated.  The softmax runs in the log2 domain with a lazily updated
// reference max (O is rescaled only when the running max grows by > 2^8).
//
// Warp roles (512 threads; setmaxnreg moves registers to the softmax warps):
//   warp 0      TMA producer (4-stage ring of 36 KB tiles)
//   warp 1      PV MMA issuer, TMEM owner
//   warp 2      score (QK^T) MMA issuer - a separate thread, so the score tile of
//               t+1 and its exchange never wait behind tile t's PV
//   warp 3      idle
//   warps 4-11  softmax / epilogue, two warpgroups: warpgroup w handles tokens
//               [32w, +32) of every tile and output columns [128w, +128); they
//               combine partial row maxima once per tile (bounded mbarrier);
//               one-tile lookahead: tile t+1's scores leave TMEM before tile t's
//               softmax, releasing S to the score MMA
//   warps 12-15 score senders: read this CTA's partial scores out of TMEM and
//               push them to the peer, so the softmax never stalls on the link
// Every wait is bounded; on expiry the kernel records DCP_ERR_TIMEOUT, drains
// its own copies and MMAs, frees TMEM and returns.
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
constexpr int kDqk = 576, kDv = 512, kLatent = 512;
constexpr int kNt = 64;                       // tokens per KV tile (half a 128-token block)
constexpr int kStages = 4;
constexpr uint32_t kChunkBytes = kNt * 128;   // 64 tokens x 64 dims bf16, 128B rows
constexpr uint32_t kRopeBytes = kNt * 64;     // 64 tokens x 32 dims bf16, 64B rows
constexpr uint32_t kStageBytes = 4 * kChunkBytes + kRopeBytes;   // 36 KB
// Exchange buffer: each head's 64 partial scores travel as 16-bit integers
// sharing one power-of-two scale per head and tile (block floating point):
// 128 bytes per head in 8 chunks of 16 bytes, chunk-major (chunk k of head h
// at (k * 128 + h) * 16, so one warp's store or load of a chunk covers 512
// contiguous bytes), followed by the 128 per-head decode scales.  The DSMEM
// link moves ~15 B/clk per direction, so the 16.5 KB exchange of a tile takes
// ~1,100 cycles.  The scale maps the head's largest |partial| into [2^13, 2^14),
// so each received partial is off by at most max|partial| * 2^-15; each CTA
// adds its own partial unrounded (the two CTAs' softmax inputs differ in the
// last bits; each CTA normalises its own half of the output with its own sums).
constexpr int kXChunks = 8;
constexpr uint32_t kXScoreBytes = kHeads * kXChunks * 16;   // 16 KB
constexpr uint32_t kXBytes = kXScoreBytes + kHeads * 4;     // + one fp32 scale per head
constexpr uint32_t kThreads = 512;             // 4 warpgroups
// Register split (setmaxnreg) against the 384 x 168 registers of the launch:
// control warpgroup and score senders give registers up, softmax takes them.
constexpr int kLaunchRegs = 128, kCtrlRegs = 80, kSendRegs = 80, kSoftRegs = 160;
constexpr int kSplitRegs = 128 * kCtrlRegs + 256 * kSoftRegs + 128 * kSendRegs;   // 61,440
static_assert(kSplitRegs <= 512 * kLaunchRegs, "register split exceeds the launch");
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr int kLptMaxBatch = 128;
// TMEM columns
constexpr uint32_t kColQ = 0;      // 144 cols: 128 rows x 288 bf16
constexpr uint32_t kColP = 144;    // 32 cols: 128 rows x 64 bf16
constexpr uint32_t kColS = 192;    // 64 cols fp32
constexpr uint32_t kColO = 256;    // 256 cols fp32
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
  uint64_t kv_empty[kStages];
  uint64_t s_full, s_free, p_full, pv_done, drain, drain_qk;
  uint64_t recv_full[2];   // armed with a tile's bytes; the peer's async stores count them
  uint64_t sent_free[2];   // the peer has read what we stored into its buffer k
  uint64_t xchg[2];        // both softmax warpgroups posted their partial max (count 256)
  uint64_t fin;            // both softmax warpgroups posted their row sums (count 256)
  uint32_t tmem_base;
  int abort;
  int req;                    // request of this unit
  float rmax[2][2][kHeads];   // [tile parity][warpgroup][head] partial row max
  float rsum[2][kHeads];      // [warpgroup][head] row sums, combined at the end
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Block floating point for the score exchange.  Encoding adds 1.5 * 2^23 +
// 2^15 to the scaled score: the fp32 sum holds round(score * enc) + 2^15 as an
// integer in its low 16 bits.  Decoding places those bits under the exponent of
// 2^23 and subtracts (2^23 + 2^15) * dec in one exact FMA.
constexpr float kEncMagic = 12615680.0f;    // 1.5 * 2^23 + 2^15
constexpr float kDecBias = 8421376.0f;      // 2^23 + 2^15

// enc = 2^(13 - e), dec = 2^(e - 13) for the exponent e of amax (clamped so both
// stay normal), so |score| * enc < 2^14.
__device__ __forceinline__ void bfp_scales(float amax, float& enc, float& dec) {
  const int eb = min(max((int)(__float_as_uint(amax) >> 23), 30), 200);
  enc = __uint_as_float((uint32_t)(267 - eb) << 23);
  dec = __uint_as_float((uint32_t)(eb - 13) << 23);
}

// Paired fp32 arithmetic (one instruction for two lanes of a register pair;
// each half rounds exactly like the scalar fmaf / add).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// three-input maximum
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t bfp_pack2(float a, float b, float enc) {
  const float2 e = ffma2(make_float2(a, b), make_float2(enc, enc), make_float2(kEncMagic, kEncMagic));
  return __byte_perm(__float_as_uint(e.x), __float_as_uint(e.y), 0x5410);
}

// both 16-bit codes of w, decoded (exact)
__device__ __forceinline__ float2 bfp_unpack2(uint32_t w, float dec, float bias) {
  return ffma2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7610)),
                           __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632))),
               make_float2(dec, dec), make_float2(bias, bias));
}

template <bool kLpt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_attn_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;                                        // kStages x 36 KB
  float* xbuf = reinterpret_cast<float*>(base + kStages * kStageBytes);   // 2 buffers: peer's scores land here
  Smem& sm = *reinterpret_cast<Smem*>(base + kStages * kStageBytes + 2 * kXBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t cta = cluster_ctarank();          // 0 or 1
  const uint32_t peer = cta ^ 1u;
  // kLpt (batches up to kLptMaxBatch): units in longest-request-first order.
  // The block scheduler starts clusters in index order, so short units fill
  // the tail.  Rank k of the order (length descending, index ascending) is
  // found by counting; both CTAs of the pair compute the same request.  (The
  // loaded request index costs registers, so large batches keep the plain
  // order, whose indices are recomputed from the block index.)
  const long long unit = blockIdx.x >> 1;
  int b_lpt = 0;
  if (kLpt) {
    const long long per_req = (long long)p.N * p.Lq * p.n_split;
    const int k_req = (int)(unit / per_req);
    for (int j = tid; j < p.B; j += kThreads) {
      const int sj = p.seq_lens[j];
      int rank = 0;
#pragma unroll 1
      for (int i = 0; i < p.B; ++i) {
        const int si = p.seq_lens[i];
        rank += (si > sj) || (si == sj && i < j);
      }
      if (rank == k_req) sm.req = j;
    }
    __syncthreads();
    b_lpt = *(volatile int*)&sm.req;
  }
  const long long per_req = (long long)p.N * p.Lq * p.n_split;
  const long long rest = kLpt ? unit % per_req : unit;
  const int s_idx = (int)(rest % p.n_split);
  const int i_q = (int)((rest / p.n_split) % p.Lq);
  const int b = kLpt ? b_lpt : (int)((unit / ((long long)p.n_split * p.Lq)) % p.B);
  const int r = kLpt ? (int)(rest / ((long long)p.n_split * p.Lq)) : (int)(unit / ((long long)p.n_split * p.Lq * p.B));

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
      mbar_init(smem_u32(&sm.kv_empty[k]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.s_free), 384);     // both softmax warpgroups and the senders
    mbar_init(smem_u32(&sm.p_full), 256);
    mbar_init(smem_u32(&sm.xchg[0]), 256);
    mbar_init(smem_u32(&sm.xchg[1]), 256);
    mbar_init(smem_u32(&sm.fin), 256);
    mbar_init(smem_u32(&sm.pv_done), 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&sm.recv_full[k]), 1);
      mbar_init(smem_u32(&sm.sent_free[k]), 1);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    mbar_init(smem_u32(&sm.drain_qk), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // query slice of this CTA -> TMEM (row = head = TMEM lane, bf16 pairs per column)
  if (warp >= 4 && warp < 12) {      // the softmax warpgroups stage the query
    const int h = (warp & 3) * 32 + lane;
    const uint4* qrow = reinterpret_cast<const uint4*>(
        p.q + (((long long)b * p.Lq + i_q) * kHeads + h) * kDqk);
    const uint32_t lane_addr = taddr(tmem, (uint32_t)((warp & 3) * 32), 0);
    const int wq = (warp - 4) >> 2;
    for (int c = 5 * wq; c < (wq ? 9 : 5); ++c) {   // 9 x 16 columns = 288 dims, split 5 / 4
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // column block c covers dims [32c, 32c+32) of the slice: latent 256*cta + 32c
        // for c < 8, rope 512 + 32*cta for c == 8; 8 bf16 per uint4
        const int dim0 = (c < 8) ? (256 * (int)cta + 32 * c) : (kLatent + 32 * (int)cta);
        const uint4 w = __ldg(qrow + dim0 / 8 + k);
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
  cluster_sync();            // barriers of both CTAs initialised, query staged
  tc_fence_after();

  volatile int* abort_flag = &sm.abort;
  auto fail = [&](void) {
    set_status(p.status, DCP_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp < 4) {
    // ---------------- warpgroup 0: control (gives registers up) ----------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kCtrlRegs));
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && T > 0) {
      prefetch_tmap(&tm_lat);
      prefetch_tmap(&tm_rope);
      const int32_t* bt = p.block_tables + ((long long)r * p.B + b) * p.max_lb;
      int next_blk = bt[kb / 128];
      int issued[kStages];
#pragma unroll
      for (int k = 0; k < kStages; ++k) issued[k] = 0;
      for (int t = 0; t < T; ++t) {
        const int j = kb + t * kNt;
        const int blk = next_blk;
        if (t + 1 < T) next_blk = bt[(j + kNt) / 128];
        const int st = t % kStages;
        const uint32_t ph = (uint32_t)(t / kStages) & 1u;
        if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_empty[st]), ph ^ 1u, kWaitNs)) {
          fail();
          break;
        }
        if ((unsigned)blk >= (unsigned)p.num_blocks) set_status(p.status, DCP_ERR_BOUNDS);
        const int row = blk * 128 + (j & 127);   // out-of-range rows read as zeros
        const uint32_t full = smem_u32(&sm.kv_full[st]);
        uint8_t* dst = stages + st * kStageBytes;
        mbar_arrive_expect_tx(full, kStageBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tma_load_2d(smem_u32(dst + c * kChunkBytes), &tm_lat, 256 * (int)cta + 64 * c, row, full);
        tma_load_2d(smem_u32(dst + 4 * kChunkBytes), &tm_rope, kLatent + 32 * (int)cta, row, full);
        ++issued[st];
      }
      if (*abort_flag) {
        // let every copy this thread issued land before the CTA exits
        for (int k = 0; k < kStages; ++k)
          if (issued[k] > 0)
            mbar_wait(smem_u32(&sm.kv_full[k]), (uint32_t)(issued[k] - 1) & 1u, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- PV issuer (and TMEM owner) ----------------
    // Score and PV MMAs come from two threads, so the score tile of t+1 (and
    // its exchange) never waits behind tile t's PV, which waits for the softmax.
    if (lane == 0 && T > 0) {
      const uint32_t id_pv = idesc_bf16(128, 256, true);
      bool ok = true;
      for (int t = 0; t < T; ++t) {
        if (*abort_flag || !mbar_wait(smem_u32(&sm.p_full), (uint32_t)t & 1u, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = stages + (t % kStages) * kStageBytes;
#pragma unroll
        for (int k = 0; k < kNt / 16; ++k) {
          const uint64_t bdesc = smem_desc(smem_u32(st + k * 2048), kChunkBytes, 1024, kSw128);
          mma_ts(tmem + kColO, tmem + kColP + 8 * k, bdesc, id_pv, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.pv_done));
        // the score MMAs of tile t completed before the softmax produced P_t
        mma_commit(smem_u32(&sm.kv_empty[t % kStages]));
      }
      if (!ok) fail();
      mma_commit(smem_u32(&sm.drain));
      if (!mbar_wait(smem_u32(&sm.drain), 0, kWaitNs)) fail();
    }
  } else if (warp == 2) {
    // ---------------- score (QK^T) issuer ----------------
    if (lane == 0 && T > 0) {
      const uint32_t id_qk = idesc_bf16(128, kNt, false);
      bool ok = true;
      for (int t = 0; t < T; ++t) {
        const int st = t % kStages;
        if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_full[st]), (uint32_t)(t / kStages) & 1u, kWaitNs) ||
            (t > 0 && !mbar_wait(smem_u32(&sm.s_free), (uint32_t)(t - 1) & 1u, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* sb = stages + st * kStageBytes;
#pragma unroll
        for (int k = 0; k < 18; ++k) {
          const uint64_t bdesc =
              (k < 16) ? smem_desc(smem_u32(sb + (k >> 2) * kChunkBytes + (k & 3) * 32), 16, 1024, kSw128)
                       : smem_desc(smem_u32(sb + 4 * kChunkBytes + (k - 16) * 32), 16, 512, kSw64);
          mma_ts(tmem + kColS, tmem + kColQ + 8 * k, bdesc, id_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.s_full));
      }
      if (!ok) fail();
      mma_commit(smem_u32(&sm.drain_qk));
      if (!mbar_wait(smem_u32(&sm.drain_qk), 0, kWaitNs)) fail();
    }
  }
  } else if (warp < 12) {
    // ---------------- softmax / epilogue (warps 4..11), take registers ----------------
    // Two warpgroups split every tile's 64 tokens (warpgroup w: tokens
    // [32w, +32)) and this CTA's 256 output columns (w: [128w, +128)); they
    // combine partial row maxima once per tile and row sums at the end.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kSoftRegs));
    const int w = (warp - 4) >> 2;
    const int lg = warp & 3;                       // TMEM lane group
    const int h = lg * 32 + lane;                  // query head = TMEM lane
    const int mt = tid - 128;                      // 0..255 among the softmax threads
    const uint32_t lane_addr = taddr(tmem, (uint32_t)(lg * 32), 0);
    const uint32_t peer_sent_free = mapa(smem_u32(&sm.sent_free[0]), peer);
    float m_ref = -INFINITY, l = 0.f;              // l over this warpgroup's tokens
    bool ok = true;
    // waits and the abort flag are made warp-uniform: the tcgen05 ld/st below
    // are .sync.aligned and need every lane
    auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, kWaitNs));
    };
    // One-tile lookahead: tile t+1's partial scores are read out of TMEM (and
    // S released to the score MMA) before tile t's softmax is computed.
    float nx[32];
    auto load_scores = [&](int t) -> bool {
      if (!wwait(smem_u32(&sm.s_full), (uint32_t)t & 1u)) return false;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(lane_addr + kColS + 32 * w, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k) nx[k] = __uint_as_float(v[k]);
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_free));
      return true;
    };
    if (T > 0 && !load_scores(0)) ok = false;
    for (int t = 0; t < T && ok; ++t) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      float x[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) x[k] = nx[k];
      // the sender warpgroup has pushed our partial scores of tile t to the
      // peer; the peer's partial of tile t arrives in exchange buffer t & 1
      const int xb = t & 1;
      if (mt == 0) mbar_arrive_expect_tx(smem_u32(&sm.recv_full[xb]), kXBytes);
      if (!wwait(smem_u32(&sm.recv_full[xb]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
      {
        // peer's partial (tokens [32w, +32): chunks [4w, +4)) plus our own
        const float* xrow = xbuf + xb * (kXBytes / 4);
        const uint4* theirs = reinterpret_cast<const uint4*>(xrow) + h;
        const float dec = xrow[kXScoreBytes / 4 + h];
        const float bias = -kDecBias * dec;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 q4 = theirs[(4 * w + k) * kHeads];
          const uint32_t wq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 s = fadd2(make_float2(x[8 * k + 2 * j], x[8 * k + 2 * j + 1]), bfp_unpack2(wq[j], dec, bias));
            x[8 * k + 2 * j] = s.x;
            x[8 * k + 2 * j + 1] = s.y;
          }
        }
      }
      // online softmax in the log2 domain on raw scores (scale > 0 is folded
      // into the exponent); tree reductions keep dependency chains short
      const int valid = min(kNt, ke - (kb + t * kNt)) - 32 * w;   // may be <= 0
      const bool full = valid >= 32;
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int k = 0; k < 32; k += 8)
#pragma unroll
          for (int j = 0; j < 4; ++j) m4[j] = fmax3(m4[j], x[k + j], x[k + 4 + j]);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) m4[k & 3] = fmaxf(m4[k & 3], (k < valid) ? x[k] : -INFINITY);
      }
      const float pmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
      // post the partial max; the barrier also tells us both warpgroups have
      // read exchange buffer xb, so the peer may refill it
      sm.rmax[xb][w][h] = pmax;
      mbar_arrive(smem_u32(&sm.xchg[xb]));
      if (!wwait(smem_u32(&sm.xchg[xb]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
      if (mt == 0) mbar_arrive_remote_signal(peer_sent_free + 8 * xb);
      const float tmax = fmaxf(pmax, sm.rmax[xb][w ^ 1][h]);
      if (t + 1 < T && !load_scores(t + 1)) { ok = false; break; }
      const bool grow = tmax > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - tmax);
        m_ref = tmax;
      }
      const float sl2 = p.scale_log2, nm = -m_ref;
      uint32_t pk[16];
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
      if (full) {
        float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 y = ffma2(make_float2(x[k], x[k + 1]), make_float2(sl2, sl2), make_float2(nm, nm));
          const float p0 = ex2(y.x);
          const float p1 = ex2(y.y);
          if ((k >> 1) & 1) lb = fadd2(lb, make_float2(p0, p1));
          else la = fadd2(la, make_float2(p0, p1));
          pk[k / 2] = pack_bf16x2(p0, p1);
        }
        l4[0] = la.x; l4[1] = la.y; l4[2] = lb.x; l4[3] = lb.y;
      } else {
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float p0 = (k < valid) ? ex2(fmaf(x[k], sl2, nm)) : 0.f;
          const float p1 = (k + 1 < valid) ? ex2(fmaf(x[k + 1], sl2, nm)) : 0.f;
          l4[(k >> 1) & 3] += p0 + p1;
          pk[k / 2] = pack_bf16x2(p0, p1);
        }
      }
      l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
      // PV of the previous tile must be done before O is rescaled or P rewritten
      if (t > 0) {
        if (!wwait(smem_u32(&sm.pv_done), (uint32_t)(t - 1) & 1u)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
          for (int c = 0; c < 128; c += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + kColO + 128 * w + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(lane_addr + kColO + 128 * w + c, v);
          }
        }
      }
      const int tv = min(kNt, ke - (kb + t * kNt));
      if (tv < kNt) {
        // ragged last tile: rows past the sequence hold whatever the cache
        // block holds; zero their value part so 0 * (NaN/Inf) cannot reach O.
        // Whole 128-byte rows, so the swizzle does not matter.
        uint4* st = reinterpret_cast<uint4*>(stages + (t % kStages) * kStageBytes);
        const int n16 = (kNt - tv) * 8;                  // uint4 per chunk
        for (int idx = mt; idx < 4 * n16; idx += 256) {
          const int c = idx / n16, q = idx % n16;
          st[(c * kChunkBytes) / 16 + tv * 8 + q] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tmem_st16(lane_addr + kColP + 16 * w, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full));
    }
    if (!ok) fail();
    // epilogue: combine the warpgroups' row sums, normalise, write columns
    // [128w, +128) of this CTA's half of the output dims
    sm.rsum[w][h] = l;
    mbar_arrive(smem_u32(&sm.fin));
    bool have = ok && T > 0 && wwait(smem_u32(&sm.fin), 0u);
    if (have) {
      have = wwait(smem_u32(&sm.pv_done), (uint32_t)(T - 1) & 1u);
      if (!have) fail();
    }
    tc_fence_after();
    const long long urow = (((((long long)r * p.B + b) * p.Lq + i_q) * p.n_split + s_idx) * kHeads + h);
    float* orow = p.dst_o + urow * kDv + 256 * cta + 128 * w;
    const float l_tot = have ? sm.rsum[0][h] + sm.rsum[1][h] : 0.f;
    if (have && l_tot > 0.f) {
      const float inv = 1.f / l_tot;
      for (int c = 0; c < 128; c += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + kColO + 128 * w + c, v);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(orow + c);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                               __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
      }
      if (cta == 0 && w == 0) p.dst_lse[urow] = (m_ref + log2f(l_tot)) * 0.69314718055994531f;
    } else {
      float4* dst = reinterpret_cast<float4*>(orow);
      for (int k = 0; k < 32; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (cta == 0 && w == 0) p.dst_lse[urow] = -INFINITY;
    }
  } else {
    // ---------------- score senders (warps 12..15), give registers up ----------------
    // Each tile's partial scores go to the peer as 16-byte async stores that
    // count bytes on the peer's barrier; a dedicated warpgroup does it so the
    // softmax warps never stall on the DSMEM link.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kSendRegs));
    const int lg = warp & 3;
    const int h = lg * 32 + lane;
    const uint32_t lane_addr = taddr(tmem, (uint32_t)(lg * 32), 0);
    const uint32_t peer_x = mapa(smem_u32(xbuf + 4 * h), peer);                 // chunk 0 of head h
    const uint32_t peer_xs = mapa(smem_u32(xbuf + kXScoreBytes / 4 + h), peer);  // scale of head h
    const uint32_t peer_recv_full = mapa(smem_u32(&sm.recv_full[0]), peer);
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      if (__any_sync(0xffffffffu, *abort_flag != 0) ||
          !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full), (uint32_t)t & 1u, kWaitNs))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(lane_addr + kColS, v0);
      tmem_ld32(lane_addr + kColS + 32, v1);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_free));
      const int xb = t & 1;
      if (t >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.sent_free[xb]), (uint32_t)((t >> 1) - 1) & 1u, kWaitNs))) {
        ok = false;
        break;
      }
      const uint32_t dst = peer_x + xb * kXBytes;
      const uint32_t bar = peer_recv_full + 8 * xb;
      // rows past the end of a ragged tile hold stale cache bytes: zero them so
      // they cannot set the scale (the softmax masks them anyway)
      const int tv = min(kNt, ke - (kb + t * kNt));
      if (tv < kNt) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (k >= tv) v0[k] = 0u;
          if (k + 32 >= tv) v1[k] = 0u;
        }
      }
      float a8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) a8[k] = fmaxf(fabsf(__uint_as_float(v0[k])), fabsf(__uint_as_float(v1[k])));
#pragma unroll
      for (int k = 8; k < 32; ++k)
        a8[k & 7] = fmax3(a8[k & 7], fabsf(__uint_as_float(v0[k])), fabsf(__uint_as_float(v1[k])));
      const float amax = fmaxf(fmaxf(fmaxf(a8[0], a8[1]), fmaxf(a8[2], a8[3])),
                               fmaxf(fmaxf(a8[4], a8[5]), fmaxf(a8[6], a8[7])));
      float enc, dec;
      bfp_scales(amax, enc, dec);
      // chunk k carries tokens [8k, 8k + 8): two per word
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_async_v4(dst + k * (kHeads * 16),
                    __uint_as_float(bfp_pack2(__uint_as_float(v0[8 * k]), __uint_as_float(v0[8 * k + 1]), enc)),
                    __uint_as_float(bfp_pack2(__uint_as_float(v0[8 * k + 2]), __uint_as_float(v0[8 * k + 3]), enc)),
                    __uint_as_float(bfp_pack2(__uint_as_float(v0[8 * k + 4]), __uint_as_float(v0[8 * k + 5]), enc)),
                    __uint_as_float(bfp_pack2(__uint_as_float(v0[8 * k + 6]), __uint_as_float(v0[8 * k + 7]), enc)),
                    bar);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_async_v4(dst + (k + 4) * (kHeads * 16),
                    __uint_as_float(bfp_pack2(__uint_as_float(v1[8 * k]), __uint_as_float(v1[8 * k + 1]), enc)),
                    __uint_as_float(bfp_pack2(__uint_as_float(v1[8 * k + 2]), __uint_as_float(v1[8 * k + 3]), enc)),
                    __uint_as_float(bfp_pack2(__uint_as_float(v1[8 * k + 4]), __uint_as_float(v1[8 * k + 5]), enc)),
                    __uint_as_float(bfp_pack2(__uint_as_float(v1[8 * k + 6]), __uint_as_float(v1[8 * k + 7]), enc)),
                    bar);
      st_async_b32(peer_xs + xb * kXBytes, __float_as_uint(dec), bar);
    }
    if (!ok) fail();
  }

  // teardown: the peer no longer touches our shared memory, then free TMEM
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t mla_smem_bytes() { return 1024 + (size_t)kStages * kStageBytes + 2 * kXBytes + sizeof(Smem) + 64; }

}  // namespace

bool mla_tc_supported(const AttnArgs& a) {
  return a.kind == DCP_ATTN_MLA && a.Hq == kHeads && a.Hkv == 1 && a.Dqk == kDqk && a.Dv == kDv &&
         a.bs == 128 && (long long)a.num_blocks * a.bs < (1LL << 31);
}

SplitPlan plan_attn_mla_tc(const AttnArgs& a, int sm_count) {
  return plan_splits(a, sm_count, kNt, 2 * a.Lq);
}

cudaError_t launch_attn_mla_tc(const AttnArgs& a, const SplitPlan& plan) {
  CUtensorMap tm_lat, tm_rope;
  const uint64_t dims[2] = {(uint64_t)kDqk, (uint64_t)a.num_blocks * a.bs};
  const uint64_t strides[1] = {(uint64_t)kDqk * 2};
  const uint32_t box_lat[2] = {64, kNt};
  const uint32_t box_rope[2] = {32, kNt};
  if (!make_tensor_map_bf16(&tm_lat, a.kv, 2, dims, strides, box_lat, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&tm_rope, a.kv, 2, dims, strides, box_rope, CU_TENSOR_MAP_SWIZZLE_64B))
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
  const bool lpt = a.B <= kLptMaxBatch;
  void (*kern)(const CUtensorMap, const CUtensorMap, const MlaParams) =
      lpt ? mla_attn_kernel<true> : mla_attn_kernel<false>;
  // the register split assumes the compiled launch count; refuse to launch
  // otherwise (setmaxnreg.inc would wait for registers that do not exist)
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * (int)kThreads < kSplitRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.N * a.B * a.Lq * plan.n_split;
  if (units == 0) return cudaSuccess;
  kern<<<(unsigned)(2 * units), kThreads, smem, a.stream>>>(tm_lat, tm_rope, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || plan.n_split <= 1) return e;
  return launch_split_combine(a, plan);
}

}  // namespace dcp
