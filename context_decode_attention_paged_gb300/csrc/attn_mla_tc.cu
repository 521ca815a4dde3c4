// Step a4: per-shard partial attention for MLA (one shared latent KV head of
// 576 = 512 latent + 64 rope values; the value is the first 512), on tcgen05
// tensor cores.
//
// vLLM DCP blog, "DCP 執行流程", Compute step (each shard attends the full
// query to its local KV slice and returns a partial output with its LSE) and
// section "Multi-head Latent Attention (MLA) 後端" (one low-rank latent KV head
// shared by every query head).
//
// Work unit = (shard r, request b, query i, KV split s), run by a cluster of
// two CTAs, longest request first (up to 128 requests every CTA ranks them
// itself; larger batches read the order from a pre-pass kernel).  With 128
// query heads the fp32 output (128 x 512) fills a whole SM's tensor memory and
// the bf16 query (128 x 576) does not fit next to a KV ring in shared memory,
// so the pair splits the head dimensions for the two products:
//   CTA c holds query dims D_c = latent[256c, +256) + rope[32c, +32) (latent
//   dims 64-255 of the slice in TMEM, the rest in shared memory, all staged by
//   TMA), streams the same dims of each 64-token KV tile (TMA, 128B/64B
//   swizzle; one box per tile, or one per block for blocks of 8-32 tokens),
//   computes the partial scores S_c = Q_c K_c^T (M = 128 heads, N = 64
//   tokens, K = 288; A from TMEM and shared memory) into one of two score
//   buffers, and accumulates O_c += P V_c for output dims [256c, +256)
//   (M = 128, N = 256, K = 64; P from TMEM, V read MN-major out of the latent
//   part of its tile),
// and splits the tokens for the softmax: CTA c owns tokens [32c, +32) of
// every tile.  It sends the peer its partial scores of the peer's 32 tokens
// (16-bit block floating point, one power-of-two scale per head and tile, and a
// 16-bit residual when some head's partials are large) and adds the peer's
// partial of its own 32 tokens to its own, so every score is formed,
// exponentiated and summed once per pair.  The two CTAs swap the maxima of
// their halves (one float per head) while the exponentials run, so both apply
// the same reference to the tile; the bf16 probabilities of its 32 tokens then
// go to the peer with their row sum, and each CTA writes both halves into its
// P buffer in TMEM.  Every KV byte is loaded once and no MMA is repeated.
// With fewer than 128 query heads (16 or more) the MMA rows past Hq hold the
// next query rows of the tensor: computed, never written.
//
// Reference.  P = exp2(score * scale * log2(e) - R) in the log2 domain; R(t)
// is the running maximum, updated lazily: it moves to the tile's maximum only
// when that exceeds it by more than 2^3 (then O and the row sums are rescaled
// once, after the previous PV product has landed), so P <= 2^8 and the token
// that moved R gets exactly 1.  Each probability is rounded to bf16 once.
//
// Warp roles (512 threads; setmaxnreg moves registers to the softmax warps):
//   warp 0      TMA producer (5-stage ring of 36 KB tiles)
//   warp 1      PV MMA issuer, TMEM owner; PV(t) goes out once the score MMAs
//               of tile t+1 are issued, so that each tile's score MMAs run
//               back to back and PV fills the gap while the scores are read
//   warp 2      score (QK^T) MMA issuer
//   warps 4-7   softmax warpgroup 0: tiles 0, 2, 4, ...
//   warps 8-11  softmax warpgroup 1: tiles 1, 3, 5, ...  The two warpgroups
//               overlap on consecutive tiles: while one waits for the peer's
//               half of its tile, the other computes the next; R(t) passes
//               from one to the other through shared memory.  At the end
//               they stage O in the idle ring, from where TMA stores it
//   warps 12-15 score senders: read the peer's half of every tile's partial
//               scores out of TMEM and push them to the peer
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
constexpr int kNt = 64;                        // tokens per KV tile
constexpr int kHalf = 32;                      // tokens of a tile whose softmax a CTA owns
constexpr int kStages = 5;
constexpr uint32_t kChunkBytes = kNt * 128;    // 64 tokens x 64 dims bf16, 128B rows
constexpr uint32_t kRopeBytes = kNt * 64;      // 64 tokens x 32 dims bf16, 64B rows
constexpr uint32_t kStageBytes = 4 * kChunkBytes + kRopeBytes;   // 36 KB
// Messages between the two CTAs (each a 16-byte st.async per head and chunk,
// counted on the receiver's mbarrier).  Chunk k of head h sits at
// (k * 128 + h) * 16, so a warp's 32 heads of one chunk are 512 contiguous
// bytes.  Four chunks carry a head's 32 tokens (two per 32-bit word).  Scores
// and probabilities have one slot each (the sender of tile t waits until the
// receiver has read tile t-1; the barriers alternate by tile parity); the
// residual of a flagged tile goes into the score
// slot once the receiving warp has read the main codes (a per-warp handshake;
// flagged tiles are rare).
constexpr uint32_t kMsgCodes = kHeads * 4 * 16;             // 8 KB
constexpr uint32_t kScMsgBytes = kMsgCodes + kHeads * 4;    // + one decode scale per head
constexpr uint32_t kPmMsgBytes = kMsgCodes + kHeads * 4;    // + one row sum per head
constexpr uint32_t kMxMsgBytes = kHeads * 4;                // one local maximum per head
// Each warp of a quadrant (32 heads) exchanges its part of a message with the
// same quadrant's warp of the peer, on barriers of its own.
constexpr uint32_t kScWarpBytes = kScMsgBytes / 4;
constexpr uint32_t kPmWarpBytes = kPmMsgBytes / 4;
constexpr uint32_t kQRopeBytes = kHeads * 64;               // query rope dims, 64B rows
constexpr uint32_t kQLat0Bytes = kHeads * 128;              // query latent dims 0-63 of the slice, 128B rows
constexpr uint32_t kThreads = 512;                          // 4 warpgroups
// Register split (setmaxnreg) against the 512 x 128 registers of the launch:
// control warpgroup and score senders give registers up, softmax takes them.
constexpr int kLaunchRegs = 128, kCtrlRegs = 48, kSendRegs = 96, kSoftRegs = 176;
constexpr int kSplitRegs = 128 * kCtrlRegs + 256 * kSoftRegs + 128 * kSendRegs;   // 63,488
static_assert(kSplitRegs <= 512 * kLaunchRegs, "register split exceeds the launch");
constexpr int kLptMaxBatch = 128;        // up to this batch every CTA ranks the requests itself
constexpr int kLptOrderMaxBatch = 16384; // up to this batch a pre-pass writes the order
// TMEM columns (512 allocated)
constexpr uint32_t kColQ = 0;      // 96 cols: 128 rows x latent dims 64-255 of the slice, bf16
constexpr uint32_t kColS = 96;     // 2 x 64 cols fp32: partial scores of tile t in buffer t & 1
constexpr uint32_t kColP = 224;    // 32 cols: P (128 rows x 64 bf16)
constexpr uint32_t kColO = 256;    // 256 cols fp32 output
constexpr float kLazyLog2 = 8.0f;       // R moves when scores pass it by more than this
constexpr float kResidualLog2 = 8.0f;   // |partial| * scale above this (log2 units): send a residual
constexpr uint32_t kBarEpi = 1;         // named barrier of the two softmax warpgroups (epilogue)
constexpr uint32_t kOBoxBytes = kHeads * 128;   // staged output box: 128 rows x 32 fp32
constexpr int kPvGate = 1;              // PV(t) waits for the score MMAs of tile t + kPvGate

struct MlaParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* order;   // longest-first request order from the pre-pass (null: rank in the kernel)
  float* dst_o;        // partial_out, or the split workspace
  float* dst_lse;
  int* status;
  int B, Lq, Hq, N, I, max_lb, bs, num_blocks, n_split, split_tokens;
  float scale_log2;    // scale * log2(e)
  unsigned long long wait_ns;   // limit of every bounded wait
  int skip_tile;                // test hook: CTA 0 never loads this tile (-1: off)
};

struct Smem {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];      // partial scores of tile t in score buffer t & 1
  uint64_t s_free[2];      // senders (128) and the tile's softmax warpgroup (128) have read them
  uint64_t sc_recv[2][4];  // [tile parity][quadrant] the peer's partial scores of tile t arrived
  uint64_t sc_res[2][4];   // [warpgroup][quadrant] the residual of a flagged tile arrived
  uint64_t sc_mfree[2][4]; // [warpgroup][quadrant] the peer has read the main codes of a flagged tile
  uint64_t sc_free[2][4];  // [tile parity][quadrant] the peer has read the scores of tile t we stored
  uint64_t pm_recv[2][4];  // [tile parity][quadrant] the peer's probabilities of tile t arrived
  uint64_t pm_free[2][4];  // [tile parity][quadrant] the peer has read the probabilities of tile t we stored
  uint64_t mx_recv[2][4];  // [tile parity][quadrant] the peer's half maxima of tile t arrived
  uint64_t p_full[2];      // both halves of P(t) are in the P buffer (128; by t & 1)
  uint64_t pv_done[2];     // PV(t) complete (commit)
  uint64_t r_pub[2][4];    // [tile parity][quadrant] R(t) published by tile t's warp of the quadrant
  uint64_t fin;            // both softmax warpgroups posted their row sums (256)
  uint64_t q_full;         // the query slice of the unit has landed (TMA)
  uint64_t drain, drain_qk;
  uint32_t tmem_base;
  int abort;
  int qk_issued;               // last tile whose score MMAs are issued
  int req;                     // request of this unit
  float rref[2][kHeads];       // R(t) by tile parity
  float lw[2][kHeads];         // final: each warpgroup's row sum
  float rlast[2][kHeads];      // final: the reference of that row sum
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kQRopeBytes + kQLat0Bytes + kScMsgBytes +
                              kPmMsgBytes + 2 * kMxMsgBytes + sizeof(Smem) + 64;
static_assert(kSmemBytes <= 232448, "shared memory of the MLA kernel");
static_assert(8 * kOBoxBytes <= kStages * kStageBytes, "the staged output fits the ring");

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
// stay normal, and enc * 2^15 too), so |score| * enc < 2^14.
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

// 16-bit codes of a and b (low, high half of the word)
__device__ __forceinline__ uint32_t bfp_pack2(float a, float b, float enc) {
  const float2 e = ffma2(make_float2(a, b), make_float2(enc, enc), make_float2(kEncMagic, kEncMagic));
  return __byte_perm(__float_as_uint(e.x), __float_as_uint(e.y), 0x5410);
}

// What the receiver decodes for a and b (exact): round(x * enc) * dec.
__device__ __forceinline__ float2 bfp_round2(float a, float b, float enc, float dec) {
  const float2 e = ffma2(make_float2(a, b), make_float2(enc, enc), make_float2(kEncMagic, kEncMagic));
  return make_float2((e.x - kEncMagic) * dec, (e.y - kEncMagic) * dec);
}

// both 16-bit codes of w, decoded (exact)
__device__ __forceinline__ float2 bfp_unpack2(uint32_t w, float dec, float bias) {
  return ffma2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7610)),
                           __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632))),
               make_float2(dec, dec), make_float2(bias, bias));
}

struct Unit {
  int r, b, i_q, s_idx, kb, ke, T;
};

// valid tokens of tile t in half `half` (tokens [32 half, +32)) of the tile
__device__ __forceinline__ int valid_of_half(const Unit& u, int t, int half) {
  const int tv = min(kNt, u.ke - (u.kb + t * kNt));
  return min(kHalf, max(0, tv - kHalf * half));
}

// ---------------------------------------------------------------------------
// softmax warpgroup w (tiles w, w + 2, ...)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void softmax_wg(const MlaParams& p, const CUtensorMap& tm_out, Smem& sm, const Unit& u,
                                           uint8_t* stages,
                                           const uint8_t* scbuf, const uint8_t* pmbuf, const float* mxbuf,
                                           uint32_t tmem, uint32_t cta, int warp, int lane) {
  const uint32_t peer = cta ^ 1u;
  const int w = (warp - 4) >> 2;                   // warpgroup 0 / 1
  const int lg = warp & 3;                         // TMEM lane quadrant
  const int h = lg * 32 + lane;                    // head = TMEM lane
  const int mt = (warp & 3) * 32 + lane;           // 0..127 within the warpgroup
  const uint32_t lane_addr = taddr(tmem, (uint32_t)(lg * 32), 0);
  const float sl2 = p.scale_log2;
  const int T = u.T;
  volatile int* abort_flag = &sm.abort;
  // remote addresses in the peer CTA
  const uint32_t peer_pm = mapa(smem_u32(pmbuf) + (uint32_t)h * 16u, peer);
  const uint32_t peer_pm_sum = mapa(smem_u32(pmbuf) + kMsgCodes + (uint32_t)h * 4u, peer);
  const uint32_t peer_mx = mapa(smem_u32(mxbuf + h), peer);
  const uint32_t peer_mx_recv = mapa(smem_u32(&sm.mx_recv[0][lg]), peer);
  const uint32_t peer_pm_recv = mapa(smem_u32(&sm.pm_recv[0][lg]), peer);   // + 32 * parity
  const uint32_t peer_sc_free = mapa(smem_u32(&sm.sc_free[0][lg]), peer);
  const uint32_t peer_pm_free = mapa(smem_u32(&sm.pm_free[0][lg]), peer);

  bool ok = true;
  auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, par, p.wait_ns));
  };

  float lw = 0.f, rw = -INFINITY;     // this warpgroup's row sum, at the reference of its last tile
  int nres = 0;                       // residual messages this warp received
  const uint32_t peer_mfree = mapa(smem_u32(&sm.sc_mfree[w][lg]), peer);

  for (int t = w; t < T; t += 2) {
    if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
    const int xb = t & 1;
    // own-token partial scores of tile t (releases the score buffer)
    if (!wwait(smem_u32(&sm.s_full[xb]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
    float x[32];
    {
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(lane_addr + kColS + 64u * (uint32_t)xb + (uint32_t)kHalf * cta, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(v[k]);
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_free[xb]));
    }
    // plus the peer's partial of the same tokens
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(&sm.sc_recv[xb][lg]), kScWarpBytes);
      mbar_arrive_expect_tx(smem_u32(&sm.pm_recv[xb][lg]), kPmWarpBytes);
      mbar_arrive_expect_tx(smem_u32(&sm.mx_recv[xb][lg]), 32 * 4);
    }
    if (!wwait(smem_u32(&sm.sc_recv[xb][lg]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
    {
      const uint8_t* slot = scbuf;
      float dec = reinterpret_cast<const float*>(slot + kMsgCodes)[h];
      const bool flagged = dec < 0.f;               // same for every head of the tile
      dec = fabsf(dec);
      const float bias = -kDecBias * dec;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 q4 = reinterpret_cast<const uint4*>(slot)[k * kHeads + h];
        const uint32_t wq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 s = fadd2(make_float2(x[8 * k + 2 * j], x[8 * k + 2 * j + 1]), bfp_unpack2(wq[j], dec, bias));
          x[8 * k + 2 * j] = s.x;
          x[8 * k + 2 * j + 1] = s.y;
        }
      }
      if (__any_sync(0xffffffffu, flagged)) {
        // large partials of this warp's heads: the 16-bit residual of every
        // code follows in the same slot once this warp has read the codes
        const unsigned used = __ballot_sync(0xffffffffu, x[0] + x[31] > 0.f);
        asm volatile("" :: "r"(used));
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&sm.sc_res[w][lg]), 32 * 4 * 16);
          mbar_arrive_remote(peer_mfree);
        }
        if (!wwait(smem_u32(&sm.sc_res[w][lg]), (uint32_t)nres & 1u)) { ok = false; break; }
        ++nres;
        const uint8_t* rs = scbuf;
        const float decr = dec * (1.0f / 32768.0f);
        const float biasr = -kDecBias * decr;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 q4 = reinterpret_cast<const uint4*>(rs)[k * kHeads + h];
          const uint32_t wq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 s = fadd2(make_float2(x[8 * k + 2 * j], x[8 * k + 2 * j + 1]), bfp_unpack2(wq[j], decr, biasr));
            x[8 * k + 2 * j] = s.x;
            x[8 * k + 2 * j + 1] = s.y;
          }
        }
      }
    }
    // local maximum of the valid tokens (log2 units)
    const int valid = valid_of_half(u, t, (int)cta);
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (valid == kHalf) {
#pragma unroll
      for (int k = 0; k < 32; k += 8)
#pragma unroll
        for (int j = 0; j < 4; ++j) m4[j] = fmax3(m4[j], x[k + j], x[k + 4 + j]);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) m4[k & 3] = fmaxf(m4[k & 3], (k < valid) ? x[k] : -INFINITY);
    }
    const float ml = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
    // every received score has been used (the maximum depends on all of
    // them, and the vote on all lanes' maxima): the peer may refill this slot
    {
      const unsigned used = __ballot_sync(0xffffffffu, ml > 0.f);
      asm volatile("" :: "r"(used));
      if (lane == 0) mbar_arrive_remote_signal(peer_sc_free + 32 * xb);
    }
    st_async_b32(peer_mx + (uint32_t)xb * (kHeads * 4), __float_as_uint(ml), peer_mx_recv + 32u * (uint32_t)xb);
    // exponentials against this half's own maximum (fp32, <= 1; masked tokens 0)
    // while the peer's maximum is on its way
    const float nml = (ml == -INFINITY) ? 0.f : -ml;
    float e[32];
    float l4[4] = {0.f, 0.f, 0.f, 0.f};
    if (valid == kHalf) {
      float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float2 y = ffma2(make_float2(x[k], x[k + 1]), make_float2(sl2, sl2), make_float2(nml, nml));
        e[k] = ex2(y.x);
        e[k + 1] = ex2(y.y);
        if ((k >> 1) & 1) lb = fadd2(lb, make_float2(e[k], e[k + 1]));
        else la = fadd2(la, make_float2(e[k], e[k + 1]));
      }
      l4[0] = la.x; l4[1] = la.y; l4[2] = lb.x; l4[3] = lb.y;
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        e[k] = (k < valid) ? ex2(fmaf(x[k], sl2, nml)) : 0.f;
        l4[k & 3] += e[k];
      }
    }
    const float l_e = (l4[0] + l4[1]) + (l4[2] + l4[3]);
    // R(t) moves lazily from R(t-1) (published by the other warpgroup's warp of
    // this quadrant) to the tile's maximum over both halves (the peer's half
    // maximum arrives while the exponentials run)
    float r_prev = -INFINITY;
    if (t >= 1) {
      if (!wwait(smem_u32(&sm.r_pub[(t - 1) & 1][lg]), (uint32_t)((t - 1) >> 1) & 1u)) { ok = false; break; }
      r_prev = sm.rref[(t - 1) & 1][h];
    }
    if (!wwait(smem_u32(&sm.mx_recv[xb][lg]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
    const float gmax = fmaxf(ml, mxbuf[xb * kHeads + h]);
    const float R = (gmax > r_prev + kLazyLog2) ? gmax : r_prev;
    sm.rref[xb][h] = R;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.r_pub[xb][lg]));
    // P = e * 2^(ml - R) <= 2^8, rounded to bf16 once
    const float f = (ml == -INFINITY) ? 0.f : ex2(ml - R);
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      const float2 pp2 = ffma2(make_float2(e[k], e[k + 1]), make_float2(f, f), make_float2(0.f, 0.f));
      pk[k / 2] = pack_bf16x2(pp2.x, pp2.y);
    }
    const float lsum = l_e * f;
    {
      // the peer has read our probabilities of tile t-1 out of its one slot
      if (t >= 1 && !wwait(smem_u32(&sm.pm_free[(t - 1) & 1][lg]), (uint32_t)((t - 1) >> 1) & 1u)) { ok = false; break; }
      const uint32_t bar = peer_pm_recv + 32u * (uint32_t)xb;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_async_v4(peer_pm + k * (kHeads * 16), __uint_as_float(pk[4 * k]), __uint_as_float(pk[4 * k + 1]),
                    __uint_as_float(pk[4 * k + 2]), __uint_as_float(pk[4 * k + 3]), bar);
      st_async_b32(peer_pm_sum, __float_as_uint(lsum), bar);
    }
    // the peer's probabilities of its tokens of tile t
    if (!wwait(smem_u32(&sm.pm_recv[xb][lg]), (uint32_t)(t >> 1) & 1u)) { ok = false; break; }
    uint32_t pp[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = reinterpret_cast<const uint4*>(pmbuf)[k * kHeads + h];
      pp[4 * k] = v.x; pp[4 * k + 1] = v.y; pp[4 * k + 2] = v.z; pp[4 * k + 3] = v.w;
    }
    const float l_peer = reinterpret_cast<const float*>(pmbuf + kMsgCodes)[h];
    lw = lw * ex2(rw - R) + (lsum + l_peer);
    rw = R;
    // the P buffer and O: PV(t-1) must be done (it implies every earlier PV,
    // and the wait for PV(t-3) before tile t-2's P keeps the parity unambiguous)
    if (t >= 1 && !wwait(smem_u32(&sm.pv_done[xb ^ 1]), (uint32_t)((t - 1) >> 1) & 1u)) { ok = false; break; }
    // O moves from R(t-1) to R(t) (rare)
    const float alpha = ex2(r_prev - R);
    if (t >= 1 && __any_sync(0xffffffffu, R != r_prev)) {
      tc_fence_after();
      for (int c = 0; c < 256; c += 32) {
        uint32_t v[32];
        tmem_ld32(lane_addr + kColO + c, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
        tmem_st32(lane_addr + kColO + c, v);
      }
    }
    // ragged last tile: value rows past the range hold whatever the cache block
    // holds; zero them so that 0 * (NaN/Inf) cannot reach O (whole 128-byte
    // rows, so the swizzle does not matter)
    const int tv = min(kNt, u.ke - (u.kb + t * kNt));
    if (tv < kNt) {
      uint4* st = reinterpret_cast<uint4*>(stages + (t % kStages) * kStageBytes);
      const int n16 = (kNt - tv) * 8;
      for (int idx = mt; idx < 4 * n16; idx += 128) {
        const int c = idx / n16, q = idx % n16;
        st[(c * kChunkBytes) / 16 + tv * 8 + q] = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    tc_fence_after();
    tmem_st16(lane_addr + kColP + 16u * cta, pk);
    tmem_st16(lane_addr + kColP + 16u * peer, pp);
    tmem_wait_st();
    // the peer's probabilities are in TMEM: it may refill our slot
    __syncwarp();
    if (lane == 0) mbar_arrive_remote_signal(peer_pm_free + 32 * xb);
    tc_fence_before();
    mbar_arrive(smem_u32(&sm.p_full[xb]));
  }
  if (!ok) {
    set_status(p.status, DCP_ERR_TIMEOUT);
    *abort_flag = 1;
  }
  // epilogue: both warpgroups' row sums at the last tile's reference
  sm.lw[w][h] = lw;
  sm.rlast[w][h] = rw;
  mbar_arrive(smem_u32(&sm.fin));
  bool have = ok && T > 0 && wwait(smem_u32(&sm.fin), 0u);
  if (have) have = __all_sync(0xffffffffu, *abort_flag == 0);
  if (have) {
    have = wwait(smem_u32(&sm.pv_done[(T - 1) & 1]), (uint32_t)((T - 1) >> 1) & 1u);
    if (!have) {
      set_status(p.status, DCP_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }
  // one decision for the CTA (both warpgroups): every PV landed, nothing aborted
  have = !bar_red_or(kBarEpi, 256, !have);
  tc_fence_after();
  float l_tot = 0.f, r_fin = -INFINITY;
  if (have) {
    r_fin = sm.rlast[(T - 1) & 1][h];
    l_tot = sm.lw[0][h] * ex2(sm.rlast[0][h] - r_fin) + sm.lw[1][h] * ex2(sm.rlast[1][h] - r_fin);
  }
  const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
  const long long row0 = ((((long long)u.r * p.B + u.b) * p.Lq + u.i_q) * p.n_split + u.s_idx) * p.Hq;
  if (have) {
    // this CTA's 256 output dims of head h, scaled by 1 / l, into shared
    // memory as eight boxes of 32 dims x 128 rows under the 128-byte swizzle
    // (the ring is idle once every PV has landed; the swizzle spreads a
    // warp's 32 rows over the banks) ...
    uint8_t* ostage = stages;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t v[32];
      tmem_ld32(lane_addr + kColO + 128 * w + c, v);
      tmem_wait_ld();
      uint8_t* row = ostage + (4 * w + c / 32) * kOBoxBytes + h * 128;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4*>(row + ((k ^ (h & 7)) << 4)) =
            make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                        __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
    }
    fence_proxy_async_smem();
    named_bar_sync(kBarEpi, 256);
    // ... and out to HBM by TMA: one thread stores the boxes (Hq rows each:
    // with fewer than 128 query heads the MMA rows past Hq hold the next query
    // rows of the tensor, computed and never written) and waits only until
    // they have been read out of shared memory
    if (w == 0 && lg == 0 && lane == 0) {
#pragma unroll 1
      for (int k = 0; k < 8; ++k)
        tma_store_2d(&tm_out, smem_u32(ostage + k * kOBoxBytes), 256 * (int)cta + 32 * k, (int32_t)row0);
      bulk_commit();
      bulk_wait_read0();
    }
  } else {
    // no product (an empty range, a skipped or an aborted unit): zeros, by
    // plain stores (copies of an aborted unit may still be landing in the ring)
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int hr = 16 * (4 * w + lg); hr < min(16 * (4 * w + lg) + 16, p.Hq); ++hr) {
      float4* g = reinterpret_cast<float4*>(p.dst_o + (row0 + hr) * kDv + 256 * cta);
      g[lane] = z;
      g[32 + lane] = z;
    }
  }
  if (cta == 0 && w == 0 && h < p.Hq)
    p.dst_lse[row0 + h] = (have && l_tot > 0.f) ? (r_fin + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
}

// ---------------------------------------------------------------------------
// score senders (warps 12..15): the peer's 32 tokens of every tile
// ---------------------------------------------------------------------------
__device__ __forceinline__ void score_sender(const MlaParams& p, Smem& sm, const Unit& u, const uint8_t* scbuf,
                                             uint32_t tmem, uint32_t cta, int warp, int lane) {
  const uint32_t peer = cta ^ 1u;
  const int lg = warp & 3;                          // this warp's heads [32 lg, +32)
  const int h = lg * 32 + lane;
  const uint32_t lane_addr = taddr(tmem, (uint32_t)(lg * 32), 0);
  const uint32_t peer_x = mapa(smem_u32(scbuf) + (uint32_t)h * 16u, peer);
  const uint32_t peer_xs = mapa(smem_u32(scbuf) + kMsgCodes + (uint32_t)h * 4u, peer);
  const uint32_t peer_recv = mapa(smem_u32(&sm.sc_recv[0][lg]), peer);   // + 32 * parity
  volatile int* abort_flag = &sm.abort;
  const float sl2 = p.scale_log2;
  int nflag[2] = {0, 0};                            // flagged tiles of each warpgroup's parity
  bool bad = false;
  for (int t = 0; t < u.T; ++t) {
    const int xb = t & 1;
    if (!__all_sync(0xffffffffu, *abort_flag == 0 &&
                                     mbar_wait(smem_u32(&sm.s_full[xb]), (uint32_t)(t >> 1) & 1u, p.wait_ns))) {
      bad = true;
      break;
    }
    uint32_t v[32];
    tc_fence_after();
    tmem_ld32(lane_addr + kColS + 64u * (uint32_t)xb + (uint32_t)kHalf * peer, v);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(smem_u32(&sm.s_free[xb]));
    // columns past the end of a ragged tile hold scores of stale cache rows:
    // zero them so they cannot set the scale (the peer masks them anyway)
    const int vp = valid_of_half(u, t, (int)peer);
    if (vp < kHalf) {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k >= vp) v[k] = 0u;
    }
    float a8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a8[k] = fmaxf(fabsf(__uint_as_float(v[k])), fabsf(__uint_as_float(v[k + 8])));
#pragma unroll
    for (int k = 16; k < 32; k += 8)
#pragma unroll
      for (int j = 0; j < 8; ++j) a8[j] = fmaxf(a8[j], fabsf(__uint_as_float(v[k + j])));
    const float amax =
        fmaxf(fmaxf(fmaxf(a8[0], a8[1]), fmaxf(a8[2], a8[3])), fmaxf(fmaxf(a8[4], a8[5]), fmaxf(a8[6], a8[7])));
    // large partials in this warp's heads: the residual follows (same for the warp)
    const bool flag = __any_sync(0xffffffffu, amax * sl2 > kResidualLog2);
    float enc, dec;
    bfp_scales(amax, enc, dec);
    // the peer has read tile t-1 out of its one slot
    if (t >= 1 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.sc_free[(t - 1) & 1][lg]), (uint32_t)((t - 1) >> 1) & 1u, p.wait_ns))) {
      bad = true;
      break;
    }
    const uint32_t bar = peer_recv + 32u * (uint32_t)xb;
    // chunk k carries tokens [8k, 8k + 8): two per word
#pragma unroll
    for (int k = 0; k < 4; ++k)
      st_async_v4(peer_x + k * (kHeads * 16),
                  __uint_as_float(bfp_pack2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1]), enc)),
                  __uint_as_float(bfp_pack2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3]), enc)),
                  __uint_as_float(bfp_pack2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5]), enc)),
                  __uint_as_float(bfp_pack2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7]), enc)),
                  bar);
    st_async_b32(peer_xs, __float_as_uint(flag ? -dec : dec), bar);
    if (flag) {
      // once the peer's warp has read the codes: the residual of every code,
      // v - round(v * enc) * dec (exact), coded with 2^15 times the scale
      // (|residual| * enc * 2^15 <= 2^14), into the same slot
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.sc_mfree[xb][lg]), (uint32_t)nflag[xb] & 1u, p.wait_ns))) {
        bad = true;
        break;
      }
      ++nflag[xb];
      const float enc_r = enc * 32768.0f;
      const uint32_t barr = mapa(smem_u32(&sm.sc_res[xb][lg]), peer);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t wd[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a = __uint_as_float(v[8 * k + 2 * j]), b = __uint_as_float(v[8 * k + 2 * j + 1]);
          const float2 q = bfp_round2(a, b, enc, dec);
          wd[j] = bfp_pack2(a - q.x, b - q.y, enc_r);
        }
        st_async_v4(peer_x + k * (kHeads * 16), __uint_as_float(wd[0]), __uint_as_float(wd[1]),
                    __uint_as_float(wd[2]), __uint_as_float(wd[3]), barr);
      }
    }
  }
  if (bad) {
    set_status(p.status, DCP_ERR_TIMEOUT);
    *abort_flag = 1;
  }
}

template <bool kLpt, bool kSmallBlocks>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_attn_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                const __grid_constant__ CUtensorMap tm_qlat, const __grid_constant__ CUtensorMap tm_qrope,
                const __grid_constant__ CUtensorMap tm_out,
                const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;                                        // kStages x 36 KB
  uint8_t* qlat0 = stages + kStages * kStageBytes;               // 16 KB, 1024-aligned
  uint8_t* qrope = qlat0 + kQLat0Bytes;                          // 8 KB, 1024-aligned
  uint8_t* scbuf = qrope + kQRopeBytes;                          // score message slot
  uint8_t* pmbuf = scbuf + kScMsgBytes;                          // probability message slot
  float* mxbuf = reinterpret_cast<float*>(pmbuf + kPmMsgBytes);  // 2 local-maximum slots
  Smem& sm = *reinterpret_cast<Smem*>(pmbuf + kPmMsgBytes + 2 * kMxMsgBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t cta = cluster_ctarank();          // 0 or 1
  // kLpt: units in longest-request-first order (length descending, index
  // ascending).  The block scheduler starts clusters in index order, so short
  // units fill the tail.  Batches up to kLptMaxBatch find rank k by counting
  // in the kernel; larger ones read it from the pre-pass's order.  Both CTAs
  // of the pair take the same request.
  const long long unit = blockIdx.x >> 1;
  int b_lpt = 0;
  if (kLpt) {
    const long long per_req = (long long)p.N * p.Lq * p.n_split;
    const int k_req = (int)(unit / per_req);
    if (p.order != nullptr && tid == 0) sm.req = p.order[k_req];
    for (int j = tid; p.order == nullptr && j < p.B; j += kThreads) {
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
  Unit u;
  {
    // 32-bit index arithmetic (the launcher keeps units below 2^31)
    const unsigned un = (unsigned)unit, per_q = (unsigned)(p.n_split * p.Lq);
    const unsigned rest = kLpt ? un % ((unsigned)p.N * per_q) : un;
    u.s_idx = (int)(rest % (unsigned)p.n_split);
    u.i_q = (int)((rest / (unsigned)p.n_split) % (unsigned)p.Lq);
    u.b = kLpt ? b_lpt : (int)((un / per_q) % (unsigned)p.B);
    u.r = kLpt ? (int)(rest / per_q) : (int)(un / (per_q * (unsigned)p.B));
  }
  // barriers and tensor memory first: they depend on no loaded data
  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) {
      mbar_init(smem_u32(&sm.kv_full[k]), 1);
      mbar_init(smem_u32(&sm.kv_empty[k]), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&sm.s_free[k]), 256);     // senders and the tile's softmax warpgroup
      mbar_init(smem_u32(&sm.s_full[k]), 1);

      for (int q = 0; q < 4; ++q) {
        mbar_init(smem_u32(&sm.sc_recv[k][q]), 1);
        mbar_init(smem_u32(&sm.sc_free[k][q]), 1);
        mbar_init(smem_u32(&sm.pm_recv[k][q]), 1);
        mbar_init(smem_u32(&sm.pm_free[k][q]), 1);
        mbar_init(smem_u32(&sm.r_pub[k][q]), 1);
        mbar_init(smem_u32(&sm.sc_res[k][q]), 1);
        mbar_init(smem_u32(&sm.sc_mfree[k][q]), 1);
        mbar_init(smem_u32(&sm.mx_recv[k][q]), 1);
      }

      mbar_init(smem_u32(&sm.p_full[k]), 128);
      mbar_init(smem_u32(&sm.pv_done[k]), 1);

    }
    mbar_init(smem_u32(&sm.fin), 256);
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.drain), 1);
    mbar_init(smem_u32(&sm.drain_qk), 1);
    sm.abort = 0;
    sm.qk_issued = -1;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), 512);

  // key range of this unit (shard-local indices [kb, ke))
  const int S = p.seq_lens[u.b];
  const bool bad_len = S < p.Lq;
  int L = bad_len ? 0 : local_len(S, u.r, p.I, p.N);
  const bool short_table = (long long)L > (long long)p.max_lb * p.bs;
  if (short_table) L = p.max_lb * p.bs;
  const int vis = bad_len ? 0 : min(L, local_count_upto((long long)S - p.Lq + u.i_q, u.r, p.I, p.N));
  u.kb = min(vis, u.s_idx * p.split_tokens);
  u.ke = min(vis, u.kb + p.split_tokens);
  u.T = (u.ke - u.kb + kNt - 1) / kNt;
  if (tid == 0 && cta == 0 && (bad_len || short_table)) set_status(p.status, DCP_ERR_BOUNDS);
  {
    // a block id past the pool among the query's visible keys skips the unit
    // (every KV split of it: zero partial, -inf LSE) and reports
    // DCP_ERR_BOUNDS; both CTAs of the pair read the same entries
    const int32_t* bt = p.block_tables + ((long long)u.r * p.B + u.b) * p.max_lb;
    bool bad_blk = false;
    for (int jb = tid; jb < (vis + p.bs - 1) / p.bs; jb += (int)kThreads)   // every split of the query
      bad_blk |= (unsigned)bt[jb] >= (unsigned)p.num_blocks;
    if (__syncthreads_or(bad_blk)) {
      u.T = 0;
      if (tid == 0 && cta == 0) set_status(p.status, DCP_ERR_BOUNDS);
    }
  }
  const int T = u.T;
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;     // the barrier above made the allocation visible

  // TMA producer state (warp 0, lane 0): the first stages are issued before
  // the query is staged, so their HBM latency overlaps the set-up
  volatile int* abort_flag = &sm.abort;
  const int32_t* bt_row = p.block_tables + ((long long)u.r * p.B + u.b) * p.max_lb;
  int issued[kStages];
#pragma unroll
  for (int k = 0; k < kStages; ++k) issued[k] = 0;
  auto issue_tile = [&](int t) {
    // test hook: CTA 0 never loads this tile, so the bounded waits on it run
    // out and the unit unwinds
    if (t == p.skip_tile && cta == 0) return;
    const int st = t % kStages;
    const uint32_t full = smem_u32(&sm.kv_full[st]);
    uint8_t* dst = stages + st * kStageBytes;
    mbar_arrive_expect_tx(full, kStageBytes);
    if (!kSmallBlocks) {
      // blocks of 64 tokens or a multiple: the tile is one box inside one block
      const int j = u.kb + t * kNt;
      const int row = bt_row[j / p.bs] * p.bs + (j % p.bs);   // ids checked against the pool above
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_load_2d(smem_u32(dst + c * kChunkBytes), &tm_lat, 256 * (int)cta + 64 * c, row, full);
      tma_load_2d(smem_u32(dst + 4 * kChunkBytes), &tm_rope, kLatent + 32 * (int)cta, row, full);
    } else {
      // blocks of 8, 16 or 32 tokens: one box per block; boxes past the key
      // range read pool row 0 (masked, values zeroed) so that no stale table
      // entry is followed
      for (int k = 0; k < kNt / p.bs; ++k) {
        const int j = u.kb + t * kNt + k * p.bs;
        const int row = j < u.ke ? bt_row[j / p.bs] * p.bs : 0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tma_load_2d(smem_u32(dst + c * kChunkBytes + k * p.bs * 128), &tm_lat, 256 * (int)cta + 64 * c, row, full);
        tma_load_2d(smem_u32(dst + 4 * kChunkBytes + k * p.bs * 64), &tm_rope, kLatent + 32 * (int)cta, row, full);
      }
    }
    ++issued[st];
  };
  // the query slice by TMA: latent dims 0-63 and the rope dims straight into
  // their shared-memory operands, latent dims 64-255 into ring stages 3-4
  // (idle until the first tiles have been issued) for the copy into TMEM
  uint8_t* qstage = stages + (kStages - 2) * kStageBytes;
  const int t_early = min(T, kStages - 2);
  if (warp == 0 && lane == 0 && T > 0) {
    prefetch_tmap(&tm_lat);
    prefetch_tmap(&tm_rope);
    const int32_t qr = (int32_t)(((long long)u.b * p.Lq + u.i_q) * p.Hq);
    const uint32_t qf = smem_u32(&sm.q_full);
    mbar_arrive_expect_tx(qf, kQLat0Bytes * 4 + kQRopeBytes);
    tma_load_2d(smem_u32(qlat0), &tm_qlat, 256 * (int)cta, qr, qf);
#pragma unroll
    for (int c = 1; c < 4; ++c) tma_load_2d(smem_u32(qstage + (c - 1) * kQLat0Bytes), &tm_qlat, 256 * (int)cta + 64 * c, qr, qf);
    tma_load_2d(smem_u32(qrope), &tm_qrope, kLatent + 32 * (int)cta, qr, qf);
    for (int t = 0; t < t_early; ++t) issue_tile(t);
  }
  // latent dims 64-255 of the slice -> TMEM (row = head = TMEM lane, bf16
  // pairs per column): the two softmax warps of a lane quadrant take 12 of the
  // 24 16-byte chunks of each row (128B-swizzled, so a warp's reads of one
  // chunk spread over the banks)
  bool q_ok = true;
  if (warp >= 4 && warp < 12 && T > 0) {
    q_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full), 0u, p.wait_ns));
    if (q_ok) {
      const int h = (warp & 3) * 32 + lane;
      const uint32_t lane_addr = taddr(tmem, (uint32_t)((warp & 3) * 32), 0);
      const int j0 = 12 * ((warp - 4) >> 2);
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        uint32_t v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int jg = j0 + 4 * i + k;                         // chunk of dims [64 + 8 jg, +8)
          const uint4 w4 = *reinterpret_cast<const uint4*>(qstage + (jg >> 3) * kQLat0Bytes + h * 128 +
                                                           (((jg & 7) ^ (h & 7)) << 4));
          v[4 * k + 0] = w4.x;
          v[4 * k + 1] = w4.y;
          v[4 * k + 2] = w4.z;
          v[4 * k + 3] = w4.w;
        }
        tmem_st16(lane_addr + kColQ + 4 * (j0 + 4 * i), v);
      }
      tmem_wait_st();
      fence_proxy_async_smem();     // stages 3-4 are reloaded by TMA after the barrier below
    }
  }
  if (!q_ok) {
    set_status(p.status, DCP_ERR_TIMEOUT);
    *abort_flag = 1;
  }
  tc_fence_before();
  cluster_sync();            // barriers of both CTAs initialised, query staged
  tc_fence_after();

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
        for (int t = t_early; t < T; ++t) {
          const int st = t % kStages;
          const uint32_t ph = (uint32_t)(t / kStages) & 1u;
          if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_empty[st]), ph ^ 1u, p.wait_ns)) {
            fail();
            break;
          }
          issue_tile(t);
        }
        if (*abort_flag) {
          // let every copy this thread issued land before the CTA exits
          for (int k = 0; k < kStages; ++k)
            if (issued[k] > 0) mbar_wait(smem_u32(&sm.kv_full[k]), (uint32_t)(issued[k] - 1) & 1u, p.wait_ns);
        }
      }
    } else if (warp == 1) {
      // ---------------- PV issuer (and TMEM owner) ----------------
      if (lane == 0 && T > 0) {
        const uint32_t id_pv = idesc_bf16(128, 256, true);
        bool ok = true;
        for (int t = 0; t < T; ++t) {
          if (*abort_flag || !mbar_wait(smem_u32(&sm.p_full[t & 1]), (uint32_t)(t >> 1) & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          // the score MMAs of tile t+2 go first (bounded spin on the QK issuer's count)
          const int need = min(t + kPvGate, T - 1);
          const uint64_t g0 = globaltimer_ns();
          while (*(volatile int*)&sm.qk_issued < need) {
            if (*abort_flag || globaltimer_ns() - g0 > p.wait_ns) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          tc_fence_after();
          const uint8_t* st = stages + (t % kStages) * kStageBytes;
#pragma unroll
          for (int k = 0; k < kNt / 16; ++k) {
            const uint64_t bdesc = smem_desc(smem_u32(st + k * 2048), kChunkBytes, 1024, kSw128);
            mma_ts(tmem + kColO, tmem + kColP + 8 * k, bdesc, id_pv, (t > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm.pv_done[t & 1]));
          // the score MMAs of tile t completed before its softmax produced P(t)
          mma_commit(smem_u32(&sm.kv_empty[t % kStages]));
        }
        if (!ok) fail();
        mma_commit(smem_u32(&sm.drain));
        if (!mbar_wait(smem_u32(&sm.drain), 0, p.wait_ns)) fail();
      }
    } else if (warp == 2) {
      // ---------------- score (QK^T) issuer ----------------
      if (lane == 0 && T > 0) {
        const uint32_t id_qk = idesc_bf16(128, kNt, false);
        // the query's shared-memory parts came by TMA (already waited for by
        // the softmax warps before the cluster barrier)
        bool ok = mbar_wait(smem_u32(&sm.q_full), 0u, p.wait_ns);
        for (int t = 0; t < T && ok; ++t) {
          const int st = t % kStages;
          if (*abort_flag || !mbar_wait(smem_u32(&sm.kv_full[st]), (uint32_t)(t / kStages) & 1u, p.wait_ns) ||
              (t >= 2 && !mbar_wait(smem_u32(&sm.s_free[t & 1]), (uint32_t)((t >> 1) - 1) & 1u, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* sb = stages + st * kStageBytes;
          const uint32_t dS = tmem + kColS + 64u * (uint32_t)(t & 1);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(dS, smem_desc(smem_u32(qlat0 + k * 32), 16, 1024, kSw128),
                   smem_desc(smem_u32(sb + k * 32), 16, 1024, kSw128), id_qk, k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 4; k < 16; ++k) {
            const uint64_t bdesc = smem_desc(smem_u32(sb + (k >> 2) * kChunkBytes + (k & 3) * 32), 16, 1024, kSw128);
            mma_ts(dS, tmem + kColQ + 8 * (k - 4), bdesc, id_qk, 1u);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_ss(dS, smem_desc(smem_u32(qrope + k * 32), 16, 512, kSw64),
                   smem_desc(smem_u32(sb + 4 * kChunkBytes + k * 32), 16, 512, kSw64), id_qk, 1u);
          mma_commit(smem_u32(&sm.s_full[t & 1]));
          *(volatile int*)&sm.qk_issued = t;
        }
        if (!ok) fail();
        mma_commit(smem_u32(&sm.drain_qk));
        if (!mbar_wait(smem_u32(&sm.drain_qk), 0, p.wait_ns)) fail();
      }
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kSoftRegs));
    softmax_wg(p, tm_out, sm, u, stages, scbuf, pmbuf, mxbuf, tmem, cta, warp, lane);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kSendRegs));
    score_sender(p, sm, u, scbuf, tmem, cta, warp, lane);
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

// Longest-first order of the requests: order[rank] = j, rank = number of
// requests longer than j, or as long with a smaller index (each rank once).
__global__ void __launch_bounds__(256) lpt_order_kernel(const int32_t* seq_lens, int B, int32_t* order) {
  __shared__ int tile[256];
  const int j = blockIdx.x * 256 + threadIdx.x;
  const int sj = j < B ? seq_lens[j] : 0;
  int rank = 0;
  for (int base = 0; base < B; base += 256) {
    __syncthreads();
    if (base + threadIdx.x < B) tile[threadIdx.x] = seq_lens[base + threadIdx.x];
    __syncthreads();
    const int n = min(256, B - base);
    for (int k = 0; k < n; ++k) {
      const int si = tile[k];
      rank += (si > sj) || (si == sj && base + k < j);
    }
  }
  if (j < B) order[rank] = j;
}

}  // namespace

bool mla_tc_supported(const AttnArgs& a) {
  // 16 to 128 query heads; the query box is 128 rows, so the query tensor
  // must hold at least that many
  return a.kind == DCP_ATTN_MLA && a.Hq >= 16 && a.Hq <= kHeads && (long long)a.B * a.Lq * a.Hq >= kHeads &&
         a.Hkv == 1 && a.Dqk == kDqk && a.Dv == kDv &&
         (a.bs == 8 || a.bs == 16 || a.bs == 32 || a.bs % kNt == 0) &&
         (long long)a.num_blocks * a.bs < (1LL << 31);
}

SplitPlan plan_attn_mla_tc(const AttnArgs& a, int sm_count) {
  SplitPlan pl = plan_splits(a, sm_count, kNt, 2 * a.Lq);
  if (a.B > kLptMaxBatch && a.B <= kLptOrderMaxBatch) {
    pl.lpt_order = true;
    pl.order_offset = (pl.ws_bytes + 255) & ~size_t(255);
    pl.ws_bytes = pl.order_offset + (((size_t)a.B * 4 + 255) & ~size_t(255));
  }
  return pl;
}

cudaError_t launch_attn_mla_tc(const AttnArgs& a, const SplitPlan& plan) {
  CUtensorMap tm_lat, tm_rope;
  const uint64_t dims[2] = {(uint64_t)kDqk, (uint64_t)a.num_blocks * a.bs};
  const uint64_t strides[1] = {(uint64_t)kDqk * 2};
  const uint32_t box_rows = (uint32_t)(a.bs < kNt ? a.bs : kNt);
  const uint32_t box_lat[2] = {64, box_rows};
  const uint32_t box_rope[2] = {32, box_rows};
  if (!make_tensor_map_bf16(&tm_lat, a.kv, 2, dims, strides, box_lat, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&tm_rope, a.kv, 2, dims, strides, box_rope, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  // the query as [B * Lq * Hq][576]: one box of 128 head rows per chunk
  CUtensorMap tm_qlat, tm_qrope;
  const uint64_t qdims[2] = {(uint64_t)kDqk, (uint64_t)a.B * a.Lq * a.Hq};
  const uint32_t qbox_lat[2] = {64, kHeads};
  const uint32_t qbox_rope[2] = {32, kHeads};
  if (!make_tensor_map_bf16(&tm_qlat, a.q, 2, qdims, strides, qbox_lat, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&tm_qrope, a.q, 2, qdims, strides, qbox_rope, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  MlaParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.status = a.status;
  p.B = a.B;
  p.Lq = a.Lq;
  p.Hq = a.Hq;
  p.N = a.N;
  p.I = a.I;
  p.max_lb = a.max_lb;
  p.bs = a.bs;
  p.num_blocks = a.num_blocks;
  p.n_split = plan.n_split;
  p.split_tokens = plan.split_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = test_hooks().wait_ns;
  p.skip_tile = test_hooks().skip_tile;
  if (plan.n_split > 1) {
    const size_t rows = (size_t)a.N * a.B * a.Lq * a.Hq;
    const size_t o_bytes = rows * plan.n_split * a.Dv * sizeof(float);
    p.dst_o = static_cast<float*>(a.workspace);
    p.dst_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ((o_bytes + 255) & ~size_t(255)));
  } else {
    p.dst_o = a.partial_out;
    p.dst_lse = a.lse;
  }
  // the fp32 output rows [units x Hq][512], stored in 32-dim x Hq-row boxes
  // (row coordinates are 32-bit)
  const long long units = (long long)a.N * a.B * a.Lq * plan.n_split;
  if (units == 0) return cudaSuccess;
  if (units * a.Hq >= (1LL << 31)) return cudaErrorInvalidValue;
  CUtensorMap tm_out;
  const uint64_t odims[2] = {(uint64_t)kDv, (uint64_t)a.N * a.B * a.Lq * plan.n_split * a.Hq};
  const uint64_t ostrides[1] = {(uint64_t)kDv * 4};
  const uint32_t obox[2] = {32, (uint32_t)a.Hq};
  if (!make_tensor_map(&tm_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dst_o, 2, odims, ostrides, obox,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const bool lpt = a.B <= kLptOrderMaxBatch, small = a.bs < kNt;
  p.order = nullptr;
  if (plan.lpt_order) {
    if (a.workspace == nullptr || a.workspace_bytes < plan.ws_bytes) return cudaErrorInvalidValue;
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(a.workspace) + plan.order_offset);
    lpt_order_kernel<<<(unsigned)((a.B + 255) / 256), 256, 0, a.stream>>>(a.seq_lens, a.B, order);
    cudaError_t eo = cudaGetLastError();
    if (eo != cudaSuccess) return eo;
    p.order = order;
  }
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const MlaParams) =
      lpt ? (small ? mla_attn_kernel<true, true> : mla_attn_kernel<true, false>)
          : (small ? mla_attn_kernel<false, true> : mla_attn_kernel<false, false>);
  // the register split assumes the compiled launch count; refuse to launch
  // otherwise (setmaxnreg.inc would wait for registers that do not exist)
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * (int)kThreads < kSplitRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  if (units > (1LL << 30)) return cudaErrorInvalidValue;   // two CTAs a unit; 32-bit unit indices
  kern<<<(unsigned)(2 * units), kThreads, kSmemBytes, a.stream>>>(tm_lat, tm_rope, tm_qlat, tm_qrope, tm_out, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || plan.n_split <= 1) return e;
  return launch_split_combine(a, plan);
}

}  // namespace dcp
