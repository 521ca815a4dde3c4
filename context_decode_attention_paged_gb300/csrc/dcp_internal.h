// Internal interface between the C-ABI layer (dcp_api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dcp.h"

namespace dcp {

// Everything a decode-attention kernel needs, validated by the API layer.
struct AttnArgs {
  int kind;              // DCP_ATTN_GQA / DCP_ATTN_MLA
  int B, Lq, Hq, Hkv, Dqk, Dv, bs, num_blocks, max_lb;
  int N, I;              // dcp_size, interleave
  float scale;
  const void* q;         // bf16 [B][Lq][Hq][Dqk]
  const void* kv;        // bf16 cache (see dcp.h)
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* partial_out;    // fp32 [N][B][Lq][Hq][Dv]
  float* lse;            // fp32 [N][B][Lq][Hq]
  void* workspace;
  size_t workspace_bytes;
  int* status;           // device status word
  cudaStream_t stream;
};

// How a call is cut into work units along the local KV axis.
struct SplitPlan {
  int n_split;           // KV splits per (shard, request[, query]) unit
  int split_tokens;      // local tokens per split (multiple of the kernel tile)
  size_t ws_bytes;       // workspace bytes (split partials, request order)
  bool lpt_order;        // a pre-pass writes the longest-first request order
  size_t order_offset;   // where it goes in the workspace (int32 [B])
};

// Workspace layout when n_split > 1:
//   ws_o   fp32 [N][B][Lq][n_split][Hq][Dv]
//   ws_lse fp32 [N][B][Lq][n_split][Hq]       (after ws_o, 256-byte aligned)
// then, 256-byte aligned, the request order when lpt_order is set.
SplitPlan plan_splits(const AttnArgs& a, int sm_count, int tile_tokens, int units_per_split);

int device_sm_count();

// Test-only knobs of the attention kernels, read at each launch: the limit of
// every bounded wait (default 2 s) and a tile that the first CTA's TMA
// producer of every work unit never loads (-1: none), so that the kernels'
// own bounded waits run out and their abort paths run.  Set through
// dcp_testing_set_hooks, an exported symbol the public header does not
// declare; nothing in the library changes them.
struct TestHooks {
  unsigned long long wait_ns;
  int skip_tile;
};
TestHooks test_hooks();

// Launchers; each returns a cudaError_t from the launch.
cudaError_t launch_slot_map(const int32_t* seq_lens, int B, int bs, int I, int N,
                            int32_t* local_seq_lens, int32_t* local_num_blocks,
                            int32_t* shard_of, int32_t* local_pos, int max_seq, int* status,
                            cudaStream_t stream);

cudaError_t launch_merge(const float* partial_out, const float* lse, int N, int B, int Lq,
                         int Hq, int Dv, void* out, float* out_lse, cudaStream_t stream);

// Store the newest n_new tokens of every request in their shards' cache cells.
cudaError_t launch_kv_write(const void* new_k, const void* new_v, void* kv_cache, const int32_t* block_tables,
                            const int32_t* seq_lens, int B, int n_new, int N, int I, int bs, int max_lb,
                            int num_blocks, int row_bytes, int* status, cudaStream_t stream);

// Combine n_split workspace partials into partial_out / lse (row a5).
cudaError_t launch_split_combine(const AttnArgs& a, const SplitPlan& p);

// Generic SIMT kernel (any head dims); used for shapes the tensor-core kernels
// do not take.
cudaError_t launch_attn_simt(const AttnArgs& a, const SplitPlan& p);
SplitPlan plan_attn_simt(const AttnArgs& a, int sm_count);

// MLA on tcgen05 (Hq 128, Dqk 576, Dv 512, block 128): cluster-pair kernel.
bool mla_tc_supported(const AttnArgs& a);
SplitPlan plan_attn_mla_tc(const AttnArgs& a, int sm_count);
cudaError_t launch_attn_mla_tc(const AttnArgs& a, const SplitPlan& p);

// GQA on tcgen05 (head dim 64/128, any Lq * Hq/Hkv in row tiles of up to 64, block size a
// multiple of 8 that divides or is a multiple of 128).
bool gqa_tc_supported(const AttnArgs& a);
SplitPlan plan_attn_gqa_tc(const AttnArgs& a, int sm_count);
cudaError_t launch_attn_gqa_tc(const AttnArgs& a, const SplitPlan& p);

}  // namespace dcp
