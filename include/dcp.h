/*
 * dcp.h - C ABI of libdcp: Decode Context Parallelism (DCP) decode attention
 * for one GB300 (sm_103a).
 *
 * What the library computes (vLLM Decode Context Parallelism blog, agentlenshq,
 * zh-TW, sections "解碼上下文並行 (DCP) 原理解析" and "DCP 執行流程"): the paged KV
 * cache of each request is split along the sequence into dcp_size shards; the
 * full query attends to each shard's keys alone, giving a partial output and
 * its log-sum-exp (LSE); the partials are merged by LSE reweighting (the
 * online-softmax rule) and each shard index r receives the slice of heads it
 * owns.  On one GPU the shards are partitions of one device pool and the
 * "exchange" is a device buffer read by dcp_merge.
 *
 * Token -> shard rule (the interleave flag cp_kv_cache_interleave_size of the
 * vLLM Ascend "Context Parallel Guide", section "Decode Context Parallel"):
 *     shard(t) = (t / interleave) % dcp_size
 *     local(t) = (t / (interleave * dcp_size)) * interleave + t % interleave
 * Tokens of one shard are stored densely in increasing global order.
 *
 * Conventions for every call
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *    The library never allocates, frees or keeps them.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Work is enqueued on it; no call synchronises the host except
 *    dcp_get_last_device_status.
 *  - Arguments are checked on the host first; a bad argument returns an error
 *    code and launches nothing.  Errors found on the device (a sequence shorter
 *    than its query, a block id out of range, a bounded wait that expired) set
 *    the status word of the stream the call was enqueued on, read by
 *    dcp_get_last_device_status(stream); the kernels then skip the offending
 *    work unit (its partial output 0, its LSE -inf).  Each stream has its own
 *    word, so concurrent streams do not see or clear each other's errors, up to
 *    DCP_STATUS_STREAMS - 1 streams per device; further streams share one word.
 *  - The first call of any entry point on a device looks up the status words'
 *    device address; make it before any stream capture.  A captured call keeps
 *    the status word of the stream it was captured on: errors of its replays
 *    are read through that stream's handle.
 *  - Every call is wrapped in an NVTX range named after it.
 *  - No C++ exception crosses this interface.
 *  - Integer tensors are int32, row-major (C order), without padding.
 */
#ifndef DCP_H_
#define DCP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DCP_API __attribute__((visibility("default")))
#else
#define DCP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DCP_OK = 0,
  DCP_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape          */
  DCP_ERR_UNSUPPORTED = 2,  /* valid request the library has no kernel for   */
  DCP_ERR_CUDA = 3,         /* a CUDA runtime call failed                      */
  DCP_ERR_TIMEOUT = 4,      /* a device-side bounded wait expired              */
  DCP_ERR_BOUNDS = 5        /* device-side range check failed (see above)     */
} dcp_status_t;

typedef enum { DCP_ATTN_GQA = 0, DCP_ATTN_MLA = 1 } dcp_attn_kind_t;

/* Status words per device: one per stream, in order of first use. */
#define DCP_STATUS_STREAMS 64

/* The kernel dcp_decode_attn runs for a shape (dcp_decode_attn_kernel_kind). */
typedef enum {
  DCP_KERNEL_NONE = 0,     /* the shape is rejected                                   */
  DCP_KERNEL_MLA_TC = 1,   /* tensor-core MLA kernel: Hq 16-128 (B * Lq * Hq >= 128),
                              Dqk 576, Dv 512, block size 8, 16, 32 or a multiple of 64 */
  DCP_KERNEL_GQA_TC = 2,   /* tensor-core GQA kernel: head dim 64 or 128, block size a
                              multiple of 8 that divides or is a multiple of 128       */
  DCP_KERNEL_SIMT = 3      /* generic CUDA-core kernel for every other shape; an order of
                              magnitude slower than the tensor-core kernels on the
                              large shapes                                            */
} dcp_kernel_kind_t;

/* Shape of one decode-attention call.
 *  kind            DCP_ATTN_GQA or DCP_ATTN_MLA
 *  batch           B, number of requests
 *  q_len           Lq, query tokens per request (1 = plain decode; 4 = MTP
 *                  verify with 3 speculative tokens, causal within the Lq)
 *  num_q_heads     Hq
 *  num_kv_heads    Hkv (MLA: 1); query head h reads KV head h / (Hq / Hkv)
 *  head_dim_qk     Dqk (MLA: 576 = 512 latent + 64 rope)
 *  head_dim_v      Dv  (MLA: 512, the value is the first Dv entries of the row)
 *  block_size      tokens per cache block
 *  num_blocks      blocks in the cache pool (block ids are < num_blocks)
 *  max_local_blocks  third dimension of block_tables                       */
typedef struct {
  int32_t kind;
  int32_t batch;
  int32_t q_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim_qk;
  int32_t head_dim_v;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_local_blocks;
} dcp_attn_desc_t;

/* Step a1: the token -> shard map.
 * Source: DCP principle section of the vLLM DCP blog (each rank holds a range
 * of token positions; worked example 200K tokens on 4 ranks) and the interleave
 * flag of the vLLM Ascend Context Parallel Guide.
 *  seq_lens          [B]            context length of each request
 *  local_seq_lens    [dcp][B] out   tokens held by shard r
 *  local_num_blocks  [dcp][B] out   ceil(local_seq_lens / block_size)
 *  shard_of, local_pos  [B][max_seq] out, optional (both NULL or both set):
 *                    owning shard and shard-local index of token t, -1 for
 *                    t >= seq_lens[b]
 *  max_seq           row length of shard_of/local_pos (ignored when NULL)
 * Errors: INVALID_ARG for batch < 0, block_size/interleave/dcp_size < 1, NULL
 * required pointers, exactly one of shard_of/local_pos NULL, max_seq < 1 with
 * the maps requested.  A seq_len < 0 sets DCP_ERR_BOUNDS on the device.      */
DCP_API dcp_status_t dcp_build_slot_map(const int32_t* seq_lens, int32_t batch, int32_t block_size,
                                int32_t interleave, int32_t dcp_size,
                                int32_t* local_seq_lens, int32_t* local_num_blocks,
                                int32_t* shard_of, int32_t* local_pos, int32_t max_seq,
                                void* stream);

/* Bytes of device scratch dcp_decode_attn needs for this shape (0 is
 * possible): the partial outputs of KV splits when a shard's keys are split
 * across several work units (small batches, long contexts), and for MLA
 * batches of 129 to 16384 requests the longest-first request order (4 bytes a
 * request) that a pre-pass writes.  Depends on the shape only (not on the
 * contents of seq_lens).  Returns 0 and sets nothing for an invalid
 * descriptor. */
DCP_API size_t dcp_decode_attn_workspace_size(const dcp_attn_desc_t* d, int32_t dcp_size);

/* Steps a2-a5: per-shard partial attention with LSE.
 * Source: "DCP 執行流程" of the vLLM DCP blog: the full query (AllGather Q)
 * attends to the shard's local KV slice only (Compute).
 * For shard r, request b, query i (position p = seq_lens[b] - Lq + i), head h:
 *   s_t = scale * q[b][i][h] . k_t  over the keys t of shard r with t <= p
 *   lse[r][b][i][h]         = log sum_t exp(s_t)               (natural log)
 *   partial_out[r][b][i][h] = sum_t exp(s_t - lse) * v_t
 * A shard with no visible key gives partial_out = 0 and lse = -inf.
 *  q             bf16 [B][Lq][Hq][Dqk]
 *  kv_cache      bf16, GQA [2][num_blocks][block_size][Hkv][Dqk] (K pool, then
 *                V pool; requires Dv == Dqk); MLA [num_blocks][block_size][Dqk]
 *  block_tables  [dcp][B][max_local_blocks]: shard r's j-th local token of
 *                request b is at block block_tables[r][b][j / block_size],
 *                slot j % block_size
 *  seq_lens      [B], each >= Lq (checked on the device)
 *  causal_q_len  must equal d->q_len
 *  partial_out   fp32 [dcp][B][Lq][Hq][Dv] out;  lse fp32 [dcp][B][Lq][Hq] out
 *  workspace     >= dcp_decode_attn_workspace_size(d, dcp_size) bytes, 256-byte
 *                aligned (may be NULL when that size is 0); its contents on entry
 *                do not matter
 * Alignment: q, kv_cache, partial_out 16 bytes.
 * Errors: INVALID_ARG (NULL pointers, sizes < 1, Hq % Hkv != 0, MLA with
 * Hkv != 1 or Dv > Dqk, GQA with Dv != Dqk, causal_q_len != q_len, small
 * workspace, misalignment); UNSUPPORTED (head dims without a kernel); CUDA.
 * Arithmetic and accuracy: products of the bf16 inputs accumulate in fp32;
 * the softmax runs in fp32 in the log2 domain.  Each probability is rounded to
 * bf16 once before the value product (the GQA tensor-core kernel carries it as
 * two bf16 terms, hi + lo, so about 16 bits reach the product).  Against the
 * fp64 definition above, partial_out is within 2e-3 absolute + 1e-2 relative
 * and lse within 1e-3 absolute; the tests hold that bar for softmaxes
 * dominated by one or a few keys and for scaled scores of 30-60 (sinks).
 * The MLA tensor-core kernel forms every score from two halves computed on
 * the two CTAs of a cluster pair; a half crosses the pair as a 16-bit code
 * with one power-of-two scale per head and 64-key tile (absolute error at most
 * 2^-14 * the head's largest |half| in that tile).  When some head's largest
 * |half| * scale * log2(e) exceeds 8, the 16-bit residual of every code is
 * sent as well, and the error drops to at most 2^-29 * that largest |half|,
 * below fp32 rounding of the score itself.  Magnitude limit: halves up to
 * 2^74 in magnitude (|q . k| about 1.9e22) are encoded; past that the
 * received score is undefined.  A half sums 288 products, so queries and
 * keys with every |q_d|, |k_d| <= 2^31 stay inside the limit.  */
DCP_API dcp_status_t dcp_decode_attn(const dcp_attn_desc_t* d, const void* q, const void* kv_cache,
                             const int32_t* block_tables, const int32_t* seq_lens,
                             int32_t dcp_size, int32_t interleave, float scale,
                             int32_t causal_q_len, float* partial_out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Step a6: LSE merge and head-slice return.
 * Source: "DCP 執行流程" of the vLLM DCP blog, AllGather + ReduceScatter: the
 * partials and LSEs are shared, reweighted with the online-softmax rule and
 * summed, and each rank gets only its head slice.
 *   LSE = m + log sum_r exp(lse_r - m),  m = max_r lse_r
 *   o   = sum_r exp(lse_r - LSE) * partial_out_r
 * out[r][b][i][h'] = o[b][i][r * Hq/dcp + h'] (bf16, round to nearest even).
 * All shards -inf gives out = 0 and out_lse = -inf.
 *  partial_out fp32 [dcp][B][Lq][Hq][Dv], lse fp32 [dcp][B][Lq][Hq]
 *  out     bf16 [dcp][B][Lq][Hq/dcp][Dv] out
 *  out_lse fp32 [dcp][B][Lq][Hq/dcp] out, optional (NULL to skip)
 * Alignment: partial_out 16 bytes, out 8 bytes; Dv % 4 == 0.
 * Errors: INVALID_ARG (NULL, sizes < 1, Hq % dcp != 0 - the one-GPU form of
 * the pages' TP/DCP divisibility constraints -, Dv % 4 != 0, alignment).     */
DCP_API dcp_status_t dcp_merge(const float* partial_out, const float* lse, int32_t dcp_size,
                       int32_t batch, int32_t q_len, int32_t num_q_heads, int32_t head_dim_v,
                       void* out, float* out_lse, void* stream);

/* dcp_decode_attn for callers that cannot allocate device memory.
 * No counterpart in the pages: this is a library convenience, not a step of
 * the method.  dcp_decode_attn takes caller-allocated scratch when it splits a
 * shard's keys over several CTAs (small batches with long contexts).  Callers
 * that may not call cudaMalloc at that point - code inside another runtime's
 * memory pool, plugins that are handed only their input and output buffers, a
 * serving loop that forbids allocation on the decode path - use this call
 * instead: the scratch is a fixed array of DCP_NOALLOC_SCRATCH_BYTES compiled
 * into the library, held on every GPU that loads the library until exit.
 * Arguments, results and errors are those of dcp_decode_attn, without the
 * workspace.  Extra rules:
 *  - a shape whose dcp_decode_attn_workspace_size exceeds
 *    DCP_NOALLOC_SCRATCH_BYTES is rejected with DCP_ERR_INVALID_ARG before any
 *    launch (check that size first to tell this case apart);
 *  - every call shares the one array, which keeps the last call's contents
 *    (nothing in it needs to start at zero); calls whose kernels overlap on
 *    the GPU - on different streams or from different host threads - race on
 *    it and give wrong results; calls ordered on one stream are safe;
 *  - the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 * It calls no allocator (no cudaMalloc/cudaFree) itself.                     */
#define DCP_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
DCP_API dcp_status_t dcp_decode_attn_noalloc(const dcp_attn_desc_t* d, const void* q,
                                             const void* kv_cache, const int32_t* block_tables,
                                             const int32_t* seq_lens, int32_t dcp_size,
                                             int32_t interleave, float scale,
                                             int32_t causal_q_len, float* partial_out, float* lse,
                                             void* stream);

/* Storing the newest tokens of every request in the sharded cache (the step
 * before a2-a5 of a decode step).
 * Source: "Context Parallel Guide", section "Overview" (DCP shards the KV cache
 * storage among the ranks of the DCP group, so a token's KV is stored once, by
 * the rank owning its position) and section "Decode Context Parallel" (the
 * interleave flag); vLLM DCP blog, "解碼上下文並行 (DCP) 原理解析" (each rank
 * holds a range of token positions).
 * Token i of request b (0 <= i < n_new) has position t = seq_lens[b] - n_new + i
 * (seq_lens already count the new tokens); its row goes to shard r = shard(t),
 * local index j = local(t), i.e. block block_tables[r][b][j / block_size],
 * slot j % block_size - the cells dcp_decode_attn reads it from.
 *  d             shape: kind, batch, num_kv_heads, head_dim_qk, block_size,
 *                num_blocks, max_local_blocks are used
 *  new_k         bf16, GQA [B][n_new][Hkv][Dqk]; MLA [B][n_new][Dqk] (the row)
 *  new_v         bf16, GQA [B][n_new][Hkv][Dqk]; MLA must be NULL
 *  kv_cache      bf16, as in dcp_decode_attn; written in place (only the
 *                B * n_new target rows of each pool)
 *  block_tables  [dcp][B][max_local_blocks];  seq_lens [B]
 * Alignment: new_k, new_v, kv_cache 16 bytes; a token row (Hkv * Dqk bf16,
 * MLA Dqk) must be a multiple of 16 bytes.
 * Errors: INVALID_ARG (NULL pointers, sizes < 1, new_v NULL for GQA or set for
 * MLA, row size or alignment); on the device, a seq_len < n_new, a local index
 * past the block table or a block id >= num_blocks sets DCP_ERR_BOUNDS and
 * that token is skipped.                                                      */
DCP_API dcp_status_t dcp_kv_cache_write(const dcp_attn_desc_t* d, const void* new_k,
                                        const void* new_v, void* kv_cache,
                                        const int32_t* block_tables, const int32_t* seq_lens,
                                        int32_t dcp_size, int32_t interleave, int32_t n_new,
                                        void* stream);

/* Which kernel dcp_decode_attn would run for this shape (a dcp_kernel_kind_t;
 * DCP_KERNEL_NONE for an invalid descriptor).  Host only, no GPU work: lets a
 * caller see in advance that a shape falls back to the CUDA-core kernel. */
DCP_API int32_t dcp_decode_attn_kernel_kind(const dcp_attn_desc_t* d, int32_t dcp_size);

/* How many kernels one dcp_decode_attn call enqueues for this shape: the
 * attention kernel, plus the combine of KV splits when a shard is split, plus
 * the request-order pre-pass of the MLA tensor-core kernel for batches of
 * 129 to 16384 requests.  0 for an invalid descriptor.  Host only. */
DCP_API int32_t dcp_decode_attn_launches(const dcp_attn_desc_t* d, int32_t dcp_size);

/* Reads `stream`'s status word (the first device-side error of the calls
 * enqueued on that stream since the last read; DCP_OK if none) and clears it.
 * The read and the clear are enqueued on `stream` and the call then waits for
 * that stream only (no device-wide synchronisation). */
DCP_API dcp_status_t dcp_get_last_device_status(void* stream);

/* Static, human-readable name of a status code. */
DCP_API const char* dcp_status_string(dcp_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* DCP_H_ */
