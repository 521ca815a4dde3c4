"""CPU oracle for Decode Context Parallelism (DCP) decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` use it.  It shares no code, constants or helpers with the
CUDA library.

Everything here is plain numpy in float64.  bf16 inputs are widened exactly
(every bf16 value is an fp64 value), so the only rounding is fp64 rounding.

What the method computes, and where the pages say so
----------------------------------------------------
* "vLLM Decode Context Parallelism blog" (agentlenshq, zh-TW), section
  "解碼上下文並行 (DCP) 原理解析": the KV cache is split along the sequence
  (context) dimension, each rank holding a range of token positions of the same
  request; its worked example gives, for a 200K-token request on four ranks,
  rank 0 tokens 0-50K, rank 1 tokens 50K-100K and so on.
* Same page, section "DCP 執行流程": (1) the full query is made available on
  every rank (AllGather Q); (2) each rank computes attention of that query
  against its local KV slice only; (3) the partial outputs and their
  log-sum-exp values are shared, the partials are re-weighted and merged with
  the online-softmax rule, and each rank receives only its head slice
  (AllGather + ReduceScatter).
* "Context Parallel Guide" (vLLM Ascend docs), section "Decode Context
  Parallel": the interleave flag ``cp_kv_cache_interleave_size`` sets how many
  consecutive tokens go to one rank before moving to the next; the token-to-rank
  rule used here is shard(t) = (t // interleave) % dcp_size, which the worked
  example above is the interleave = 50K, dcp_size = 4 case of.

Readings where the pages are silent:
* tokens of one shard are stored densely in increasing global order;
* seq_len counts the query tokens (their KV is already cached); query i of a
  request of length S sits at position S - Lq + i and sees keys at positions
  <= that position;
* lse is the natural log of the sum of exp of the *scaled* scores;
* an empty shard (or one with no visible key) yields o = 0, lse = -inf, and
  weight 0 in the merge;
* rank r's head slice is heads [r*Hq/N, (r+1)*Hq/N);
* GQA: query head h reads KV head h // (Hq / Hkv);
* MLA: one latent KV row of Dqk = 576 values (512 latent + 64 rope) per token;
  the value is its first Dv = 512 values; the query is already absorbed.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")


# ---------------------------------------------------------------------------
# Step 1 - token -> shard map (DCP principle section; interleave flag)
# ---------------------------------------------------------------------------

def shard_token_lists(seq_len: int, interleave: int, dcp_size: int) -> list[np.ndarray]:
    """Global positions held by each shard, in increasing order.

    Enumeration of every position t < seq_len with shard(t) = (t // I) % N.
    Shard r's local index j is the position of t within its list.
    """
    t = np.arange(seq_len, dtype=np.int64)
    owner = (t // interleave) % dcp_size
    return [t[owner == r] for r in range(dcp_size)]


def ref_slot_map(seq_lens, interleave: int, dcp_size: int, block_size: int):
    """Slot map by enumeration.

    Returns a dict with
      shard_of   int32 [B][max_seq]  owning shard of each token (-1 past the end)
      local_pos  int32 [B][max_seq]  index of the token inside its shard
      local_seq_lens   int32 [N][B]  tokens held by shard r for sequence b
      local_num_blocks int32 [N][B]  ceil(local_seq_lens / block_size)
    """
    seq_lens = [int(s) for s in seq_lens]
    B = len(seq_lens)
    max_seq = max(seq_lens) if B else 0
    shard_of = np.full((B, max_seq), -1, dtype=np.int32)
    local_pos = np.full((B, max_seq), -1, dtype=np.int32)
    local_seq_lens = np.zeros((dcp_size, B), dtype=np.int32)
    for b, S in enumerate(seq_lens):
        for r, toks in enumerate(shard_token_lists(S, interleave, dcp_size)):
            shard_of[b, toks] = r
            local_pos[b, toks] = np.arange(len(toks), dtype=np.int32)
            local_seq_lens[r, b] = len(toks)
    local_num_blocks = (local_seq_lens + block_size - 1) // block_size
    return {
        "shard_of": shard_of,
        "local_pos": local_pos,
        "local_seq_lens": local_seq_lens,
        "local_num_blocks": local_num_blocks.astype(np.int32),
    }


# ---------------------------------------------------------------------------
# Attention over one set of keys (plain definition of softmax attention)
# ---------------------------------------------------------------------------

def _attend(qh: np.ndarray, keys: np.ndarray, vals: np.ndarray, scale: float):
    """softmax(scale * q . k_t)-weighted sum of v_t, and the log-sum-exp.

    qh [H][Dqk] (query heads that read the same KV head), keys [n][Dqk],
    vals [n][Dv].  Returns o [H][Dv], lse [H].  n == 0 gives (0, -inf).
    """
    H = qh.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((H, vals.shape[1])), np.full(H, NEG_INF)
    s = scale * (qh @ keys.T)                 # [H][n]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1)
    return (p @ vals) / l[:, None], m[:, 0] + np.log(l)


def _head_groups(num_q_heads: int, num_kv_heads: int):
    """(kv head g, query heads of g): query head h reads KV head h // (Hq/Hkv)."""
    g_size = num_q_heads // num_kv_heads
    return [(g, slice(g * g_size, (g + 1) * g_size)) for g in range(num_kv_heads)]


# ---------------------------------------------------------------------------
# Unsharded attention from the logical (unpaged) per-sequence K/V
# ---------------------------------------------------------------------------

def ref_attn_unsharded(q, keys, values, seq_lens, scale: float, q_len: int):
    """Unsharded decode attention.

    q      [B][Lq][Hq][Dqk]
    keys   list over b of [S_b][Hkv][Dqk]
    values list over b of [S_b][Hkv][Dv]
    Returns out [B][Lq][Hq][Dv], lse [B][Lq][Hq] (float64).
    Query i sees positions t <= S_b - Lq + i.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Lq, Hq, _ = q.shape
    assert Lq == q_len
    Hkv = keys[0].shape[1]
    Dv = values[0].shape[2]
    out = np.zeros((B, Lq, Hq, Dv))
    lse = np.full((B, Lq, Hq), NEG_INF)
    for b in range(B):
        S = int(seq_lens[b])
        Kb = np.asarray(keys[b], dtype=np.float64)
        Vb = np.asarray(values[b], dtype=np.float64)
        for i in range(Lq):
            last = S - Lq + i  # last visible position
            for g, hs in _head_groups(Hq, Hkv):
                out[b, i, hs], lse[b, i, hs] = _attend(
                    q[b, i, hs], Kb[: last + 1, g], Vb[: last + 1, g], scale)
    return out, lse


# ---------------------------------------------------------------------------
# Storing new tokens into the sharded cache (the step before the Compute step)
# ---------------------------------------------------------------------------

def ref_kv_cache_write(kind: str, kv_cache, new_k, new_v, block_tables, seq_lens,
                       dcp_size: int, interleave: int, block_size: int, n_new: int):
    """The cache after storing the newest n_new tokens of every request.

    "Context Parallel Guide", section "Overview": DCP shards the KV cache
    storage among the ranks of the DCP group, so each new token's KV row is
    stored once, in the shard that owns its position (section "Decode Context
    Parallel": the interleave flag; blog, section "解碼上下文並行 (DCP) 原理解析":
    each rank holds a range of token positions).  Token i of request b sits at
    global position t = seq_lens[b] - n_new + i (seq_lens count the new
    tokens); its shard r and local index j come from enumerating the shard's
    positions (shard_token_lists); its slot is block_tables[r][b][j // bs],
    row j % bs.

    kind 'gqa': kv_cache [2][nb][bs][Hkv][D], new_k/new_v [B][n_new][Hkv][D]
    kind 'mla': kv_cache [nb][bs][Dqk],      new_k [B][n_new][Dqk], new_v None
    Returns a new array; the input cache is not modified.
    """
    out = np.array(kv_cache, copy=True)
    bt = np.asarray(block_tables)
    for b, S in enumerate(int(x) for x in seq_lens):
        lists = shard_token_lists(S, interleave, dcp_size)
        where = {}
        for r, toks in enumerate(lists):
            for j, t in enumerate(toks[max(0, len(toks) - n_new):].tolist(), start=max(0, len(toks) - n_new)):
                where[t] = (r, j)
        for i in range(n_new):
            r, j = where[S - n_new + i]
            blk, row = int(bt[r, b, j // block_size]), j % block_size
            if kind == "gqa":
                out[0, blk, row] = new_k[b, i]
                out[1, blk, row] = new_v[b, i]
            else:
                out[blk, row] = new_k[b, i]
    return out


# ---------------------------------------------------------------------------
# Per-shard partial attention read through the paged pool (Compute step)
# ---------------------------------------------------------------------------

def gather_shard_kv(kind: str, kv_cache, block_table_row, n_local: int, block_size: int):
    """Local keys/values of one shard of one sequence, in local order.

    kind 'gqa': kv_cache [2][nb][bs][Hkv][D] -> K, V of [n][Hkv][D]
    kind 'mla': kv_cache [nb][bs][Dqk]       -> K [n][1][Dqk], V [n][1][Dv]
    """
    j = np.arange(n_local, dtype=np.int64)
    blk = np.asarray(block_table_row, dtype=np.int64)[j // block_size]
    off = j % block_size
    if kind == "gqa":
        K = kv_cache[0][blk, off]
        V = kv_cache[1][blk, off]
        return K, V
    rows = kv_cache[blk, off]
    return rows[:, None, :], None  # V is a prefix of K, cut by the caller


def ref_attn_shard(kind: str, q, kv_cache, block_tables, seq_lens, shard: int,
                   dcp_size: int, interleave: int, block_size: int, scale: float,
                   q_len: int, head_dim_v: int):
    """Partial output and LSE of one shard.

    kv_cache must already be float64 (see ``to_f64``).  block_tables
    [N][B][max_local_blocks].  Returns o_r [B][Lq][Hq][Dv], lse_r [B][Lq][Hq].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Lq, Hq, _ = q.shape
    out = np.zeros((B, Lq, Hq, head_dim_v))
    lse = np.full((B, Lq, Hq), NEG_INF)
    for b in range(B):
        S = int(seq_lens[b])
        toks = shard_token_lists(S, interleave, dcp_size)[shard]
        K, V = gather_shard_kv(kind, kv_cache, block_tables[shard][b], len(toks), block_size)
        if kind == "mla":
            V = K[:, :, :head_dim_v]
        Hkv = K.shape[1]
        for i in range(Lq):
            visible = toks <= S - Lq + i
            for g, hs in _head_groups(Hq, Hkv):
                out[b, i, hs], lse[b, i, hs] = _attend(
                    q[b, i, hs], K[visible, g], V[visible, g], scale)
    return out, lse


# ---------------------------------------------------------------------------
# LSE merge and head-slice return (AllGather + ReduceScatter step)
# ---------------------------------------------------------------------------

def ref_merge(partial_out, lse):
    """Merge shard partials by LSE reweighting; return head slices.

    partial_out [N][B][Lq][Hq][Dv], lse [N][B][Lq][Hq]
    -> out [N][B][Lq][Hq/N][Dv], out_lse [N][B][Lq][Hq/N]
    LSE = log sum_r exp(lse_r) (shifted by the max), weight_r = exp(lse_r - LSE).
    """
    partial_out = np.asarray(partial_out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    N, B, Lq, Hq, Dv = partial_out.shape
    assert Hq % N == 0
    full = np.zeros((B, Lq, Hq, Dv))
    full_lse = np.full((B, Lq, Hq), NEG_INF)
    for b in range(B):
        for i in range(Lq):
            for h in range(Hq):
                ls = lse[:, b, i, h]
                if np.all(ls == NEG_INF):
                    continue
                m = ls.max()
                w = np.exp(ls - m)
                tot = w.sum()
                full_lse[b, i, h] = m + math.log(tot)
                full[b, i, h] = (w[:, None] * partial_out[:, b, i, h]).sum(axis=0) / tot
    return head_slices(full, N), head_slices(full_lse, N)


def head_slices(full, dcp_size: int):
    """[B][Lq][Hq](...) -> [N][B][Lq][Hq/N](...): rank r gets heads r*Hq/N .. ."""
    B, Lq, Hq = full.shape[:3]
    hs = Hq // dcp_size
    return np.stack([full[:, :, r * hs:(r + 1) * hs] for r in range(dcp_size)])


# ---------------------------------------------------------------------------
# Whole DCP decode step: every shard, then the merge
# ---------------------------------------------------------------------------

def ref_dcp_decode(kind: str, q, kv_cache, block_tables, seq_lens, dcp_size: int,
                   interleave: int, block_size: int, scale: float, q_len: int,
                   head_dim_v: int):
    """All shard partials and the merged head-sliced output."""
    parts, lses = [], []
    for r in range(dcp_size):
        o, l = ref_attn_shard(kind, q, kv_cache, block_tables, seq_lens, r, dcp_size,
                              interleave, block_size, scale, q_len, head_dim_v)
        parts.append(o)
        lses.append(l)
    partial_out = np.stack(parts)
    lse = np.stack(lses)
    out, out_lse = ref_merge(partial_out, lse)
    return {"partial_out": partial_out, "lse": lse, "out": out, "out_lse": out_lse}


def to_f64(t):
    """torch tensor (any float dtype, e.g. bf16) or array -> float64 numpy (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)
