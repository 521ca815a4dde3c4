"""Test glue: build seeded instances with the oracle's slot map and run the oracle."""

from __future__ import annotations

import numpy as np
import torch

from context_decode_attention_paged_gb300 import workloads as wl
from oracle import dcp_oracle as orc


def build_instance(w: wl.Workload, device="cpu", seq_lens=None) -> wl.Instance:
    """Instance whose block tables are sized by the oracle's enumerated slot map."""
    if seq_lens is None:
        seq_lens = wl.make_seq_lens(w)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32)
    sm = orc.ref_slot_map(seq_lens.tolist(), w.interleave, w.dcp_size, w.block_size)
    return wl.make_instance(w, sm["local_num_blocks"], device=device, seq_lens=seq_lens)


def oracle_inputs(inst: wl.Instance):
    q = orc.to_f64(inst.q)
    kv = orc.to_f64(inst.kv_cache)
    bt = inst.block_tables.cpu().numpy()
    sl = inst.seq_lens.cpu().numpy()
    return q, kv, bt, sl


def oracle_decode(inst: wl.Instance, dcp_size=None, interleave=None):
    w = inst.w
    q, kv, bt, sl = oracle_inputs(inst)
    return orc.ref_dcp_decode(w.kind, q, kv, bt, sl, dcp_size or w.dcp_size,
                              interleave or w.interleave, w.block_size, w.scale,
                              w.q_len, w.head_dim_v)


def logical_kv(inst: wl.Instance):
    """Per-sequence K/V in global token order, read back out of the paged pool.

    Returns lists over b of K [S][Hkv][Dqk] and V [S][Hkv][Dv] (float64).
    """
    w = inst.w
    _, kv, bt, sl = oracle_inputs(inst)
    Ks, Vs = [], []
    for b, S in enumerate(sl):
        S = int(S)
        lists = orc.shard_token_lists(S, w.interleave, w.dcp_size)
        if w.kind == "gqa":
            K = np.zeros((S, w.num_kv_heads, w.head_dim_qk))
            V = np.zeros((S, w.num_kv_heads, w.head_dim_v))
        else:
            K = np.zeros((S, 1, w.head_dim_qk))
        for r, toks in enumerate(lists):
            k, v = orc.gather_shard_kv(w.kind, kv, bt[r][b], len(toks), w.block_size)
            K[toks] = k
            if w.kind == "gqa":
                V[toks] = v
        if w.kind == "mla":
            V = K[:, :, : w.head_dim_v]
        Ks.append(K)
        Vs.append(V)
    return Ks, Vs


def small(w_name: str, **kw) -> wl.Workload:
    """A named workload with some fields overridden (small test sizes)."""
    return wl.WORKLOADS[w_name].with_(**kw)


def repage(inst: wl.Instance, w2: wl.Workload) -> wl.Instance:
    """Same q and logical K/V as ``inst``, laid out under w2's shard rule.

    Used to compare different dcp_size / interleave on identical data.
    """
    w = inst.w
    Ks, Vs = logical_kv(inst)
    sl = inst.seq_lens.cpu()
    sm = orc.ref_slot_map(sl.tolist(), w2.interleave, w2.dcp_size, w2.block_size)
    new = wl.make_instance(w2, sm["local_num_blocks"], device="cpu", seq_lens=sl)
    kv = new.kv_cache
    bt = new.block_tables.numpy()
    for b, S in enumerate(sl.tolist()):
        for r, toks in enumerate(orc.shard_token_lists(S, w2.interleave, w2.dcp_size)):
            j = np.arange(len(toks))
            blk = torch.from_numpy(bt[r][b][j // w2.block_size].astype(np.int64))
            off = torch.from_numpy(j % w2.block_size)
            if w2.kind == "gqa":
                kv[0][blk, off] = torch.from_numpy(Ks[b][toks]).to(kv.dtype)
                kv[1][blk, off] = torch.from_numpy(Vs[b][toks]).to(kv.dtype)
            else:
                kv[blk, off] = torch.from_numpy(Ks[b][toks][:, 0]).to(kv.dtype)
    new.q.copy_(inst.q.cpu())
    return new



def scale_keys_by_position(inst: wl.Instance, factor, value_scale: float = 1.0,
                           key_dims: slice = slice(None)) -> wl.Instance:
    """Multiply the dims ``key_dims`` of every cached key row at global position
    t of a request of length S by factor(t / S), and every value row by
    ``value_scale``, in place (MLA: scale only the rope dims to leave the
    values alone).  Scores that grow along the sequence move the running
    reference max many times, tile after tile."""
    w = inst.w
    kv = inst.kv_cache
    bt = inst.block_tables.numpy()
    for b, S in enumerate(inst.seq_lens.tolist()):
        for r, toks in enumerate(orc.shard_token_lists(S, w.interleave, w.dcp_size)):
            if not len(toks):
                continue
            j = np.arange(len(toks))
            blk = torch.from_numpy(bt[r][b][j // w.block_size].astype(np.int64))
            off = torch.from_numpy(j % w.block_size)
            f = torch.as_tensor(factor(np.asarray(toks, dtype=np.float64) / S))
            if w.kind == "gqa":
                rows = kv[0][blk, off].double()
                rows[..., key_dims] *= f.view(-1, 1, 1)
                kv[0][blk, off] = rows.to(kv.dtype)
                kv[1][blk, off] = (kv[1][blk, off].double() * value_scale).to(kv.dtype)
            else:
                rows = kv[blk, off].double()
                rows[..., key_dims] *= f.view(-1, 1)
                kv[blk, off] = rows.to(kv.dtype)
    return inst


# ---------------------------------------------------------------------------
# Stress inputs: peaked softmaxes, attention sinks, poisoned unused cache slots
# ---------------------------------------------------------------------------

def _cell_of(inst: wl.Instance, b: int, t: int):
    """(block id, row in block) that holds global position t of request b."""
    w = inst.w
    r = (t // w.interleave) % w.dcp_size
    toks = orc.shard_token_lists(int(inst.seq_lens[b]), w.interleave, w.dcp_size)[r]
    j = int(np.searchsorted(toks, t))
    assert toks[j] == t
    return int(inst.block_tables[r, b, j // w.block_size]), j % w.block_size


def _bf16(x) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)


def plant_dominant_keys(inst: wl.Instance, lifts=(12.0, 12.25, 11.5, 11.7), seed: int = 7) -> wl.Instance:
    """Peaked softmaxes at the workload's own value scale, in place.

    For every request, len(lifts) keys at seeded positions (visible to every
    query) are rewritten so that the scaled score of every query row at key k
    is lifts[k] (natural-log units; the other keys of these workloads score
    about N(0, 1)).  Their value rows come in opposite-sign pairs (u, -u, w, -w,
    u, w ~ N(0, std^2)), so the dominant keys' contributions nearly cancel and
    the output is small: the absolute part of the tolerance is what binds, and
    any rounding of the probabilities of the dominant keys shows up in full.

    GQA: each dominant key row of KV head g is the minimum-norm solution of
    q_h . k = lifts[k] / scale over the group's query rows.  MLA: the key row is
    shared by all 128 heads and its first Dv values are the value, so the rope
    part carries the score: the queries' rope dims become a shared direction
    plus noise, the dominant rope rows point along it, and the dominant latent
    rows (the values) are projected off the span of the query latents.
    """
    w = inst.w
    rng = np.random.default_rng(seed)
    n = len(lifts)
    Dv, Dqk = w.head_dim_v, w.head_dim_qk
    q = orc.to_f64(inst.q)                                   # [B][Lq][Hq][Dqk]
    for b in range(w.batch):
        S = int(inst.seq_lens[b])
        last = S - w.q_len                                   # seen by every query of b
        if last + 1 < n:
            continue
        pos = rng.choice(last + 1, size=n, replace=False)
        vals = []
        for k in range(0, n, 2):
            u = rng.standard_normal(Dv) * w.std
            vals += [u, -u]
        if w.kind == "gqa":
            gsize = w.num_q_heads // w.num_kv_heads
            for g in range(w.num_kv_heads):
                Q = q[b, :, g * gsize:(g + 1) * gsize, :].reshape(-1, Dqk)
                for k, t in enumerate(pos):
                    target = np.full(Q.shape[0], lifts[k] / w.scale)
                    krow = np.linalg.lstsq(Q, target, rcond=None)[0]
                    blk, row = _cell_of(inst, b, int(t))
                    inst.kv_cache[0, blk, row, g] = _bf16(krow)
                    inst.kv_cache[1, blk, row, g] = _bf16(vals[k])
        else:
            r_dir = rng.standard_normal(Dqk - Dv) * w.std
            noise = rng.standard_normal(q[b, :, :, Dv:].shape) * w.std * 0.3
            q[b, :, :, Dv:] = r_dir + noise
            inst.q[b, :, :, Dv:] = _bf16(q[b, :, :, Dv:])
            qlat = orc.to_f64(inst.q[b, :, :, :Dv]).reshape(-1, Dv)
            basis = np.linalg.svd(qlat, full_matrices=False)[2]   # rows span the query latents
            for k, t in enumerate(pos):
                u = vals[k] - basis.T @ (basis @ vals[k])
                rope = (lifts[k] / w.scale) * r_dir / float(r_dir @ r_dir)
                blk, row = _cell_of(inst, b, int(t))
                inst.kv_cache[blk, row] = _bf16(np.concatenate([u, rope]))
    return inst


def plant_sinks(inst: wl.Instance, totals=(30.0, 45.0, 60.0), seed: int = 11) -> wl.Instance:
    """Attention-sink scores on an MLA instance, in place.

    Request b gets one key at position 0 (the first token, as a sink usually
    is) whose scaled score is totals[b % len(totals)] for every head, split
    unevenly between the two halves of the rope dims: the first half carries
    -10 and the second total + 10, or the other way round, or half each.  The
    queries' rope halves become shared directions plus noise so that every
    head sees the sink.  Every other key keeps its N(0, std^2) row.
    """
    w = inst.w
    assert w.kind == "mla"
    rng = np.random.default_rng(seed)
    Dv, Dqk = w.head_dim_v, w.head_dim_qk
    half = (Dqk - Dv) // 2
    for b in range(w.batch):
        total = totals[b % len(totals)]
        split = [(-10.0, total + 10.0), (total + 10.0, -10.0), (total / 2, total / 2)][b % 3]
        q = orc.to_f64(inst.q[b])
        rope = np.zeros(Dqk - Dv)
        for hh, part in enumerate(split):
            sl = slice(Dv + hh * half, Dv + (hh + 1) * half)
            d = rng.standard_normal(half) * w.std
            q[:, :, sl] = d + rng.standard_normal(q[:, :, sl].shape) * w.std * 0.3
            rope[hh * half:(hh + 1) * half] = (part / w.scale) * d / float(d @ d)
        inst.q[b] = _bf16(q)
        blk, row = _cell_of(inst, b, 0)
        u = rng.standard_normal(Dv) * w.std
        inst.kv_cache[blk, row] = _bf16(np.concatenate([u, rope]))
    return inst


def poison_unused_slots(inst: wl.Instance) -> wl.Instance:
    """Fill every cache row no live token occupies with bf16 NaN, +Inf and -Inf
    (cycling), in place: the rows past each shard's length in its last block
    and every block no table references.  A kernel that lets a stale row reach
    the output (0 * NaN, 0 * Inf) fails the comparison; the oracle reads live
    rows only."""
    w = inst.w
    nb = inst.kv_cache.shape[1] if w.kind == "gqa" else inst.kv_cache.shape[0]
    live = np.zeros((nb, w.block_size), dtype=bool)
    bt = inst.block_tables.numpy()
    for b, S in enumerate(inst.seq_lens.tolist()):
        for r, toks in enumerate(orc.shard_token_lists(int(S), w.interleave, w.dcp_size)):
            j = np.arange(len(toks))
            live[bt[r][b][j // w.block_size], j % w.block_size] = True
    dead = torch.from_numpy(~live)
    bad = torch.tensor([float("nan"), float("inf"), float("-inf")], dtype=torch.bfloat16)
    idx = torch.nonzero(dead)
    fill = bad[torch.arange(idx.shape[0]) % 3]
    if w.kind == "gqa":
        for p in range(2):
            view = inst.kv_cache[p]
            view[idx[:, 0], idx[:, 1]] = fill.view(-1, 1, 1).expand(-1, w.num_kv_heads, w.head_dim_qk)
    else:
        inst.kv_cache[idx[:, 0], idx[:, 1]] = fill.view(-1, 1).expand(-1, w.head_dim_qk)
    return inst
