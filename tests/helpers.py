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
