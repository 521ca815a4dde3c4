"""Pins for the oracle's cache write (storing each request's newest tokens in
the shard that owns their positions), pinned by what does not depend on it:

* round trip through the read path the attention oracle uses: after the write,
  the logical sequence read back out of the paged pool holds the new rows at
  positions S - n_new .. S - 1 and the old rows everywhere else;
* only B * n_new cache rows change;
* dcp_size 1: token t sits at local index t (closed form);
* the blog's worked example (200K tokens, 4 ranks, runs of 50K): the newest
  token belongs to rank 3 at local index 49,999;
* planted mistakes in the position, the owner or the local index are caught.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from oracle import dcp_oracle as orc
import helpers as H


def _new_rows(w, n_new, seed):
    g = torch.Generator().manual_seed(seed)
    if w.kind == "gqa":
        shape = (w.batch, n_new, w.num_kv_heads, w.head_dim_qk)
        k = torch.randn(shape, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, generator=g).to(torch.bfloat16)
        return orc.to_f64(k), orc.to_f64(v)
    k = torch.randn((w.batch, n_new, w.head_dim_qk), generator=g).to(torch.bfloat16)
    return orc.to_f64(k), None


def _with_cache(inst, kv):
    return dataclasses.replace(inst, kv_cache=torch.from_numpy(np.ascontiguousarray(kv)))


def check_round_trip(write_fn, name, kw, n_new):
    inst = H.build_instance(H.small(name, **kw))
    w = inst.w
    _, kv, bt, sl = H.oracle_inputs(inst)
    new_k, new_v = _new_rows(w, n_new, seed=77)
    after = write_fn(w.kind, kv, new_k, new_v, bt, sl, w.dcp_size, w.interleave, w.block_size, n_new)
    K0, V0 = H.logical_kv(inst)
    K1, V1 = H.logical_kv(_with_cache(inst, after))
    for b, S in enumerate(int(x) for x in sl):
        old = slice(0, S - n_new)
        assert np.array_equal(K1[b][old], K0[b][old]), f"request {b}: old keys changed"
        if w.kind == "gqa":
            assert np.array_equal(K1[b][S - n_new:], new_k[b]), f"request {b}: new keys"
            assert np.array_equal(V1[b][S - n_new:], new_v[b]), f"request {b}: new values"
            assert np.array_equal(V1[b][old], V0[b][old]), f"request {b}: old values changed"
        else:
            assert np.array_equal(K1[b][S - n_new:, 0], new_k[b]), f"request {b}: new rows"
    return kv, after


KV_CASES = [
    ("tiny_gqa", dict(batch=3, lengths=("uniform", 5, 700), dcp_size=4, interleave=3), 1),
    ("tiny_gqa", dict(batch=2, q_len=4, lengths=("uniform", 4, 300), dcp_size=2, interleave=16), 4),
    ("qwen_gqa", dict(batch=2, num_q_heads=8, lengths=("uniform", 300, 900), dcp_size=4), 2),
    ("mla_32", dict(batch=2, num_q_heads=4, lengths=("uniform", 129, 600), dcp_size=8, interleave=1), 3),
    ("mla_32", dict(batch=1, num_q_heads=4, lengths=("fixed", 257), dcp_size=2, interleave=128), 1),
]


@pytest.mark.parametrize("name,kw,n_new", KV_CASES)
def test_kv_write_round_trip_through_the_read_path(name, kw, n_new):
    before, after = check_round_trip(orc.ref_kv_cache_write, name, kw, n_new)
    w = H.small(name, **kw)
    row = before.shape[-1] * (before.shape[-2] if w.kind == "gqa" else 1)   # values of one token row
    changed = (after.reshape(-1, row) != before.reshape(-1, row)).any(axis=-1).sum()
    # random new rows differ from the old ones in every row (probability 1 at these sizes)
    per_token = 2 if w.kind == "gqa" else 1
    assert changed == w.batch * n_new * per_token


def test_kv_write_single_shard_is_position_indexed():
    w = H.small("mla_32", batch=2, num_q_heads=4, lengths=("uniform", 200, 700), dcp_size=1, interleave=5)
    inst = H.build_instance(w)
    _, kv, bt, sl = H.oracle_inputs(inst)
    new_k, _ = _new_rows(w, 3, seed=5)
    after = orc.ref_kv_cache_write("mla", kv, new_k, None, bt, sl, 1, 5, w.block_size, 3)
    for b, S in enumerate(int(x) for x in sl):
        for i in range(3):
            t = S - 3 + i
            assert np.array_equal(after[bt[0, b, t // w.block_size], t % w.block_size], new_k[b, i])


def test_kv_write_blog_worked_example():
    """200K tokens on 4 ranks in runs of 50K: position 199,999 is rank 3's 50,000th token."""
    S, N, I, bs, D = 200_000, 4, 50_000, 128, 8
    nb_per = -(-50_000 // bs)
    bt = np.arange(N * nb_per, dtype=np.int32).reshape(N, 1, nb_per)
    kv = np.zeros((N * nb_per, bs, D))
    new_k = np.arange(D, dtype=np.float64).reshape(1, 1, D) + 1.0
    after = orc.ref_kv_cache_write("mla", kv, new_k, None, bt, [S], N, I, bs, 1)
    j = 49_999
    assert np.array_equal(after[bt[3, 0, j // bs], j % bs], new_k[0, 0])
    assert np.count_nonzero(after) == D


def _write_with(mistake):
    def fn(kind, kv_cache, new_k, new_v, block_tables, seq_lens, N, I, bs, n_new):
        out = np.array(kv_cache, copy=True)
        for b, S in enumerate(int(x) for x in seq_lens):
            lists = orc.shard_token_lists(S, I, N)
            for i in range(n_new):
                t = S - n_new + i + (1 if mistake == "position_plus_one" else 0)
                t = min(t, S - 1)
                r = (t // I) % N
                if mistake == "owner_rotated":
                    r = (r + 1) % N
                j = t if mistake == "global_index" else int(np.searchsorted(lists[(t // I) % N], t))
                j = min(j, len(lists[r]) - 1) if len(lists[r]) else 0
                blk, row = int(block_tables[r, b, j // bs]), j % bs
                if kind == "gqa":
                    out[0, blk, row] = new_k[b, i]
                    out[1, blk, row] = new_v[b, i]
                else:
                    out[blk, row] = new_k[b, i]
        return out
    return fn


@pytest.mark.parametrize("mistake", ["position_plus_one", "owner_rotated", "global_index"])
def test_planted_kv_write_mistakes_are_caught(mistake):
    with pytest.raises(AssertionError):
        check_round_trip(_write_with(mistake), "tiny_gqa",
                         dict(batch=3, lengths=("uniform", 40, 700), dcp_size=4, interleave=3), 2)
    check_round_trip(_write_with("none"), "tiny_gqa",
                     dict(batch=3, lengths=("uniform", 40, 700), dcp_size=4, interleave=3), 2)
