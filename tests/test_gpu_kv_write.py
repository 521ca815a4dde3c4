"""GPU parity of the cache write (storing each request's newest tokens in the
shard that owns their positions): bit-exact against the oracle at test sizes,
and at the full workload sizes every target cell holds its new row and no other
row of the pool changed."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import helpers as H
from context_decode_attention_paged_gb300 import workloads as wl
from oracle import dcp_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()


def _new_rows(w, n_new, seed, device):
    g = torch.Generator(device=device).manual_seed(seed)
    if w.kind == "gqa":
        shape = (w.batch, n_new, w.num_kv_heads, w.head_dim_qk)
        k = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
        v = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
        return k, v
    return torch.randn((w.batch, n_new, w.head_dim_qk), generator=g, device=device).to(torch.bfloat16), None


CASES = [
    ("tiny_gqa", dict(batch=3, lengths=("uniform", 5, 700), dcp_size=4, interleave=3), 1),
    ("tiny_gqa", dict(batch=2, q_len=4, lengths=("uniform", 4, 300), dcp_size=2, interleave=16), 4),
    ("tiny_gqa", dict(batch=2, lengths=("fixed", 1), dcp_size=2, interleave=1), 1),
    ("qwen_gqa", dict(batch=4, lengths=("uniform", 300, 5000), dcp_size=4), 2),
    ("mla_32", dict(batch=3, num_q_heads=4, lengths=("uniform", 129, 3000), dcp_size=8, interleave=1), 3),
    ("mla_32", dict(batch=2, num_q_heads=4, lengths=("fixed", 257), dcp_size=2, interleave=128), 1),
    ("mla_mtp", dict(num_q_heads=4, lengths=("fixed", 40000)), 4),
]


@pytest.mark.parametrize("name,kw,n_new", CASES)
def test_kv_write_bit_exact(name, kw, n_new):
    from context_decode_attention_paged_gb300 import binding as dcp
    inst = H.build_instance(H.small(name, **kw))
    w = inst.w
    new_k, new_v = _new_rows(w, n_new, seed=11, device="cpu")
    ref = orc.ref_kv_cache_write(w.kind, orc.to_f64(inst.kv_cache), orc.to_f64(new_k),
                                 None if new_v is None else orc.to_f64(new_v),
                                 inst.block_tables.numpy(), inst.seq_lens.numpy(), w.dcp_size,
                                 w.interleave, w.block_size, n_new)
    dev = torch.device("cuda:0")
    kv = inst.kv_cache.to(dev)
    dcp.dcp_kv_cache_write(w.kind, new_k.to(dev), None if new_v is None else new_v.to(dev), kv,
                           inst.block_tables.to(dev), inst.seq_lens.to(dev), w.dcp_size, w.interleave)
    torch.cuda.synchronize()
    assert dcp.dcp_get_last_device_status() == dcp.DCP_OK
    assert np.array_equal(orc.to_f64(kv.cpu()), ref)


def test_kv_write_short_sequence_sets_bounds_status():
    from context_decode_attention_paged_gb300 import binding as dcp
    inst = H.build_instance(H.small("tiny_gqa", batch=2, lengths=("fixed", 64)))
    w = inst.w
    dev = torch.device("cuda:0")
    kv = inst.kv_cache.to(dev)
    before = kv.clone()
    sl = inst.seq_lens.to(dev).clone()
    sl[1] = 1                                         # shorter than its 2 new tokens
    new_k, new_v = _new_rows(w, 2, seed=3, device=dev)
    dcp.dcp_kv_cache_write("gqa", new_k, new_v, kv, inst.block_tables.to(dev), sl, w.dcp_size, w.interleave)
    assert dcp.dcp_get_last_device_status() == dcp.DCP_ERR_BOUNDS
    changed = (kv != before).flatten(3).any(-1).sum().item()   # token rows, both pools
    assert changed == 2 * 2                           # request 0's two tokens, K and V


@pytest.mark.parametrize("name", ["qwen_gqa", "mla_512"])
def test_kv_write_full_size(name):
    from context_decode_attention_paged_gb300 import binding as dcp
    w = wl.WORKLOADS[name]
    inst = bench.setup_gpu(w, 0)
    try:
        n_new = max(1, w.q_len)
        before = inst.kv_cache.clone()
        new_k, new_v = _new_rows(w, n_new, seed=29, device=inst.kv_cache.device)
        dcp.dcp_kv_cache_write(w.kind, new_k, new_v, inst.kv_cache, inst.block_tables, inst.seq_lens,
                               w.dcp_size, w.interleave)
        torch.cuda.synchronize()
        assert dcp.dcp_get_last_device_status() == dcp.DCP_OK
        # target cells from the oracle's enumeration of each shard's positions
        bt = inst.block_tables.cpu().numpy()
        cells = []
        for b, S in enumerate(inst.seq_lens.cpu().tolist()):
            lists = orc.shard_token_lists(S, w.interleave, w.dcp_size)
            for i in range(n_new):
                t = S - n_new + i
                r = (t // w.interleave) % w.dcp_size
                j = int(np.searchsorted(lists[r], t))
                assert lists[r][j] == t
                cells.append((b, i, int(bt[r, b, j // w.block_size]), j % w.block_size))
        blk = torch.tensor([c[2] for c in cells], device=inst.kv_cache.device)
        row = torch.tensor([c[3] for c in cells], device=inst.kv_cache.device)
        if w.kind == "gqa":
            got_k = inst.kv_cache[0][blk, row]
            got_v = inst.kv_cache[1][blk, row]
            assert torch.equal(got_k, new_k.reshape(-1, *new_k.shape[2:]))
            assert torch.equal(got_v, new_v.reshape(-1, *new_v.shape[2:]))
            changed = (inst.kv_cache != before).flatten(3).any(-1).sum().item()
            assert changed == 2 * w.batch * n_new
        else:
            got = inst.kv_cache[blk, row]
            assert torch.equal(got, new_k.reshape(-1, new_k.shape[-1]))
            changed = (inst.kv_cache != before).any(-1).sum().item()
            assert changed == w.batch * n_new
    finally:
        del inst
        torch.cuda.empty_cache()
