"""The decode step is stream-ordered and allocation-free, so it can be captured
in a CUDA graph: attention (including the split-combine launch) and merge
captured once, replayed, give the eager results bit for bit, and a replay after
the query is rewritten in place gives the new eager results."""

from __future__ import annotations

import pytest
import torch

import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()


CASES = [
    ("qwen_gqa", dict(batch=2, lengths=("uniform", 300, 2000), dcp_size=4)),
    ("mla_32", dict(batch=2, lengths=("uniform", 900, 3000))),
    ("mla_mtp", dict(lengths=("fixed", 40000))),          # KV splits: three launches per step
]


@pytest.mark.parametrize("name,kw", CASES)
def test_decode_step_replays_from_a_cuda_graph(name, kw):
    from context_decode_attention_paged_gb300 import binding as dcp
    inst = H.build_instance(H.small(name, **kw))
    w = inst.w
    dev = torch.device("cuda:0")
    q, kv = inst.q.to(dev), inst.kv_cache.to(dev)
    bt, sl = inst.block_tables.to(dev), inst.seq_lens.to(dev)
    B, Lq, Hq, _ = q.shape
    N, Dv = w.dcp_size, w.head_dim_v
    po = torch.empty((N, B, Lq, Hq, Dv), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, Lq, Hq), dtype=torch.float32, device=dev)
    out = torch.empty((N, B, Lq, Hq // N, Dv), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty((N, B, Lq, Hq // N), dtype=torch.float32, device=dev)
    desc = dcp.desc_from_tensors(w.kind, q, kv, bt, Dv)
    ws_bytes = dcp.dcp_decode_attn_workspace_size(desc, N)
    ws = torch.empty((max(ws_bytes, 1),), dtype=torch.uint8, device=dev)

    def step():
        dcp.dcp_decode_attn(w.kind, q, kv, bt, sl, N, w.interleave, w.scale, w.q_len, Dv,
                            partial_out=po, lse=lse, workspace=ws if ws_bytes else None)
        dcp.dcp_merge(po, lse, N, out=out, out_lse=out_lse)

    step()                                           # eager (also warms the library's caches)
    torch.cuda.synchronize()
    assert dcp.dcp_get_last_device_status() == dcp.DCP_OK
    eager = (po.clone(), lse.clone(), out.clone(), out_lse.clone())

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for t in (po, lse, out, out_lse):
            t.zero_()
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert dcp.dcp_get_last_device_status(s) == dcp.DCP_OK      # the captured calls' status word
    for a, b in zip((po, lse, out, out_lse), eager):
        assert torch.equal(a, b)

    # new query values in the same buffer: the replay follows them
    q.copy_(torch.flip(q, dims=[2]))
    step()
    torch.cuda.synchronize()
    eager2 = (po.clone(), lse.clone(), out.clone(), out_lse.clone())
    for t in (po, lse, out, out_lse):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip((po, lse, out, out_lse), eager2):
        assert torch.equal(a, b)
    assert not torch.equal(eager2[2], eager[2])
