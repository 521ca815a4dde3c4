"""dcp_decode_attn_noalloc: the entry point for callers that cannot allocate.

Some callers may not call cudaMalloc when they run attention (a plugin that
is given only its input and output buffers, code inside another runtime's
memory pool, a decode loop that forbids allocation).  For them the library
takes the split scratch from an array compiled into it.  These checks call it
through the raw C ABI and compare it with dcp_decode_attn, which uses a
caller-allocated workspace, on shapes that do need scratch; two calls in a
row, so the second one runs on the first one's leftover scratch contents.
This file sorts last so that a run stopping at the first failure has already
run every other test.
"""

from __future__ import annotations

import ctypes
import re
import os

import numpy as np
import pytest
import torch

import helpers as H
from gpu_common import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def scratch_limit() -> int:
    src = open(os.path.join(ROOT, "include", "dcp.h")).read()
    m = re.search(r"#define DCP_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", src)
    return int(m.group(1)) * int(m.group(2)) * int(m.group(3))


@pytest.fixture(scope="module")
def dcp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()
    from context_decode_attention_paged_gb300 import binding
    raw = binding.raw_lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    raw.dcp_decode_attn_noalloc.restype = i32
    raw.dcp_decode_attn_noalloc.argtypes = [ctypes.POINTER(binding.DcpAttnDesc), vp, vp, vp, vp,
                                            i32, i32, ctypes.c_float, i32, vp, vp, vp]
    return binding


def call_noalloc(dcp, w, desc, q, kv, bt, sl, po, lse):
    raw = dcp.raw_lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return raw.dcp_decode_attn_noalloc(ctypes.byref(desc), q.data_ptr(), kv.data_ptr(),
                                       bt.data_ptr(), sl.data_ptr(), w.dcp_size, w.interleave,
                                       w.scale, w.q_len, po.data_ptr(), lse.data_ptr(), stream)


CASES = [
    ("qwen_gqa", dict(batch=2, lengths=("uniform", 3000, 8000))),       # tensor-core kernel, splits
    ("mla_32", dict(batch=1, lengths=("fixed", 40000))),                # tensor-core kernel, splits
]


@pytest.mark.parametrize("name,kw", CASES)
def test_noalloc_matches_dcp_decode_attn(dcp, name, kw):
    w = H.small(name, **kw)
    inst = H.build_instance(w)
    dev = torch.device("cuda:0")
    q, kv = inst.q.to(dev), inst.kv_cache.to(dev)
    bt, sl = inst.block_tables.to(dev), inst.seq_lens.to(dev)
    desc = dcp.desc_from_tensors(w.kind, q, kv, bt, w.head_dim_v)
    need = dcp.dcp_decode_attn_workspace_size(desc, w.dcp_size)
    assert 0 < need <= scratch_limit(), need            # the case does use scratch

    ref_po, ref_lse = dcp.dcp_decode_attn(w.kind, q, kv, bt, sl, w.dcp_size, w.interleave,
                                          w.scale, w.q_len, w.head_dim_v)
    torch.cuda.synchronize()
    for _ in range(2):
        po = torch.full_like(ref_po, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = call_noalloc(dcp, w, desc, q, kv, bt, sl, po, lse)
        assert rc == dcp.DCP_OK, dcp.status_string(rc)
        torch.cuda.synchronize()
        assert dcp.dcp_get_last_device_status() == dcp.DCP_OK
        assert_close(po.cpu().numpy(), ref_po.cpu().numpy(), "partial_out (no-alloc)")
        assert_lse_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), "lse (no-alloc)")


def test_noalloc_rejects_shapes_beyond_its_scratch(dcp):
    """MLA, 4 requests x 4 query tokens at 200k context needs more split scratch
    than the built-in array; the call is refused before anything is written."""
    w = H.small("mla_mtp", batch=4)
    N, max_lb = w.dcp_size, 196                       # 200000 / 8 tokens per shard, 128 per block
    nb = N * w.batch * max_lb
    dev = torch.device("cuda:0")
    q = torch.zeros((w.batch, w.q_len, 128, 576), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((nb, 128, 576), dtype=torch.bfloat16, device=dev)
    bt = torch.arange(nb, dtype=torch.int32, device=dev).reshape(N, w.batch, max_lb)
    sl = torch.full((w.batch,), 200000, dtype=torch.int32, device=dev)
    po = torch.full((N, w.batch, w.q_len, 128, 512), float("nan"), device=dev)
    lse = torch.full((N, w.batch, w.q_len, 128), float("nan"), device=dev)
    desc = dcp.desc_from_tensors("mla", q, kv, bt, 512)
    assert dcp.dcp_decode_attn_workspace_size(desc, N) > scratch_limit()
    rc = call_noalloc(dcp, w, desc, q, kv, bt, sl, po, lse)
    assert rc == dcp.DCP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(po).all() and torch.isnan(lse).all()
