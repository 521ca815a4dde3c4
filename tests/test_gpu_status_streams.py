"""Device status words are per stream: an error found by a kernel on one stream
is reported by dcp_get_last_device_status for that stream only, and reading one
stream's word neither waits for nor clears another's."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import helpers as H
from gpu_common import run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()


def test_status_of_one_stream_does_not_reach_another():
    from context_decode_attention_paged_gb300 import binding as dcp
    bad = H.build_instance(H.small("tiny_gqa", batch=2, q_len=4, lengths=("fixed", 64)))
    bad.seq_lens[1] = 2                           # shorter than its 4 query tokens
    good = H.build_instance(H.small("tiny_gqa", batch=2, lengths=("fixed", 300)))
    s_bad, s_good = torch.cuda.Stream(), torch.cuda.Stream()
    got_bad = run_gpu(bad, stream=s_bad)            # reads and clears s_bad's word
    assert got_bad["status"] == dcp.DCP_ERR_BOUNDS
    # the error is raised again on s_bad; s_good, read before and after, stays clean
    w = bad.w
    dev = torch.device("cuda:0")
    q, kv, bt, sl = bad.q.to(dev), bad.kv_cache.to(dev), bad.block_tables.to(dev), bad.seq_lens.to(dev)
    torch.cuda.synchronize()
    dcp.dcp_decode_attn(w.kind, q, kv, bt, sl, w.dcp_size, w.interleave, w.scale, w.q_len, w.head_dim_v,
                        stream=s_bad)
    got_good = run_gpu(good, stream=s_good)
    assert got_good["status"] == dcp.DCP_OK
    assert dcp.dcp_get_last_device_status(s_good) == dcp.DCP_OK
    assert dcp.dcp_get_last_device_status(s_bad) == dcp.DCP_ERR_BOUNDS
    assert dcp.dcp_get_last_device_status(s_bad) == dcp.DCP_OK          # cleared by the read
    ref = H.oracle_decode(good)
    assert np.abs(got_good["out"] - ref["out"]).max() < 2e-3 + 1e-2 * np.abs(ref["out"]).max()
