"""Failure detection inside the attention kernels, without a GPU fault.

A test-only hook (dcp_testing_set_hooks, exported by the library but not
declared in include/dcp.h) shortens every bounded wait to a few milliseconds
and makes the TMA producer of the work unit skip one tile: that tile never
arrives, so the waits on it run out.  The kernel must then unwind on its own:
record DCP_ERR_TIMEOUT, leave the unit's outputs at zero / -inf, drain its
copies and MMAs, free its tensor memory and release the peer CTA of its
cluster.  An ordinary launch on the same context right after must still match
the oracle (nothing left waiting, TMEM free).
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import helpers as H
from gpu_common import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()
    from context_decode_attention_paged_gb300 import binding as dcp
    lib = dcp.raw_lib()
    lib.dcp_testing_set_hooks.restype = None
    lib.dcp_testing_set_hooks.argtypes = [ctypes.c_ulonglong, ctypes.c_int32]
    yield lib.dcp_testing_set_hooks
    lib.dcp_testing_set_hooks(0, -1)


# MLA with one shard and one request (one cluster pair), GQA with one shard,
# one request and one KV head (one CTA); then two MLA paths of their own
CASES = [
    ("mla_32", dict(batch=1, lengths=("fixed", 300), dcp_size=1)),
    ("mla_32", dict(batch=1, lengths=("fixed", 100), dcp_size=1)),
    ("qwen_gqa", dict(batch=1, num_q_heads=16, num_kv_heads=1, lengths=("fixed", 700), dcp_size=1)),
    # the MLA instance for small blocks (four TMA boxes a tile)
    ("mla_32", dict(batch=1, block_size=16, lengths=("fixed", 300), dcp_size=1, interleave=16)),
    # an MLA batch above 128: units in the order a pre-pass writes (every unit
    # times out; they run in two waves of clusters)
    ("mla_32", dict(batch=130, lengths=("uniform", 100, 200), dcp_size=1)),
]


@pytest.mark.parametrize("name,kw", CASES)
def test_kernel_wait_runs_out_and_the_unit_unwinds(hooks, name, kw):
    from context_decode_attention_paged_gb300 import binding as dcp
    inst = H.build_instance(H.small(name, **kw))
    hooks(5_000_000, 1)                     # 5 ms waits; tile 1 is never loaded
    try:
        got = run_gpu(inst)
    finally:
        hooks(0, -1)
    assert got["status"] == dcp.DCP_ERR_TIMEOUT, dcp.status_string(got["status"])
    assert (got["lse"] == -np.inf).all()
    assert (got["partial_out"] == 0).all()
    assert (got["out"] == 0).all()
    # the same context right after: an ordinary launch matches the oracle
    check_against_oracle(inst)
