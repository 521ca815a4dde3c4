"""GPU parity on inputs that stress the numerics and the edge handling, through
the C ABI, against the oracle, at the unchanged tolerances.

* Peaked softmaxes at the workloads' own value scale (GQA N(0,1), MLA
  N(0,0.5)): a few keys per row score 11-12 above the rest and their values
  cancel in pairs, so the output is small and the rounding of the dominant
  probabilities is what the absolute bound sees.
* Attention sinks on MLA: one key per request with a scaled score of 30-60,
  split unevenly between the two halves of the rope dims.
* Poisoned cache: every row no live token occupies holds bf16 NaN / +Inf / -Inf
  (the rows past a shard's length in its last block and every unreferenced
  block); shard lengths leave ragged last tiles of 1, 63, 65 and 127 keys.
* Long causal queries on MLA (chunked prefill, Lq 16 and 64).
* A block table entry past the pool: the unit that owns it is skipped (zero
  partial, -inf LSE) and DCP_ERR_BOUNDS is reported; every other unit matches.

"Context Parallel Guide", section "Overview" (DCP shards the KV-cache storage;
unused slots of a block hold whatever was there) and section "Decode Context
Parallel" (chunked prefill with DCP); vLLM DCP blog, "DCP 執行流程" (Compute
step and the LSE merge).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import helpers as H
from gpu_common import assert_close, assert_lse_close, check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()


DOMINANT_CASES = [
    ("qwen_gqa", dict(batch=3, lengths=("uniform", 1500, 4000), dcp_size=2)),
    ("qwen_gqa", dict(batch=2, q_len=4, lengths=("uniform", 800, 3000), dcp_size=4, interleave=64)),
    ("tiny_gqa", dict(batch=3, lengths=("uniform", 300, 1500), dcp_size=2)),
    ("mla_32", dict(batch=3, lengths=("uniform", 1500, 5000), dcp_size=4)),
    ("mla_32", dict(batch=2, q_len=2, lengths=("uniform", 700, 3000), dcp_size=2, interleave=1)),
]


@pytest.mark.parametrize("name,kw", DOMINANT_CASES)
def test_dominant_keys_at_workload_value_scale(name, kw):
    inst = H.plant_dominant_keys(H.build_instance(H.small(name, **kw)))
    check_against_oracle(inst)


@pytest.mark.parametrize("kw", [
    dict(batch=3, lengths=("uniform", 2000, 6000), dcp_size=2),
    dict(batch=6, lengths=("uniform", 300, 3000), dcp_size=8),
    dict(batch=3, q_len=4, lengths=("fixed", 2500), dcp_size=4, interleave=1),
])
def test_attention_sink_scores_30_to_60(kw):
    inst = H.plant_sinks(H.build_instance(H.small("mla_32", **kw)))
    check_against_oracle(inst)


# local lengths with ragged last tiles: 128k + {1, 63, 65, 127} keys per shard
RAGGED = [128 * 3 + 1, 128 * 2 + 63, 128 * 5 + 65, 128 * 4 + 127]
POISON_CASES = [
    ("qwen_gqa", dict(batch=4, dcp_size=1, interleave=128)),                   # tensor-core GQA
    ("qwen_gqa", dict(batch=4, dcp_size=2, interleave=128, block_size=32)),
    ("tiny_gqa", dict(batch=4, dcp_size=2, interleave=16)),                    # bs 16, D 64
    ("mla_32", dict(batch=4, dcp_size=1, interleave=128)),                     # tensor-core MLA
    ("mla_32", dict(batch=4, dcp_size=4, interleave=1, q_len=4)),
    ("mla_32", dict(batch=4, dcp_size=2, interleave=16, block_size=16)),      # four boxes per tile
    ("mla_32", dict(batch=4, dcp_size=1, interleave=64, block_size=64)),
    ("tiny_gqa", dict(batch=4, dcp_size=2, interleave=16, head_dim_qk=96, head_dim_v=96)),   # SIMT
    ("mla_32", dict(batch=4, dcp_size=2, interleave=128, num_q_heads=16, head_dim_qk=72,
                    head_dim_v=64)),                                           # SIMT, MLA layout
]


@pytest.mark.parametrize("name,kw", POISON_CASES)
def test_poisoned_unused_cache_rows_do_not_reach_the_output(name, kw):
    w = H.small(name, **kw)
    # shard 0 of request b holds RAGGED[b] keys (the other shards hold the rest)
    lens = []
    for L in RAGGED[: w.batch]:
        if w.dcp_size == 1:
            lens.append(L)
        else:
            period = w.interleave * w.dcp_size
            lens.append((L // w.interleave) * period + L % w.interleave)
    inst = H.build_instance(w, seq_lens=np.array(lens, dtype=np.int32))
    H.poison_unused_slots(inst)
    check_against_oracle(inst)


@pytest.mark.parametrize("kw", [
    dict(batch=1, q_len=16, lengths=("fixed", 2100), dcp_size=2, interleave=1),
    dict(batch=2, q_len=16, lengths=("uniform", 900, 2500), dcp_size=4, interleave=128),
    dict(batch=1, q_len=64, lengths=("fixed", 1500), dcp_size=2, interleave=128),
    dict(batch=1, q_len=64, lengths=("fixed", 700), dcp_size=2, interleave=1),
])
def test_mla_long_causal_queries(kw):
    check_against_oracle(H.build_instance(H.small("mla_32", **kw)))


@pytest.mark.parametrize("name,kw", [
    ("qwen_gqa", dict(batch=3, lengths=("uniform", 500, 1500), dcp_size=2)),
    ("mla_32", dict(batch=3, lengths=("uniform", 500, 1500), dcp_size=2)),
    ("tiny_gqa", dict(batch=3, lengths=("uniform", 200, 600), dcp_size=2, head_dim_qk=96, head_dim_v=96)),
])
def test_block_id_past_the_pool_skips_its_unit(name, kw):
    from context_decode_attention_paged_gb300 import binding as dcp
    inst = H.build_instance(H.small(name, **kw))
    ref = H.oracle_decode(inst)
    nb = inst.kv_cache.shape[1] if inst.w.kind == "gqa" else inst.kv_cache.shape[0]
    inst.block_tables[1, 1, 1] = nb + 5              # shard 1 of request 1, its second block
    got = run_gpu(inst)
    assert got["status"] == dcp.DCP_ERR_BOUNDS
    assert (got["lse"][1, 1] == -np.inf).all()
    assert (got["partial_out"][1, 1] == 0).all()
    keep = np.ones(got["lse"].shape[:2], dtype=bool)
    keep[1, 1] = False
    assert_close(got["partial_out"][keep], ref["partial_out"][keep], "partial_out (other units)")
    assert_lse_close(got["lse"][keep], ref["lse"][keep], "lse (other units)")
