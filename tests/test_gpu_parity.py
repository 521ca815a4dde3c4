"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Sizes are small enough for the oracle to finish in seconds but span several
kernel tiles and a ragged tail; edge cases cover empty shards, a single token,
seq_len == q_len, interleave 1 and interleave >= seq_len.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import helpers as H
from gpu_common import check_against_oracle, run_gpu
from oracle import dcp_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()


# ---------------------------------------------------------------------------
# a1: slot map, bit-exact
# ---------------------------------------------------------------------------

SLOT_CASES = [
    ([1024], 16, 2, 16),
    ([1, 2, 3, 17, 128, 129, 1000], 16, 2, 16),
    ([200000], 1, 8, 128),
    ([200000], 50000, 4, 128),
    ([5, 300, 64], 1000, 4, 16),
    ([8192, 32768, 12345], 128, 4, 128),
    ([0, 7, 4096], 7, 3, 5),
]


@pytest.mark.parametrize("lens,I,N,bs", SLOT_CASES)
def test_slot_map_bit_exact(lens, I, N, bs):
    from context_decode_attention_paged_gb300 import binding as dcp
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    max_seq = max(lens) + 3
    lsl, lnb, shard, local = dcp.dcp_build_slot_map(sl, bs, I, N, max_seq=max_seq)
    torch.cuda.synchronize()
    assert dcp.dcp_get_last_device_status() == dcp.DCP_OK
    ref = orc.ref_slot_map(lens, I, N, bs)
    assert np.array_equal(lsl.cpu().numpy(), ref["local_seq_lens"])
    assert np.array_equal(lnb.cpu().numpy(), ref["local_num_blocks"])
    rs = np.full((len(lens), max_seq), -1, dtype=np.int32)
    rl = np.full((len(lens), max_seq), -1, dtype=np.int32)
    rs[:, : ref["shard_of"].shape[1]] = ref["shard_of"]
    rl[:, : ref["local_pos"].shape[1]] = ref["local_pos"]
    assert np.array_equal(shard.cpu().numpy(), rs)
    assert np.array_equal(local.cpu().numpy(), rl)


def test_slot_map_negative_len_sets_bounds_status():
    from context_decode_attention_paged_gb300 import binding as dcp
    sl = torch.tensor([5, -3], dtype=torch.int32, device="cuda")
    lsl, lnb, _, _ = dcp.dcp_build_slot_map(sl, 16, 4, 2)
    assert dcp.dcp_get_last_device_status() == dcp.DCP_ERR_BOUNDS
    assert lsl.cpu()[:, 1].tolist() == [0, 0]
    assert dcp.dcp_get_last_device_status() == dcp.DCP_OK   # cleared by the read


# ---------------------------------------------------------------------------
# a3-a6: attention + merge
# ---------------------------------------------------------------------------

ATTN_CASES = [
    ("tiny_gqa", {}),                                                  # the full tiny config
    ("tiny_gqa", dict(batch=3, lengths=("uniform", 1, 700), dcp_size=4, interleave=3)),
    ("tiny_gqa", dict(lengths=("fixed", 40), dcp_size=4, interleave=64)),   # empty shards
    ("tiny_gqa", dict(batch=2, q_len=3, lengths=("uniform", 3, 300))),      # causal Lq=3
    ("tiny_gqa", dict(lengths=("fixed", 1))),                               # single token
    ("qwen_gqa", dict(batch=2, lengths=("uniform", 300, 2000), dcp_size=4)),
    ("qwen_gqa", dict(batch=1, q_len=2, lengths=("fixed", 1153), dcp_size=2, interleave=1)),
    ("mla_32", dict(batch=2, lengths=("uniform", 900, 3000))),
    ("mla_32", dict(batch=1, lengths=("fixed", 129), dcp_size=2, interleave=128)),
    ("mla_mtp", dict(lengths=("fixed", 2500))),
    ("mla_mtp", dict(lengths=("fixed", 4))),                                # S == Lq
    ("mla_mtp", dict(lengths=("fixed", 300), dcp_size=1)),
    ("mla_mtp", dict(lengths=("fixed", 40000))),                            # KV splits + combine
    ("mla_32", dict(batch=3, lengths=("uniform", 1, 700), dcp_size=4, interleave=3)),
    # GQA tensor-core kernel: one and two 64-row query tiles (Lq 4 and 8 x 16 heads)
    ("qwen_gqa", dict(batch=2, q_len=4, lengths=("uniform", 200, 1500), dcp_size=2)),
    ("qwen_gqa", dict(batch=1, q_len=8, lengths=("fixed", 3000), dcp_size=2, interleave=64)),
    # long causal queries (chunked prefill): several 64-row tiles per KV head
    ("qwen_gqa", dict(batch=2, q_len=16, lengths=("uniform", 300, 1500), dcp_size=2)),
    ("qwen_gqa", dict(batch=1, q_len=40, lengths=("fixed", 2100), dcp_size=4, interleave=64)),
    ("tiny_gqa", dict(batch=2, q_len=64, lengths=("uniform", 64, 900), dcp_size=2, interleave=16)),
    # head dims without a tensor-core kernel run on the generic SIMT kernel
    ("tiny_gqa", dict(head_dim_qk=96, head_dim_v=96, lengths=("fixed", 500))),
    # GQA block sizes: several TMA boxes per 128-key tile (8, 32, 64), a block
    # spanning two tiles (256), and one the tensor-core kernel declines (48)
    ("qwen_gqa", dict(batch=2, block_size=8, lengths=("uniform", 300, 1300), dcp_size=2)),
    ("qwen_gqa", dict(batch=2, block_size=32, lengths=("uniform", 300, 1300), dcp_size=4, interleave=32)),
    ("qwen_gqa", dict(batch=2, block_size=64, lengths=("uniform", 700, 2000), dcp_size=2, interleave=64)),
    ("qwen_gqa", dict(batch=2, block_size=256, lengths=("uniform", 700, 3000), dcp_size=2, interleave=256)),
    ("tiny_gqa", dict(block_size=48, lengths=("fixed", 700), dcp_size=2, interleave=48)),
    # MLA block sizes: one TMA box per block in a 64-key tile (8, 16, 32), one
    # block per tile (64), a block spanning four tiles (256), with ragged tails
    # and a KV split; 48 is declined by the tensor-core kernel
    ("mla_32", dict(batch=2, block_size=8, lengths=("uniform", 300, 1300), dcp_size=2, interleave=8)),
    ("mla_32", dict(batch=2, block_size=16, lengths=("uniform", 300, 1300), dcp_size=4, interleave=1)),
    ("mla_32", dict(batch=3, block_size=32, q_len=2, lengths=("uniform", 200, 2000), dcp_size=2,
                    interleave=32)),
    ("mla_32", dict(batch=2, block_size=64, lengths=("uniform", 700, 3000), dcp_size=2, interleave=64)),
    ("mla_32", dict(batch=1, block_size=64, lengths=("fixed", 9000), dcp_size=1)),
    ("mla_32", dict(batch=2, block_size=256, lengths=("uniform", 700, 3000), dcp_size=2, interleave=256)),
    ("mla_32", dict(batch=2, block_size=48, lengths=("uniform", 100, 700), dcp_size=2, interleave=48)),
    # MLA with fewer query heads per rank (the MMA rows past Hq hold other
    # queries' rows, computed and discarded), odd counts included
    ("mla_32", dict(batch=3, num_q_heads=64, lengths=("uniform", 300, 2000), dcp_size=4)),
    ("mla_32", dict(batch=2, num_q_heads=16, q_len=4, lengths=("uniform", 300, 1500), dcp_size=2,
                    interleave=1)),
    ("mla_32", dict(batch=3, num_q_heads=40, lengths=("uniform", 700, 3000), dcp_size=8)),
    # combinations: a batch ordered by the pre-pass with 64 heads; 16-token
    # blocks under causal MTP queries at interleave 1; 32 heads with KV splits
    # (a long single request) and their combine
    ("mla_32", dict(batch=130, num_q_heads=64, lengths=("uniform", 64, 400), dcp_size=2)),
    ("mla_32", dict(batch=2, block_size=16, q_len=4, lengths=("uniform", 500, 2500), dcp_size=4,
                    interleave=1)),
    ("mla_mtp", dict(num_q_heads=32, lengths=("fixed", 40000), dcp_size=8)),
    # group sizes: 1 (one real row of a 16-row tile) and 8 with Lq 3 (24 rows of a 32-row tile)
    ("qwen_gqa", dict(batch=2, num_q_heads=8, num_kv_heads=8, lengths=("uniform", 300, 900), dcp_size=2)),
    ("qwen_gqa", dict(batch=2, num_q_heads=32, num_kv_heads=4, q_len=3, lengths=("uniform", 300, 900),
                      dcp_size=4)),
    ("mla_32", dict(batch=2, num_q_heads=16, head_dim_qk=72, head_dim_v=64,
                    lengths=("uniform", 100, 900), dcp_size=4)),
]


@pytest.mark.parametrize("name,kw", ATTN_CASES)
def test_attention_matches_oracle(name, kw):
    inst = H.build_instance(H.small(name, **kw))
    check_against_oracle(inst)


GROWING_CASES = [
    ("qwen_gqa", dict(batch=2, lengths=("uniform", 1500, 4000), dcp_size=2)),
    ("qwen_gqa", dict(batch=1, q_len=4, lengths=("fixed", 3000), dcp_size=2, interleave=64)),
    ("tiny_gqa", dict(batch=2, lengths=("uniform", 700, 1500), dcp_size=2, interleave=16)),
    ("mla_32", dict(batch=2, lengths=("uniform", 2000, 5000), dcp_size=4)),
]


@pytest.mark.parametrize("name,kw", GROWING_CASES)
def test_attention_with_scores_growing_along_the_sequence(name, kw):
    """GQA keys scaled up to 8x (16x in a spike near the end): each row's running
    max moves past its lazy-rescale threshold in later tiles, not only the first.
    The values keep the workload's scale (N(0,1)), so the peaked softmaxes put
    the dominant probabilities' rounding straight into the output.  MLA grows
    only its 64 rope dims (up to 16x, no spike), which leaves the values (the
    latent) alone.  A wrong rescale errs by the size of the output itself."""
    inst = H.build_instance(H.small(name, **kw))

    def factor(u):
        return np.where(u > 0.97, 16.0, 1.0 + 7.0 * u * u)

    if inst.w.kind == "gqa":
        H.scale_keys_by_position(inst, factor)
    else:
        H.scale_keys_by_position(inst, lambda u: 1.0 + 15.0 * u * u, key_dims=slice(inst.w.head_dim_v, None))
    check_against_oracle(inst)


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_mtp_merge_invariance_sweep(N):
    """MTP verify (Lq 4, interleave 1): merged output equals the oracle at every dcp_size."""
    w = H.small("mla_mtp", lengths=("fixed", 1500), dcp_size=N)
    check_against_oracle(H.build_instance(w))


def test_seq_shorter_than_query_sets_bounds_status():
    from context_decode_attention_paged_gb300 import binding as dcp
    w = H.small("tiny_gqa", batch=2, q_len=4, lengths=("fixed", 64))
    inst = H.build_instance(w)
    inst.seq_lens[1] = 2                       # shorter than its 4 query tokens
    got = run_gpu(inst)
    assert got["status"] == dcp.DCP_ERR_BOUNDS
    assert (got["lse"][:, 1] == -np.inf).all()
    assert np.isfinite(got["lse"][:, 0]).all()
