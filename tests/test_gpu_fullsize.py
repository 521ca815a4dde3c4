"""GPU parity at the full sizes of the workload configurations, in the launch
configuration bench.py times.

The whole decode step (all shards, one attention launch, one merge launch) runs
on the device over the full synthetic workload, generated exactly as the
benchmark generates it.  Every request (at batch 512 a seeded 64 of the 512,
always including the longest and the shortest) is
then checked element by element against the oracle, run a few requests at a
time on a compact host copy of their cache blocks; properties that hold at any size are checked on
every output: everything finite, every partial LSE finite (every shard of these
workloads has keys), and every output bounded by the largest |entry| of the
value cache (the output is a convex combination of value rows).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
from context_decode_attention_paged_gb300 import workloads as wl
from gpu_common import assert_close, assert_lse_close
from oracle import dcp_oracle as orc

pytestmark = pytest.mark.gpu

FULL = ["qwen_gqa", "mla_32", "mla_mtp", "mla_512", "mla_512_s1", "mla_chunk64"]
# long query chunks: these query rows of every request are checked; query i
# at position S - Lq + i sees what a one-token decode of context S - Lq + i + 1
# sees, which keeps the oracle's work to a few decodes per request
CHUNK_ROWS = (0, 1, 31, 62, 63)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from context_decode_attention_paged_gb300 import build
    build.build()


def _checked_requests(w: wl.Workload):
    """Every request, except at batch 512: a seeded subset of 64 that always
    holds the longest and the shortest request."""
    if w.batch <= 64:
        return list(range(w.batch))
    rng = np.random.default_rng(20260 + w.batch)
    idx = set(rng.choice(w.batch, size=62, replace=False).tolist())
    lens = wl.make_seq_lens(w)
    idx.add(int(torch.argmax(lens)))
    idx.add(int(torch.argmin(lens)))
    while len(idx) < 64:
        idx.add(int(rng.integers(w.batch)))
    return sorted(idx)


@pytest.mark.parametrize("name", FULL)
def test_full_size_against_oracle(name):
    from context_decode_attention_paged_gb300 import binding as dcp
    w = wl.WORKLOADS[name]
    inst = bench.setup_gpu(w, 0)
    try:
        po, lse = dcp.dcp_decode_attn(w.kind, inst.q, inst.kv_cache, inst.block_tables, inst.seq_lens,
                                      w.dcp_size, w.interleave, w.scale, w.q_len, w.head_dim_v)
        out, out_lse = dcp.dcp_merge(po, lse, w.dcp_size)
        torch.cuda.synchronize()
        assert dcp.dcp_get_last_device_status() == dcp.DCP_OK

        # properties over every output
        assert torch.isfinite(po).all() and torch.isfinite(lse).all()
        assert torch.isfinite(out.float()).all() and torch.isfinite(out_lse).all()
        vals = inst.kv_cache[1] if w.kind == "gqa" else inst.kv_cache     # (MLA: latent and rope)
        vmax = torch.maximum(vals.amax().float().abs(), vals.amin().float().abs())
        assert out.float().abs().max() <= vmax * (1 + 1e-2)

        # requests element by element, a few at a time (bounded host memory)
        idx_all = _checked_requests(w)
        if w.q_len > 4:
            _check_chunk_rows(w, inst, po, lse, out, out_lse, idx_all)
            return
        for c0 in range(0, len(idx_all), 8):
            idx = idx_all[c0:c0 + 8]
            q, kv, bt, sl = bench.host_sample(inst, idx)
            ref = orc.ref_dcp_decode(w.kind, orc.to_f64(q), orc.to_f64(kv), bt, sl, w.dcp_size, w.interleave,
                                     w.block_size, w.scale, w.q_len, w.head_dim_v)
            sel = torch.as_tensor(idx, device=po.device)
            tag = f"{name} requests {idx[0]}..{idx[-1]}"
            assert_close(out.index_select(1, sel).float().cpu().numpy(), ref["out"], f"{tag} out")
            assert_lse_close(out_lse.index_select(1, sel).cpu().numpy(), ref["out_lse"], f"{tag} out_lse")
            assert_close(po.index_select(1, sel).cpu().numpy(), ref["partial_out"], f"{tag} partial_out")
            assert_lse_close(lse.index_select(1, sel).cpu().numpy(), ref["lse"], f"{tag} lse")
    finally:
        del inst
        torch.cuda.empty_cache()


def _check_chunk_rows(w, inst, po, lse, out, out_lse, idx_all):
    """Sampled query rows of a long causal chunk, each against the oracle's
    one-token decode of the context that row sees."""
    for b in idx_all:
        q, kv, bt, sl = bench.host_sample(inst, [b])
        for i in CHUNK_ROWS:
            s_i = np.array([int(sl[0]) - w.q_len + i + 1], dtype=sl.dtype)
            ref = orc.ref_dcp_decode(w.kind, orc.to_f64(q[:, i:i + 1]), orc.to_f64(kv), bt, s_i, w.dcp_size,
                                     w.interleave, w.block_size, w.scale, 1, w.head_dim_v)
            tag = f"{w.name} request {b} query {i}"
            assert_close(out[:, b:b + 1, i:i + 1].float().cpu().numpy(), ref["out"], f"{tag} out")
            assert_lse_close(out_lse[:, b:b + 1, i:i + 1].cpu().numpy(), ref["out_lse"], f"{tag} out_lse")
            assert_close(po[:, b:b + 1, i:i + 1].cpu().numpy(), ref["partial_out"], f"{tag} partial_out")
            assert_lse_close(lse[:, b:b + 1, i:i + 1].cpu().numpy(), ref["lse"], f"{tag} lse")
