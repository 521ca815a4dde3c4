"""Shared pieces of the GPU parity tests: run the library on an instance and
compare with the oracle under the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

from oracle import dcp_oracle as orc
import helpers as H

# Tolerances of the target statement: bf16 inputs, fp32 accumulation.
OUT_ABS = 2e-3      # max-abs error of outputs
OUT_REL = 1e-2      # max-abs error relative to the largest |reference| value
LSE_ABS = 1e-3


def run_gpu(inst, dcp_size=None, interleave=None, stream=None):
    from context_decode_attention_paged_gb300 import binding as dcp
    w = inst.w
    N = dcp_size or w.dcp_size
    I = interleave or w.interleave
    dev = torch.device("cuda:0")
    q, kv = inst.q.to(dev), inst.kv_cache.to(dev)
    bt, sl = inst.block_tables.to(dev), inst.seq_lens.to(dev)
    po, lse = dcp.dcp_decode_attn(w.kind, q, kv, bt, sl, N, I, w.scale, w.q_len, w.head_dim_v,
                                  stream=stream)
    out, out_lse = dcp.dcp_merge(po, lse, N, stream=stream)
    torch.cuda.synchronize()
    status = dcp.dcp_get_last_device_status()
    return {"partial_out": po.cpu().numpy(), "lse": lse.cpu().numpy(),
            "out": out.float().cpu().numpy(), "out_lse": out_lse.cpu().numpy(),
            "status": status}


def assert_close(got, ref, what, abs_tol=OUT_ABS, rel_tol=OUT_REL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref).max() if got.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err <= abs_tol, f"{what}: max-abs error {err:.3e} > {abs_tol:.1e}"
    if scale > 0:
        assert err / scale <= rel_tol, f"{what}: relative error {err / scale:.3e} > {rel_tol:.1e}"
    return err


def assert_lse_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ninf_g, ninf_r = got == -np.inf, ref == -np.inf
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    assert np.isfinite(got[fin]).all(), f"{what}: non-finite values"
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    assert err <= LSE_ABS, f"{what}: LSE error {err:.3e} > {LSE_ABS:.1e}"
    return err


def check_against_oracle(inst, check_partials=True):
    from context_decode_attention_paged_gb300 import binding as dcp
    got = run_gpu(inst)
    assert got["status"] == dcp.DCP_OK, dcp.status_string(got["status"])
    ref = H.oracle_decode(inst)
    e_out = assert_close(got["out"], ref["out"], "out")
    e_lse = assert_lse_close(got["out_lse"], ref["out_lse"], "out_lse")
    if check_partials:
        assert_close(got["partial_out"], ref["partial_out"], "partial_out")
        assert_lse_close(got["lse"], ref["lse"], "lse")
    return e_out, e_lse
