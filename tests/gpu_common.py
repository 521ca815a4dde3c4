"""Shared pieces of the GPU parity tests: run the library on an instance and
compare with the oracle under the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

from oracle import dcp_oracle as orc
import helpers as H

# Tolerances of the target statement: bf16 inputs, fp32 accumulation.
OUT_ABS = 2e-3      # absolute part of the element-wise bound
OUT_REL = 1e-2      # relative part: |err| <= OUT_ABS + OUT_REL * |ref|
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
    status = dcp.dcp_get_last_device_status(stream)
    return {"partial_out": po.cpu().numpy(), "lse": lse.cpu().numpy(),
            "out": out.float().cpu().numpy(), "out_lse": out_lse.cpu().numpy(),
            "status": status}


def assert_close(got, ref, what, abs_tol=OUT_ABS, rel_tol=OUT_REL):
    """Element-wise |got - ref| <= abs_tol + rel_tol * |ref| (numpy allclose form).

    A flat 2e-3 bound alone is finer than bf16 itself for |out| >= 0.5 (half
    an ulp there is 2^-9 * 2^e >= 1e-3), so the relative term carries the large
    values and the absolute term the small ones.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if not got.size:
        return 0.0
    err = np.abs(got - ref)
    bound = abs_tol + rel_tol * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (
        f"{what}: |err| {err[worst]:.3e} > {bound[worst]:.3e} at {worst} "
        f"(got {got[worst]:.6g}, ref {ref[worst]:.6g}); max-abs {err.max():.3e}")
    return float(err.max())


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
