"""The seeded length mixes follow their stated distributions (CPU only).

The blog's agentic trace (median input ~67k tokens, "性能基準測試") is not
available; log-normal lengths with that median stand in for it.  These checks pin
the generator's parameters, not the method.
"""

import math

import torch

from context_decode_attention_paged_gb300 import workloads as wl


def _log_stats(name):
    w = wl.WORKLOADS[name]
    s = wl.make_seq_lens(w).to(torch.float64)
    lo, hi = w.lengths[3], w.lengths[4]
    assert int(s.min()) >= lo and int(s.max()) <= hi
    ls = torch.log(s)
    return w, s, float(ls.median()), float(ls.std())


def test_mla_512_lengths_are_lognormal_with_the_trace_median():
    w, s, med, sd = _log_stats("mla_512")
    assert abs(med - math.log(67000)) < 0.05
    assert abs(sd - 0.25) < 0.03
    kv_gb = float(s.sum()) * w.head_dim_qk * 2 / 1e9
    assert 38.0 < kv_gb < 43.0            # "~40 GB" of latent cache


def test_stress_variant_has_sigma_one_and_the_same_median():
    w, s, med, sd = _log_stats("mla_512_s1")
    assert abs(med - math.log(67000)) < 0.25
    assert 0.8 < sd < 1.05                # clipping at [4096, 200000] trims the tails
    base = wl.WORKLOADS["mla_512"]
    same = ("kind", "batch", "q_len", "num_q_heads", "head_dim_qk", "head_dim_v", "block_size",
            "dcp_size", "interleave", "scale", "std")
    assert all(getattr(w, f) == getattr(base, f) for f in same)


def test_seeds_are_distinct():
    seeds = [w.seed for w in wl.WORKLOADS.values()]
    assert len(seeds) == len(set(seeds))
