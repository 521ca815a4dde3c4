"""Seeded synthetic workloads for DCP decode attention.

This module only draws random numbers and lays them out in the paged-cache
format.  It holds none of the method's arithmetic: the number of cache blocks
each shard needs is an *input* (``local_num_blocks``), computed by whoever calls
it (the library's own slot-map call in the benchmark, the CPU oracle in tests).

Workloads (shapes, distributions, seeds) follow the pages' settings:
* "vLLM Decode Context Parallelism blog", section "性能基準測試": an agentic
  long-context trace with a median input of about 67k tokens; the trace itself
  is not available, so log-normal lengths with that median stand in for it;
* same page, sections on the MLA and GQA backends: DeepSeek-style MLA (one
  shared latent KV head) and Qwen3-235B-style GQA shapes;
* same page, "未來發展藍圖" / speculative decoding with MTP: 1 + 3 speculative
  tokens, causal within the four (query length 4).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "gqa" or "mla"
    batch: int
    q_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    block_size: int
    dcp_size: int
    interleave: int
    scale: float
    std: float                # standard deviation of q and of the cache values
    lengths: tuple            # ("fixed", S) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    permute_blocks: bool
    seed: int
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_gqa": Workload(
        "tiny_gqa", "gqa", batch=1, q_len=1, num_q_heads=8, num_kv_heads=2,
        head_dim_qk=64, head_dim_v=64, block_size=16, dcp_size=2, interleave=16,
        scale=1.0 / 8.0, std=1.0, lengths=("fixed", 1024), permute_blocks=False,
        seed=1000),
    "qwen_gqa": Workload(
        "qwen_gqa", "gqa", batch=64, q_len=1, num_q_heads=64, num_kv_heads=4,
        head_dim_qk=128, head_dim_v=128, block_size=128, dcp_size=4, interleave=128,
        scale=1.0 / math.sqrt(128.0), std=1.0, lengths=("uniform", 8192, 32768),
        permute_blocks=True, seed=1001),
    "mla_32": Workload(
        "mla_32", "mla", batch=32, q_len=1, num_q_heads=128, num_kv_heads=1,
        head_dim_qk=576, head_dim_v=512, block_size=128, dcp_size=8, interleave=128,
        scale=1.0 / math.sqrt(192.0), std=0.5,
        lengths=("lognormal", 67000, 0.25, 4096, 200000), permute_blocks=True, seed=1002),
    "mla_mtp": Workload(
        "mla_mtp", "mla", batch=1, q_len=4, num_q_heads=128, num_kv_heads=1,
        head_dim_qk=576, head_dim_v=512, block_size=128, dcp_size=8, interleave=1,
        scale=1.0 / math.sqrt(192.0), std=0.5, lengths=("fixed", 200000),
        permute_blocks=True, seed=1003),
    "mla_512": Workload(
        "mla_512", "mla", batch=512, q_len=1, num_q_heads=128, num_kv_heads=1,
        head_dim_qk=576, head_dim_v=512, block_size=128, dcp_size=8, interleave=128,
        scale=1.0 / math.sqrt(192.0), std=0.5,
        lengths=("lognormal", 67000, 0.25, 4096, 200000), permute_blocks=True, seed=1004),
    # chunked prefill under DCP: 64 causal query tokens per request attend to
    # the sharded cache; the 64 queries of a shard read the same keys
    "mla_chunk64": Workload(
        "mla_chunk64", "mla", batch=4, q_len=64, num_q_heads=128, num_kv_heads=1,
        head_dim_qk=576, head_dim_v=512, block_size=128, dcp_size=8, interleave=128,
        scale=1.0 / math.sqrt(192.0), std=0.5,
        lengths=("lognormal", 67000, 0.25, 4096, 200000), permute_blocks=True, seed=1006),
    # length stress variant of mla_512: log-normal sigma 1.0 (same median and
    # clip), ~51 GB of cache; reported beside the main workload
    "mla_512_s1": Workload(
        "mla_512_s1", "mla", batch=512, q_len=1, num_q_heads=128, num_kv_heads=1,
        head_dim_qk=576, head_dim_v=512, block_size=128, dcp_size=8, interleave=128,
        scale=1.0 / math.sqrt(192.0), std=0.5,
        lengths=("lognormal", 67000, 1.0, 4096, 200000), permute_blocks=True, seed=1005),
}


def make_seq_lens(w: Workload) -> torch.Tensor:
    """int32 [B] context lengths (each includes the q_len query tokens)."""
    g = torch.Generator().manual_seed(w.seed)
    kind = w.lengths[0]
    if kind == "fixed":
        s = torch.full((w.batch,), int(w.lengths[1]), dtype=torch.int64)
    elif kind == "uniform":
        lo, hi = w.lengths[1], w.lengths[2]
        s = torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64)
    elif kind == "lognormal":
        median, sigma, lo, hi = w.lengths[1:]
        z = torch.randn((w.batch,), generator=g, dtype=torch.float64)
        s = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi).to(torch.int64)
    else:
        raise ValueError(kind)
    return s.to(torch.int32)


def cache_shape(w: Workload, num_blocks: int) -> tuple:
    if w.kind == "gqa":
        return (2, num_blocks, w.block_size, w.num_kv_heads, w.head_dim_qk)
    return (num_blocks, w.block_size, w.head_dim_qk)


def _normal_bf16(shape, std, gen, device) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16; chunked along dim 0 to bound memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    chunk = 1 << 27
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn((e - s,), generator=gen, dtype=torch.float32, device=device)
        flat[s:e] = (x * std).to(torch.bfloat16)
    return out


@dataclass
class Instance:
    """One generated input set (all tensors on ``device``)."""
    w: Workload
    seq_lens: torch.Tensor        # int32 [B]
    q: torch.Tensor               # bf16 [B][Lq][Hq][Dqk]
    kv_cache: torch.Tensor        # bf16, gqa [2][nb][bs][Hkv][D] / mla [nb][bs][Dqk]
    block_tables: torch.Tensor    # int32 [N][B][max_local_blocks]
    local_num_blocks: torch.Tensor  # int32 [N][B] (the input it was built from)


def make_instance(w: Workload, local_num_blocks, device="cpu", seq_lens=None) -> Instance:
    """Draw q and the paged cache, and lay out block tables.

    ``local_num_blocks`` [N][B] is how many cache blocks shard r needs for
    sequence b.  Block ids are handed out in (r, b, j) order, through a random
    permutation of the pool when ``w.permute_blocks``; unused table entries are 0.
    """
    if seq_lens is None:
        seq_lens = make_seq_lens(w)
    lnb = torch.as_tensor(local_num_blocks, dtype=torch.int64).cpu()
    N, B = w.dcp_size, w.batch
    assert tuple(lnb.shape) == (N, B)
    total = int(lnb.sum())
    max_lb = max(1, int(lnb.max()))
    g_host = torch.Generator().manual_seed(w.seed + 7)
    ids = torch.randperm(total, generator=g_host) if w.permute_blocks else torch.arange(total)
    tables = torch.zeros((N, B, max_lb), dtype=torch.int32)
    pos = 0
    for r in range(N):
        for b in range(B):
            n = int(lnb[r, b])
            tables[r, b, :n] = ids[pos:pos + n].to(torch.int32)
            pos += n
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(w.seed + 11)
    q = _normal_bf16((B, w.q_len, w.num_q_heads, w.head_dim_qk), w.std, gen, dev)
    kv = _normal_bf16(cache_shape(w, max(total, 1)), w.std, gen, dev)
    return Instance(w, seq_lens.to(dev), q, kv, tables.to(dev), lnb.to(torch.int32))
