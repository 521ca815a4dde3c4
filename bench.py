"""Benchmark: DCP-sharded decode attention + LSE merge on one GB300.

One step = dcp_decode_attn (all shards) + dcp_merge over one decode batch of
the named workload (default: MLA, batch 512, Lq 1, dcp_size 8, interleave 128,
log-normal context lengths with median 67k; about 40 GB of bf16 latent cache).
The cache is resident in HBM; the default one is far larger than L2, so steps
run back to back.  A cache under 4x L2 (the MTP and tiny workloads) gets a
1 GB write before each timed step so that no step is served from L2.  Prints
one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Metric: KV-cache GB/s (algorithmic cache bytes of the step / step time), with
the step's fraction of its HBM/tensor roofline and query-tokens/s alongside.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from context_decode_attention_paged_gb300 import workloads as wl  # noqa: E402

METRIC = "KV GB/s & % roofline, DCP-sharded MLA/GQA decode attn + LSE merge, 1xGB300"
L2_FLUSH_BELOW = 4 * 129e6          # flush L2 between steps when the cache is smaller than 4x L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# roofline arithmetic (per unit of work: cache bytes per token, fixed bytes per launch)
# ---------------------------------------------------------------------------

def kv_bytes_per_token(w: wl.Workload) -> int:
    """Cache bytes one token contributes (MLA: the value is a prefix of the key row)."""
    if w.kind == "mla":
        return w.head_dim_qk * 2
    return w.num_kv_heads * (w.head_dim_qk + w.head_dim_v) * 2


def visible_keys(w: wl.Workload, seq_lens) -> int:
    """Sum over (b, i) of keys query i sees (S - Lq + i + 1)."""
    s = np.asarray(seq_lens, dtype=np.int64)
    return int(sum((s - w.q_len + i + 1).sum() for i in range(w.q_len)))


def algorithmic(w: wl.Workload, seq_lens) -> dict:
    B, Lq, Hq, N = w.batch, w.q_len, w.num_q_heads, w.dcp_size
    tokens = int(np.asarray(seq_lens, dtype=np.int64).sum())
    kv = tokens * kv_bytes_per_token(w)
    q = B * Lq * Hq * w.head_dim_qk * 2
    partials = N * B * Lq * Hq * (w.head_dim_v + 1) * 4          # written once, read once
    out = B * Lq * Hq * w.head_dim_v * 2 + B * Lq * Hq * 4
    flops = 2 * (w.head_dim_qk + w.head_dim_v) * Hq * visible_keys(w, seq_lens)
    return {"kv_bytes": kv, "tokens": tokens,
            "attn_bytes": kv + q + partials,                       # the attention kernel
            "merge_bytes": partials + out,
            "step_bytes": kv + q + 2 * partials + out,
            "flops": flops}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one attention
# launch, as a multiple of its algorithmic bytes, from an ncu capture of a
# smaller case of the same kernel (traffic scales with the cache bytes
# processed): MLA from the batch-32 workload, GQA from the Qwen-like one, and
# the 64-token chunk workload from its own capture (its 64 queries per shard
# share the key stream through L2, so its ratio differs).  Keyed by the kernel
# source the counters were taken on: once the source changes, traffic is
# reported as null.
NCU_TRAFFIC_RATIO = {
    "mla": ("08235e44124c0ac7", 1.00528, "attn_mla_tc.cu"),
    "gqa": ("f6e04d4ccaedbfff", 1.00386, "attn_gqa_tc.cu"),
    "mla_chunk64": ("08235e44124c0ac7", 1.03412, "attn_mla_tc.cu"),
}


def measured_traffic(w: wl.Workload, alg_bytes: int):
    sha, ratio, fname = NCU_TRAFFIC_RATIO.get(w.name, NCU_TRAFFIC_RATIO[w.kind])
    path = os.path.join(ROOT, "context_decode_attention_paged_gb300", "csrc", fname)
    with open(path, "rb") as f:
        cur = hashlib.sha256(f.read()).hexdigest()[:16]
    return int(round(ratio * alg_bytes)) if cur == sha else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload set-up (GPU leg): block counts come from the library's slot map
# ---------------------------------------------------------------------------

def setup_gpu(w: wl.Workload, rank: int):
    from context_decode_attention_paged_gb300 import binding as dcp
    seq_lens = wl.make_seq_lens(w)
    sl_dev = seq_lens.cuda()
    _, lnb, _, _ = dcp.dcp_build_slot_map(sl_dev, w.block_size, w.interleave, w.dcp_size)
    torch.cuda.synchronize()
    inst = wl.make_instance(w, lnb.cpu(), device="cuda", seq_lens=seq_lens)
    return inst


def step_fn(inst, po, lse, out, out_lse, ws):
    from context_decode_attention_paged_gb300 import binding as dcp
    w = inst.w

    def attn():
        dcp.dcp_decode_attn(w.kind, inst.q, inst.kv_cache, inst.block_tables, inst.seq_lens,
                            w.dcp_size, w.interleave, w.scale, w.q_len, w.head_dim_v,
                            partial_out=po, lse=lse, workspace=ws)

    def merge():
        dcp.dcp_merge(po, lse, w.dcp_size, out=out, out_lse=out_lse)

    return attn, merge


def kv_write_timing(inst, reps: int):
    """dcp_kv_cache_write of one decode step's new tokens (B x Lq rows), timed on
    its own with CUDA events (the step before attention; not part of `value`)."""
    from context_decode_attention_paged_gb300 import binding as dcp
    w = inst.w
    dev = inst.kv_cache.device
    g = torch.Generator(device=dev).manual_seed(w.seed + 7)
    if w.kind == "gqa":
        shape = (w.batch, w.q_len, w.num_kv_heads, w.head_dim_qk)
        new_k = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
        new_v = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
        row_bytes = 2 * w.num_kv_heads * w.head_dim_qk * 2          # K and V rows of a token
    else:
        new_k = torch.randn((w.batch, w.q_len, w.head_dim_qk), generator=g, device=dev).to(torch.bfloat16)
        new_v = None
        row_bytes = w.head_dim_qk * 2

    def call():
        dcp.dcp_kv_cache_write(w.kind, new_k, new_v, inst.kv_cache, inst.block_tables, inst.seq_lens,
                               w.dcp_size, w.interleave)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    st = dcp.dcp_get_last_device_status()
    if st != dcp.DCP_OK:
        raise RuntimeError(f"device status after the cache write: {dcp.status_string(st)}")
    ms = e0.elapsed_time(e1) / reps
    rows = w.batch * w.q_len
    alg = 2 * rows * row_bytes                                          # rows read + cells written
    return {"kernel": "dcp_kv_cache_write", "ms_per_call": round(ms, 5), "tokens": rows,
            "alg_bytes": alg, "achieved_gbs": round(alg / (ms * 1e-3) / 1e9, 2),
            "reps": reps, "bound": "launch latency (a step writes a few hundred KB)"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as td
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if td.get_backend() == "nccl" else "cpu")
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(local_units: float, local_ms: float, world: int):
    """Weak scaling: every rank runs its own full workload, so the job's rate is
    the units of all ranks over the slowest rank's time.  Returns (units per
    second, slowest ms)."""
    ms = max_over_ranks(local_ms, world)
    return sum_over_ranks(float(local_units), world) / (ms * 1e-3), ms


def rank_workload(name: str, rank: int) -> wl.Workload:
    """Rank r's workload: the named configuration with its own seed (same
    shapes and length distribution, different draws)."""
    w = wl.WORKLOADS[name]
    return w.with_(seed=w.seed + rank)


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as td
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if td.get_backend() == "nccl" else "cpu")
    td.all_reduce(t, op=td.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as td
        td.barrier()


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def host_sample(inst, idx):
    """q, a compact host copy of the blocks the sampled requests use, remapped
    block tables and lengths for the requests ``idx``."""
    w = inst.w
    bt = inst.block_tables.cpu()[:, idx]                     # [N][b][max_lb]
    sl = inst.seq_lens.cpu()[idx]
    from oracle import dcp_oracle as orc
    used, tables = [], torch.zeros_like(bt)
    for r in range(w.dcp_size):
        for k, b in enumerate(idx):
            n_local = len(orc.shard_token_lists(int(sl[k]), w.interleave, w.dcp_size)[r])
            nb = -(-n_local // w.block_size)
            ids = bt[r, k, :nb]
            tables[r, k, :nb] = torch.arange(len(used), len(used) + nb, dtype=torch.int32)
            used.extend(ids.tolist())
    ids = torch.tensor(used, dtype=torch.int64, device=inst.kv_cache.device)
    if w.kind == "gqa":
        kv = inst.kv_cache[:, ids].cpu()
    else:
        kv = inst.kv_cache[ids].cpu()
    q = inst.q[torch.as_tensor(idx, device=inst.q.device)].cpu()
    return q, kv, tables.numpy(), sl.numpy()


def oracle_time(inst, budget_s: float, max_seqs: int):
    """Run the oracle over requests 0, 1, ... until ``budget_s`` of CPU time;
    returns (seconds, cache bytes covered, requests, query tokens)."""
    from oracle import dcp_oracle as orc
    w = inst.w
    done, secs, kv_bytes, qtok = 0, 0.0, 0, 0
    while done < min(max_seqs, w.batch) and (secs < budget_s or done < 1):
        q, kv, bt, sl = host_sample(inst, [done])
        q64, kv64 = orc.to_f64(q), orc.to_f64(kv)
        t0 = time.perf_counter()
        orc.ref_dcp_decode(w.kind, q64, kv64, bt, sl, w.dcp_size, w.interleave, w.block_size,
                           w.scale, w.q_len, w.head_dim_v)
        secs += time.perf_counter() - t0
        kv_bytes += int(sl.sum()) * kv_bytes_per_token(w)
        qtok += w.q_len
        done += 1
    return secs, kv_bytes, done, qtok


def cpu_threads() -> int:
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = [i.get("num_threads") for i in info if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# main legs
# ---------------------------------------------------------------------------

# The other workload configurations, measured in the same run after the headline
# one and reported beside it (single GPU).
OTHER_CONFIGS = ("tiny_gqa", "qwen_gqa", "mla_32", "mla_mtp", "mla_chunk64")


def roofline_of(w, alg, attn_ms: float, peaks) -> dict:
    """Roofline record of the attention launch: HBM when its algorithmic bytes at
    the copy rate take longer than its flops at the bf16 rate, else tensor."""
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    gbs = alg["attn_bytes"] / (attn_ms * 1e-3) / 1e9
    tfs = alg["flops"] / (attn_ms * 1e-3) / 1e12
    if alg["attn_bytes"] / hbm >= alg["flops"] / (tflops * 1e3):
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4)}
    return {"bound": "tensor", "achieved": round(tfs, 1), "peak": tflops, "unit": "TFLOP/s",
            "frac": round(tfs / tflops, 4)}


def measure_config(name: str, steps: int, warmup: int, dev, peaks) -> dict:
    """One workload configuration, timed like the headline one: attention +
    merge per step, CUDA events on the launching stream, L2 flushed before each
    step when the cache is small enough to stay in it."""
    from context_decode_attention_paged_gb300 import binding as dcp
    w = wl.WORKLOADS[name]
    inst = setup_gpu(w, 0)
    N, B, Lq, Hq, Dv = w.dcp_size, w.batch, w.q_len, w.num_q_heads, w.head_dim_v
    po = torch.empty((N, B, Lq, Hq, Dv), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, Lq, Hq), dtype=torch.float32, device=dev)
    out = torch.empty((N, B, Lq, Hq // N, Dv), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty((N, B, Lq, Hq // N), dtype=torch.float32, device=dev)
    desc = dcp.desc_from_tensors(w.kind, inst.q, inst.kv_cache, inst.block_tables, Dv)
    ws_bytes = dcp.dcp_decode_attn_workspace_size(desc, N)
    ws = torch.empty((max(ws_bytes, 1),), dtype=torch.uint8, device=dev) if ws_bytes else None
    attn, merge = step_fn(inst, po, lse, out, out_lse, ws)
    alg = algorithmic(w, inst.seq_lens.cpu().numpy())
    for _ in range(warmup):
        attn()
        merge()
    torch.cuda.synchronize()
    flush = alg["kv_bytes"] <= L2_FLUSH_BELOW
    scratch = torch.empty((1 << 30,), dtype=torch.uint8, device=dev) if flush else None
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for k in range(steps):
        if flush:
            scratch.fill_(k & 0xFF)
        ev[k][0].record(stream)
        attn()
        ev[k][1].record(stream)
        merge()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    st = dcp.dcp_get_last_device_status()
    if st != dcp.DCP_OK:
        raise RuntimeError(f"{name}: device status {dcp.status_string(st)}")
    attn_ms = [e[0].elapsed_time(e[1]) for e in ev]
    step_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    attn_avg = statistics.mean(attn_ms)
    rec = {"workload": name, "kind": w.kind, "batch": B, "q_len": Lq, "dcp_size": N,
           "interleave": w.interleave, "kv_tokens": alg["tokens"], "kv_bytes": alg["kv_bytes"],
           "step_ms": round(step_ms, 4), "kv_gbs": round(alg["kv_bytes"] / (step_ms * 1e-3) / 1e9, 2),
           "query_tokens_per_s": round(B * Lq / (step_ms * 1e-3), 1),
           "attn_ms": round(attn_avg, 4), "attn_ms_median": round(statistics.median(attn_ms), 4),
           "alg_bytes_per_launch": alg["attn_bytes"], "alg_flops_per_launch": alg["flops"],
           "roofline": roofline_of(w, alg, attn_avg, peaks),
           "l2": "L2 flushed before each timed step (1 GB write, untimed)" if flush
           else "inputs larger than L2 (cache resident, no flush)",
           "steps": steps, "warmup": warmup}
    del inst, po, lse, out, out_lse, ws, scratch
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl")
    torch.cuda.set_device(local)
    from context_decode_attention_paged_gb300 import binding as dcp
    w = rank_workload(args.workload, rank)
    inst = setup_gpu(w, rank)
    N, B, Lq, Hq, Dv = w.dcp_size, w.batch, w.q_len, w.num_q_heads, w.head_dim_v
    dev = torch.device("cuda", local)
    po = torch.empty((N, B, Lq, Hq, Dv), dtype=torch.float32, device=dev)
    lse = torch.empty((N, B, Lq, Hq), dtype=torch.float32, device=dev)
    out = torch.empty((N, B, Lq, Hq // N, Dv), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty((N, B, Lq, Hq // N), dtype=torch.float32, device=dev)
    desc = dcp.desc_from_tensors(w.kind, inst.q, inst.kv_cache, inst.block_tables, Dv)
    ws_bytes = dcp.dcp_decode_attn_workspace_size(desc, N)
    ws = torch.empty((max(ws_bytes, 1),), dtype=torch.uint8, device=dev) if ws_bytes else None
    attn, merge = step_fn(inst, po, lse, out, out_lse, ws)
    launches_per_step = dcp.dcp_decode_attn_launches(desc, N) + 1          # + the merge
    alg = algorithmic(w, inst.seq_lens.cpu().numpy())

    for _ in range(args.warmup):
        attn()
        merge()
    torch.cuda.synchronize()
    st = dcp.dcp_get_last_device_status()
    if st != dcp.DCP_OK:
        raise RuntimeError(f"device status after warm-up: {dcp.status_string(st)}")

    stream = torch.cuda.current_stream()
    # a cache that fits a few times in L2 would be served from it on repeated
    # steps: write a 1 GB scratch buffer before each such step (outside its
    # timing) so every step reads HBM
    flush = alg["kv_bytes"] <= L2_FLUSH_BELOW
    scratch = torch.empty((1 << 30,), dtype=torch.uint8, device=dev) if flush else None
    barrier(world)
    torch.cuda.synchronize()
    if flush:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        with ClockSampler(local) as clocks:
            for k in range(args.steps):
                scratch.fill_(k & 0xFF)
                ev[k][0].record(stream)
                attn()
                ev[k][1].record(stream)
                merge()
                ev[k][2].record(stream)
            torch.cuda.synchronize()
        barrier(world)
        attn_ms = [e[0].elapsed_time(e[1]) for e in ev]
        merge_ms = [e[1].elapsed_time(e[2]) for e in ev]
        total_ms = sum(e[0].elapsed_time(e[2]) for e in ev)
        del scratch
    else:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps + 1)]
        with ClockSampler(local) as clocks:
            ev[0].record(stream)
            for k in range(args.steps):
                attn()
                ev[2 * k + 1].record(stream)
                merge()
                ev[2 * k + 2].record(stream)
            torch.cuda.synchronize()
        barrier(world)
        total_ms = ev[0].elapsed_time(ev[-1])
        attn_ms = [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(args.steps)]
        merge_ms = [ev[2 * k + 1].elapsed_time(ev[2 * k + 2]) for k in range(args.steps)]
    st = dcp.dcp_get_last_device_status()
    if st != dcp.DCP_OK:
        raise RuntimeError(f"device status after timing: {dcp.status_string(st)}")

    # e2e through the same calls with host buffers: every step copies its q,
    # block tables and lengths in from pinned memory and reads its merged
    # output back.  Two sets of step buffers let step k+1's upload and step
    # k-1's download run beside step k's kernels (one copy stream each way,
    # ordered by events); the timed region brackets every copy.
    q_h = inst.q.cpu().pin_memory()
    bt_h = inst.block_tables.cpu().pin_memory()
    sl_h = inst.seq_lens.cpu().pin_memory()
    sets = [(inst.q, inst.block_tables, inst.seq_lens, out, out_lse),
            (torch.empty_like(inst.q), torch.empty_like(inst.block_tables), torch.empty_like(inst.seq_lens),
             torch.empty_like(out), torch.empty_like(out_lse))]
    outs_h = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
               torch.empty(out_lse.shape, dtype=out_lse.dtype).pin_memory()) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(k):
        qd, btd, sld, od, old = sets[k % 2]
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(in_free[k % 2])             # step k-2 has read this input set
            qd.copy_(q_h, non_blocking=True)
            btd.copy_(bt_h, non_blocking=True)
            sld.copy_(sl_h, non_blocking=True)
            in_ready[k % 2].record(h2d_s)
        stream.wait_event(in_ready[k % 2])
        stream.wait_event(out_free[k % 2])               # step k-2's output has been read back
        dcp.dcp_decode_attn(w.kind, qd, inst.kv_cache, btd, sld, w.dcp_size, w.interleave, w.scale, w.q_len,
                            w.head_dim_v, partial_out=po, lse=lse, workspace=ws)
        in_free[k % 2].record(stream)
        dcp.dcp_merge(po, lse, w.dcp_size, out=od, out_lse=old)
        out_ready[k % 2].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[k % 2])
            outs_h[k % 2][0].copy_(od, non_blocking=True)
            outs_h[k % 2][1].copy_(old, non_blocking=True)
            out_free[k % 2].record(d2h_s)

    e2e_steps = max(4, min(args.steps, 10))
    for k in range(2):
        e2e_step(k)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    t0.record(stream)
    h2d_s.wait_event(t0)
    for k in range(e2e_steps):
        e2e_step(k)
    stream.wait_event(out_free[(e2e_steps - 1) % 2])
    stream.wait_event(out_free[(e2e_steps - 2) % 2])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if not torch.equal(outs_h[(e2e_steps - 1) % 2][0], out.cpu()):
        raise RuntimeError("e2e output differs from the device-timed step's output")
    e2e_ms = t0.elapsed_time(t1) / e2e_steps
    h2d = q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + sl_h.numel() * 4
    d2h = out.numel() * 2 + out_lse.numel() * 4

    kv_write = kv_write_timing(inst, reps=max(args.steps, 20))

    kv_rate, ms_per_step = whole_job_rate(alg["kv_bytes"], total_ms / args.steps, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    kv_all = sum_over_ranks(float(alg["kv_bytes"]), world)
    qtok_all = sum_over_ranks(float(B * Lq), world)
    value = kv_rate / 1e9
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    attn_avg = statistics.mean(attn_ms)
    attn_gbs = alg["attn_bytes"] / (attn_avg * 1e-3) / 1e9
    attn_tfs = alg["flops"] / (attn_avg * 1e-3) / 1e12
    t_roof_ms = max(alg["step_bytes"] / (hbm * 1e9), alg["flops"] / (tflops * 1e12)) * 1e3
    bound = "hbm" if alg["attn_bytes"] / hbm >= alg["flops"] / (tflops * 1e3) else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(attn_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(attn_gbs / hbm, 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(attn_tfs, 1), "peak": tflops,
                "unit": "TFLOP/s", "frac": round(attn_tfs / tflops, 4)}
    roof.update({"traffic": measured_traffic(w, alg["attn_bytes"]), "peak_source": f"{peak_src} (MEASURED_PEAKS.json)"
                 if peak_src == "measured" else "fallback",
                 "kernel": "dcp_decode_attn", "attn_ms": round(attn_avg, 4),
                 "attn_ms_median": round(statistics.median(attn_ms), 4),
                 "merge_ms": round(statistics.mean(merge_ms), 4),
                 "alg_bytes_per_launch": alg["attn_bytes"], "alg_flops_per_launch": alg["flops"],
                 "step_frac_of_roofline": round(t_roof_ms / (ms_per_step), 4)})

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; log-normal lengths stand in for the blog's agentic trace)",
        "config": {"workload": w.name, "kind": w.kind, "batch": B, "q_len": Lq,
                   "num_q_heads": Hq, "num_kv_heads": w.num_kv_heads,
                   "head_dim_qk": w.head_dim_qk, "head_dim_v": Dv, "block_size": w.block_size,
                   "dcp_size": N, "interleave": w.interleave,
                   "kv_tokens": alg["tokens"], "kv_bytes": alg["kv_bytes"],
                   "l2": "inputs larger than L2 (cache resident, no flush)"
                   if not flush else "L2 flushed before each timed step (1 GB write, untimed)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "query_tokens_per_s": round(qtok_all / (ms_per_step * 1e-3), 1),
        "roofline": roof,
        "clocks": clocks.summary(),
        "e2e": {"value": round(kv_all / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "kv_write": kv_write,
    }
    if world == 1 and not args.no_other_configs:
        others = {}
        for name in OTHER_CONFIGS:
            if name != w.name:
                others[name] = measure_config(name, args.steps, args.warmup, dev, peaks)
        result["configs"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, kvb, nseq, qtok = oracle_time(inst, args.cpu_budget, args.cpu_max_seqs)
        result["cpu_baseline"] = {
            "value": round(kvb / secs / 1e9, 4), "unit": "GB/s", "cores": cpu_threads(),
            "kind": "oracle", "cpu_count": os.cpu_count(),
            "omp_num_threads": os.environ.get("OMP_NUM_THREADS"),
            "sample": f"{nseq} request(s) of {w.name} ({kvb / 1e9:.2f} GB of cache, all "
                      f"{w.dcp_size} shards + merge), numpy fp64, {secs:.1f} s",
            "query_tokens_per_s": round(qtok / secs, 4)}
    if world > 1:
        import torch.distributed as td
        td.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_reference(args):
    """The CPU oracle on the host cores, timed as the reference arm."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    if torch.cuda.is_available():
        torch.cuda.set_device(0)
    inst = setup_reference_inputs(w)
    alg = algorithmic(w, inst.seq_lens.cpu().numpy())
    budget = max(2.0, args.cpu_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_time(inst, budget, args.cpu_max_seqs)
    secs = kvb = qtok = 0
    nseq = 0
    for _ in range(args.steps):
        s, k, n, qt = oracle_time(inst, budget, args.cpu_max_seqs)
        secs += s
        kvb += k
        nseq += n
        qtok += qt
    value = kvb / secs / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "kind": w.kind, "batch": w.batch, "q_len": w.q_len,
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim_qk": w.head_dim_qk, "head_dim_v": w.head_dim_v,
                   "block_size": w.block_size, "dcp_size": w.dcp_size, "interleave": w.interleave,
                   "kv_tokens": alg["tokens"], "kv_bytes": alg["kv_bytes"],
                   "l2": "not applicable (host oracle)", "parallelism": "host cores (numpy)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_threads(),
                         "kind": "oracle", "cpu_count": os.cpu_count(),
                         "omp_num_threads": os.environ.get("OMP_NUM_THREADS"),
                         "sample": f"{nseq} request(s) of {w.name} over {args.steps} steps "
                                   f"({kvb / 1e9:.2f} GB of cache)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def setup_reference_inputs(w):
    """Same seeded workload as the GPU leg, block counts from the oracle."""
    from oracle import dcp_oracle as orc
    seq_lens = wl.make_seq_lens(w)
    lnb = np.zeros((w.dcp_size, w.batch), dtype=np.int32)
    for b, S in enumerate(seq_lens.tolist()):
        for r, toks in enumerate(orc.shard_token_lists(S, w.interleave, w.dcp_size)):
            lnb[r, b] = -(-len(toks) // w.block_size)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    return wl.make_instance(w, lnb, device=dev, seq_lens=seq_lens)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mla_512", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the CPU baseline sample")
    ap.add_argument("--cpu-max-seqs", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="measure only the named workload (the other configurations are reported by default)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
