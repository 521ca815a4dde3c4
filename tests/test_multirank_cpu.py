"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The decode path shards by independent requests, so ranks exchange only timing
scalars: the max of the per-rank step times and the sum of the per-rank work.
These tests run that logic across two gloo processes, and run the reference
arm under torchrun to check that rank 0 alone prints its JSON line.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as td
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        mx = bench.max_over_ranks(10.0 + rank * 5.0, world)     # rank times 10, 15
        sm = bench.sum_over_ranks(100.0 * (rank + 1), world)    # rank work 100, 200
        # the job's rate: all ranks' work over the slowest rank's time
        rate, slow = bench.whole_job_rate(100.0 * (rank + 1), 10.0 + rank * 5.0, world)
        # every rank draws its own workload of the same shape
        w = bench.rank_workload("mla_512", rank)
        lens = bench.wl.make_seq_lens(w)
        bench.barrier(world)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": mx, "sum": sm, "rate": rate, "slow": slow, "seed": w.seed,
                       "batch": w.batch, "lens_head": lens[:4].tolist()}, f)
    finally:
        td.destroy_process_group()


def test_rank_reductions_gloo(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for g in got:
        assert g["max"] == 15.0 and g["sum"] == 300.0
        assert g["rate"] == 300.0 / 15e-3 and g["slow"] == 15.0
    assert got[0]["batch"] == got[1]["batch"] == 512
    assert got[0]["seed"] + 1 == got[1]["seed"]
    assert got[0]["lens_head"] != got[1]["lens_head"]      # independent draws


def test_single_rank_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)


def test_reference_arm_rank0_only_under_torchrun():
    """Two ranks: rank 0 prints one JSON line for the oracle arm, rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_gqa", "--steps", "1", "--warmup", "0", "--cpu-budget", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    # the same workload description as the GPU arm's line
    cfg = rec["config"]
    for key in ("workload", "kind", "batch", "q_len", "num_q_heads", "num_kv_heads", "head_dim_qk",
                "head_dim_v", "block_size", "dcp_size", "interleave", "kv_tokens", "kv_bytes"):
        assert key in cfg, key
    assert cfg["workload"] == "tiny_gqa" and cfg["kv_tokens"] == 1024
    assert rec["higher_is_better"] is True and rec["steps"] == 1
