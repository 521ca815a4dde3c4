"""C ABI checks that need no GPU: the library loads, exports every declared
symbol, and rejects bad arguments on the host before any launch."""

from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dcp.h")


def declared_symbols():
    src = open(HEADER).read()
    return re.findall(r"DCP_API[^;(]*?\b(dcp_\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    from context_decode_attention_paged_gb300 import build
    build.build()
    from context_decode_attention_paged_gb300 import binding
    return binding


def test_header_declares_the_calls():
    syms = declared_symbols()
    for s in ("dcp_build_slot_map", "dcp_decode_attn", "dcp_merge",
              "dcp_decode_attn_workspace_size", "dcp_get_last_device_status",
              "dcp_status_string", "dcp_kv_cache_write"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    raw = lib.raw_lib()
    for s in declared_symbols():
        assert hasattr(raw, s), s


def test_status_strings(lib):
    assert lib.status_string(0) == "DCP_OK"
    assert lib.status_string(1) == "DCP_ERR_INVALID_ARG"
    assert lib.status_string(5) == "DCP_ERR_BOUNDS"
    assert lib.status_string(99) == "DCP_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x10000)   # 256-byte aligned, never dereferenced: the calls below
                                  # must fail validation before touching memory


def _attn(lib, desc, dcp_size=2, interleave=16, scale=0.125, causal=None, q=FAKE, kv=FAKE,
          po=FAKE):
    raw = lib.raw_lib()
    return raw.dcp_decode_attn(ctypes.byref(desc), q, kv, FAKE, FAKE, dcp_size, interleave,
                               scale, desc.q_len if causal is None else causal, po, FAKE, FAKE,
                               0, None)


def _desc(lib, **kw):
    base = dict(kind="gqa", batch=1, q_len=1, num_q_heads=8, num_kv_heads=2, head_dim_qk=64,
                head_dim_v=64, block_size=16, num_blocks=64, max_local_blocks=32)
    base.update(kw)
    return lib.make_desc(**base)


@pytest.mark.parametrize("kw,extra", [
    (dict(num_q_heads=7), {}),                      # Hq % Hkv != 0
    (dict(batch=0), {}),
    (dict(q_len=0), {}),
    (dict(block_size=0), {}),
    (dict(kind=7), {}),
    (dict(kind="mla", num_kv_heads=2), {}),         # MLA has one latent head
    (dict(kind="mla", num_kv_heads=1, head_dim_v=600, head_dim_qk=576), {}),
    (dict(head_dim_v=32), {}),                      # GQA needs Dv == Dqk
    ({}, dict(dcp_size=0)),
    ({}, dict(dcp_size=33)),
    ({}, dict(interleave=0)),
    ({}, dict(scale=0.0)),
    ({}, dict(causal=2)),                           # causal_q_len must equal q_len
    ({}, dict(q=ctypes.c_void_p(0x10002))),         # misaligned q
    ({}, dict(kv=ctypes.c_void_p(0x10008))),        # misaligned cache
    ({}, dict(q=None)),
])
def test_decode_attn_rejects_bad_arguments(lib, kw, extra):
    assert _attn(lib, _desc(lib, **kw), **extra) == lib.DCP_ERR_INVALID_ARG


def test_decode_attn_unsupported_head_dim(lib):
    assert _attn(lib, _desc(lib, head_dim_qk=60, head_dim_v=60)) == lib.DCP_ERR_UNSUPPORTED


def test_merge_rejects_bad_arguments(lib):
    raw = lib.raw_lib()
    ok = dict(N=2, B=1, Lq=1, Hq=8, Dv=64)

    def call(N, B, Lq, Hq, Dv, po=FAKE, out=FAKE):
        return raw.dcp_merge(po, FAKE, N, B, Lq, Hq, Dv, out, None, None)

    assert call(**{**ok, "Hq": 6, "N": 4}) == lib.DCP_ERR_INVALID_ARG   # Hq % N != 0
    assert call(**{**ok, "Dv": 62}) == lib.DCP_ERR_INVALID_ARG
    assert call(**{**ok, "N": 0}) == lib.DCP_ERR_INVALID_ARG
    assert call(**{**ok, "B": 0}) == lib.DCP_ERR_INVALID_ARG
    assert call(**ok, po=ctypes.c_void_p(0x10004)) == lib.DCP_ERR_INVALID_ARG
    assert call(**ok, out=None) == lib.DCP_ERR_INVALID_ARG


def test_slot_map_rejects_bad_arguments(lib):
    raw = lib.raw_lib()
    assert raw.dcp_build_slot_map(FAKE, 1, 0, 16, 2, FAKE, FAKE, None, None, 0, None) == 1
    assert raw.dcp_build_slot_map(FAKE, 1, 16, 0, 2, FAKE, FAKE, None, None, 0, None) == 1
    assert raw.dcp_build_slot_map(FAKE, 1, 16, 16, 0, FAKE, FAKE, None, None, 0, None) == 1
    assert raw.dcp_build_slot_map(FAKE, -1, 16, 16, 2, FAKE, FAKE, None, None, 0, None) == 1
    assert raw.dcp_build_slot_map(FAKE, 1, 16, 16, 2, FAKE, FAKE, FAKE, None, 8, None) == 1
    assert raw.dcp_build_slot_map(FAKE, 1, 16, 16, 2, FAKE, FAKE, FAKE, FAKE, 0, None) == 1
    assert raw.dcp_build_slot_map(None, 1, 16, 16, 2, FAKE, FAKE, None, None, 0, None) == 1
    # an empty batch is a no-op success
    assert raw.dcp_build_slot_map(None, 0, 16, 16, 2, None, None, None, None, 0, None) == 0


def test_workspace_size_of_invalid_desc_is_zero(lib):
    assert lib.dcp_decode_attn_workspace_size(_desc(lib, num_q_heads=7), 2) == 0


def _kvw(lib, desc, new_k=FAKE, new_v=FAKE, cache=FAKE, dcp_size=2, interleave=16, n_new=1):
    raw = lib.raw_lib()
    return raw.dcp_kv_cache_write(ctypes.byref(desc), new_k, new_v, cache, FAKE, FAKE, dcp_size,
                                  interleave, n_new, None)


@pytest.mark.parametrize("kw,extra", [
    ({}, dict(new_v=None)),                                        # GQA needs the V rows
    (dict(kind="mla", num_kv_heads=1, head_dim_qk=576, head_dim_v=512), {}),   # MLA takes no V
    (dict(kind="mla", num_kv_heads=2, head_dim_qk=576, head_dim_v=512), dict(new_v=None)),
    ({}, dict(n_new=0)),
    ({}, dict(dcp_size=0)),
    ({}, dict(interleave=0)),
    (dict(batch=0), {}),
    (dict(block_size=0), {}),
    (dict(num_blocks=0), {}),
    (dict(num_kv_heads=1, head_dim_qk=4, head_dim_v=4), {}),       # 8-byte rows
    ({}, dict(new_k=ctypes.c_void_p(0x10008))),                    # misaligned
    ({}, dict(cache=None)),
    (dict(kind=7), {}),
])
def test_kv_cache_write_rejects_bad_arguments(lib, kw, extra):
    assert _kvw(lib, _desc(lib, **kw), **extra) == lib.DCP_ERR_INVALID_ARG


def _sm_count():
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(0).multi_processor_count
    return 148          # the library's answer when no device is visible


def _wave_model_splits(base_units, max_local, tile, sm):
    """The split count the planner documents: fewest waves x (tiles per split
    + 4 tiles of start-up) over 1..32 splits, when the units fill less than two
    waves; then rounded to whole tiles per split."""
    n = 1
    if base_units < 2 * sm and max_local > 4 * tile:
        tiles = -(-max_local // tile)
        best = None
        for c in range(1, max(1, min(32, max_local // (4 * tile))) + 1):
            cost = -(-base_units * c // sm) * (-(-tiles // c) + 4)
            if best is None or cost < best:
                best, n = cost, c
    per = -(-max_local // n)
    per = max(tile, -(-per // tile) * tile)
    return -(-max_local // per)


@pytest.mark.parametrize("kw,N,tile,units_per_split", [
    # MLA long MTP request: 8 shards x 4 queries, clusters of two CTAs, 64-token tiles
    (dict(kind="mla", batch=1, q_len=4, num_q_heads=128, num_kv_heads=1, head_dim_qk=576, head_dim_v=512,
          block_size=128, num_blocks=8 * 196, max_local_blocks=196), 8, 64, 8),
    # Qwen-like GQA, two short requests: 4 shards x 4 KV heads, 128-key tiles
    (dict(kind="gqa", batch=2, q_len=1, num_q_heads=64, num_kv_heads=4, head_dim_qk=128, head_dim_v=128,
          block_size=128, num_blocks=4 * 2 * 20, max_local_blocks=20), 4, 128, 4),
])
def test_split_planner_follows_the_wave_model(lib, kw, N, tile, units_per_split):
    desc = _desc(lib, **kw)
    ws = lib.raw_lib().dcp_decode_attn_workspace_size(ctypes.byref(desc), N)
    n = _wave_model_splits(N * kw["batch"] * units_per_split, kw["max_local_blocks"] * kw["block_size"], tile,
                           _sm_count())
    rows = N * kw["batch"] * kw["q_len"] * kw["num_q_heads"]
    want = 0 if n == 1 else ((rows * n * kw["head_dim_v"] * 4 + 255) & ~255) + rows * n * 4
    assert n > 1
    assert ws == want, (ws, want, n)


@pytest.mark.parametrize("shape,N,want", [
    (("mla", 4, 1, 128, 1, 576, 512, 128, 100, 10), 8, "MLA_TC"),
    (("mla", 4, 4, 128, 1, 576, 512, 128, 100, 10), 8, "MLA_TC"),
    (("mla", 4, 1, 64, 1, 576, 512, 128, 100, 10), 8, "MLA_TC"),    # 64 heads: MMA rows past 64 unused
    (("mla", 1, 1, 64, 1, 576, 512, 128, 100, 10), 8, "SIMT"),      # a query tensor under 128 rows
    (("mla", 4, 1, 8, 1, 576, 512, 128, 100, 10), 8, "SIMT"),       # under 16 heads
    (("mla", 4, 1, 128, 1, 576, 512, 64, 100, 10), 8, "MLA_TC"),    # block size 64
    (("mla", 4, 1, 128, 1, 576, 512, 16, 100, 10), 8, "MLA_TC"),    # block size 16 (four boxes a tile)
    (("mla", 4, 1, 128, 1, 576, 512, 48, 100, 10), 8, "SIMT"),      # block size 48
    (("gqa", 4, 1, 64, 4, 128, 128, 128, 100, 10), 4, "GQA_TC"),
    (("gqa", 4, 1, 8, 2, 64, 64, 16, 100, 10), 2, "GQA_TC"),
    (("gqa", 4, 1, 8, 2, 96, 96, 16, 100, 10), 2, "SIMT"),          # head dim 96
    (("gqa", 4, 1, 8, 2, 64, 64, 48, 100, 10), 2, "SIMT"),          # block size 48
    (("gqa", 4, 1, 8, 3, 64, 64, 16, 100, 10), 2, "NONE"),          # Hq % Hkv != 0
    (("mla", 4, 1, 128, 2, 576, 512, 128, 100, 10), 8, "NONE"),     # MLA with 2 KV heads
])
def test_kernel_kind_reports_the_kernel_a_shape_runs(lib, shape, N, want):
    """The host-side query names the kernel dcp_decode_attn selects, so a caller
    sees a fall-back to the CUDA-core kernel before launching."""
    desc = lib.make_desc(*shape)
    assert lib.dcp_decode_attn_kernel_kind(desc, N) == getattr(lib, "DCP_KERNEL_" + want)


@pytest.mark.parametrize("shape,N,want_launches,want_ws", [
    # MLA batch 512: the longest-first request order comes from a pre-pass
    # into the workspace (int32 per request)
    (("mla", 512, 1, 128, 1, 576, 512, 128, 512 * 8 * 80, 80), 8, 2, 2048),
    # MLA batch 32 ranks its requests in the kernel: nothing extra
    (("mla", 32, 1, 128, 1, 576, 512, 128, 32 * 8 * 80, 80), 8, 1, 0),
    # a small batch with long shards also splits them: attention + combine
    (("mla", 1, 4, 128, 1, 576, 512, 128, 8 * 196, 196), 8, 2, None),
    (("gqa", 64, 1, 64, 4, 128, 128, 128, 64 * 4 * 60, 60), 4, 1, 0),
])
def test_launch_count_and_workspace(lib, shape, N, want_launches, want_ws):
    """The kernels a call enqueues, as the benchmark counts them, and the
    workspace the MLA request order takes."""
    desc = lib.make_desc(*shape)
    assert lib.dcp_decode_attn_launches(desc, N) == want_launches
    ws = lib.raw_lib().dcp_decode_attn_workspace_size(ctypes.byref(desc), N)
    if want_ws is not None:
        assert ws == want_ws
    else:
        assert ws > 0
    assert lib.dcp_decode_attn_launches(lib.make_desc("mla", 4, 1, 128, 2, 576, 512, 128, 100, 10), N) == 0
