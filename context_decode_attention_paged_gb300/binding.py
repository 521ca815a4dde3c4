"""Thin ctypes binding over libdcp.so (declared in include/dcp.h).

Argument marshalling only: tensors are passed as raw device pointers together
with ``torch.cuda.current_stream()``; every step of the computation runs in the
library's CUDA kernels.  Output tensors are allocated here with torch when the
caller does not pass them (torch is used for device memory only).

Importing this module loads the library and raises ``ImportError`` when it has
not been built: there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdcp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libdcp.so is not built ({LIB_PATH}); run "
                      "`python -m context_decode_attention_paged_gb300.build`")

_lib = ctypes.CDLL(LIB_PATH)

DCP_OK, DCP_ERR_INVALID_ARG, DCP_ERR_UNSUPPORTED, DCP_ERR_CUDA, DCP_ERR_TIMEOUT, DCP_ERR_BOUNDS = range(6)
DCP_ATTN_GQA, DCP_ATTN_MLA = 0, 1
DCP_KERNEL_NONE, DCP_KERNEL_MLA_TC, DCP_KERNEL_GQA_TC, DCP_KERNEL_SIMT = range(4)
KINDS = {"gqa": DCP_ATTN_GQA, "mla": DCP_ATTN_MLA}


class DcpAttnDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kind", "batch", "q_len", "num_q_heads", "num_kv_heads", "head_dim_qk", "head_dim_v",
        "block_size", "num_blocks", "max_local_blocks")]


_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_lib.dcp_build_slot_map.restype = _i32
_lib.dcp_build_slot_map.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp]
_lib.dcp_decode_attn_workspace_size.restype = _sz
_lib.dcp_decode_attn_workspace_size.argtypes = [ctypes.POINTER(DcpAttnDesc), _i32]
_lib.dcp_decode_attn.restype = _i32
_lib.dcp_decode_attn.argtypes = [ctypes.POINTER(DcpAttnDesc), _vp, _vp, _vp, _vp, _i32, _i32,
                                 _f32, _i32, _vp, _vp, _vp, _sz, _vp]
_lib.dcp_decode_attn_noalloc.restype = _i32
_lib.dcp_decode_attn_noalloc.argtypes = [ctypes.POINTER(DcpAttnDesc), _vp, _vp, _vp, _vp, _i32,
                                         _i32, _f32, _i32, _vp, _vp, _vp]
_lib.dcp_kv_cache_write.restype = _i32
_lib.dcp_kv_cache_write.argtypes = [ctypes.POINTER(DcpAttnDesc), _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                    _i32, _vp]
_lib.dcp_merge.restype = _i32
_lib.dcp_merge.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]
_lib.dcp_decode_attn_kernel_kind.restype = _i32
_lib.dcp_decode_attn_kernel_kind.argtypes = [ctypes.POINTER(DcpAttnDesc), _i32]
_lib.dcp_decode_attn_launches.restype = _i32
_lib.dcp_decode_attn_launches.argtypes = [ctypes.POINTER(DcpAttnDesc), _i32]
_lib.dcp_get_last_device_status.restype = _i32
_lib.dcp_get_last_device_status.argtypes = [_vp]
_lib.dcp_status_string.restype = ctypes.c_char_p
_lib.dcp_status_string.argtypes = [_i32]


class DcpError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)}")


def status_string(code: int) -> str:
    return _lib.dcp_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, what: str):
    if code != DCP_OK:
        raise DcpError(code, what)


def make_desc(kind, batch, q_len, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v,
              block_size, num_blocks, max_local_blocks) -> DcpAttnDesc:
    return DcpAttnDesc(KINDS.get(kind, kind), batch, q_len, num_q_heads, num_kv_heads,
                       head_dim_qk, head_dim_v, block_size, num_blocks, max_local_blocks)


def desc_from_tensors(kind, q, kv_cache, block_tables, head_dim_v) -> DcpAttnDesc:
    B, Lq, Hq, Dqk = q.shape
    if KINDS.get(kind, kind) == DCP_ATTN_GQA:
        _, nb, bs, Hkv, _ = kv_cache.shape
    else:
        nb, bs, _ = kv_cache.shape
        Hkv = 1
    return make_desc(kind, B, Lq, Hq, Hkv, Dqk, head_dim_v, bs, nb, block_tables.shape[2])


def dcp_build_slot_map(seq_lens, block_size, interleave, dcp_size, max_seq=None, stream=None):
    """Returns (local_seq_lens [N][B], local_num_blocks [N][B], shard_of, local_pos);
    the last two are [B][max_seq] when ``max_seq`` is given, else None."""
    B = seq_lens.shape[0]
    dev = seq_lens.device
    lsl = torch.empty((dcp_size, B), dtype=torch.int32, device=dev)
    lnb = torch.empty((dcp_size, B), dtype=torch.int32, device=dev)
    shard_of = local_pos = None
    if max_seq is not None:
        shard_of = torch.empty((B, max_seq), dtype=torch.int32, device=dev)
        local_pos = torch.empty((B, max_seq), dtype=torch.int32, device=dev)
    _check(_lib.dcp_build_slot_map(_ptr(seq_lens), B, block_size, interleave, dcp_size,
                                   _ptr(lsl), _ptr(lnb), _ptr(shard_of), _ptr(local_pos),
                                   int(max_seq or 0), _stream(stream)), "dcp_build_slot_map")
    return lsl, lnb, shard_of, local_pos


def dcp_decode_attn_workspace_size(desc: DcpAttnDesc, dcp_size: int) -> int:
    return int(_lib.dcp_decode_attn_workspace_size(ctypes.byref(desc), dcp_size))


def dcp_decode_attn_launches(desc: DcpAttnDesc, dcp_size: int) -> int:
    """Kernels one dcp_decode_attn call enqueues for this shape (0: invalid)."""
    return int(_lib.dcp_decode_attn_launches(ctypes.byref(desc), dcp_size))


def dcp_decode_attn_kernel_kind(desc: DcpAttnDesc, dcp_size: int) -> int:
    """Which kernel dcp_decode_attn runs for this shape (DCP_KERNEL_*)."""
    return int(_lib.dcp_decode_attn_kernel_kind(ctypes.byref(desc), dcp_size))


def dcp_decode_attn(kind, q, kv_cache, block_tables, seq_lens, dcp_size, interleave, scale,
                    causal_q_len, head_dim_v, partial_out=None, lse=None, workspace=None,
                    stream=None):
    """Per-shard partial outputs fp32 [N][B][Lq][Hq][Dv] and lse fp32 [N][B][Lq][Hq]."""
    desc = desc_from_tensors(kind, q, kv_cache, block_tables, head_dim_v)
    B, Lq, Hq, _ = q.shape
    dev = q.device
    if partial_out is None:
        partial_out = torch.empty((dcp_size, B, Lq, Hq, head_dim_v), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((dcp_size, B, Lq, Hq), dtype=torch.float32, device=dev)
    ws_bytes = dcp_decode_attn_workspace_size(desc, dcp_size)
    if workspace is None and ws_bytes:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    _check(_lib.dcp_decode_attn(ctypes.byref(desc), _ptr(q), _ptr(kv_cache), _ptr(block_tables),
                                _ptr(seq_lens), dcp_size, interleave, float(scale),
                                causal_q_len, _ptr(partial_out), _ptr(lse), _ptr(workspace),
                                workspace.numel() if workspace is not None else 0,
                                _stream(stream)), "dcp_decode_attn")
    return partial_out, lse


def dcp_decode_attn_noalloc(kind, q, kv_cache, block_tables, seq_lens, dcp_size, interleave,
                            scale, causal_q_len, head_dim_v, partial_out, lse, stream=None):
    """dcp_decode_attn without a workspace argument: split scratch comes from the
    library's built-in array (for callers that may not allocate device memory).
    Outputs must be passed in; calls overlapping on the GPU share that array."""
    desc = desc_from_tensors(kind, q, kv_cache, block_tables, head_dim_v)
    _check(_lib.dcp_decode_attn_noalloc(ctypes.byref(desc), _ptr(q), _ptr(kv_cache),
                                        _ptr(block_tables), _ptr(seq_lens), dcp_size, interleave,
                                        float(scale), causal_q_len, _ptr(partial_out), _ptr(lse),
                                        _stream(stream)), "dcp_decode_attn_noalloc")
    return partial_out, lse


def dcp_kv_cache_write(kind, new_k, new_v, kv_cache, block_tables, seq_lens, dcp_size, interleave,
                       stream=None):
    """Store the newest n_new tokens of every request in their shards' cache cells
    (kv_cache is written in place).  new_k/new_v: GQA [B][n_new][Hkv][D];
    MLA new_k [B][n_new][Dqk] and new_v None."""
    B, n_new = new_k.shape[0], new_k.shape[1]
    if KINDS.get(kind, kind) == DCP_ATTN_GQA:
        _, nb, bs, Hkv, D = kv_cache.shape
    else:
        nb, bs, D = kv_cache.shape
        Hkv = 1
    desc = make_desc(kind, B, n_new, Hkv, Hkv, D, D, bs, nb, block_tables.shape[2])
    _check(_lib.dcp_kv_cache_write(ctypes.byref(desc), _ptr(new_k), _ptr(new_v), _ptr(kv_cache),
                                   _ptr(block_tables), _ptr(seq_lens), dcp_size, interleave, n_new,
                                   _stream(stream)), "dcp_kv_cache_write")
    return kv_cache


def dcp_merge(partial_out, lse, dcp_size, out=None, out_lse=None, want_lse=True, stream=None):
    """out bf16 [N][B][Lq][Hq/N][Dv] (+ out_lse fp32 [N][B][Lq][Hq/N])."""
    N, B, Lq, Hq, Dv = partial_out.shape
    assert N == dcp_size
    dev = partial_out.device
    if out is None:
        out = torch.empty((N, B, Lq, Hq // N, Dv), dtype=torch.bfloat16, device=dev)
    if out_lse is None and want_lse:
        out_lse = torch.empty((N, B, Lq, Hq // N), dtype=torch.float32, device=dev)
    _check(_lib.dcp_merge(_ptr(partial_out), _ptr(lse), dcp_size, B, Lq, Hq, Dv, _ptr(out),
                          _ptr(out_lse), _stream(stream)), "dcp_merge")
    return out, out_lse


def dcp_get_last_device_status(stream=None) -> int:
    return int(_lib.dcp_get_last_device_status(_stream(stream)))


def raw_lib():
    """The ctypes library handle (for tests of the raw C ABI)."""
    return _lib
