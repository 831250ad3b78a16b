"""Python binding of libdcp's C ABI (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks dtypes/devices/contiguity, turns torch
tensors into raw pointers and passes them on. There is no fallback: if the
compiled library is missing the import of this module's functions raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdcp.so")
_lib = None

DCP_OK = 0
DCP_ERR_INVALID_ARG = -1
DCP_ERR_SHAPE = -2
DCP_ERR_UNSUPPORTED = -3
DCP_ERR_CUDA = -4
DCP_ERR_WORKSPACE = -5
DCP_ERR_SCRATCH_LIMIT = -6
DCP_NOALLOC_SCRATCH_BYTES = 64 << 20

DCP_DEVERR_BLOCK_RANGE = 1
DCP_DEVERR_TABLE_RANGE = 2
DCP_DEVERR_POSITION = 4
DCP_DEVERR_TIMEOUT = 8

DCP_MAX_SHARDS = 32
DCP_MAX_QUERY_TOKENS = 8192
DCP_KIND_GQA = 0
DCP_KIND_MLA = 1
DCP_KV_BF16 = 0
DCP_KV_FP8_E4M3 = 1

EXPORTED = ("dcp_status_string", "dcp_version", "dcp_shard_plan", "dcp_kv_append", "dcp_workspace_size",
            "dcp_workspace_size_mtp", "dcp_decode_partial", "dcp_decode_partial_all", "dcp_decode_partial_all_mtp",
            "dcp_attention_all",
            "dcp_decode_partial_all_noalloc", "dcp_merge")


class DcpError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {dcp_status_string(status)} ({status})")
        self.status = status


class _Desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim_k", ctypes.c_int), ("head_dim_v", ctypes.c_int), ("block_size", ctypes.c_int),
                ("scale", ctypes.c_float), ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


class _Shard(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("max_blocks_per_seq", ctypes.c_int32)]


@dataclass(frozen=True)
class AttnDesc:
    kind: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_k: int
    head_dim_v: int
    block_size: int
    scale: float
    kv_dtype: int = DCP_KV_BF16
    k_scale: float = 1.0
    v_scale: float = 1.0

    def c(self) -> _Desc:
        return _Desc(self.kind, self.num_q_heads, self.num_kv_heads, self.head_dim_k, self.head_dim_v,
                     self.block_size, self.scale, self.kv_dtype, self.k_scale, self.v_scale)

    @property
    def kv_torch_dtype(self):
        """torch dtype of pools and appended rows: bf16, or uint8 E4M3 codes."""
        return torch.uint8 if self.kv_dtype == DCP_KV_FP8_E4M3 else torch.bfloat16


@dataclass
class Shard:
    """One shard's pool(s) and block table (device tensors)."""
    k_pool: torch.Tensor
    v_pool: torch.Tensor | None
    block_table: torch.Tensor

    def c(self) -> _Shard:
        if self.k_pool.dtype not in (torch.bfloat16, torch.uint8):
            raise TypeError("k_pool must be bf16 or uint8 (E4M3 codes)")
        _check(self.k_pool, self.k_pool.dtype, "k_pool")
        if self.v_pool is not None:
            _check(self.v_pool, self.k_pool.dtype, "v_pool")
        _check(self.block_table, torch.int32, "block_table")
        return _Shard(self.k_pool.data_ptr(), self.v_pool.data_ptr() if self.v_pool is not None else None,
                      int(self.k_pool.shape[0]), self.block_table.data_ptr(), int(self.block_table.shape[1]))


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libdcp.so (built in-tree by build.py); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libdcp.so not built ({_LIB_PATH}); run sequence_sharded_decode_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    pdesc, pshard = ctypes.POINTER(_Desc), ctypes.POINTER(_Shard)
    lib.dcp_status_string.restype = ctypes.c_char_p
    lib.dcp_status_string.argtypes = [i32]
    lib.dcp_version.restype = i32
    lib.dcp_version.argtypes = []
    lib.dcp_shard_plan.restype = i32
    lib.dcp_shard_plan.argtypes = [vp, i32, i32, i32, i32, vp, vp]
    lib.dcp_kv_append.restype = i32
    lib.dcp_kv_append.argtypes = [pdesc, pshard, i32, vp, i32, vp, vp, vp, vp, i32, vp, vp]
    lib.dcp_workspace_size.restype = sz
    lib.dcp_workspace_size.argtypes = [pdesc, i32, i32]
    lib.dcp_workspace_size_mtp.restype = sz
    lib.dcp_workspace_size_mtp.argtypes = [pdesc, i32, i32, i32]
    lib.dcp_decode_partial.restype = i32
    lib.dcp_decode_partial.argtypes = [pdesc, vp, pshard, vp, vp, i32, vp, vp, vp, sz, vp, vp]
    lib.dcp_decode_partial_all.restype = i32
    lib.dcp_decode_partial_all.argtypes = [pdesc, vp, pshard, i32, vp, vp, i32, vp, vp, vp, sz, vp, vp]
    lib.dcp_decode_partial_all_mtp.restype = i32
    lib.dcp_decode_partial_all_mtp.argtypes = [pdesc, vp, pshard, i32, vp, vp, i32, i32, vp, vp, vp, sz, vp, vp]
    lib.dcp_attention_all.restype = i32
    lib.dcp_attention_all.argtypes = [pdesc, vp, pshard, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.dcp_decode_partial_all_noalloc.restype = i32
    lib.dcp_decode_partial_all_noalloc.argtypes = [pdesc, vp, pshard, i32, vp, vp, i32, vp, vp, vp, vp]
    lib.dcp_merge.restype = i32
    lib.dcp_merge.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
    _lib = lib
    return lib


def _check(t: torch.Tensor, dtype, name: str, cuda: bool = True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _shards(shards) -> ctypes.Array:
    arr = (_Shard * len(shards))()
    for i, s in enumerate(shards):
        arr[i] = s.c()
    return arr


def _raise(rc: int, where: str):
    if rc != DCP_OK:
        raise DcpError(rc, where)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def dcp_status_string(status: int) -> str:
    return load().dcp_status_string(int(status)).decode()


def dcp_version() -> int:
    return load().dcp_version()


def dcp_shard_plan(ctx_lens, n_shards: int, block_size: int, reserve_tokens: int):
    """Host routing plan: (shard_starts int32 [B, N], blocks_needed int32 [B, N])."""
    ctx = np.ascontiguousarray(np.asarray(ctx_lens, dtype=np.int32).reshape(-1))
    B = ctx.shape[0]
    starts = np.zeros((B, n_shards), dtype=np.int32)
    blocks = np.zeros((B, n_shards), dtype=np.int32)
    rc = load().dcp_shard_plan(ctx.ctypes.data, B, n_shards, block_size, reserve_tokens,
                               starts.ctypes.data, blocks.ctypes.data)
    _raise(rc, "dcp_shard_plan")
    return starts, blocks


def dcp_kv_append(desc: AttnDesc, shards, shard_starts: torch.Tensor, positions: torch.Tensor,
                  k_new: torch.Tensor, v_new: torch.Tensor | None, seq_ids: torch.Tensor | None = None,
                  err: torch.Tensor | None = None, stream=None):
    _check(shard_starts, torch.int32, "shard_starts")
    _check(positions, torch.int32, "positions")
    _check(k_new, desc.kv_torch_dtype, "k_new")
    if v_new is not None:
        _check(v_new, desc.kv_torch_dtype, "v_new")
    if seq_ids is not None:
        _check(seq_ids, torch.int32, "seq_ids")
    if err is not None:
        _check(err, torch.int32, "err")
    B = int(shard_starts.shape[0])
    T = int(positions.numel())
    arr = _shards(shards)
    rc = load().dcp_kv_append(ctypes.byref(desc.c()), arr, len(shards), shard_starts.data_ptr(), B,
                              _ptr(seq_ids), positions.data_ptr(), k_new.data_ptr(), _ptr(v_new), T,
                              _ptr(err), _stream(stream))
    _raise(rc, "dcp_kv_append")


def dcp_workspace_size(desc: AttnDesc, batch: int, n_shards: int) -> int:
    return int(load().dcp_workspace_size(ctypes.byref(desc.c()), batch, n_shards))


def dcp_workspace_size_mtp(desc: AttnDesc, batch: int, q_len: int, n_shards: int) -> int:
    return int(load().dcp_workspace_size_mtp(ctypes.byref(desc.c()), batch, q_len, n_shards))


def dcp_decode_partial(desc: AttnDesc, q: torch.Tensor, shard: Shard, seq_lens: torch.Tensor,
                       shard_range: torch.Tensor, o_part: torch.Tensor, lse: torch.Tensor,
                       workspace: torch.Tensor, err: torch.Tensor | None = None, stream=None):
    _check(q, torch.bfloat16, "q")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(shard_range, torch.int32, "shard_range")
    _check(o_part, torch.float32, "o_part")
    _check(lse, torch.float32, "lse")
    _check(workspace, torch.uint8, "workspace")
    if err is not None:
        _check(err, torch.int32, "err")
    arr = _shards([shard])
    rc = load().dcp_decode_partial(ctypes.byref(desc.c()), q.data_ptr(), arr, seq_lens.data_ptr(),
                                   shard_range.data_ptr(), int(q.shape[0]), o_part.data_ptr(), lse.data_ptr(),
                                   workspace.data_ptr(), workspace.numel(), _ptr(err), _stream(stream))
    _raise(rc, "dcp_decode_partial")


def dcp_decode_partial_all(desc: AttnDesc, q: torch.Tensor, shards, seq_lens: torch.Tensor,
                           shard_starts: torch.Tensor, o_parts: torch.Tensor, lses: torch.Tensor,
                           workspace: torch.Tensor, err: torch.Tensor | None = None, stream=None):
    _check(q, torch.bfloat16, "q")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(shard_starts, torch.int32, "shard_starts")
    _check(o_parts, torch.float32, "o_parts")
    _check(lses, torch.float32, "lses")
    _check(workspace, torch.uint8, "workspace")
    if err is not None:
        _check(err, torch.int32, "err")
    arr = _shards(shards)
    rc = load().dcp_decode_partial_all(ctypes.byref(desc.c()), q.data_ptr(), arr, len(shards),
                                       seq_lens.data_ptr(), shard_starts.data_ptr(), int(q.shape[0]),
                                       o_parts.data_ptr(), lses.data_ptr(), workspace.data_ptr(),
                                       workspace.numel(), _ptr(err), _stream(stream))
    _raise(rc, "dcp_decode_partial_all")


def dcp_decode_partial_all_mtp(desc: AttnDesc, q: torch.Tensor, shards, seq_lens: torch.Tensor,
                               shard_starts: torch.Tensor, o_parts: torch.Tensor, lses: torch.Tensor,
                               workspace: torch.Tensor, err: torch.Tensor | None = None, stream=None):
    """q [B, q_len, Hq, Dk] bf16: q_len new tokens per sequence, query token j
    at position seq_lens[b] - q_len + j, causal among the new tokens.
    o_parts [N, B, q_len, Hq, Dv], lses [N, B, q_len, Hq]; the workspace is
    dcp_workspace_size_mtp(desc, B, q_len, N) bytes."""
    _check(q, torch.bfloat16, "q")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(shard_starts, torch.int32, "shard_starts")
    _check(o_parts, torch.float32, "o_parts")
    _check(lses, torch.float32, "lses")
    _check(workspace, torch.uint8, "workspace")
    if err is not None:
        _check(err, torch.int32, "err")
    if q.dim() != 4:
        raise ValueError("q must be [B, q_len, Hq, Dk]")
    arr = _shards(shards)
    rc = load().dcp_decode_partial_all_mtp(ctypes.byref(desc.c()), q.data_ptr(), arr, len(shards),
                                           seq_lens.data_ptr(), shard_starts.data_ptr(), int(q.shape[0]),
                                           int(q.shape[1]), o_parts.data_ptr(), lses.data_ptr(),
                                           workspace.data_ptr(), workspace.numel(), _ptr(err), _stream(stream))
    _raise(rc, "dcp_decode_partial_all_mtp")


def dcp_attention_all(desc: AttnDesc, q: torch.Tensor, shards, seq_lens: torch.Tensor, shard_starts: torch.Tensor,
                      o_parts: torch.Tensor, lses: torch.Tensor, o: torch.Tensor, lse_out: torch.Tensor | None,
                      workspace: torch.Tensor, err: torch.Tensor | None = None, stream=None):
    """Partial attention of every shard and the merge in one call. q is
    [B, Hq, Dk] (one-token decode) or [B, q_len, Hq, Dk]; o_parts / lses are
    scratch of the shards' partial rows; o [B, (q_len,) Hq, Dv], lse_out
    [B, (q_len,) Hq] or None receive the merged result."""
    _check(q, torch.bfloat16, "q")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(shard_starts, torch.int32, "shard_starts")
    _check(o_parts, torch.float32, "o_parts")
    _check(lses, torch.float32, "lses")
    _check(o, torch.float32, "o")
    if lse_out is not None:
        _check(lse_out, torch.float32, "lse_out")
    _check(workspace, torch.uint8, "workspace")
    if err is not None:
        _check(err, torch.int32, "err")
    q_len = 1 if q.dim() == 3 else int(q.shape[1])
    arr = _shards(shards)
    rc = load().dcp_attention_all(ctypes.byref(desc.c()), q.data_ptr(), arr, len(shards), seq_lens.data_ptr(),
                                  shard_starts.data_ptr(), int(q.shape[0]), q_len, o_parts.data_ptr(),
                                  lses.data_ptr(), o.data_ptr(), _ptr(lse_out), workspace.data_ptr(),
                                  workspace.numel(), _ptr(err), _stream(stream))
    _raise(rc, "dcp_attention_all")


def dcp_decode_partial_all_noalloc(desc: AttnDesc, q: torch.Tensor, shards, seq_lens: torch.Tensor,
                                   shard_starts: torch.Tensor, o_parts: torch.Tensor, lses: torch.Tensor,
                                   err: torch.Tensor | None = None, stream=None):
    """dcp_decode_partial_all without a caller workspace: the library's fixed
    device scratch (DCP_NOALLOC_SCRATCH_BYTES) is used instead."""
    _check(q, torch.bfloat16, "q")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(shard_starts, torch.int32, "shard_starts")
    _check(o_parts, torch.float32, "o_parts")
    _check(lses, torch.float32, "lses")
    if err is not None:
        _check(err, torch.int32, "err")
    arr = _shards(shards)
    rc = load().dcp_decode_partial_all_noalloc(ctypes.byref(desc.c()), q.data_ptr(), arr, len(shards),
                                               seq_lens.data_ptr(), shard_starts.data_ptr(), int(q.shape[0]),
                                               o_parts.data_ptr(), lses.data_ptr(), _ptr(err), _stream(stream))
    _raise(rc, "dcp_decode_partial_all_noalloc")


def dcp_merge(o_parts: torch.Tensor, lses: torch.Tensor, o: torch.Tensor, lse_out: torch.Tensor | None = None,
              stream=None):
    """o_parts [N, ..., Hq, Dv] fp32, lses [N, ..., Hq] fp32 -> o [..., Hq, Dv] (+ lse_out [..., Hq]);
    the middle dimensions (sequences, or sequences x query tokens) are merged row by row."""
    _check(o_parts, torch.float32, "o_parts")
    _check(lses, torch.float32, "lses")
    _check(o, torch.float32, "o")
    if lse_out is not None:
        _check(lse_out, torch.float32, "lse_out")
    if o_parts.dim() < 4:
        raise ValueError("o_parts must be [N, ..., Hq, Dv]")
    N, Hq, Dv = int(o_parts.shape[0]), int(o_parts.shape[-2]), int(o_parts.shape[-1])
    B = o_parts.numel() // max(1, N * Hq * Dv)
    rc = load().dcp_merge(o_parts.data_ptr(), lses.data_ptr(), N, B, Hq, Dv, o.data_ptr(), _ptr(lse_out),
                          _stream(stream))
    _raise(rc, "dcp_merge")
