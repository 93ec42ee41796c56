"""ctypes binding of libmla_gb300.so (argument marshalling only).

Every function mirrors one C entry point of ``include/mla_gb300.h``: torch
tensors are checked for dtype / device / contiguity, their device pointers and
the current CUDA stream are passed through, and a non-OK status raises
``MLAError``.  All compute happens in the library's CUDA kernels; there is no
fallback path.  Call ``mla_decode_speculative_gb300.build.build()`` first (or
``__graft_entry__.build()``); loading a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

D_QK = 576
D_V = 512

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_CHECK = 5

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_MERGE_SEGMENTS = 0
MLA_MERGE_STATES = 1
MLA_DECODE_SKIP_MERGE = 1
MLA_DECODE_UNIFORM_SEGMENTS = 2
MLA_DECODE_FUSED_MERGE = 4

DEVICE_ERRORS = {0: "MLA_DEV_OK", 1: "MLA_DEV_BAD_INDPTR", 2: "MLA_DEV_BAD_QLEN",
                 3: "MLA_DEV_BAD_BLOCK_ID", 4: "MLA_DEV_LEN_BOUND", 5: "MLA_DEV_BAD_SUBPAGE",
                 6: "MLA_DEV_WAIT_TIMEOUT"}


class MLAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class DecodeArgs(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int), ("num_rows", ctypes.c_int),
                ("num_heads", ctypes.c_int), ("max_qlen", ctypes.c_int),
                ("kv_dtype", ctypes.c_int), ("sm_scale", ctypes.c_float),
                ("kv_scale", ctypes.c_float), ("q", ctypes.c_void_p),
                ("kv_cache", ctypes.c_void_p), ("num_cache_rows", ctypes.c_int64),
                ("qo_indptr", ctypes.c_void_p), ("row_len", ctypes.c_void_p),
                ("subpage_table", ctypes.c_void_p), ("subpage_stride", ctypes.c_int),
                ("page_size", ctypes.c_int), ("num_segments", ctypes.c_int),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("flags", ctypes.c_int),
                ("num_views", ctypes.c_int), ("wait_cycles", ctypes.c_int64)]


class MergeArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("num_rows", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("num_parts", ctypes.c_int), ("segm_out", ctypes.c_void_p),
                ("segm_max", ctypes.c_void_p), ("segm_sum", ctypes.c_void_p),
                ("qo_indptr", ctypes.c_void_p), ("num_reqs", ctypes.c_int),
                ("max_qlen", ctypes.c_int), ("num_views", ctypes.c_int), ("part_out", ctypes.c_void_p), ("part_lse", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()
EXPORTS = ("mla_page_size", "mla_plan_rows", "mla_shard_row_view", "mla_shard_row_views",
           "mla_decode_verify_workspace",
           "mla_decode_verify", "mla_decode_verify_noalloc", "mla_write_kv", "mla_merge_segments", "mla_get_device_error",
           "mla_last_error_string", "mla_status_string", "mla_abi_version")


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libmla_gb300.so not built ({path}); run "
                               "mla_decode_speculative_gb300.build.build() first")
        L = ctypes.CDLL(path)
        i32p, vp, c_int = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
        L.mla_page_size.argtypes = [c_int]
        L.mla_page_size.restype = c_int
        L.mla_plan_rows.argtypes = [c_int, c_int, i32p, i32p, i32p, i32p, i32p, c_int, c_int, c_int,
                                    i32p, c_int, vp]
        L.mla_plan_rows.restype = c_int
        L.mla_shard_row_view.argtypes = [c_int, c_int, i32p, i32p, c_int, c_int, c_int, i32p, i32p,
                                         c_int, c_int, c_int, i32p, c_int, vp]
        L.mla_shard_row_view.restype = c_int
        L.mla_shard_row_views.argtypes = [c_int, c_int, i32p, i32p, c_int, c_int, i32p, i32p, c_int,
                                          c_int, c_int, i32p, c_int, vp]
        L.mla_shard_row_views.restype = c_int
        L.mla_decode_verify_workspace.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.mla_decode_verify_workspace.restype = ctypes.c_size_t
        L.mla_decode_verify.argtypes = [ctypes.POINTER(DecodeArgs), vp, ctypes.c_size_t, vp]
        L.mla_decode_verify.restype = c_int
        L.mla_decode_verify_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), vp]
        L.mla_decode_verify_noalloc.restype = c_int
        L.mla_write_kv.argtypes = [c_int, c_int, i32p, i32p, vp, c_int, c_int, c_int, i32p, c_int,
                                   c_int, c_int, vp, c_int, ctypes.c_float, ctypes.c_int64, vp]
        L.mla_write_kv.restype = c_int
        L.mla_merge_segments.argtypes = [ctypes.POINTER(MergeArgs), vp]
        L.mla_merge_segments.restype = c_int
        L.mla_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
        L.mla_get_device_error.restype = c_int
        L.mla_last_error_string.restype = ctypes.c_char_p
        L.mla_status_string.argtypes = [c_int]
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_abi_version.restype = c_int
        _lib = L
        return _lib


def _check(status: int, what: str):
    if status != MLA_OK:
        L = lib()
        raise MLAError(status, f"{what}: {L.mla_status_string(status).decode()}: "
                               f"{L.mla_last_error_string().decode()}")


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def page_size(block_size: int) -> int:
    return int(lib().mla_page_size(int(block_size)))


def plan_rows(seq_lens: torch.Tensor, qo_indptr: torch.Tensor, num_rows: int,
              block_table: Optional[torch.Tensor] = None, num_blocks: int = 0,
              block_size: int = 0, subpage_stride: int = 0, row_len=None, row_req=None,
              subpage_table=None, stream=None):
    """mla_plan_rows.  Returns (row_len [T], row_req [T], subpage_table [B, stride] or None)."""
    B = int(seq_lens.shape[0])
    dev = seq_lens.device
    if row_len is None:
        row_len = torch.empty(num_rows, dtype=torch.int32, device=dev)
    if row_req is None:
        row_req = torch.empty(num_rows, dtype=torch.int32, device=dev)
    bt_stride = 0
    if block_table is not None:
        bt_stride = int(block_table.shape[1])
        if subpage_table is None:
            subpage_table = torch.empty((B, subpage_stride), dtype=torch.int32, device=dev)
    _check(lib().mla_plan_rows(B, int(num_rows), _ptr(seq_lens, torch.int32, "seq_lens"),
                               _ptr(qo_indptr, torch.int32, "qo_indptr"),
                               _ptr(row_len, torch.int32, "row_len"),
                               _ptr(row_req, torch.int32, "row_req"),
                               _ptr(block_table, torch.int32, "block_table"), bt_stride,
                               int(num_blocks), int(block_size),
                               _ptr(subpage_table, torch.int32, "subpage_table"),
                               int(subpage_stride), _stream(stream)), "mla_plan_rows")
    return row_len, row_req, subpage_table


def shard_row_view(qo_indptr: torch.Tensor, row_len_global: torch.Tensor, world_size: int,
                   rank: int, interleave: int = 1, block_table: Optional[torch.Tensor] = None,
                   num_blocks: int = 0, block_size: int = 0, subpage_stride: int = 0,
                   row_len_local=None, subpage_table=None, stream=None):
    """mla_shard_row_view.  Returns (row_len_local [T], subpage_table or None)."""
    B = int(qo_indptr.shape[0]) - 1
    T = int(row_len_global.shape[0])
    dev = row_len_global.device
    if row_len_local is None:
        row_len_local = torch.empty(T, dtype=torch.int32, device=dev)
    bt_stride = 0
    if block_table is not None:
        bt_stride = int(block_table.shape[1])
        if subpage_table is None:
            subpage_table = torch.empty((B, subpage_stride), dtype=torch.int32, device=dev)
    _check(lib().mla_shard_row_view(B, T, _ptr(qo_indptr, torch.int32, "qo_indptr"),
                                    _ptr(row_len_global, torch.int32, "row_len_global"),
                                    int(world_size), int(rank), int(interleave),
                                    _ptr(row_len_local, torch.int32, "row_len_local"),
                                    _ptr(block_table, torch.int32, "block_table"), bt_stride,
                                    int(num_blocks), int(block_size),
                                    _ptr(subpage_table, torch.int32, "subpage_table"),
                                    int(subpage_stride), _stream(stream)), "mla_shard_row_view")
    return row_len_local, subpage_table


def shard_row_views(qo_indptr: torch.Tensor, row_len_global: torch.Tensor, world_size: int,
                    interleave: int = 1, block_tables: Optional[torch.Tensor] = None,
                    num_blocks: int = 0, block_size: int = 0, subpage_stride: int = 0,
                    row_len_local=None, subpage_tables=None, stream=None):
    """mla_shard_row_views: all W views in one launch.  block_tables [W, B, width];
    returns (row_len_local [W, T], subpage_tables [W, B, stride] or None)."""
    B = int(qo_indptr.shape[0]) - 1
    T = int(row_len_global.shape[0])
    W = int(world_size)
    dev = row_len_global.device
    if row_len_local is None:
        row_len_local = torch.empty((W, T), dtype=torch.int32, device=dev)
    bt_stride = 0
    if block_tables is not None:
        bt_stride = int(block_tables.shape[-1])
        if subpage_tables is None:
            subpage_tables = torch.empty((W, B, subpage_stride), dtype=torch.int32, device=dev)
    _check(lib().mla_shard_row_views(B, T, _ptr(qo_indptr, torch.int32, "qo_indptr"),
                                     _ptr(row_len_global, torch.int32, "row_len_global"), W,
                                     int(interleave), _ptr(row_len_local, torch.int32, "row_len_local"),
                                     _ptr(block_tables, torch.int32, "block_tables"), bt_stride,
                                     int(num_blocks), int(block_size),
                                     _ptr(subpage_tables, torch.int32, "subpage_tables"),
                                     int(subpage_stride), _stream(stream)), "mla_shard_row_views")
    return row_len_local, subpage_tables


def make_decode_args(q, kv_cache, qo_indptr, row_len, subpage_table, page_size_, num_segments,
                     max_qlen, sm_scale, kv_scale=1.0, out=None, lse=None, flags=0,
                     num_views=1, wait_cycles=0) -> DecodeArgs:
    T, H, dk = q.shape
    if dk != D_QK:
        raise ValueError("q must be [T, H, 576]")
    fp8 = kv_cache.dtype == torch.uint8
    if kv_cache.dtype not in (torch.uint8, torch.bfloat16) or kv_cache.shape[-1] != D_QK:
        raise ValueError("kv_cache must be [N, 576] bf16 or uint8 (e4m3 codes)")
    a = DecodeArgs()
    a.num_reqs = int(qo_indptr.shape[0]) - 1
    a.num_rows = int(T)
    a.num_heads = int(H)
    a.max_qlen = int(max_qlen)
    a.kv_dtype = MLA_KV_FP8_E4M3 if fp8 else MLA_KV_BF16
    a.sm_scale = float(sm_scale)
    a.kv_scale = float(kv_scale)
    a.q = _ptr(q, torch.bfloat16, "q")
    a.kv_cache = _ptr(kv_cache, None, "kv_cache")
    a.num_cache_rows = int(kv_cache.numel() // D_QK)
    a.qo_indptr = _ptr(qo_indptr, torch.int32, "qo_indptr")
    a.row_len = _ptr(row_len, torch.int32, "row_len")
    a.subpage_table = _ptr(subpage_table, torch.int32, "subpage_table")
    a.subpage_stride = int(subpage_table.shape[-1])
    a.page_size = int(page_size_)
    a.num_segments = int(num_segments)
    a.out = _ptr(out, torch.bfloat16, "out")
    a.lse = _ptr(lse, torch.float32, "lse")
    a.flags = int(flags)
    a.num_views = int(num_views)
    a.wait_cycles = int(wait_cycles)
    return a


def decode_verify_workspace_bytes(a: DecodeArgs) -> int:
    return int(lib().mla_decode_verify_workspace(ctypes.byref(a)))


def decode_verify(q, kv_cache, qo_indptr, row_len, subpage_table, page_size_, num_segments,
                  max_qlen, sm_scale, kv_scale=1.0, out=None, lse=None, workspace=None,
                  stream=None, skip_merge=False, num_views=1, uniform_segments=False,
                  wait_cycles=0, fused_merge=False):
    """mla_decode_verify.  Returns (out [T, H, 512] bf16, lse [T, H] f32, workspace).
    skip_merge: leave the segment partials in the workspace (MLA_DECODE_SKIP_MERGE).
    uniform_segments: the pages' equal split per request (MLA_DECODE_UNIFORM_SEGMENTS)
    instead of the balanced split.
    num_views V > 1: row_len [V, T], subpage_table [V, B, stride]; out [V, T, H, 512],
    lse [V, T, H] (V row views of the same queries, one launch).
    wait_cycles: bound on each in-kernel wait in SM cycles (0 = the library default).
    fused_merge: merge the balanced split's parts inside the decode kernel
    (MLA_DECODE_FUSED_MERGE) instead of a separate merge launch."""
    T, H, _ = q.shape
    V = max(1, int(num_views))
    lead = (V, T) if V > 1 else (T,)
    if out is None:
        out = torch.empty((*lead, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((*lead, H), dtype=torch.float32, device=q.device)
    a = make_decode_args(q, kv_cache, qo_indptr, row_len, subpage_table, page_size_,
                         num_segments, max_qlen, sm_scale, kv_scale, out, lse,
                         (MLA_DECODE_SKIP_MERGE if skip_merge else 0) |
                         (MLA_DECODE_UNIFORM_SEGMENTS if uniform_segments else 0) |
                         (MLA_DECODE_FUSED_MERGE if fused_merge else 0), num_views=V,
                         wait_cycles=wait_cycles)
    need = decode_verify_workspace_bytes(a)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace, torch.uint8, "workspace") if need else None
    _check(lib().mla_decode_verify(ctypes.byref(a), ws_ptr, need, _stream(stream)),
           "mla_decode_verify")
    return out, lse, workspace


STATIC_SCRATCH_BYTES = 80 * 1024 * 1024


def decode_verify_noalloc(q, kv_cache, qo_indptr, row_len, subpage_table, page_size_,
                          num_segments, max_qlen, sm_scale, kv_scale=1.0, out=None, lse=None,
                          stream=None):
    """mla_decode_verify_noalloc: the library's own static device scratch instead of a
    caller workspace, for callers that cannot allocate device memory at the call (serving
    runtimes that reserve all device memory at start-up, C or plugin hosts without a device
    allocator).  Calls that overlap on the GPU share that scratch and must be serialised.
    Returns (out, lse)."""
    T, H, _ = q.shape
    if out is None:
        out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    a = make_decode_args(q, kv_cache, qo_indptr, row_len, subpage_table, page_size_,
                         num_segments, max_qlen, sm_scale, kv_scale, out, lse)
    _check(lib().mla_decode_verify_noalloc(ctypes.byref(a), _stream(stream)),
           "mla_decode_verify_noalloc")
    return out, lse


def row_blocks(max_qlen: int, num_heads: int) -> int:
    """RB: 64-row blocks per request in the segment-partial layout."""
    return -(-max_qlen * num_heads // 64)


def workspace_views(workspace: torch.Tensor, num_reqs: int, max_qlen: int, num_rows: int,
                    num_heads: int, num_segments: int, num_views: int = 1):
    """The documented workspace layout (num_views = 1): (segm_out [B, RB, S, 8, 512, 8] bf16
    blocks -- row octet, dim, row in octet --, segm_max [T, H, S], segm_sum [T, H, S]); V
    views stack V such layouts."""
    num_reqs, num_rows = num_reqs * num_views, num_rows * num_views
    items = num_rows * num_heads * num_segments
    blocks = num_reqs * row_blocks(max_qlen, num_heads) * num_segments
    a256 = lambda x: (x + 255) & ~255
    o_bytes = a256(blocks * 512 * 64 * 2)
    m_bytes = a256(items * 4)
    segm_out = workspace[:blocks * 512 * 64 * 2].view(torch.bfloat16).view(
        num_reqs, row_blocks(max_qlen, num_heads), num_segments, 8, 512, 8)
    segm_max = workspace[o_bytes:o_bytes + items * 4].view(torch.float32).view(num_rows, num_heads, num_segments)
    segm_sum = workspace[o_bytes + m_bytes:o_bytes + m_bytes + items * 4].view(torch.float32).view(
        num_rows, num_heads, num_segments)
    return segm_out, segm_max, segm_sum


def merge_segments(segm_out, segm_max, segm_sum, qo_indptr, max_qlen, out=None, lse=None,
                   stream=None, num_views=1):
    """mla_merge_segments, segment mode: bf16 partial blocks [V*B, RB, S, 8, 512, 8] (the
    decode workspace layout) + [V*T, H, S] f32 base-2 stats; qo_indptr [B + 1] int32.
    num_views V > 1: out [V, T, H, 512], lse [V, T, H] (the V row views of one decode)."""
    VT, H, S = segm_max.shape
    V = max(1, int(num_views))
    T = VT // V
    lead = (V, T) if V > 1 else (T,)
    if out is None:
        out = torch.empty((*lead, H, D_V), dtype=torch.bfloat16, device=segm_out.device)
    if lse is None:
        lse = torch.empty((*lead, H), dtype=torch.float32, device=segm_out.device)
    m = MergeArgs()
    m.mode, m.num_rows, m.num_heads, m.num_parts = MLA_MERGE_SEGMENTS, T, H, S
    m.segm_out = _ptr(segm_out, torch.bfloat16, "segm_out")
    m.qo_indptr = _ptr(qo_indptr, torch.int32, "qo_indptr")
    m.num_reqs = int(qo_indptr.shape[0]) - 1
    m.max_qlen = int(max_qlen)
    m.num_views = V
    m.segm_max = _ptr(segm_max, torch.float32, "segm_max")
    m.segm_sum = _ptr(segm_sum, torch.float32, "segm_sum")
    m.out = _ptr(out, torch.bfloat16, "out")
    m.lse = _ptr(lse, torch.float32, "lse")
    _check(lib().mla_merge_segments(ctypes.byref(m), _stream(stream)), "mla_merge_segments")
    return out, lse


def merge_states(part_out, part_lse, out=None, lse=None, stream=None):
    """mla_merge_segments, state mode: [W,T,H,512] bf16 + [W,T,H] natural-log LSE."""
    W, T, H, dv = part_out.shape
    if out is None:
        out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=part_out.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=part_out.device)
    m = MergeArgs()
    m.mode, m.num_rows, m.num_heads, m.num_parts = MLA_MERGE_STATES, T, H, W
    m.part_out = _ptr(part_out, torch.bfloat16, "part_out")
    m.part_lse = _ptr(part_lse, torch.float32, "part_lse")
    m.out = _ptr(out, torch.bfloat16, "out")
    m.lse = _ptr(lse, torch.float32, "lse")
    _check(lib().mla_merge_segments(ctypes.byref(m), _stream(stream)), "mla_merge_segments")
    return out, lse


def write_kv(seq_lens, qo_indptr, kv_new, kv_cache, block_table, num_blocks, block_size,
             world_size=1, rank=0, kv_scale=1.0, interleave=1, stream=None):
    """mla_write_kv: owner-filtered paged write of the new tokens (kv_new [T, 576]
    bf16) into this rank's cache (bf16 [N, 576], or uint8 e4m3 codes)."""
    fp8 = kv_cache.dtype == torch.uint8
    _check(lib().mla_write_kv(int(seq_lens.shape[0]), int(kv_new.shape[0]),
                              _ptr(seq_lens, torch.int32, "seq_lens"),
                              _ptr(qo_indptr, torch.int32, "qo_indptr"),
                              _ptr(kv_new, torch.bfloat16, "kv_new"), int(world_size), int(rank),
                              int(interleave), _ptr(block_table, torch.int32, "block_table"),
                              int(block_table.shape[1]), int(num_blocks), int(block_size),
                              _ptr(kv_cache, None, "kv_cache"),
                              MLA_KV_FP8_E4M3 if fp8 else MLA_KV_BF16, float(kv_scale),
                              int(kv_cache.numel() // D_QK), _stream(stream)), "mla_write_kv")
    return kv_cache


def get_device_error(stream=None) -> int:
    """mla_get_device_error: synchronises, returns and clears the device error code."""
    code = ctypes.c_int32(0)
    st = lib().mla_get_device_error(ctypes.byref(code), _stream(stream))
    if st not in (MLA_OK, MLA_ERR_DEVICE_CHECK):
        _check(st, "mla_get_device_error")
    return int(code.value)
