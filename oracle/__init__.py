"""Float64 CPU oracle for absorbed-form MLA decode / causal speculative verify.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``mla_decode_speculative_gb300``) never imports it and shares no
code with it: the arithmetic lives in ``mla_oracle.c`` (plain C, float64,
OpenMP over (row, head)), compiled here with gcc and called through ctypes.

Page abbreviations in the docstrings:
  [vLLM #51705]   ROCm AITER MLA: causal multi-token speculative verification
                  under DCP (pull request digest)
  [sglang #34432] [AMD][DCP 1/N] add dcp support for aiter backend
  [vLLM #51011]   fix silent wrong decoding of the fp8 KV cache on ROCm AITER MLA

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

D_K = 576
D_V = 512


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into oracle/_build/liboracle.so (gcc, -fopenmp)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            f64p = ctypes.POINTER(ctypes.c_double)
            vp = ctypes.c_void_p
            c_int, c_i64, c_dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_num_threads.restype = c_int
            lib.oracle_page_size.argtypes = [c_int]
            lib.oracle_page_size.restype = c_int
            lib.oracle_plan_rows.argtypes = [c_int, i32p, i32p, c_int, i32p, i32p, i32p]
            lib.oracle_plan_rows.restype = c_int
            lib.oracle_rr_local_len.argtypes = [c_i64, c_int, c_int]
            lib.oracle_rr_local_len.restype = c_i64
            lib.oracle_il_local_len.argtypes = [c_i64, c_int, c_int, c_int]
            lib.oracle_il_local_len.restype = c_i64
            lib.oracle_il_owner.argtypes = [c_i64, c_int, c_int]
            lib.oracle_il_owner.restype = c_int
            lib.oracle_il_local_index.argtypes = [c_i64, c_int, c_int]
            lib.oracle_il_local_index.restype = c_i64
            lib.oracle_shard_row_view.argtypes = [c_int, i32p, c_int, c_int, c_int, i32p]
            lib.oracle_shard_row_view.restype = c_int
            lib.oracle_subpage_table.argtypes = [c_int, i32p, i32p, c_int, c_int, c_int, i32p, c_int]
            lib.oracle_subpage_table.restype = c_int
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = c_dbl
            lib.oracle_attention.argtypes = [c_int, c_int, i32p, i32p, vp, vp, c_int, c_i64,
                                             c_dbl, c_dbl, i32p, c_int, c_int, c_int, i32p, i32p,
                                             f64p, f64p]
            lib.oracle_attention.restype = c_int
            lib.oracle_segment_partials.argtypes = [c_int, c_int, i32p, i32p, vp, vp, c_int, c_i64,
                                                    c_dbl, c_dbl, i32p, c_int, c_int, c_int, c_int,
                                                    f64p, f64p, f64p]
            lib.oracle_segment_partials.restype = c_int
            lib.oracle_range_partials.argtypes = [c_int, c_int, c_int, i32p, i32p, vp, vp, c_int, c_i64,
                                                  c_dbl, c_dbl, i32p, c_int, c_int, c_int,
                                                  ctypes.POINTER(ctypes.c_int64), f64p, f64p, f64p]
            lib.oracle_range_partials.restype = c_int
            lib.oracle_merge_segments.argtypes = [c_i64, c_int, f64p, f64p, f64p, f64p, f64p]
            lib.oracle_merge_segments.restype = None
            lib.oracle_merge_states.argtypes = [c_i64, c_int, f64p, f64p, f64p, f64p]
            lib.oracle_merge_states.restype = None
            lib.oracle_e4m3_encode_rne_sat.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode_rne_sat.restype = ctypes.c_uint8
            lib.oracle_write_kv.argtypes = [c_int, i32p, i32p, vp, c_int, c_int, c_int, i32p, c_int, c_int,
                                            vp, c_int, ctypes.c_float, c_i64]
            lib.oracle_write_kv.restype = c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(code, what):
    if code != 0:
        raise OracleError(f"{what}: oracle error code {code}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def page_size(block_size: int) -> int:
    """Sub-page size P = min(128, largest power-of-two divisor of block_size)
    [vLLM #51705, 实现拆解 3]; -1 for block_size <= 0."""
    return int(_load().oracle_page_size(int(block_size)))


def plan_rows(seq_lens, qo_indptr, num_rows=None):
    """Per verify row: global window length L - qlen + 1 + t, request, t
    [vLLM #51705, 实现拆解 2].  Returns (row_len, row_req, row_t)."""
    seq, sp = _i32(seq_lens)
    ind, ip = _i32(qo_indptr)
    B = seq.shape[0]
    T = int(ind[-1]) if num_rows is None else int(num_rows)
    row_len = np.zeros(T, np.int32)
    row_req = np.zeros(T, np.int32)
    row_t = np.zeros(T, np.int32)
    _, lp = _i32(row_len)
    _, rp = _i32(row_req)
    _, tp = _i32(row_t)
    _check(_load().oracle_plan_rows(B, sp, ip, T, lp, rp, tp), "plan_rows")
    return row_len, row_req, row_t


def rr_local_len(w: int, world_size: int, rank: int) -> int:
    """floor((w-1-r)/W)+1 when non-negative, else 0 [vLLM #51705, row view]."""
    return int(_load().oracle_rr_local_len(int(w), int(world_size), int(rank)))


def il_local_len(w: int, world_size: int, rank: int, interleave: int) -> int:
    """Positions g < w that rank r holds under round-robin with interleave I
    (runs of I positions dealt in turn; the pages support only I = 1)."""
    return int(_load().oracle_il_local_len(int(w), int(world_size), int(rank), int(interleave)))


def il_owner(g: int, world_size: int, interleave: int) -> int:
    """Rank holding global position g: (g div I) mod W."""
    return int(_load().oracle_il_owner(int(g), int(world_size), int(interleave)))


def il_local_index(g: int, world_size: int, interleave: int) -> int:
    """Local index of global position g on its rank: (g div (I*W)) * I + g mod I."""
    return int(_load().oracle_il_local_index(int(g), int(world_size), int(interleave)))


def shard_row_view(row_len_global, world_size, rank, interleave=1):
    """Per-row shard-local lengths counted from each row's global window
    [vLLM #51705, 实现拆解 2]; interleave I >= 1 (I = 1 is the pages' form)."""
    g, gp = _i32(row_len_global)
    out = np.zeros_like(g)
    _, op = _i32(out)
    _check(_load().oracle_shard_row_view(g.shape[0], gp, int(world_size), int(rank),
                                         int(interleave), op), "shard_row_view")
    return out


def subpage_table(kv_len, block_table, num_blocks, block_size, width):
    """Sub-page expansion of a physical block table [vLLM #51705, 实现拆解 3]."""
    kl, kp = _i32(kv_len)
    bt, bp = _i32(block_table)
    B = kl.shape[0]
    out = np.zeros((B, width), np.int32)
    _, op = _i32(out)
    _check(_load().oracle_subpage_table(B, kp, bp, bt.shape[1], int(num_blocks),
                                        int(block_size), op, int(width)), "subpage_table")
    return out


def e4m3_to_double(code: int) -> float:
    """OCP e4m3 ("fn") code -> exact value."""
    return float(_load().oracle_e4m3_to_double(int(code) & 0xFF))


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_to_double(c) for c in range(256)], dtype=np.float64)


def _kv_args(kv):
    kv = np.ascontiguousarray(kv)
    if kv.dtype == np.uint16:
        dt = 0
    elif kv.dtype == np.uint8:
        dt = 1
    else:
        raise TypeError("kv must be uint16 (bf16 bits) or uint8 (e4m3 codes)")
    assert kv.ndim == 2 and kv.shape[1] == D_K
    return kv, dt


def attention(qo_indptr, row_len, q_bits, kv, kv_scale, sm_scale, block_table,
              block_size, sel=None):
    """Plain softmax attention over each row's visible tokens, walking the
    physical block table; returns (out float64, lse float64).

    q_bits: uint16 [T, H, 576] (bf16 bit patterns); kv: uint16 [rows, 576]
    (bf16 bits) or uint8 [rows, 576] (e4m3 codes, multiplied by kv_scale).
    sel: None for every (row, head) -> out [T, H, 512], lse [T, H]; or an
    int array [n, 2] of (row, head) pairs -> out [n, 512], lse [n].
    """
    ind, ip = _i32(qo_indptr)
    rl, rp = _i32(row_len)
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    T, H, dk = q.shape
    assert dk == D_K
    kv, dt = _kv_args(kv)
    bt, bp = _i32(block_table)
    B = ind.shape[0] - 1
    if sel is None:
        n_sel = -1
        out = np.zeros((T, H, D_V), np.float64)
        lse = np.zeros((T, H), np.float64)
        sr = sh = np.zeros(1, np.int32)
    else:
        sel = np.asarray(sel, dtype=np.int32).reshape(-1, 2)
        n_sel = sel.shape[0]
        out = np.zeros((n_sel, D_V), np.float64)
        lse = np.zeros((n_sel,), np.float64)
        sr = np.ascontiguousarray(sel[:, 0])
        sh = np.ascontiguousarray(sel[:, 1])
    _, srp = _i32(sr)
    _, shp = _i32(sh)
    _, outp = _f64(out)
    _, lsep = _f64(lse)
    code = _load().oracle_attention(B, H, ip, rp, q.ctypes.data, kv.ctypes.data, dt,
                                    kv.shape[0], float(kv_scale), float(sm_scale), bp,
                                    bt.shape[1], int(block_size), n_sel, srp, shp, outp, lsep)
    _check(code, "attention")
    return out, lse


def segment_partials(qo_indptr, row_len, q_bits, kv, kv_scale, sm_scale, block_table,
                     block_size, num_segments, tile_size):
    """Base-2 split-K partials per (row, head, segment) under the partition
    tiles_per_segment = cdiv(len, S * TILE) [vLLM #51705, 实现拆解 4].
    Returns (acc [T,H,S,512], m [T,H,S], l [T,H,S])."""
    ind, ip = _i32(qo_indptr)
    rl, rp = _i32(row_len)
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    T, H, _ = q.shape
    kv, dt = _kv_args(kv)
    bt, bp = _i32(block_table)
    B = ind.shape[0] - 1
    S = int(num_segments)
    acc = np.zeros((T, H, S, D_V), np.float64)
    mx = np.zeros((T, H, S), np.float64)
    sm = np.zeros((T, H, S), np.float64)
    _, ap = _f64(acc)
    _, mp = _f64(mx)
    _, smp = _f64(sm)
    code = _load().oracle_segment_partials(B, H, ip, rp, q.ctypes.data, kv.ctypes.data, dt,
                                           kv.shape[0], float(kv_scale), float(sm_scale), bp,
                                           bt.shape[1], int(block_size), S, int(tile_size),
                                           ap, mp, smp)
    _check(code, "segment_partials")
    return acc, mx, sm


def range_partials(qo_indptr, row_len, q_bits, kv, kv_scale, sm_scale, block_table,
                   block_size, ranges):
    """Base-2 partials per (row, head, slot) over given token ranges
    [vLLM #51705, 实现拆解 4: a segment's local max, exp2 sum and output]:
    ranges [B, G, S, 2] int64 = [lo, hi) of slot s for the 64-row group g of
    request b (row (t, h) of b is in group ((t - q0) * H + h) // 64).
    Returns (acc [T,H,S,512], m [T,H,S], l [T,H,S])."""
    ind, ip = _i32(qo_indptr)
    rl, rp = _i32(row_len)
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    T, H, _ = q.shape
    kv, dt = _kv_args(kv)
    bt, bp = _i32(block_table)
    rg = np.ascontiguousarray(ranges, dtype=np.int64)
    B, G, S, two = rg.shape
    if B != ind.shape[0] - 1 or two != 2:
        raise ValueError("ranges must be [B, G, S, 2]")
    acc = np.zeros((T, H, S, D_V), np.float64)
    mx = np.zeros((T, H, S), np.float64)
    sm = np.zeros((T, H, S), np.float64)
    _, ap = _f64(acc)
    _, mp = _f64(mx)
    _, smp = _f64(sm)
    code = _load().oracle_range_partials(B, H, G, ip, rp, q.ctypes.data, kv.ctypes.data, dt,
                                         kv.shape[0], float(kv_scale), float(sm_scale), bp,
                                         bt.shape[1], int(block_size), S,
                                         rg.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                         ap, mp, smp)
    _check(code, "range_partials")
    return acc, mx, sm


def merge_segments(acc, mx, sm):
    """Base-2 segment stats -> (out, natural-log lse) [vLLM #51705, 实现拆解 4].
    acc [..., S, 512], m/l [..., S]; returns out [..., 512], lse [...]."""
    acc = np.asarray(acc, np.float64)
    lead = acc.shape[:-2]
    S = acc.shape[-2]
    n = int(np.prod(lead)) if lead else 1
    a, ap = _f64(acc.reshape(n, S, D_V))
    m, mp = _f64(np.asarray(mx, np.float64).reshape(n, S))
    s, sp = _f64(np.asarray(sm, np.float64).reshape(n, S))
    out = np.zeros((n, D_V), np.float64)
    lse = np.zeros((n,), np.float64)
    _, op = _f64(out)
    _, lp = _f64(lse)
    _load().oracle_merge_segments(n, S, ap, mp, sp, op, lp)
    return out.reshape(*lead, D_V), lse.reshape(lead)


def merge_states(out_parts, lse_parts):
    """Natural-log LSE merge of W partial states [vLLM #51705 功能与动机;
    sglang #34432 merge_state_triton].  out_parts [W, ..., 512], lse_parts
    [W, ...]; returns (out [..., 512], lse [...])."""
    op_ = np.asarray(out_parts, np.float64)
    W = op_.shape[0]
    lead = op_.shape[1:-1]
    n = int(np.prod(lead)) if lead else 1
    o, opp = _f64(op_.reshape(W, n, D_V))
    l, lpp = _f64(np.asarray(lse_parts, np.float64).reshape(W, n))
    out = np.zeros((n, D_V), np.float64)
    lse = np.zeros((n,), np.float64)
    _, outp = _f64(out)
    _, lsep = _f64(lse)
    _load().oracle_merge_states(n, W, opp, lpp, outp, lsep)
    return out.reshape(*lead, D_V), lse.reshape(lead)


def sharded_attention(qo_indptr, row_len_global, q_bits, kv, kv_scale, sm_scale,
                      shard_block_tables, block_size, world_size, sel=None, interleave=1):
    """DCP verify as the pages describe it: every shard r attends the tokens
    it holds within each row's global window (counted by the shard row view),
    reading its own block table; the W partial states are merged in the
    natural-log domain.  shard_block_tables: [W, B, max_blocks] over the one
    cache ``kv``.  Returns (out, lse, per-shard (out_r, lse_r) lists)."""
    parts_out, parts_lse = [], []
    for r in range(world_size):
        local = shard_row_view(row_len_global, world_size, r, interleave)
        o, l = attention(qo_indptr, local, q_bits, kv, kv_scale, sm_scale,
                         shard_block_tables[r], block_size, sel=sel)
        parts_out.append(o)
        parts_lse.append(l)
    out, lse = merge_states(np.stack(parts_out), np.stack(parts_lse))
    return out, lse, parts_out, parts_lse


def e4m3_encode(x: float) -> int:
    """float32 value -> e4m3 code, round to nearest even, saturating at 448."""
    return int(_load().oracle_e4m3_encode_rne_sat(float(x)))


def write_kv(seq_lens, qo_indptr, kv_new_bits, world_size, rank, block_table, block_size,
             cache, kv_scale=1.0, interleave=1):
    """Owner-filtered paged write of the new verify tokens into one rank's cache
    [sglang #34432, 实现拆解 4, set_mla_kv_buffer].  cache (uint16 bf16 bits or
    uint8 e4m3 codes, [rows, 576]) is updated in place."""
    seq, sp = _i32(seq_lens)
    ind, ip = _i32(qo_indptr)
    kvn = np.ascontiguousarray(kv_new_bits, dtype=np.uint16)
    bt, bp = _i32(block_table)
    assert cache.flags["C_CONTIGUOUS"] and cache.shape[1] == D_K
    dt = 0 if cache.dtype == np.uint16 else 1
    _check(_load().oracle_write_kv(seq.shape[0], sp, ip, kvn.ctypes.data, int(world_size), int(rank),
                                   int(interleave), bp, bt.shape[1], int(block_size), cache.ctypes.data, dt,
                                   float(kv_scale), cache.shape[0]), "write_kv")
    return cache
