"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/mla_gb300.h declares, and rejects bad
arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from mla_decode_speculative_gb300 import build, mla

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "mla_gb300.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return mla.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_plan_rows", "mla_shard_row_view", "mla_decode_verify", "mla_merge_segments",
              "mla_decode_verify_workspace", "mla_get_device_error", "mla_page_size"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in mla_gb300.h but not exported"
    assert L.mla_abi_version() == 5


def test_page_size_matches_rule(L):
    for bs, p in [(16, 16), (64, 64), (256, 128), (96, 32), (1, 1), (0, -1), (-8, -1), (1000, 8)]:
        assert L.mla_page_size(bs) == p


def test_status_strings(L):
    assert mla.lib().mla_status_string(0) == b"MLA_OK"
    assert mla.lib().mla_status_string(2) == b"MLA_ERR_UNSUPPORTED"


def test_host_validation_without_cuda(L):
    vp = ctypes.c_void_p
    # shard view: interleave < 1 is invalid, checked before anything else
    st = L.mla_shard_row_view(1, 1, vp(8), vp(8), 4, 0, 0, vp(8), None, 0, 0, 0, None, 0, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    assert b"interleave" in L.mla_last_error_string()
    st = L.mla_shard_row_view(1, 1, vp(8), vp(8), 4, 4, 1, vp(8), None, 0, 0, 0, None, 0, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    # all views in one launch: world size and interleave checked first
    assert L.mla_shard_row_views(1, 1, vp(8), vp(8), 0, 1, vp(8), None, 0, 0, 0, None, 0, None) == 1
    assert L.mla_shard_row_views(1, 1, vp(8), vp(8), 4, 0, vp(8), None, 0, 0, 0, None, 0, None) == 1
    assert L.mla_shard_row_views(1, 1, vp(8), vp(8), 4, 1, vp(8), vp(8), 4, 4, 0, vp(8), 4, None) == 1
    # plan rows: negative sizes, non-positive block size
    assert L.mla_plan_rows(-1, 1, vp(8), vp(8), vp(8), vp(8), None, 0, 0, 0, None, 0, None) == 1
    assert L.mla_plan_rows(1, 1, vp(8), vp(8), vp(8), vp(8), vp(8), 4, 4, 0, vp(8), 4, None) == 1
    # decode: page size 4 unsupported, bad dtype, missing workspace
    a = mla.DecodeArgs()
    a.num_reqs, a.num_rows, a.num_heads, a.max_qlen = 1, 1, 16, 1
    a.kv_dtype, a.sm_scale, a.kv_scale = 0, 0.07, 1.0
    a.q = a.kv_cache = a.qo_indptr = a.row_len = a.subpage_table = a.out = a.lse = 256
    a.num_cache_rows, a.subpage_stride, a.page_size, a.num_segments = 64, 4, 4, 1
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_UNSUPPORTED
    a.page_size = 16
    a.kv_dtype = 7
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_UNSUPPORTED
    a.kv_dtype = 0
    a.num_segments = 4
    assert L.mla_decode_verify_workspace(ctypes.byref(a)) > 0
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_WORKSPACE
    # the split flag is a known flag (the call then stops at the missing workspace);
    # an unknown flag bit is rejected before anything else happens
    a.flags = mla.MLA_DECODE_UNIFORM_SEGMENTS | mla.MLA_DECODE_SKIP_MERGE
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_WORKSPACE
    a.flags = 8
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_INVALID_ARG
    assert b"flags" in L.mla_last_error_string()
    # the in-kernel merge needs the balanced split: not with the pages' split,
    # not when the partials are kept for the caller, not with one segment
    for f in (mla.MLA_DECODE_FUSED_MERGE | mla.MLA_DECODE_UNIFORM_SEGMENTS,
              mla.MLA_DECODE_FUSED_MERGE | mla.MLA_DECODE_SKIP_MERGE):
        a.flags = f
        assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_UNSUPPORTED
    a.flags, a.num_segments = mla.MLA_DECODE_FUSED_MERGE, 1
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_UNSUPPORTED
    a.flags, a.num_segments = mla.MLA_DECODE_FUSED_MERGE, 4
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_WORKSPACE
    a.flags = 0
    a.q = 258  # misaligned
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_INVALID_ARG
    a.q = 256
    # a qlen bound above the row capacity, and one whose rows overflow int32
    a.max_qlen = 2
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_INVALID_ARG
    assert b"max_qlen" in L.mla_last_error_string()
    a.num_rows, a.max_qlen = 1 << 27, 1 << 27
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_INVALID_ARG
    a.num_rows, a.max_qlen = 1, 1
    a.wait_cycles = -5
    assert L.mla_decode_verify(ctypes.byref(a), None, 0, None) == mla.MLA_ERR_INVALID_ARG
    assert b"wait_cycles" in L.mla_last_error_string()
    a.wait_cycles = 0
    # merge: unknown mode
    m = mla.MergeArgs()
    m.mode, m.num_rows, m.num_heads, m.num_parts = 9, 1, 1, 1
    m.out = m.lse = 256
    assert L.mla_merge_segments(ctypes.byref(m), None) == mla.MLA_ERR_INVALID_ARG


def test_workspace_size_formula(L):
    a = mla.DecodeArgs()
    a.num_reqs, a.max_qlen, a.num_rows, a.num_heads, a.num_segments = 40, 5, 128, 16, 16
    items = 128 * 16 * 16
    blocks = 40 * 2 * 16  # RB = ceil(5 * 16 / 64) = 2 row blocks per request
    r256 = lambda x: (x + 255) // 256 * 256
    units = 40 * 2  # one 32-bit part counter per (request, row block) unit
    assert L.mla_decode_verify_workspace(ctypes.byref(a)) == \
        r256(blocks * 512 * 64 * 2) + 2 * r256(items * 4) + 256 + r256(units * 4)
    a.num_segments = 1
    assert L.mla_decode_verify_workspace(ctypes.byref(a)) == 256


def test_argument_structs_match_the_header(tmp_path):
    """The ctypes mirrors of mla_decode_args / mla_merge_args have the C
    layout: a tiny C program built against the header prints sizeof and the
    offset of every field."""
    import subprocess
    fields = {"mla_decode_args": [f for f, _ in mla.DecodeArgs._fields_],
              "mla_merge_args": [f for f, _ in mla.MergeArgs._fields_]}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_gb300.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for st, cls in (("mla_decode_args", mla.DecodeArgs), ("mla_merge_args", mla.MergeArgs)):
        assert int(got[st]) == ctypes.sizeof(cls), st
        for f, _ in cls._fields_:
            assert int(got[f"{st}.{f}"]) == getattr(cls, f).offset, f"{st}.{f}"
