"""Decode / causal verify through the C ABI against the float64 oracle.

Every (row, head) is compared, on small workloads and on the full-size
configured workloads in the launch configuration the benchmark times (the
qlen-4 verify over 1k-8k contexts, the fp8 cache with mixed qlen, and the
8-way sharded 128k-context verify).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, balanced_parts, blocks_to_rows, oracle_reference, run_gpu, run_gpu_partials
from mla_decode_speculative_gb300 import mla, runner, workloads

pytestmark = pytest.mark.gpu


def _full_check(wl, what, num_segments=None, uniform=False):
    out, lse, _ = run_gpu(wl, num_segments, uniform_segments=uniform)
    assert mla.get_device_error() == 0
    ref_o, ref_l = oracle_reference(wl)
    return assert_close(out, lse, ref_o, ref_l, what)


# ------------------------------------------------------------------ small, every pair

def test_decode_qlen1_bf16_full():
    _full_check(workloads.decode_qlen1_bf16(), "qlen=1 bf16 decode, batch 2, L 256, block 16")


@pytest.mark.parametrize("S", [1, 3, 16])
@pytest.mark.parametrize("uniform", [False, True])
def test_verify_mtp4_small_every_pair(S, uniform):
    wl = workloads.verify_mtp4_bf16(seed=1, batch=5, lo=130, hi=1500, num_segments=S)
    _full_check(wl, f"verify qlen=4, S={S}, uniform={uniform}", uniform=uniform)


def test_fp8_small_every_pair():
    wl = workloads.fp8_mixed_qlen(seed=2, batch=7, lo=100, hi=2500, num_segments=3)
    _full_check(wl, "fp8 e4m3 verify, qlen 1-3, 12 heads")


def test_dcp_small_every_pair():
    wl = workloads.dcp8_verify_bf16(seed=3, batch=3, context=3000, world_size=8, num_segments=2)
    _full_check(wl, "8-way round-robin sharded verify")


@pytest.mark.parametrize("block_size", [16, 64, 256])
def test_block_sizes_and_subpages(block_size):
    rng = np.random.default_rng(block_size)
    L = rng.integers(5, 900, 6)
    wl = workloads.make_workload(f"bs{block_size}", L, np.minimum(L, 4), 16, block_size,
                                 num_segments=2, seed=block_size)
    _full_check(wl, f"block_size {block_size}")


@pytest.mark.parametrize("block_size", [16, 256])
def test_fp8_block_sizes_every_pair(block_size):
    """fp8 through both load paths: 16-row pages (one 2-D box per chunk and
    page, packed into the stage's upper half) and 128-row sub-pages (one 3-D
    box per 64-token tile, a sub-page spanning two tiles)."""
    rng = np.random.default_rng(300 + block_size)
    L = rng.integers(5, 1200, 5)
    wl = workloads.make_workload(f"fp8_bs{block_size}", L, np.minimum(L, 3), 12, block_size,
                                 kv_dtype="fp8", num_segments=2, seed=block_size)
    _full_check(wl, f"fp8 block_size {block_size}")


@pytest.mark.parametrize("W,I", [(8, 4), (3, 16), (2, 64)])
def test_dcp_interleaved_every_pair(W, I):
    """Interleave I > 1 (runs of I positions dealt to the shards in turn):
    row views, shard decodes and the state merge against the oracle."""
    wl = workloads.make_workload("dcp_interleaved", [700, 90, 1500, 33], [4, 3, 8, 2], 16, 16,
                                 world_size=W, num_segments=3, seed=W + I, interleave=I)
    _full_check(wl, f"DCP W={W} interleave={I}")


@pytest.mark.parametrize("S", [1, 3])
def test_row_views_in_one_launch_equal_separate_calls(S):
    """num_views = W decodes the W shard row views in one launch.  With the
    pages' split every view's output equals, bit for bit, its own single-view
    call (each work item runs the same arithmetic either way); the balanced
    split cuts a different set of chunks, so there both agree with the oracle's
    shard states."""
    W = 4
    wl = workloads.make_workload("views", [700, 90, 1500, 33], [4, 3, 8, 2], 16, 16,
                                 world_size=W, num_segments=S, seed=11)
    step = runner.step_for_workload(wl, "cuda")
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step(q, kv, seq, ind, bt, wl.sm_scale)  # fills the row views and sub-page tables
    torch.cuda.synchronize()
    Q = int(wl.qlens.max())
    all_out, all_lse, _ = mla.decode_verify(q, kv, ind, step.row_len_local, step.subpage, step.P, S, Q,
                                            wl.sm_scale, num_views=W, uniform_segments=True)
    bal_out, bal_lse, _ = mla.decode_verify(q, kv, ind, step.row_len_local, step.subpage, step.P, S, Q,
                                            wl.sm_scale, num_views=W)
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    _, _, ref_po, ref_pl = oracle.sharded_attention(wl.qo_indptr, row_len, wl.q_bits(), wl.kv_host(),
                                                    wl.kv_scale, wl.sm_scale, wl.block_tables,
                                                    wl.block_size, W)
    for r in range(W):
        o, l, _ = mla.decode_verify(q, kv, ind, step.row_len_local[r], step.subpage[r], step.P, S, Q,
                                    wl.sm_scale, uniform_segments=True)
        torch.cuda.synchronize()
        assert torch.equal(o, all_out[r]) and torch.equal(l, all_lse[r]), f"view {r}"
        assert_close(bal_out[r], bal_lse[r], ref_po[r], ref_pl[r], f"balanced, view {r}")
    assert mla.get_device_error() == 0


def test_many_rows_per_request_and_short_windows():
    # 32 heads x qlen 6 = 192 rows (three 64-row blocks); qlen == seq_len rows
    wl = workloads.make_workload("wide", [6, 300, 77], [6, 6, 5], 32, 16, num_segments=2, seed=9)
    _full_check(wl, "192 rows per request, window of 1 token")


def test_single_token_and_tiny_lengths():
    wl = workloads.make_workload("tiny", [1, 2, 3, 129, 128], [1, 2, 1, 1, 3], 16, 16,
                                 num_segments=4, seed=4)
    _full_check(wl, "tiny windows")


def test_dcp_windows_shorter_than_world():
    # seq_len < W: several shards see no token for some rows
    wl = workloads.make_workload("dcp_short", [3, 5, 9], [3, 2, 4], 16, 16, world_size=8,
                                 num_segments=1, seed=5, max_kv_len=2)
    _full_check(wl, "windows shorter than the shard count")


def test_nan_in_unused_cache_slots_is_never_read():
    wl = workloads.make_workload("nan_slots", [70, 200, 33], [3, 4, 2], 16, 64, num_segments=2,
                                 seed=6)
    # poison every cache row no request can see
    visible = np.zeros(wl.kv_rows, bool)
    for b in range(wl.num_reqs):
        for j in range(int(wl.seq_lens[b])):
            blk = wl.block_tables[0, b, j // wl.block_size]
            visible[blk * wl.block_size + j % wl.block_size] = True
    kv = wl.kv.clone()
    kv[torch.as_tensor(~visible)] = float("nan")
    wl.kv = kv
    _full_check(wl, "NaN in invisible cache rows")


def test_segment_partials_match_oracle():
    wl = workloads.verify_mtp4_bf16(seed=7, batch=3, lo=300, hi=1300, num_segments=5)
    out, lse, step = run_gpu(wl, uniform_segments=True)  # the pages' split, slot by slot
    segm_out, segm_max, segm_sum = mla.workspace_views(step.workspace, wl.num_reqs, int(wl.qlens.max()),
                                                       wl.num_rows, wl.num_heads, 5)
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    acc, mx, sm = oracle.segment_partials(wl.qo_indptr, row_len, wl.q_bits(), wl.kv_host(), 1.0,
                                          wl.sm_scale, wl.block_tables[0], wl.block_size, 5,
                                          oracle.page_size(wl.block_size))
    gm, gs = segm_max.cpu().numpy(), segm_sum.cpu().numpy()
    go = blocks_to_rows(segm_out.float().cpu().numpy(), wl.qo_indptr, wl.num_heads, wl.num_rows)  # bf16 blocks
    live = sm > 0
    assert (np.isneginf(gm) == ~live).all(), "GPU and oracle disagree on which segments are empty"
    # normalised segment output and segment LSE (invariant to the reference max)
    norm_ref = acc[live] / sm[live][:, None]
    norm_gpu = go[live] / gs[live][:, None]
    scale = np.abs(norm_ref).max(axis=-1)
    assert (np.abs(norm_gpu - norm_ref).max(axis=-1) / scale).max() <= 1e-2
    lse2_ref = mx[live] + np.log2(sm[live])
    lse2_gpu = gm[live] + np.log2(gs[live])
    assert np.abs(lse2_gpu - lse2_ref).max() * math.log(2) <= 1e-3


@pytest.mark.parametrize("S", [2, 5, 16])
def test_balanced_split_slots_and_merge(S):
    """Balanced split (the default): which (row, slot) pairs hold a part is
    fixed by the rule above, slots past a unit's parts are empty (max = -inf,
    sum = 0), and merging the kernel's own bf16 partials in float64 gives the
    oracle's attention -- every visible token counted once."""
    wl = workloads.verify_mtp4_bf16(seed=11, batch=9, lo=40, hi=5000, num_segments=S)
    step = run_gpu_partials(wl)
    assert mla.get_device_error() == 0
    H, B = wl.num_heads, wl.num_reqs
    RB = mla.row_blocks(int(wl.qlens.max()), H)
    segm_out, segm_max, segm_sum = mla.workspace_views(step.workspace, B, int(wl.qlens.max()),
                                                       wl.num_rows, H, S)
    gm, gs = segm_max.cpu().numpy(), segm_sum.cpu().numpy()
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    ind = wl.qo_indptr
    units = []
    for b in range(B):
        ln = int(max(row_len[ind[b]:ind[b + 1]]))
        rows = (ind[b + 1] - ind[b]) * H
        units += [(-(-ln // 64)) if rb * 64 < rows else 0 for rb in range(RB)]
    grid = min(torch.cuda.get_device_properties(0).multi_processor_count, B * RB * S)
    parts = balanced_parts(units, S, grid)
    assert max(len(v) for v in parts.values()) <= S
    for b in range(B):
        for t in range(ind[b], ind[b + 1]):
            for h in range(H):
                rr = (t - ind[b]) * H + h
                pl = parts[b * RB + rr // 64]
                for s in range(S):
                    live = s < len(pl) and pl[s][0] * 64 < row_len[t]
                    assert np.isneginf(gm[t, h, s]) == (not live), (b, t, h, s)
                    if not live:
                        assert gs[t, h, s] == 0.0
    go = blocks_to_rows(segm_out.float().cpu().numpy(), ind, H, wl.num_rows)
    live = ~np.isneginf(gm)
    acc = np.where(live[..., None], go, 0.0).astype(np.float64)
    mo, ml = oracle.merge_segments(acc, np.where(live, gm, -np.inf).astype(np.float64),
                                   np.where(live, gs, 0.0).astype(np.float64))
    ref_o, ref_l = oracle_reference(wl)
    assert_close(torch.tensor(mo), torch.tensor(ml), ref_o, ref_l, f"merged kernel partials, S={S}")


def _multi_block_workload(S):
    """64 heads x qlen 1-4 mixed: up to four 64-row blocks per request, so a
    block's own rows can be shorter than its unit's tile count (parts with no
    visible token for some rows) and blocks past a request's rows are empty
    units."""
    rng = np.random.default_rng(15)
    L = rng.integers(40, 2500, 7)
    ql = rng.integers(1, 5, 7)
    return workloads.make_workload("multi_block", L, ql, 64, 64, num_segments=S, seed=15)


@pytest.mark.parametrize("S,shape", [(3, "verify"), (16, "verify"), (4, "multi_block"), (9, "multi_block")])
def test_balanced_parts_match_oracle_slot_by_slot(S, shape):
    """Every part of the balanced split against the oracle's partial over the
    part's token range (the rule restated above): same empty slots, the
    normalised part output to the output tolerance, the part's log-sum-exp to
    the LSE tolerance."""
    wl = (workloads.verify_mtp4_bf16(seed=14, batch=6, lo=40, hi=3000, num_segments=S)
          if shape == "verify" else _multi_block_workload(S))
    step = run_gpu_partials(wl)
    assert mla.get_device_error() == 0
    H, B, Q = wl.num_heads, wl.num_reqs, int(wl.qlens.max())
    RB = mla.row_blocks(Q, H)
    segm_out, segm_max, segm_sum = mla.workspace_views(step.workspace, B, Q, wl.num_rows, H, S)
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    ind = wl.qo_indptr
    units = []
    for b in range(B):
        ln = int(max(row_len[ind[b]:ind[b + 1]]))
        rows = (ind[b + 1] - ind[b]) * H
        units += [(-(-ln // 64)) if rb * 64 < rows else 0 for rb in range(RB)]
    grid = min(torch.cuda.get_device_properties(0).multi_processor_count, B * RB * S)
    parts = balanced_parts(units, S, grid)
    ranges = np.zeros((B, RB, S, 2), np.int64)
    for b in range(B):
        for rb in range(RB):
            for s_, (lo, hi) in enumerate(parts[b * RB + rb]):
                ranges[b, rb, s_] = [lo * 64, hi * 64]
    acc, mx, sm = oracle.range_partials(ind, row_len, wl.q_bits(), wl.kv_host(), wl.kv_scale, wl.sm_scale,
                                        wl.block_tables[0], wl.block_size, ranges)
    gm, gs = segm_max.cpu().numpy(), segm_sum.cpu().numpy()
    go = blocks_to_rows(segm_out.float().cpu().numpy(), ind, H, wl.num_rows)
    live = sm > 0
    assert (np.isneginf(gm) == ~live).all(), "GPU and oracle disagree on which parts are empty"
    norm_ref = acc[live] / sm[live][:, None]
    norm_gpu = go[live] / gs[live][:, None]
    scale = np.abs(norm_ref).max(axis=-1)
    assert (np.abs(norm_gpu - norm_ref).max(axis=-1) / scale).max() <= 1e-2
    lse2_ref = mx[live] + np.log2(sm[live])
    lse2_gpu = gm[live] + np.log2(gs[live])
    assert np.abs(lse2_gpu - lse2_ref).max() * math.log(2) <= 1e-3


@pytest.mark.parametrize("uniform", [False, True])
def test_poisoned_workspace_is_never_read(uniform):
    """Every segment slot the merge reads is written by the call: a workspace
    full of NaN bit patterns beforehand changes nothing."""
    wl = workloads.dcp8_verify_bf16(seed=12, batch=3, context=2500, world_size=4, num_segments=6)
    step = runner.step_for_workload(wl, "cuda", uniform_segments=uniform)
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step.workspace.fill_(0xFF)
    out, lse = step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)
    torch.cuda.synchronize()
    assert mla.get_device_error() == 0
    ref_o, ref_l = oracle_reference(wl)
    assert_close(out, lse, ref_o, ref_l, f"poisoned workspace, uniform={uniform}")


def test_more_units_than_the_balanced_table_uses_the_uniform_split():
    """1030 requests of one row each (more (view, request, row block) units
    than the balanced split tabulates): the call takes the pages' split."""
    rng = np.random.default_rng(13)
    L = rng.integers(1, 200, 1030)
    wl = workloads.make_workload("many_units", L, np.ones(1030, np.int64), 4, 16, num_segments=3, seed=13)
    _full_check(wl, "1030 single-row requests, S=3")


def test_static_bound_does_not_change_results():
    wl = workloads.verify_mtp4_bf16(seed=8, batch=4, lo=100, hi=700, num_segments=4)
    out1, lse1, _ = run_gpu(wl)
    wl2 = workloads.verify_mtp4_bf16(seed=8, batch=4, lo=100, hi=700, num_segments=4)
    wl2.max_kv_len = 4096  # wider sub-page table, same data
    out2, lse2, _ = run_gpu(wl2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


# ------------------------------------------------------------------ full size, every pair

def test_repeated_steps_are_bit_identical():
    """Each work item is computed start to finish by one CTA in a fixed
    arithmetic order, whichever CTA claims it, so repeated steps must agree
    bit for bit.  Many repetitions, some behind an L2 flush and some back to
    back, shift the timing between the kernel's warp roles: a missing or
    mis-phased barrier shows up as a mismatch here even when one run happens
    to pass the oracle comparison."""
    from mla_decode_speculative_gb300 import runner
    for wl in (workloads.verify_mtp4_bf16(seed=4, batch=6, lo=64, hi=3000, num_segments=3),
               workloads.fp8_mixed_qlen(seed=5, batch=5, lo=64, hi=2000, num_segments=2),
               workloads.decode_qlen1_bf16()):
        step = runner.step_for_workload(wl, "cuda")
        q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
        flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
        first = None
        for it in range(40):
            if it % 3 == 0:
                flush.fill_(float(it))
            out, lse = step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)
            if first is None:
                first = (out.clone(), lse.clone())
                continue
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1]), f"{wl.name}: run {it} differs"
        assert mla.get_device_error() == 0
        ref_o, ref_l = oracle_reference(wl)
        assert_close(first[0], first[1], ref_o, ref_l, wl.name)


def test_verify_mtp4_full_size_every_pair():
    _full_check(workloads.verify_mtp4_bf16(), "verify qlen=4 batch 32 L 1k-8k S=16")


def test_fp8_full_size_every_pair():
    _full_check(workloads.fp8_mixed_qlen(), "fp8 batch 64 L 512-32k")


def test_dcp8_full_size_every_pair():
    _full_check(workloads.dcp8_verify_bf16(device="cuda"), "dcp8 batch 16 context 128k")


# ------------------------------------------------------------------ in-kernel split-K merge

FUSED_CASES = {
    # the configured qlen-4 verify and the 8-way sharded 128k-context verify
    "verify_mtp4": lambda: workloads.verify_mtp4_bf16(),
    "dcp8": lambda: workloads.dcp8_verify_bf16(device="cuda"),
    # one long request cut into 14 chunks: a unit with more parts than the
    # eight 64-dim output blocks, so some holders merge nothing
    "one_long_request": lambda: workloads.make_workload("fused_long", [100000], [4], 16, 64,
                                                        num_segments=16, seed=41, device="cuda"),
    # many short requests: most units lie inside one chunk (out written
    # straight from the accumulator), the rest span two
    "many_short": lambda: workloads.make_workload(
        "fused_short", np.random.default_rng(42).integers(64, 900, 100), [2] * 100, 16, 64,
        num_segments=4, seed=42),
    # four shard views in one launch, several row blocks per request
    "views_row_blocks": lambda: workloads.make_workload("fused_views", [7000, 300, 12000], [4, 3, 8], 32, 64,
                                                        world_size=4, num_segments=6, seed=43),
    "fp8": lambda: workloads.fp8_mixed_qlen(seed=44, batch=20, lo=200, hi=20000, num_segments=8),
    # sweep corner: 128 heads x qlen 8, 16 row blocks per request
    "wide_rows": lambda: workloads.make_workload("fused_wide", [9000, 12000, 7000], [8, 8, 8], 128, 64,
                                                 num_segments=8, seed=46, device="cuda"),
}


def _fused_and_two_step(wl):
    """(fused out, fused lse, two-step out, two-step lse) for every view of a
    workload whose row plan / shard views are prepared by its step."""
    step = runner.step_for_workload(wl, "cuda")
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)
    W, Q = wl.world_size, step.max_qlen
    row_len = step.row_len if W == 1 else step.row_len_local
    sp = step.subpage[0] if W == 1 else step.subpage
    fo, fl, _ = mla.decode_verify(q, kv, ind, row_len, sp, step.P, step.S, Q, wl.sm_scale, wl.kv_scale,
                                  num_views=W, fused_merge=True)
    two_o, two_l, ws = mla.decode_verify(q, kv, ind, row_len, sp, step.P, step.S, Q, wl.sm_scale,
                                         wl.kv_scale, skip_merge=True, num_views=W)
    so, sm, ss = mla.workspace_views(ws, wl.num_reqs, Q, wl.num_rows, wl.num_heads, step.S, num_views=W)
    mla.merge_segments(so, sm, ss, ind, Q, out=two_o, lse=two_l, num_views=W)
    torch.cuda.synchronize()
    return fo, fl, two_o, two_l


@pytest.mark.parametrize("case", sorted(FUSED_CASES))
def test_fused_merge_matches_oracle_and_two_step_form(case):
    """MLA_DECODE_FUSED_MERGE merges the balanced split's parts inside the
    decode kernel (single-chunk units straight from the accumulator; the last
    arriving part's SM, helped by holders that wait for the unit, for the
    rest); its out / LSE must match the oracle and the pages' two-step form
    (decode with MLA_DECODE_SKIP_MERGE, then mla_merge_segments) within the
    stated tolerances, view by view."""
    wl = FUSED_CASES[case]()
    fo, fl, two_o, two_l = _fused_and_two_step(wl)
    assert mla.get_device_error() == 0
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    kvh, qb = wl.kv_host(), wl.q_bits()
    for r in range(wl.world_size):
        local = oracle.shard_row_view(row_len, wl.world_size, r, wl.interleave) if wl.world_size > 1 else row_len
        ref_o, ref_l = oracle.attention(wl.qo_indptr, local, qb, kvh, wl.kv_scale, wl.sm_scale,
                                        wl.block_tables[r], wl.block_size)
        f = (fo[r], fl[r]) if wl.world_size > 1 else (fo, fl)
        t = (two_o[r], two_l[r]) if wl.world_size > 1 else (two_o, two_l)
        assert_close(f[0], f[1], ref_o, ref_l, f"{case}: in-kernel merge, view {r}")
        assert_close(t[0], t[1], ref_o, ref_l, f"{case}: two-step, view {r}")


def test_fused_merge_repeated_launches_are_bit_identical():
    """Which holder merges which output block depends on arrival order, but
    every block is merged from the same published parts in the same order,
    so repeated launches agree bit for bit."""
    wl = workloads.verify_mtp4_bf16(seed=45, batch=12, lo=500, hi=9000, num_segments=16)
    step = runner.step_for_workload(wl, "cuda")
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step(q, kv, seq, ind, bt, wl.sm_scale)
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    first = None
    for it in range(30):
        if it % 4 == 0:
            flush.fill_(float(it))
        out, lse, _ = mla.decode_verify(q, kv, ind, step.row_len, step.subpage[0], step.P, step.S,
                                        step.max_qlen, wl.sm_scale, workspace=step.workspace,
                                        fused_merge=True)
        if first is None:
            first = (out.clone(), lse.clone())
        else:
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1]), f"launch {it} differs"
    assert mla.get_device_error() == 0


def test_fused_merge_needs_the_balanced_split():
    wl = workloads.verify_mtp4_bf16(seed=47, batch=3, lo=300, hi=900, num_segments=4)
    step = runner.step_for_workload(wl, "cuda")
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step(q, kv, seq, ind, bt, wl.sm_scale)
    for kw in (dict(uniform_segments=True), dict(skip_merge=True)):
        with pytest.raises(mla.MLAError) as e:
            mla.decode_verify(q, kv, ind, step.row_len, step.subpage[0], step.P, 4, 4, wl.sm_scale,
                              fused_merge=True, **kw)
        assert e.value.status == mla.MLA_ERR_UNSUPPORTED
