"""The decode's device checks and its timeout exit path, driven by host-made
inputs only (nothing here can fault a GPU):

* a sub-page id outside the cache is recorded as MLA_DEV_BAD_SUBPAGE and the
  page is read as zeros (the kernel points the copy past the cache's last
  row, where the tensor copy fills zeros);
* a row length beyond the static bound (table width x page size) is recorded
  as MLA_DEV_LEN_BOUND and the row is clipped to the bound;
* a wait budget far shorter than one tile load makes every CTA give up:
  MLA_DEV_WAIT_TIMEOUT is returned, the kernel drains its own copies and MMAs
  under its fixed exit bound and frees its tensor memory, and the next call
  with the default budget is correct.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, oracle_reference
from mla_decode_speculative_gb300 import mla, runner, workloads

pytestmark = pytest.mark.gpu


def _prepared(wl):
    step = runner.step_for_workload(wl, "cuda")
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)  # row plan + sub-page table
    torch.cuda.synchronize()
    assert mla.get_device_error() == 0
    return step, q, kv, ind


@pytest.mark.parametrize("S", [1, 4])
def test_subpage_outside_the_cache_is_flagged_and_read_as_zeros(S):
    wl = workloads.make_workload("bad_subpage", [300, 260], [3, 2], 16, 64, num_segments=S, seed=31)
    step, q, kv, ind = _prepared(wl)
    sp = step.subpage[0].clone()
    sp[0, 1] = 1 << 24  # page 1 of request 0: rows far past the cache
    out, lse, _ = mla.decode_verify(q, kv, ind, step.row_len, sp, step.P, S, int(wl.qlens.max()),
                                    wl.sm_scale)
    torch.cuda.synchronize()
    assert mla.get_device_error() == 5  # MLA_DEV_BAD_SUBPAGE
    assert mla.get_device_error() == 0  # cleared
    # oracle: the same page read from an all-zero block appended to the pool
    kvh = wl.kv_host()
    kvz = np.concatenate([kvh, np.zeros((wl.block_size, kvh.shape[1]), kvh.dtype)])
    bt = wl.block_tables[0].copy()
    bt[0, 1] = wl.num_blocks
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    ref_o, ref_l = oracle.attention(wl.qo_indptr, row_len, wl.q_bits(), kvz, 1.0, wl.sm_scale, bt,
                                    wl.block_size)
    assert_close(out, lse, ref_o, ref_l, f"sub-page read as zeros, S={S}")


@pytest.mark.parametrize("S", [1, 4])
def test_row_length_beyond_the_bound_is_flagged_and_clipped(S):
    wl = workloads.make_workload("len_bound", [300, 150], [2, 2], 16, 64, num_segments=S, seed=32)
    step, q, kv, ind = _prepared(wl)
    width = 3  # 3 pages of 64: the bound is 192 tokens
    sp = step.subpage[0][:, :width].contiguous()
    out, lse, _ = mla.decode_verify(q, kv, ind, step.row_len, sp, step.P, S, 2, wl.sm_scale)
    torch.cuda.synchronize()
    assert mla.get_device_error() == 4  # MLA_DEV_LEN_BOUND
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    clipped = np.minimum(row_len, width * step.P)
    ref_o, ref_l = oracle.attention(wl.qo_indptr, clipped, wl.q_bits(), wl.kv_host(), 1.0, wl.sm_scale,
                                    wl.block_tables[0], wl.block_size)
    assert_close(out, lse, ref_o, ref_l, f"rows clipped to the bound, S={S}")


@pytest.mark.parametrize("S,fp8", [(1, False), (4, False), (4, True)])
def test_wait_timeout_exit_path_then_a_correct_call(S, fp8):
    wl = workloads.make_workload("timeout", [2500, 3100, 1800, 2900], [4, 4, 4, 4], 16, 64,
                                 kv_dtype="fp8" if fp8 else "bf16", num_segments=S, seed=33)
    step, q, kv, ind = _prepared(wl)
    args = (q, kv, ind, step.row_len, step.subpage[0], step.P, S, 4, wl.sm_scale, wl.kv_scale)
    # 1000 SM cycles: far less than any tile load, so every CTA's first
    # dependent wait runs out
    for _ in range(2):
        mla.decode_verify(*args, wait_cycles=1000)
        torch.cuda.synchronize()
        assert mla.get_device_error() == 6  # MLA_DEV_WAIT_TIMEOUT
    out, lse, _ = mla.decode_verify(*args)
    torch.cuda.synchronize()
    assert mla.get_device_error() == 0
    ref_o, ref_l = oracle_reference(wl)
    assert_close(out, lse, ref_o, ref_l, f"after timeouts, S={S}, fp8={fp8}")


def test_negative_wait_budget_is_rejected_before_launch():
    wl = workloads.make_workload("neg_budget", [100], [1], 16, 64, seed=34)
    step, q, kv, ind = _prepared(wl)
    with pytest.raises(mla.MLAError) as e:
        mla.decode_verify(q, kv, ind, step.row_len, step.subpage[0], step.P, 1, 1, wl.sm_scale,
                          wait_cycles=-1)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
