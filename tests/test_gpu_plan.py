"""Row plan, shard row view and sub-page tables on the GPU: bit-exact against
the oracle on every configured workload's shape and on seeded fuzz."""
import numpy as np
import pytest
import torch

import oracle
from mla_decode_speculative_gb300 import mla, workloads

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")


def _check_plan(seq, ql, bt, num_blocks, block_size, width, extra_rows=0):
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(ind[-1]) + extra_rows
    rl, rr, sp = mla.plan_rows(_dev(seq), _dev(ind), T, _dev(bt), num_blocks, block_size, width)
    assert mla.get_device_error() == 0
    o_rl, o_rr, _ = oracle.plan_rows(seq, ind)
    P = oracle.page_size(block_size)
    o_sp = oracle.subpage_table(np.asarray(seq, np.int32), bt, num_blocks, block_size, width)
    rl, rr, sp = rl.cpu().numpy(), rr.cpu().numpy(), sp.cpu().numpy()
    n = int(ind[-1])
    assert (rl[:n] == o_rl).all() and (rr[:n] == o_rr).all()
    assert (rl[n:] == 0).all() and (rr[n:] == -1).all()
    assert (sp == o_sp).all()
    assert mla.page_size(block_size) == P


@pytest.mark.parametrize("maker", [workloads.decode_qlen1_bf16,
                                   lambda: workloads.verify_mtp4_bf16(),
                                   lambda: workloads.fp8_mixed_qlen()])
def test_plan_rows_configured_workloads(maker):
    wl = maker()
    width = -(-wl.max_kv_len // oracle.page_size(wl.block_size))
    _check_plan(wl.seq_lens, wl.qlens, wl.block_tables[0], wl.num_blocks, wl.block_size, width,
                extra_rows=3)


@pytest.mark.parametrize("seed", range(6))
def test_plan_rows_fuzz(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 40))
    block_size = int(rng.choice([8, 16, 48, 64, 96, 256, 512]))
    seq = rng.integers(1, 3000, B).astype(np.int32)
    ql = np.minimum(rng.integers(1, 9, B), seq).astype(np.int32)
    nb = [-(-int(L) // block_size) for L in seq]
    num_blocks = sum(nb) + 5
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max(nb) + 2), -1, np.int32)
    pos = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += nb[b]
    P = oracle.page_size(block_size)
    width = -(-int(seq.max()) // P) + int(rng.integers(0, 4))
    _check_plan(seq, ql, bt, num_blocks, block_size, width)


@pytest.mark.parametrize("W", [2, 3, 8])
def test_shard_row_view_matches_oracle_and_sums(W):
    rng = np.random.default_rng(W)
    B = 20
    seq = rng.integers(1, 5000, B).astype(np.int32)
    ql = np.minimum(rng.integers(1, 9, B), seq).astype(np.int32)
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(ind[-1])
    o_rl, _, _ = oracle.plan_rows(seq, ind)
    rl, _, _ = mla.plan_rows(_dev(seq), _dev(ind), T)
    block_size = 64
    P = 64
    total = np.zeros(T, np.int64)
    for r in range(W):
        local_cap = [-(-int(L) // W) for L in seq]
        nb = [-(-c // block_size) for c in local_cap]
        num_blocks = sum(nb) + 2
        perm = rng.permutation(num_blocks).astype(np.int32)
        bt = np.full((B, max(nb)), -1, np.int32)
        pos = 0
        for b in range(B):
            bt[b, :nb[b]] = perm[pos:pos + nb[b]]
            pos += nb[b]
        width = -(-max(local_cap) // P)
        loc, sp = mla.shard_row_view(_dev(ind), rl, W, r, 1, _dev(bt), num_blocks, block_size, width)
        assert mla.get_device_error() == 0
        o_loc = oracle.shard_row_view(o_rl, W, r)
        assert (loc.cpu().numpy() == o_loc).all()
        kv_len = np.array([o_loc[ind[b]:ind[b + 1]].max() for b in range(B)], np.int32)
        o_sp = oracle.subpage_table(kv_len, bt, num_blocks, block_size, width)
        assert (sp.cpu().numpy() == o_sp).all()
        total += o_loc
    assert (total == o_rl).all()


def test_shard_row_view_rejects_interleave_0():
    ind = _dev([0, 1])
    rl = _dev([5])
    with pytest.raises(mla.MLAError) as e:
        mla.shard_row_view(ind, rl, 4, 0, interleave=0)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


@pytest.mark.parametrize("W,I", [(2, 2), (3, 4), (8, 16), (8, 1)])
def test_shard_row_view_interleaved_matches_oracle(W, I):
    rng = np.random.default_rng(W * 31 + I)
    B = 24
    seq = rng.integers(1, 6000, B).astype(np.int32)
    ql = np.minimum(rng.integers(1, 9, B), seq).astype(np.int32)
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(ind[-1])
    o_rl, _, _ = oracle.plan_rows(seq, ind)
    rl, _, _ = mla.plan_rows(_dev(seq), _dev(ind), T)
    total = np.zeros(T, np.int64)
    for r in range(W):
        loc, _ = mla.shard_row_view(_dev(ind), rl, W, r, I)
        assert mla.get_device_error() == 0
        o_loc = oracle.shard_row_view(o_rl, W, r, I)
        assert (loc.cpu().numpy() == o_loc).all()
        total += o_loc
    assert (total == o_rl).all()


def test_device_checks_fire_without_faulting():
    # qlen > seq_len
    mla.plan_rows(_dev([3]), _dev([0, 4]), 4)
    assert mla.get_device_error() == 2            # MLA_DEV_BAD_QLEN
    assert mla.get_device_error() == 0            # cleared
    # block id out of range
    mla.plan_rows(_dev([100]), _dev([0, 1]), 1, _dev([[0, 9]]), 5, 64, 4)
    assert mla.get_device_error() == 3            # MLA_DEV_BAD_BLOCK_ID
    # length beyond the static bound
    mla.plan_rows(_dev([300]), _dev([0, 1]), 1, _dev([[0, 1, 2, 3, 4]]), 5, 64, 2)
    assert mla.get_device_error() == 4            # MLA_DEV_LEN_BOUND
    # bad indptr (decreasing)
    mla.plan_rows(_dev([10, 10]), _dev([0, 3, 2]), 3)
    assert mla.get_device_error() in (1, 2)


@pytest.mark.parametrize("W,I", [(8, 1), (3, 4), (2, 64)])
def test_all_shard_views_in_one_launch_bit_exact(W, I):
    """mla_shard_row_views computes every rank's view in one launch: each view
    equals the oracle's shard row view and sub-page table, and the per-rank
    call mla_shard_row_view, bit for bit."""
    rng = np.random.default_rng(70 + W * 7 + I)
    B = 17
    seq = rng.integers(1, 7000, B).astype(np.int32)
    ql = np.minimum(rng.integers(1, 9, B), seq).astype(np.int32)
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(ind[-1])
    o_rl, _, _ = oracle.plan_rows(seq, ind)
    rl, _, _ = mla.plan_rows(_dev(seq), _dev(ind), T)
    block_size = 16
    P = oracle.page_size(block_size)
    cap = [-(-int(L) // (W * I)) * I for L in seq]
    nb = [-(-c // block_size) for c in cap]
    num_blocks = W * sum(nb) + 3
    perm = rng.permutation(num_blocks).astype(np.int32)
    bts = np.full((W, B, max(nb)), -1, np.int32)
    pos = 0
    for r in range(W):
        for b in range(B):
            bts[r, b, :nb[b]] = perm[pos:pos + nb[b]]
            pos += nb[b]
    width = -(-max(cap) // P) + 1
    loc, sp = mla.shard_row_views(_dev(ind), rl, W, I, _dev(bts), num_blocks, block_size, width)
    assert mla.get_device_error() == 0
    loc, sp = loc.cpu().numpy(), sp.cpu().numpy()
    total = np.zeros(T, np.int64)
    for r in range(W):
        o_loc = oracle.shard_row_view(o_rl, W, r, I)
        assert (loc[r] == o_loc).all(), r
        kv_len = np.array([o_loc[ind[b]:ind[b + 1]].max() for b in range(B)], np.int32)
        assert (sp[r] == oracle.subpage_table(kv_len, bts[r], num_blocks, block_size, width)).all(), r
        one_loc, one_sp = mla.shard_row_view(_dev(ind), rl, W, r, I, _dev(bts[r]), num_blocks, block_size, width)
        assert (one_loc.cpu().numpy() == loc[r]).all() and (one_sp.cpu().numpy() == sp[r]).all()
        total += o_loc
    assert (total == o_rl).all()
