"""Segment merge and cross-shard state merge on the GPU against the oracle's
float64 merges, on seeded partials with empty parts."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, rows_to_blocks
from mla_decode_speculative_gb300 import mla

pytestmark = pytest.mark.gpu


# the last two cases have more than two waves of row-octet tasks, so the merge
# takes its wide shape (6-slot ring), with up to 16 / 12 live parts per row to
# wrap the ring, and partial octets (15 rows per block)
@pytest.mark.parametrize("qlens,H,S", [([1, 2], 16, 1), ([4] * 32, 16, 16), ([3, 1, 2, 1], 12, 5),
                                       ([1, 1], 4, 40), ([8, 3], 16, 3), ([4] * 160, 8, 16),
                                       ([3] * 200, 5, 12)])
def test_merge_segments_matches_oracle(qlens, H, S):
    qo = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    T = int(qo[-1])
    rng = np.random.default_rng(T * 100 + S)
    acc = rng.standard_normal((T, H, S, 512)).astype(np.float32) * 20
    m = (rng.standard_normal((T, H, S)) * 4).astype(np.float32)
    l = rng.uniform(1, 100, (T, H, S)).astype(np.float32)
    empty = rng.random((T, H, S)) < 0.3
    m[empty] = -np.inf
    l[empty] = 0
    acc[empty] = np.nan  # never read
    if S > 1:
        m[0, 0, :] = -np.inf  # a fully empty item
        l[0, 0, :] = 0
        acc[0, 0, :] = np.nan
    # segment partial outputs are bf16 in the decode workspace's block layout;
    # the oracle merges the same rounded values
    acc_r = torch.tensor(acc).to(torch.bfloat16).float().numpy()
    RB = mla.row_blocks(max(qlens), H)
    blocks = torch.tensor(rows_to_blocks(acc_r, qo, H, RB)).to(torch.bfloat16)
    out, lse = mla.merge_segments(blocks.to("cuda"), torch.tensor(m, device="cuda"),
                                  torch.tensor(l, device="cuda"), torch.tensor(qo, device="cuda"),
                                  max(qlens))
    ref_o, ref_l = oracle.merge_segments(np.nan_to_num(acc_r, nan=0.0).astype(np.float64),
                                         m.astype(np.float64), l.astype(np.float64))
    assert_close(out, lse, ref_o, ref_l, "segment merge")
    if S > 1:
        assert (out[0, 0].float() == 0).all() and torch.isneginf(lse[0, 0])


@pytest.mark.parametrize("W,T,H", [(8, 64, 16), (2, 5, 3), (3, 1, 128)])
def test_merge_states_matches_oracle(W, T, H):
    rng = np.random.default_rng(W * 10 + T)
    po = torch.tensor(rng.standard_normal((W, T, H, 512)), dtype=torch.bfloat16)
    pl = (rng.standard_normal((W, T, H)) * 3 + 5).astype(np.float32)
    empty = rng.random((W, T, H)) < 0.25
    pl[empty] = -np.inf
    po[torch.tensor(empty)] = float("nan")  # never read
    if T > 1:
        pl[:, 1, 0] = -np.inf
    out, lse = mla.merge_states(po.cuda(), torch.tensor(pl, device="cuda"))
    po64 = np.nan_to_num(po.float().numpy().astype(np.float64), nan=0.0)
    ref_o, ref_l = oracle.merge_states(po64, pl.astype(np.float64))
    assert_close(out, lse, ref_o, ref_l, "state merge")
