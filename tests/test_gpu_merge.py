"""Segment merge and cross-shard state merge on the GPU against the oracle's
float64 merges, on seeded partials with empty parts."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close
from mla_decode_speculative_gb300 import mla

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,S", [(3, 16, 1), (128, 16, 16), (7, 12, 5), (2, 4, 40)])
def test_merge_segments_matches_oracle(T, H, S):
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
    # segment partial outputs are bf16; the oracle merges the same rounded values
    acc_bf = torch.tensor(acc).to(torch.bfloat16)
    out, lse = mla.merge_segments(acc_bf.to("cuda"), torch.tensor(m, device="cuda"),
                                  torch.tensor(l, device="cuda"))
    ref_o, ref_l = oracle.merge_segments(np.nan_to_num(acc_bf.float().numpy(), nan=0.0).astype(np.float64),
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
