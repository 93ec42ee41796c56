"""Cross-check of the per-row shard row view against the two-stage verify
decomposition [sglang #34432 digest, 实现拆解 3, _forward_verify_dcp]: every
shard attends its part of the committed prefix (global positions
[0, L - qlen)); the verify window -- the qlen new tokens, replicated on all
shards -- is attended once (rank 0's job) with the causal mask row t ->
window tokens [0, t]; the W + 1 partial states are LSE-merged.  Both
decompositions run on the library's kernels and must agree with each other
and with the oracle."""
import pytest
import torch

from parity import OUT_TOL, LSE_TOL, assert_close, oracle_reference
from mla_decode_speculative_gb300 import mla, runner, workloads

pytestmark = pytest.mark.gpu


def _window_rows(wl):
    """The new tokens' cached rows (global position g of request b lives on
    shard g % W at local index g // W), gathered in verify-row order."""
    kv = wl.kv.cpu()
    rows = []
    W, bs = wl.world_size, wl.block_size
    for b in range(wl.num_reqs):
        L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
        for t in range(ql):
            g = L - ql + t
            r, j = g % W, g // W
            rows.append(kv[int(wl.block_tables[r, b, j // bs]) * bs + j % bs])
    return torch.stack(rows)


def _two_stage(wl, step, q, kv, seq, ind, bt):
    dev = q.device
    B, T, H, W = wl.num_reqs, wl.num_rows, wl.num_heads, wl.world_size
    qmax = int(wl.qlens.max())
    pages = -(-qmax // 8)
    win_pool = torch.zeros((B * pages * 8, 576), dtype=torch.bfloat16, device=dev)
    win_table = torch.arange(B * pages, dtype=torch.int32, device=dev).view(B, pages)
    qlens = ind[1:] - ind[:-1]
    # window stage: seq_len = qlen puts new token t at window index t and makes row t see [0, t]
    win_len, _, win_sp = mla.plan_rows(qlens, ind, T, win_table, B * pages, 8, pages)
    mla.write_kv(qlens, ind, _window_rows(wl).to(dev), win_pool, win_table, B * pages, 8)
    part_out = torch.empty((W + 1, T, H, 512), dtype=torch.bfloat16, device=dev)
    part_lse = torch.empty((W + 1, T, H), dtype=torch.float32, device=dev)
    mla.decode_verify(q, win_pool, ind, win_len, win_sp, 8, 1, qmax, wl.sm_scale,
                      out=part_out[W], lse=part_lse[W])
    # prefix stage on every shard: the committed prefix [0, L - qlen) of each row
    row_len, _, _ = mla.plan_rows(seq, ind, T)
    prefix = row_len - win_len
    for r in range(W):
        loc, sp = mla.shard_row_view(ind, prefix, W, r, 1, bt[r], wl.num_blocks, wl.block_size,
                                     step.sp_stride)
        mla.decode_verify(q, kv, ind, loc, sp, step.P, step.S, qmax, wl.sm_scale,
                          out=part_out[r], lse=part_lse[r])
    return mla.merge_states(part_out, part_lse)


@pytest.mark.parametrize("W,seq,ql", [(8, [300, 40, 1000, 9, 8], [4, 3, 8, 2, 8]),
                                      (2, [129, 64], [4, 1])])
def test_two_stage_equals_row_view_and_oracle(W, seq, ql):
    wl = workloads.make_workload("two_stage", seq, ql, 16, 16, world_size=W, num_segments=2,
                                 seed=W)
    step = runner.step_for_workload(wl, "cuda")
    q, kv, s, ind, bt = runner.device_inputs(wl, "cuda")
    one_out, one_lse = step(q, kv, s, ind, bt, wl.sm_scale)
    one_out, one_lse = one_out.clone(), one_lse.clone()
    two_out, two_lse = _two_stage(wl, step, q, kv, s, ind, bt)
    torch.cuda.synchronize()
    assert mla.get_device_error() == 0
    ref_o, ref_l = oracle_reference(wl)
    assert_close(one_out, one_lse, ref_o, ref_l, "row view")
    assert_close(two_out, two_lse, ref_o, ref_l, "two-stage")
    scale = one_out.float().abs().amax(-1).clamp_min(1e-30)
    assert ((two_out.float() - one_out.float()).abs().amax(-1) / scale).max() <= 2 * OUT_TOL
    assert (two_lse - one_lse).abs().max() <= 2 * LSE_TOL
