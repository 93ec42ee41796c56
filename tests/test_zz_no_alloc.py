"""The allocation-free entry point (mla_decode_verify_noalloc) against the
workspace entry point (mla_decode_verify) through the C ABI.

It serves callers that cannot allocate device memory where they call --
serving runtimes with a fixed memory budget, C hosts without a device
allocator -- by using a static scratch array inside the library.  Two calls in a row must both match the workspace path within the
tolerance the parity tests use, and oversize problems are refused before any
launch.  This file sorts last so a stopping run has covered everything else."""
import numpy as np
import pytest
import torch

from parity import OUT_TOL, LSE_TOL
from mla_decode_speculative_gb300 import build, mla, runner, workloads

pytestmark = pytest.mark.gpu


def _inputs(wl):
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    step = runner.step_for_workload(wl, "cuda")
    mla.plan_rows(seq, ind, wl.num_rows, bt[0], wl.num_blocks, wl.block_size, step.sp_stride,
                  row_len=step.row_len, row_req=step.row_req, subpage_table=step.subpage[0])
    return q, kv, ind, step


def _close(a_out, a_lse, b_out, b_lse):
    ao, bo = a_out.float(), b_out.float()
    scale = bo.abs().amax(dim=-1).clamp_min(1e-30)
    err = ((ao - bo).abs().amax(dim=-1) / scale).max().item()
    lerr = (a_lse - b_lse).abs().max().item()
    assert torch.isfinite(ao).all() and torch.isfinite(a_lse).all()
    assert err <= OUT_TOL and lerr <= LSE_TOL, (err, lerr)


@pytest.mark.parametrize("S", [16, 1])
def test_noalloc_matches_workspace_entry_point_twice(S):
    build.build()
    wl = workloads.verify_mtp4_bf16(seed=21, batch=9, lo=300, hi=5000, num_segments=S)
    q, kv, ind, step = _inputs(wl)
    ref_out, ref_lse, _ = mla.decode_verify(q, kv, ind, step.row_len, step.subpage[0], step.P, S,
                                            4, wl.sm_scale, workspace=step.workspace)
    torch.cuda.synchronize()
    for _ in range(2):
        out, lse = mla.decode_verify_noalloc(q, kv, ind, step.row_len, step.subpage[0], step.P, S,
                                             4, wl.sm_scale)
        torch.cuda.synchronize()
        assert mla.get_device_error() == 0
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    wl = workloads.verify_mtp4_bf16(seed=22, batch=2, lo=100, hi=200, num_segments=1)
    q, kv, ind, step = _inputs(wl)
    # 1024 segments: the two requests' 64-row partial blocks alone take
    # 2 x 1024 x 64 KiB = 128 MiB, beyond the 80 MiB of static scratch
    S = 1024
    a = mla.make_decode_args(q, kv, ind, step.row_len, step.subpage[0], step.P, S, 4, wl.sm_scale,
                             out=torch.empty((wl.num_rows, wl.num_heads, 512), dtype=torch.bfloat16,
                                             device="cuda"),
                             lse=torch.empty((wl.num_rows, wl.num_heads), dtype=torch.float32,
                                             device="cuda"))
    assert mla.decode_verify_workspace_bytes(a) > mla.STATIC_SCRATCH_BYTES
    with pytest.raises(mla.MLAError) as e:
        mla.decode_verify_noalloc(q, kv, ind, step.row_len, step.subpage[0], step.P, S, 4, wl.sm_scale)
    assert e.value.status == mla.MLA_ERR_WORKSPACE
