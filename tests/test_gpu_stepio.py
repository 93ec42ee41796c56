"""runner.StepIO: a step's inputs staged in one pinned block and uploaded in
one copy, out + lse read back in one copy, give exactly the outputs of the
same step fed from separately copied device tensors (unsharded and sharded,
eager and captured in a CUDA graph), and those match the oracle."""
import pytest
import torch

from parity import assert_close, oracle_reference, sample_pairs
from mla_decode_speculative_gb300 import mla, runner, workloads

pytestmark = pytest.mark.gpu


# (name, seq_lens, qlens, world size, segment slots, seed); drawn inside the test
SPECS = [
    ("stepio_w1", [700, 1300, 90, 2100], [4, 2, 1, 3], 1, 4, 61),
    ("stepio_w4", [3000, 5100, 800], [4, 4, 2], 4, 3, 62),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s[0])
@pytest.mark.parametrize("graph", [False, True])
def test_staged_io_matches_separate_copies_and_the_oracle(spec, graph):
    name, L, ql, W, S, seed = spec
    wl = workloads.make_workload(name, L, ql, 16, 64, world_size=W, num_segments=S, seed=seed, device="cuda",
                                 max_kv_len=-(-max(L) // W))
    ref_step = runner.step_for_workload(wl, "cuda")
    q, kv, seq, ind, bt = runner.device_inputs(wl, "cuda")
    ref_out, ref_lse = ref_step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)
    ref_out, ref_lse = ref_out.cpu(), ref_lse.cpu()

    step = runner.step_for_workload(wl, "cuda")
    io = runner.StepIO(step, wl.q.shape, wl.num_reqs, wl.block_tables.shape, device="cuda")
    io.stage(wl.q, wl.seq_lens, wl.qo_indptr, wl.block_tables)
    d_q, d_seq, d_ind, d_bt = io.device_inputs()

    def one():
        io.upload()
        step(d_q, kv, d_seq, d_ind, d_bt, wl.sm_scale, wl.kv_scale)
        io.download()

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        one()  # eager first call (also the warm-up before any capture)
    torch.cuda.synchronize()
    if graph:
        io.out.zero_()
        io.lse.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one()
        g.replay()
        torch.cuda.synchronize()
    assert mla.get_device_error() == 0
    assert torch.equal(io.out, ref_out) and torch.equal(io.lse, ref_lse)
    sel = sample_pairs(wl, 24, seed=wl.seed)
    o_ref, l_ref = oracle_reference(wl, sel)
    assert_close(io.out[sel[:, 0], sel[:, 1]], io.lse[sel[:, 0], sel[:, 1]], o_ref, l_ref, wl.name)
