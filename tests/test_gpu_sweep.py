"""Sweep points (heads {16,64,128}, batch 1-256, context 4k-132k, qlen
{1,2,4,8}, bf16/fp8, block {16,64,256}) through the C ABI, checked against the
oracle on sampled (row, head) pairs.  Total visible tokens per point are capped
so the suite stays quick; the corners of each factor are covered explicitly."""
import numpy as np
import pytest

from parity import assert_close, oracle_reference, run_gpu, sample_pairs
from mla_decode_speculative_gb300 import mla, workloads

pytestmark = pytest.mark.gpu

POINTS = workloads.sweep_points(100, seed=0)
# every factor value at least once, from the seeded grid
CHOSEN = []
for key, vals in (("heads", (16, 64, 128)), ("qlen", (1, 2, 4, 8)),
                  ("kv_dtype", ("bf16", "fp8")), ("block_size", (16, 64, 256))):
    for v in vals:
        cand = [p for p in POINTS if getattr(p, key) == v and p not in CHOSEN]
        CHOSEN.append(cand[0])
CORNERS = [
    workloads.SweepPoint(128, 256, 4096, 8, "bf16", 64, 901),     # widest rows, largest batch
    workloads.SweepPoint(128, 2, 135168, 8, "fp8", 256, 902),     # widest rows, longest context
    workloads.SweepPoint(16, 1, 135168, 1, "bf16", 16, 903),      # single long decode, small pages
]


@pytest.mark.parametrize("pt", CHOSEN + CORNERS, ids=lambda p: p.name())
def test_sweep_point_sampled(pt):
    wl = workloads.sweep_workload(pt, device="cuda", max_tokens=600_000)
    out, lse, _ = run_gpu(wl)
    assert mla.get_device_error() == 0
    sel = sample_pairs(wl, 48, seed=pt.seed)
    ref_o, ref_l = oracle_reference(wl, sel)
    assert_close(out[sel[:, 0], sel[:, 1]], lse[sel[:, 0], sel[:, 1]], ref_o, ref_l, pt.name())
