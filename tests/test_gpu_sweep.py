"""Sweep points (heads {16,64,128}, batch 1-256, context 4k-132k, qlen
{1,2,4,8}, bf16/fp8, block {16,64,256}) through the C ABI against the oracle.

The seeded grid's points run the direct path (one segment) with their total
visible tokens capped so the suite stays quick, every factor value at least
once, checked on sampled (row, head) pairs.  The corners run the default
balanced split-K (several segment slots) at full size and are checked on
every (row, head): the widest rows (128 heads x qlen 8 = 16 row blocks per
request), 16-token pages at 64k+ contexts, and an fp8 cache with 256-token
blocks (128-row sub-pages spanning two tiles)."""
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


# balanced split-K at the sweep's corners, full size, every (row, head)
SPLIT_CORNERS = [
    (workloads.SweepPoint(128, 6, 12000, 8, "bf16", 64, 911), 8),     # 16 row blocks per request
    (workloads.SweepPoint(64, 3, 20000, 2, "fp8", 64, 912), 6),       # 2 row blocks, fp8
    (workloads.SweepPoint(16, 3, 70000, 4, "bf16", 16, 913), 4),      # 16-token pages, 64k+ context
    (workloads.SweepPoint(16, 4, 40000, 3, "fp8", 256, 914), 8),      # fp8, 128-row sub-pages
]


@pytest.mark.parametrize("pt,S", SPLIT_CORNERS, ids=lambda x: x.name() if hasattr(x, "name") else f"S{x}")
def test_sweep_corner_balanced_split_every_pair(pt, S):
    g = np.random.default_rng(pt.seed)
    L = g.integers(max(pt.qlen, pt.context // 2), pt.context + 1, pt.batch)
    wl = workloads.make_workload(pt.name() + f"_s{S}", L, [pt.qlen] * pt.batch, pt.heads, pt.block_size,
                                 pt.kv_dtype, 1, S, pt.seed, device="cuda")
    out, lse, _ = run_gpu(wl)
    assert mla.get_device_error() == 0
    ref_o, ref_l = oracle_reference(wl)
    assert_close(out, lse, ref_o, ref_l, wl.name)
