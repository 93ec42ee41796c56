"""World-size-2 gloo runs on CPU of the multi-process host logic:
* the benchmark's replica aggregation (slowest rank's time, all ranks' bytes);
* the context-parallel exchange: each rank owns half of W round-robin shards,
  computes its shards' (out, lse) states, the states are all-gathered and
  LSE-merged -- equal to the unsharded attention (float64 oracle)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _replica_worker(rank, world, port, q):
    _init(rank, world, port)
    import bench
    local_ms = [1.5, 2.5][rank]
    q.put((rank, bench.max_over_ranks(local_ms, dist, "cpu")))
    dist.destroy_process_group()


def _dcp_worker(rank, world, port, q):
    _init(rank, world, port)
    import oracle
    from mla_decode_speculative_gb300 import workloads
    W = 4
    wl = workloads.make_workload("dcp_cpu", [37, 150, 9], [4, 2, 3], 2, 16, world_size=W,
                                 num_segments=1, seed=3)
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    qb, kv = wl.q_bits(), wl.kv_host()
    mine = [r for r in range(W) if r % world == rank]
    outs, lses = [], []
    for r in mine:
        local = oracle.shard_row_view(row_len, W, r)
        o, l = oracle.attention(wl.qo_indptr, local, qb, kv, 1.0, wl.sm_scale,
                                wl.block_tables[r], wl.block_size)
        outs.append(torch.from_numpy(o))
        lses.append(torch.from_numpy(l))
    o_local, l_local = torch.stack(outs), torch.stack(lses)
    o_all = [torch.empty_like(o_local) for _ in range(world)]
    l_all = [torch.empty_like(l_local) for _ in range(world)]
    dist.all_gather(o_all, o_local)
    dist.all_gather(l_all, l_local)
    out, lse = oracle.merge_states(torch.cat(o_all).numpy(), torch.cat(l_all).numpy())
    # unsharded reference: the oracle's own all-shard composition on one process
    ref_o, ref_l, _, _ = oracle.sharded_attention(wl.qo_indptr, row_len, qb, kv, 1.0, wl.sm_scale,
                                                  wl.block_tables, wl.block_size, W)
    q.put((rank, float(np.abs(out - ref_o).max()), float(np.abs(lse - ref_l).max())))
    dist.destroy_process_group()


def _spawn(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_replica_time_is_max_over_ranks():
    res = _spawn(_replica_worker)
    assert [r[1] for r in res] == [2.5, 2.5]


def test_dcp_state_exchange_over_two_ranks_matches_single_process():
    res = _spawn(_dcp_worker)
    for _, eo, el in res:
        assert eo < 1e-12 and el < 1e-12
