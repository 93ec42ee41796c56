#!/usr/bin/env python3
"""Benchmark of the MLA decode / causal-verify hot path on GB300.

One step = the whole path over one batch.  Default workload: the simulated
8-way round-robin context-sharded verify (batch 16, 16 heads, qlen 4, context
131072, bf16 cache, block 64): mla_plan_rows (global windows) -> the 8 shard
row views with their sub-page tables (one mla_shard_row_views launch) -> one
mla_decode_verify launch over the 8 views (balanced split-K) -> segment
merge into the 8 shard states -> cross-shard natural-log LSE merge into bf16
out + LSE.

Metric: KV-read GB/s = unique visible latent bytes (every position of every
request once, 1152 B bf16 / 576 B fp8) / step time, plus query rows / s.
Inputs are resident in HBM; L2 is flushed (256 MiB write) before every timed
step, outside each step's CUDA-event bracket; the step is one CUDA graph.
The same line carries, under "workloads", the other two bandwidth configs
(qlen-4 verify over 1k-8k contexts; fp8 e4m3 cache with mixed qlen), each
timed the same way, and under "merge" the merge kernels against HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload dcp8|verify_mtp4|fp8_mixed|decode_qlen1]

N > 1 (under torchrun): every rank runs an independent replica (weak scaling:
requests are independent, no collective on the data path); value = all
ranks' KV bytes / the slowest rank's time.  --impl reference times the float64
CPU oracle on the host cores on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode/verify KV-read GB/s (% of GB300 HBM peak) and query-rows/sec"
L2_FLUSH_BYTES = 256 << 20
WORKLOADS = ["dcp8", "verify_mtp4", "fp8_mixed", "decode_qlen1", "wide_rows"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dcp8", choices=WORKLOADS)
    ap.add_argument("--extra", default="verify_mtp4,fp8_mixed,wide_rows,decode_qlen1",
                    help="comma-separated workloads also timed into the line ('none': skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-merge", action="store_true", help="skip the bandwidth-sized merge leg")
    ap.add_argument("--no-fused", action="store_true", help="skip the in-kernel merge comparison")
    ap.add_argument("--sweep", type=int, default=100, metavar="N",
                    help="time the first N points of the seeded 100-point sweep (full size, split-K "
                         "S=16) and add per-point roofline fractions under 'sweep' (0: skip)")
    ap.add_argument("--merge-only", action="store_true",
                    help="time only the bandwidth-sized segment merge and print its figures (for profiling)")
    return ap.parse_args()


def make_workload(name, seed, device=None):
    from mla_decode_speculative_gb300 import workloads
    if name == "verify_mtp4":
        return workloads.verify_mtp4_bf16(seed=seed, device=device)
    if name == "fp8_mixed":
        return workloads.fp8_mixed_qlen(seed=seed, device=device)
    if name == "dcp8":
        return workloads.dcp8_verify_bf16(seed=seed, device=device)
    if name == "wide_rows":
        # the sweep's widest rows: 128 heads x qlen 8 (16 64-row blocks per
        # request), seq_len U{6k..12k}, bf16, block 64, 8 split-K slots
        g = np.random.default_rng(seed + 911)
        L = g.integers(6000, 12001, 6)
        return workloads.make_workload("wide_rows_bf16_b6_h128_qlen8_L6k-12k_bs64_s8", L, [8] * 6, 128, 64,
                                       "bf16", 1, 8, seed, device=device)
    return workloads.decode_qlen1_bf16(seed=seed)


def kv_bytes(wl) -> int:
    """Unique visible latent bytes of one step: each request's longest row sees
    its whole seq_len; the W shards together hold every position once."""
    per_tok = 576 if wl.kv_dtype == "fp8" else 1152
    return int(wl.seq_lens.astype(np.int64).sum()) * per_tok


def _balanced_parts(unit_tiles, S, grid):
    """Tile ranges of the balanced split's parts, per unit (the default split of
    mla_decode_verify as its header states it): each unit with t > 0 tiles is
    one overhead position then its t tiles, V positions end to end,
    n = min(grid, V // ceil(tmax / (S-1))) chunks [floor(cV/n), floor((c+1)V/n));
    a unit's part in chunk c is one segment."""
    V = int(sum(int(t) + 1 for t in unit_tiles if int(t) > 0))
    tmax = int(max(unit_tiles))
    need = max(-(-tmax // (S - 1)), 1)
    n = min(grid, max(V // need, 1)) if V else 1
    bounds = [c * V // n for c in range(n + 1)]
    parts, pos = [], 0
    for t in unit_tiles:
        t = int(t)
        lst = []
        if t:
            start = pos + 1  # past the overhead position
            c = next(c for c in range(n) if bounds[c + 1] > start)
            while c < n and bounds[c] < start + t:
                lst.append((max(bounds[c], start) - start, min(bounds[c + 1], start + t) - start))
                c += 1
            pos = start + t
        parts.append(lst)
    return parts


def _local(w, r, W, I):
    """Positions of a window of w that shard r of W holds (runs of I dealt in turn)."""
    rem = min(max(w % (I * W) - r * I, 0), I)
    return (w // (I * W)) * I + rem


def is_balanced(wl, uniform=False):
    """Whether mla_decode_verify takes the balanced split for this workload
    (S > 1, at most 1024 (view, request, row block) units, tile counts within
    int32), which MLA_DECODE_FUSED_MERGE needs."""
    P = min(128, wl.block_size & -wl.block_size)
    S = wl.num_segments
    W, B, H = wl.world_size, wl.num_reqs, wl.num_heads
    RB = -(-int(max(wl.qlens)) * H // 64)
    max_len = max(1, -(-int(wl.max_kv_len) // P)) * P  # the static bound the step passes
    return (not uniform and S > 1 and W * B * RB <= 1024
            and W * B * RB * (-(-max_len // 64) + 1) <= 2 ** 31 - 1)


def balanced_units(wl, grid=None):
    """Per (view, request, row block) unit of the balanced split: (rows of the
    unit with their visible lengths, the unit's parts as tile ranges)."""
    S = wl.num_segments
    W, I, H, B = wl.world_size, wl.interleave, wl.num_heads, wl.num_reqs
    RB = -(-int(max(wl.qlens)) * H // 64)
    if grid is None:
        grid = torch.cuda.get_device_properties(0).multi_processor_count
    grid = min(grid, W * B * RB * S)
    tiles, rows = [], []
    for r in range(W):
        for b in range(B):
            L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
            lens = [_local(L - ql + 1 + t, r, W, I) for t in range(ql)]
            for rb in range(RB):
                rl = [lens[(rb * 64 + i) // H] for i in range(64) if rb * 64 + i < ql * H]
                rows.append(rl)
                tiles.append(-(-max(lens) // 64) if rl else 0)
    return list(zip(rows, _balanced_parts(tiles, S, grid)))


def split_parts(wl, grid=None, uniform=False):
    """(active, S, balanced): active = (view, row, head, part) triples whose part
    holds at least one visible token of that row, under the split the call takes."""
    P = min(128, wl.block_size & -wl.block_size)
    S = wl.num_segments
    W, I, H, B = wl.world_size, wl.interleave, wl.num_heads, wl.num_reqs
    balanced = is_balanced(wl, uniform)
    active = 0
    if S == 1:
        return 0, 1, False
    if balanced:
        for rl, pl in balanced_units(wl, grid):
            active += sum(1 for w in rl for lo, _ in pl if lo * 64 < w)
    else:
        for r in range(W):
            for b in range(B):
                L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
                ln = max(_local(L - ql + 1 + t, r, W, I) for t in range(ql))
                seg_tok = max(1, -(-ln // (S * P))) * P
                for t in range(ql):
                    active += -(-_local(L - ql + 1 + t, r, W, I) // seg_tok) * H
    return active, S, balanced


def algorithmic_flops(wl) -> int:
    """2 * sum over (view, row, head) of the row's visible tokens * (576 + 512):
    the QK^T and PV multiply-adds of the exact causal windows (unpadded heads,
    masked keys excluded)."""
    W, I, H = wl.world_size, wl.interleave, wl.num_heads
    tot = 0
    for r in range(W):
        for b in range(wl.num_reqs):
            L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
            tot += sum(_local(L - ql + 1 + t, r, W, I) for t in range(ql))
    return 2 * H * tot * (576 + 512)


def decode_unit_bytes(wl, grid=None, uniform=False) -> dict:
    """Algorithmic bytes of one launch of the decode kernel (all shard views of
    a sharded step in the one launch): the visible KV rows, the query rows
    (once per view), and what the split writes -- an (m, l) pair for every
    (view, row, head, segment slot) and a 1 KiB bf16 vector for every
    (view, row, head, part) that holds a visible token; with one segment the
    bf16 output row + LSE of every (view, row, head)."""
    W, H = wl.world_size, wl.num_heads
    active, S, _ = split_parts(wl, grid, uniform)
    kv = kv_bytes(wl)
    q = W * wl.num_rows * H * 1152
    partial = (W * wl.num_rows * H * S * 8 + active * 1024) if S > 1 else \
        W * wl.num_rows * H * (1024 + 4)
    return {"kv": kv, "q": q, "partials": partial, "total": kv + q + partial}


def fused_decode_bytes(wl, grid=None) -> dict:
    """Algorithmic bytes of one launch of the decode kernel that also merges
    its split-K parts (MLA_DECODE_FUSED_MERGE): the visible KV rows, the
    query rows (once per view), every (view, row, head)'s bf16 output row and
    float32 LSE, and for the units cut into two or more parts the partials
    written and read back once -- a 1 KiB bf16 vector per (row, head, part)
    with a visible token, the (m, l) pairs of all S slots written (8 B each)
    and those of the unit's parts read."""
    W, H, S = wl.world_size, wl.num_heads, wl.num_segments
    kv = kv_bytes(wl)
    q = W * wl.num_rows * H * 1152
    out = W * wl.num_rows * H * (1024 + 4)
    partial = 0
    for rl, pl in balanced_units(wl, grid):
        if len(pl) < 2:
            continue
        act = sum(1 for w in rl for lo, _ in pl if lo * 64 < w)
        partial += 2 * act * 1024 + len(rl) * (S + len(pl)) * 8
    return {"kv": kv, "q": q, "out": out, "partials": partial, "total": kv + q + out + partial}


def segment_merge_bytes(wl, grid=None, uniform=False) -> dict:
    """Algorithmic bytes of the segment merge: the live partial vectors (1 KiB
    bf16 per (view, row, head, part) with a token) and every slot's (m, l)
    pair read, the bf16 output row and float32 LSE of every (view, row, head)
    written."""
    W, H = wl.world_size, wl.num_heads
    active, S, _ = split_parts(wl, grid, uniform)
    rd = active * 1024 + W * wl.num_rows * H * S * 8
    wr = W * wl.num_rows * H * (1024 + 4)
    return {"read": rd, "write": wr, "total": rd + wr, "live_parts": active}


def state_merge_bytes(wl) -> dict:
    """Algorithmic bytes of the cross-shard merge: W bf16 states + LSEs read per
    (row, head) (every shard of these long windows is non-empty), one written."""
    n = wl.num_rows * wl.num_heads
    rd = wl.world_size * n * (1024 + 4)
    wr = n * (1024 + 4)
    return {"read": rd, "write": wr, "total": rd + wr}


class ClockSampler:
    """nvidia-smi sampled every 20 ms in the background; samples are kept with
    host timestamps so the timed region can be selected afterwards."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        self.index = index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if len(win) < 3:
            win = [s for s in self.samples if t0 - 2.0 <= s[0] <= t1]
            window = "timed+preceding 2 s of warm-up under the same load"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, pw = [], [], []
        for _, p in win:
            try:
                sm.append(float(p[0]))
                smax.append(float(p[1]))
                pw.append(float(p[2]))
            except ValueError:
                pass
            for k, n in enumerate(names):
                if p[3 + k].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(win), "window": window}


# ----------------------------------------------------------------------------
# the float64 oracle on the host cores (cpu_baseline leg and --impl reference)

def _oracle_attention(wl, row_len, q, kv, ind, sel=None, nreq=None):
    """The oracle over requests [0, nreq) (or the (row, head) pairs sel): plain
    attention for an unsharded workload; for a context-sharded one the pages'
    row view [vLLM #51705, 实现拆解 2] -- every shard attends its positions of
    each row's global window through its own block table, then the shard
    states are merged -- exactly as the GPU step does it."""
    import oracle
    if nreq is not None:
        ind = ind[:nreq + 1]
        rows = int(ind[-1])
        row_len, q = row_len[:rows], q[:rows]
        tables = wl.block_tables[:, :nreq]
    else:
        tables = wl.block_tables
    if wl.world_size == 1:
        return oracle.attention(ind, row_len, q, kv, wl.kv_scale, wl.sm_scale, tables[0],
                                wl.block_size, sel=sel)
    out, lse, _, _ = oracle.sharded_attention(ind, row_len, q, kv, wl.kv_scale, wl.sm_scale, tables,
                                              wl.block_size, wl.world_size, sel=sel,
                                              interleave=wl.interleave)
    return out, lse


def oracle_cpu_baseline(wl, target_s: float):
    """Times the float64 oracle (as it stands) on a prefix of whole requests
    sized to about target_s seconds of host CPU work."""
    import oracle
    oracle.build()
    q = wl.q_bits()
    kv = wl.kv_host()
    ind = wl.qo_indptr
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, ind)

    def run(nreq):
        t0 = time.perf_counter()
        _oracle_attention(wl, row_len, q, kv, ind, nreq=nreq)
        return time.perf_counter() - t0

    t1 = run(1)
    per_tok = 576 if wl.kv_dtype == "fp8" else 1152
    L0 = int(wl.seq_lens[0])
    est = t1 / max(L0, 1)  # seconds per visible position of a request
    n, acc = 1, L0
    while n < wl.num_reqs and (acc + int(wl.seq_lens[n])) * est <= target_s:
        acc += int(wl.seq_lens[n])
        n += 1
    t = run(n)
    nb = int(wl.seq_lens[:n].astype(np.int64).sum()) * per_tok
    rows = int(ind[n])
    how = (f"{wl.world_size} shard row views + state merge, " if wl.world_size > 1 else "")
    return {"value": nb / t / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {n} of {wl.num_reqs} requests ({rows} verify rows x {wl.num_heads} heads, "
                      f"{how}{nb / 1e6:.1f} MB of visible KV), {t:.2f} s",
            "query_rows_per_s": rows / t}


def run_reference(args):
    """--impl reference: the float64 CPU oracle on the host cores, same metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = make_workload(args.workload, 0)
    q = wl.q_bits()
    kv = wl.kv_host()
    ind = wl.qo_indptr
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, ind)
    H = wl.num_heads
    per_tok = 576 if wl.kv_dtype == "fp8" else 1152
    # each (row, head) pair is charged its request's unique KV bytes / (rows x heads)
    items = np.array([(r, h) for r in range(wl.num_rows) for h in range(H)], np.int32)
    req = np.searchsorted(ind, np.arange(wl.num_rows), side="right") - 1
    charge = np.array([wl.seq_lens[req[r]] * per_tok / (wl.qlens[req[r]] * H) for r, _ in items])
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    probe = items[:16]
    t0 = time.perf_counter()
    _oracle_attention(wl, row_len, q, kv, ind, sel=probe)
    per_item = (time.perf_counter() - t0) / len(probe)
    k = max(1, min(len(items), int(budget / max(per_item, 1e-9))))
    rng = np.random.default_rng(0)
    order = rng.permutation(len(items))
    pos = 0
    tot_t, tot_b, tot_rows = 0.0, 0.0, 0.0
    for step in range(args.warmup + args.steps):
        idx = order[np.arange(pos, pos + k) % len(items)]
        pos += k
        t0 = time.perf_counter()
        _oracle_attention(wl, row_len, q, kv, ind, sel=items[idx])
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            tot_t += dt
            tot_b += float(charge[idx].sum())
            tot_rows += k / H
    value = tot_b / tot_t / 1e9
    how = (f"through the {wl.world_size} shard row views and the state merge"
           if wl.world_size > 1 else "")
    cpu = {"kind": "oracle", "cores": oracle.num_threads(), "value": value, "unit": "GB/s",
           "sample": f"{k} (row, head) pairs per step drawn from the workload {how}, each charged "
                     f"its request's visible KV bytes / (rows x heads)"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, **wl.describe()},
            "query_rows_per_s": tot_rows / tot_t, "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------------------

def source_hash() -> str:
    h = hashlib.sha256()
    for f in ("mla_decode.cu", "mla_ptx.cuh"):
        with open(os.path.join(ROOT, "mla_decode_speculative_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(kernel: str, workload: str):
    """dram read + write bytes of one launch from the committed ncu summary, when
    it was taken on this kernel source and workload (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
            tr = json.load(f)
        for ent in tr.get("entries", [tr]):
            if (ent.get("kernel_source_sha256") == source_hash() and ent.get("workload") == workload
                    and ent.get("kernel", kernel) == kernel):
                return ent.get("bytes_per_launch")
    except (OSError, ValueError, AttributeError):
        pass
    return None


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's value (max all-reduce); the identity on one process."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class Timer:
    """CUDA-event timing of graph replays on one stream, L2 flushed (a 256 MiB
    write) before every replay, outside the bracket."""

    def __init__(self, stream, device):
        self.stream = stream
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self, g, n):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        with torch.cuda.stream(self.stream):
            for k in range(n):
                # a ~50 us device spin ahead of the flush keeps the launch queue
                # ahead of the GPU, so no host-side delay falls inside a bracket
                torch.cuda._sleep(100000)
                self.flush.zero_()
                starts[k].record(self.stream)
                g.replay()
                ends[k].record(self.stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def capture(stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def launches_per_step(wl, fused=False) -> int:
    """Library kernels one step launches: plan (1), the shard row views
    (sharded: one launch for all W), decode (1), segment merge (1 if S > 1,
    unless the decode merges its parts itself), state merge (sharded)."""
    seg = 1 if wl.num_segments > 1 and not fused else 0
    if wl.world_size == 1:
        return 2 + seg
    return 1 + 1 + 1 + seg + 1


class StepBench:
    """One workload's step, its graphs (whole step, decode alone, merges alone)
    and their timings.  fused: the decode merges its split-K parts itself
    (MLA_DECODE_FUSED_MERGE) instead of the separate segment merge."""

    def __init__(self, wl, dev, stream, timer, fused=False):
        from mla_decode_speculative_gb300 import mla, runner
        self.wl, self.dev, self.stream, self.timer = wl, dev, stream, timer
        self.mla = mla
        self.step = runner.step_for_workload(wl, dev, fused_merge=fused)
        self.inputs = runner.device_inputs(wl, dev)
        st = self.step
        with torch.cuda.stream(stream):
            for _ in range(3):
                self.run()
        torch.cuda.synchronize()
        code = mla.get_device_error()
        if code:
            raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} during warm-up")
        self.graph = capture(stream, self.run)
        # the row plan / shard views of the warm-up steps stay in the step's buffers
        q, kv, seq, ind, bt = self.inputs
        W, Q = wl.world_size, st.max_qlen
        self.dgraph = self.mgraph = self.sgraph = None
        # the decode call exactly as the step makes it (a segment merge launch
        # follows unless the decode merges its parts itself)
        self.fused = fused
        skip = wl.num_segments > 1 and not self.fused
        if W == 1:
            dec = lambda: mla.decode_verify(q, kv, ind, st.row_len, st.subpage[0], st.P, st.S, Q,
                                            wl.sm_scale, wl.kv_scale, out=st.out, lse=st.lse,
                                            workspace=st.workspace, skip_merge=skip, fused_merge=fused)
            mout, mlse = st.out, st.lse
        else:
            dec = lambda: mla.decode_verify(q, kv, ind, st.row_len_local, st.subpage, st.P, st.S, Q,
                                            wl.sm_scale, wl.kv_scale, out=st.part_out,
                                            lse=st.part_lse, workspace=st.workspace,
                                            skip_merge=skip, num_views=W, fused_merge=fused)
            mout, mlse = st.part_out, st.part_lse
        self.dgraph = capture(stream, dec)
        if skip:
            so, sm, ss = mla.workspace_views(st.workspace, wl.num_reqs, Q, wl.num_rows, wl.num_heads,
                                             st.S, num_views=W)
            self.mgraph = capture(stream, lambda: mla.merge_segments(so, sm, ss, ind, Q, out=mout,
                                                                     lse=mlse, num_views=W))
        if W > 1:
            self.sgraph = capture(stream, lambda: mla.merge_states(st.part_out, st.part_lse,
                                                                   out=st.out, lse=st.lse))

    def run(self):
        q, kv, seq, ind, bt = self.inputs
        return self.step(q, kv, seq, ind, bt, self.wl.sm_scale, self.wl.kv_scale)

    def parts(self, n):
        """Mean ms of the decode alone, the segment merge alone and the state
        merge alone (each graph replayed with its inputs in place)."""
        r = {}
        for key, g in (("decode", self.dgraph), ("segment_merge", self.mgraph),
                       ("state_merge", self.sgraph)):
            if g is not None:
                r[key] = float(np.mean(self.timer(g, n)))
        return r

    def summary(self, step_ms, parts, peaks, peak_kind):
        """The per-workload figures: KV GB/s of the step, the decode kernel's
        roofline, the merges' bandwidth."""
        wl = self.wl
        kvb = kv_bytes(wl)
        hbm = peaks["hbm_gbs"]
        res = {"workload": wl.name, "ms_per_step": step_ms,
               "kv_gbs": kvb / (step_ms * 1e-3) / 1e9,
               "hbm_frac_of_measured": kvb / (step_ms * 1e-3) / 1e9 / hbm,
               "query_rows_per_s": wl.num_rows / (step_ms * 1e-3),
               "head_rows_per_s": wl.num_rows * wl.num_heads / (step_ms * 1e-3),
               "launches_per_step": launches_per_step(wl, self.fused)}
        if "decode" in parts:
            ub = fused_decode_bytes(wl) if self.fused else decode_unit_bytes(wl)
            dms = parts["decode"]
            kname = "mla_decode_kernel<bf16>" if wl.kv_dtype == "bf16" else "mla_decode_kernel<fp8>"
            achieved = ub["total"] / (dms * 1e-3) / 1e9
            fl = algorithmic_flops(wl)
            ridge = peaks["bf16_tflops"] * 1e12 / (hbm * 1e9)  # FLOP per byte where the roofs meet
            if fl / ub["kv"] > ridge:
                # heads x qlen rows against one KV tile: a dense bf16 contraction
                tf = fl / (dms * 1e-3) / 1e12
                res["roofline"] = {
                    "kernel": kname, "bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                    "peak_source": f"{peak_kind} bf16_tflops (cuBLAS, burst)", "traffic": None,
                    "algorithmic_flops": fl, "intensity_flop_per_kv_byte": fl / ub["kv"],
                    "ridge_flop_per_byte": ridge, "avg_launch_ms": dms,
                    "kv_only_gbs": ub["kv"] / (dms * 1e-3) / 1e9, "algorithmic_bytes": ub}
            else:
                res["roofline"] = {
                    "kernel": kname, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                    "traffic": recorded_traffic(kname, wl.name), "algorithmic_bytes": ub,
                    "avg_launch_ms": dms, "kv_only_gbs": ub["kv"] / (dms * 1e-3) / 1e9,
                    "kv_only_frac": ub["kv"] / (dms * 1e-3) / 1e9 / hbm}
        merges = {}
        if "segment_merge" in parts:
            mb = segment_merge_bytes(wl)
            ms = parts["segment_merge"]
            merges["segment_merge"] = {"kernel": "merge_segment_octets", "bytes": mb, "avg_launch_ms": ms,
                                       "gbs": mb["total"] / (ms * 1e-3) / 1e9,
                                       "frac": mb["total"] / (ms * 1e-3) / 1e9 / hbm}
        if "state_merge" in parts:
            mb = state_merge_bytes(wl)
            ms = parts["state_merge"]
            merges["state_merge"] = {"kernel": "merge_states_small", "bytes": mb, "avg_launch_ms": ms,
                                     "gbs": mb["total"] / (ms * 1e-3) / 1e9,
                                     "frac": mb["total"] / (ms * 1e-3) / 1e9 / hbm}
        if merges:
            res["merges"] = merges
        return res


def sweep_leg(n_points, dev, stream, timer, peaks, peak_kind, reps=10):
    """The seeded sweep (heads {16,64,128} x batch 1-256 x context 4k-132k x
    qlen {1,2,4,8} x bf16/fp8 x block {16,64,256}) at full size, each point's
    step with 16 split-K slots: per point the decode kernel's time and its
    roofline fraction (HBM-bound or tensor-bound by its intensity against the
    measured ridge), and a summary per bound."""
    from mla_decode_speculative_gb300 import workloads
    points = workloads.sweep_points(100, seed=0)[:n_points]
    if n_points >= 100:  # the sweep's largest corner: 256 requests x 128 heads x qlen 8, context to 132k
        points.append(workloads.SweepPoint(128, 256, 135168, 8, "bf16", 64, 950))
    rows = []
    for p in points:
        wl = workloads.sweep_workload(p, device=dev, num_segments=16)
        sb = StepBench(wl, dev, stream, timer)
        with torch.cuda.stream(stream):
            for _ in range(3):
                timer.flush.zero_()
                sb.graph.replay()
        step_ms = float(np.mean(timer(sb.graph, reps)))
        s = sb.summary(step_ms, sb.parts(reps), peaks, peak_kind)
        r = s["roofline"]
        rb = -(-int(max(wl.qlens)) * wl.num_heads // 64)  # 64-row blocks per request
        rows.append([p.name(), round(kv_bytes(wl) / 1e6, 1), rb, round(step_ms * 1e3, 1),
                     round(r["avg_launch_ms"] * 1e3, 1), r["bound"], round(r["frac"], 3)])
        del sb, wl
        torch.cuda.empty_cache()
    summ = {}
    groups = {}
    for name, _, rb, _, _, bound, frac in rows:
        dt = "fp8" if "_fp8_" in name else "bf16"
        groups.setdefault(f"{bound}_rb{'1' if rb == 1 else '2+'}_{dt}", []).append(frac)
    for key in sorted(groups):
        fr = sorted(groups[key])
        summ[key] = {"points": len(fr), "median_frac": fr[len(fr) // 2], "min_frac": fr[0], "max_frac": fr[-1]}
    big = sorted((x for x in rows if x[5] == "hbm" and x[2] == 1 and "_bf16_" in x[0]), key=lambda x: -x[1])[:10]
    if big:
        summ["hbm_rb1_bf16_largest10_median_frac"] = sorted(x[6] for x in big)[len(big) // 2]
    return {"summary": summ,
            "columns": ["point", "kv_mb", "row_blocks", "step_us", "decode_us", "bound", "frac"],
            "points": rows,
            "note": "decode kernel alone (CUDA events, L2 flushed before each launch); frac of measured "
                    "HBM (algorithmic bytes) or of measured bf16 (algorithmic FLOPs) by the point's "
                    "intensity against the measured ridge"}


def bandwidth_sized_merge(dev, stream, timer, n, peaks):
    """The segment merge on an instance large enough to be bandwidth-bound: the
    pages' equal split (16 segments per request, [vLLM #51705, 实现拆解 4]) of a
    qlen-4 verify batch of 256 requests, 16 heads, seq_len U{1k..8k}; the
    partials come from a real decode launch.  Its inputs (~250 MB) exceed
    twice the L2, so launches are timed back to back (20 per CUDA-event
    bracket, no flush): each launch reads its partials from DRAM, and the
    graph-launch latency of a single replay is not charged to the kernel."""
    from mla_decode_speculative_gb300 import mla, runner, workloads
    wl = workloads.verify_mtp4_bf16(seed=5, batch=256, num_segments=16, device=dev)
    st = runner.step_for_workload(wl, dev, uniform_segments=True)
    q, kv, seq, ind, bt = runner.device_inputs(wl, dev)
    with torch.cuda.stream(stream):
        st(q, kv, seq, ind, bt, wl.sm_scale)
        mla.decode_verify(q, kv, ind, st.row_len, st.subpage[0], st.P, st.S, st.max_qlen, wl.sm_scale,
                          out=st.out, lse=st.lse, workspace=st.workspace, skip_merge=True,
                          uniform_segments=True)
    torch.cuda.synchronize()
    so, sm, ss = mla.workspace_views(st.workspace, wl.num_reqs, st.max_qlen, wl.num_rows, wl.num_heads, st.S)
    g = capture(stream, lambda: mla.merge_segments(so, sm, ss, ind, st.max_qlen, out=st.out, lse=st.lse))
    per = 20
    times = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        for _ in range(max(3, n // per)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(per):
                g.replay()
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in times])) / per
    mb = segment_merge_bytes(wl, uniform=True)
    code = mla.get_device_error()
    if code:
        raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} in the merge leg")
    gbs = mb["total"] / (ms * 1e-3) / 1e9
    return {"kernel": "merge_segment_octets", "workload": wl.name + "_uniform_split",
            "bytes": mb, "avg_launch_ms": ms, "gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
            "l2": f"inputs {mb['total'] / 1e6:.0f} MB > 2 x L2; {per} launches back to back per event bracket"}


def e2e_leg(sb, dev, stream, world, dist):
    """The same metric end to end through the public API: each step copies its
    inputs (q, seq_lens, qo_indptr, block tables, packed in one pinned block)
    to the device in one copy, runs the step's library calls and copies out +
    LSE back to pinned host memory in one copy; the copies and the calls are
    captured as one CUDA graph, replayed and synchronised once per step.  The
    KV cache stays resident on the device (it is the server's state, not a
    step input)."""
    from mla_decode_speculative_gb300 import runner
    wl, st = sb.wl, sb.step
    io = runner.StepIO(st, wl.q.shape, wl.num_reqs, wl.block_tables.shape, device=dev)
    io.stage(wl.q, wl.seq_lens, wl.qo_indptr, wl.block_tables)
    d_q, d_seq, d_ind, d_bt = io.device_inputs()
    kv = sb.inputs[1]

    def api_step():
        io.upload()  # one host-to-device copy of the packed inputs
        st(d_q, kv, d_seq, d_ind, d_bt, wl.sm_scale, wl.kv_scale)
        io.download()  # one device-to-host copy of out + lse

    def run(fn, n):
        s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        with torch.cuda.stream(stream):
            for k in range(n + 3):
                sb.timer.flush.zero_()
                if k >= 3:
                    s_ev[k - 3].record(stream)
                fn()
                if k >= 3:
                    e_ev[k - 3].record(stream)
                stream.synchronize()
        return float(np.mean([s.elapsed_time(e) for s, e in zip(s_ev, e_ev)]))

    n = 200
    g = capture(stream, api_step)
    ms = max_over_ranks(run(g.replay, n), dist, dev)
    eager_ms = max_over_ranks(run(api_step, n), dist, dev)
    bi = io.in_bytes
    bo = io.host_result.numel()
    kvb = kv_bytes(wl)
    return {"value": world * kvb / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "path": "runner.VerifyStep (C ABI) with runner.StepIO: the step's inputs packed in one "
                    "pinned block (one H2D copy), the step's library calls, out + lse in one D2H "
                    "copy, captured as one CUDA graph, one synchronisation per step; KV cache "
                    "resident on the device",
            "eager": {"value": world * kvb / (eager_ms * 1e-3) / 1e9, "ms_per_step": eager_ms,
                      "path": "the same calls issued from Python every step (no graph)"}}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from mla_decode_speculative_gb300 import build, mla
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    timer = Timer(stream, dev)
    peaks, peak_kind = measured_peaks()
    if args.merge_only:
        if rank == 0:
            print(json.dumps({"merge_only": bandwidth_sized_merge(dev, stream, timer, max(20, min(args.steps, 500)),
                                                                  peaks)}))
        return
    wl = make_workload(args.workload, seed=rank, device=dev)
    sb = StepBench(wl, dev, stream, timer)

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):  # graph warm-up under the same load
            timer.flush.zero_()
            sb.graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    step_ms = timer(sb.graph, args.steps)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    mean_ms = max_over_ranks(float(np.mean(step_ms)), dist, dev)
    n_parts = max(20, min(args.steps, 500))
    parts = sb.parts(n_parts)
    clocks = sampler.summary(t_wall0, t_wall1)
    code = mla.get_device_error()
    if code:
        raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} while timing")
    head = sb.summary(mean_ms, parts, peaks, peak_kind)

    e2e = None if args.no_e2e else e2e_leg(sb, dev, stream, world, dist)

    # the other configured bandwidth workloads, timed the same way
    extra = {}
    names = [] if args.extra in ("", "none") else [w for w in args.extra.split(",") if w != args.workload]
    for name in names:
        ewl = make_workload(name, seed=rank, device=dev)
        esb = StepBench(ewl, dev, stream, timer)
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                timer.flush.zero_()
                esb.graph.replay()
        ems = max_over_ranks(float(np.mean(timer(esb.graph, args.steps))), dist, dev)
        extra[name] = esb.summary(ems, esb.parts(n_parts), peaks, peak_kind)
        code = mla.get_device_error()
        if code:
            raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} in {name}")
        del esb, ewl
        torch.cuda.empty_cache()
    # the same workloads with the split-K parts merged inside the decode kernel
    fused_cmp = {}
    if not args.no_fused:
        for name in [args.workload] + names:
            fwl = wl if name == args.workload else make_workload(name, seed=rank, device=dev)
            if not is_balanced(fwl):
                continue
            fsb = StepBench(fwl, dev, stream, timer, fused=True)
            fms = max_over_ranks(float(np.mean(timer(fsb.graph, min(args.steps, 200)))), dist, dev)
            fsum = fsb.summary(fms, fsb.parts(min(args.steps, 200)), peaks, peak_kind)
            sep = head if name == args.workload else extra[name]
            fused_cmp[name] = {"ms_per_step": fms, "kv_gbs": fsum["kv_gbs"],
                               "decode_ms": fsum["roofline"]["avg_launch_ms"],
                               "separate_merge_ms_per_step": sep["ms_per_step"],
                               "flag": "MLA_DECODE_FUSED_MERGE"}
            code = mla.get_device_error()
            if code:
                raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} in fused {name}")
            del fsb
            torch.cuda.empty_cache()
    sweep = sweep_leg(args.sweep, dev, stream, timer, peaks, peak_kind) if args.sweep > 0 else None
    merge = dict(head.get("merges", {}))
    if not args.no_merge:
        merge["bandwidth_sized"] = bandwidth_sized_merge(dev, stream, timer, n_parts, peaks)
    clocks_all = sampler.summary(t_wall0, time.time())
    sampler.stop()

    kvb = kv_bytes(wl)
    value = world * kvb / (mean_ms * 1e-3) / 1e9
    gpu_launches = launches_per_step(wl) * args.steps
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.kv_dtype == "bf16" else "fp8_e4m3 cache, bf16 MMA",
            "data": "synthetic",
            "config": {**wl.describe(), "parallelism": f"replicas x{world}" if world > 1 else "1 gpu",
                       "shards": (f"{wl.world_size} round-robin context shards simulated on one GPU "
                                  "(all shard views in one decode launch, then the state merge)"
                                  if wl.world_size > 1 else "none"),
                       "l2": "flushed (256 MiB write) before every step, outside the timed bracket",
                       "launch": "one CUDA graph per step", "seed": "rank"},
            "hbm_frac_of_measured": value / world / peaks["hbm_gbs"],
            "query_rows_per_s": world * wl.num_rows / (mean_ms * 1e-3),
            "head_rows_per_s": world * wl.num_rows * wl.num_heads / (mean_ms * 1e-3),
            "roofline": head.get("roofline"), "gpu_launches": gpu_launches,
            "clocks": clocks, "e2e": e2e, "merge": merge or None,
            "workloads": {k: v for k, v in extra.items()},
            "fused_merge": fused_cmp or None,
            "clocks_whole_run": clocks_all}
    if sweep is not None:
        line["sweep"] = sweep
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
