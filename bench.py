#!/usr/bin/env python3
"""Benchmark of the MLA decode / causal-verify hot path on GB300.

One step = the whole path over one batch: row plan + sub-page expansion
(mla_plan_rows), split-K decode (mla_decode_verify's decode kernel) and the
segment merge into bf16 out + natural-log LSE.  Default workload: causal MTP
verify, qlen 4, bf16 cache, batch 32, 16 heads, seq_len U{1k..8k}, block 64,
16 split-K segments (seeded synthetic data).

Metric: KV-read GB/s = unique visible latent bytes (sum over requests of the
longest row's window x 1152 B) / step time, plus query rows / s.  Inputs are
resident in HBM; L2 is flushed (256 MiB write) before every timed step and the
flush is outside each step's CUDA-event bracket; the step is one CUDA graph.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun): every rank runs an independent replica (weak scaling:
requests are independent, no collective on the data path); value = all
ranks' KV bytes / the slowest rank's time.  --impl reference times the float64
CPU oracle on the host cores on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="verify_mtp4",
                    choices=["verify_mtp4", "fp8_mixed", "dcp8", "decode_qlen1"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def make_workload(name, seed, device=None):
    from mla_decode_speculative_gb300 import workloads
    if name == "verify_mtp4":
        return workloads.verify_mtp4_bf16(seed=seed)
    if name == "fp8_mixed":
        return workloads.fp8_mixed_qlen(seed=seed)
    if name == "dcp8":
        return workloads.dcp8_verify_bf16(seed=seed, device=device)
    return workloads.decode_qlen1_bf16(seed=seed)


def kv_bytes(wl) -> int:
    """Unique visible latent bytes of one step: each request's longest row sees
    its whole seq_len; W shards together hold every position once."""
    per_tok = 576 if wl.kv_dtype == "fp8" else 1152
    return int(wl.seq_lens.astype(np.int64).sum()) * per_tok


def _balanced_parts(unit_tiles, S, grid):
    """Tile ranges of the balanced split's parts, per unit (the rule of
    MLA_DECODE_UNIFORM_SEGMENTS's default in the C header): the units' T tiles
    end to end, n = min(grid, T // ceil(tmax / (S-1))) chunks
    [floor(cT/n), floor((c+1)T/n)); a unit's part in chunk c is one segment."""
    T, tmax = int(sum(unit_tiles)), int(max(unit_tiles))
    need = max(-(-tmax // (S - 1)), 1)
    n = min(grid, max(T // need, 1)) if T else 1
    bounds = [c * T // n for c in range(n + 1)]
    parts, start = [], 0
    for t in unit_tiles:
        t = int(t)
        c0 = next((c for c in range(n) if bounds[c + 1] > start), n) if t else n
        lst = []
        c = c0
        while t and c < n and bounds[c] < start + t:
            lst.append((max(bounds[c], start) - start, min(bounds[c + 1], start + t) - start))
            c += 1
        parts.append(lst)
        start += t
    return parts


def decode_unit_bytes(wl, grid=None) -> dict:
    """Algorithmic bytes of one launch of the decode kernel (all shard views
    of a sharded step in the one launch): visible KV rows, the query rows
    (once per view), and the split-K partials it must write (an (m, l) pair
    for every (view, row, head, segment slot), a 1 KiB bf16 vector for every
    (row, head, part) that holds a visible token).  Parts follow the split
    the call takes: balanced (S > 1, at most 1024 (view, request, row block)
    units; grid = the launch's CTAs) or the pages' equal split."""
    P = min(128, wl.block_size & -wl.block_size)
    S = wl.num_segments
    W, I, H, B = wl.world_size, wl.interleave, wl.num_heads, wl.num_reqs

    def local(w, r):  # positions of a window of w that shard r holds (runs of I dealt in turn)
        rem = min(max(w % (I * W) - r * I, 0), I)
        return (w // (I * W)) * I + rem

    RB = -(-int(max(wl.qlens)) * H // 64)
    max_len = max(1, -(-int(wl.max_kv_len) // P)) * P  # the static bound the step passes
    balanced = S > 1 and W * B * RB <= 1024 and W * B * RB * -(-max_len // 64) <= 2 ** 31 - 1
    active = 0
    if balanced:
        if grid is None:
            import torch
            grid = torch.cuda.get_device_properties(0).multi_processor_count
        grid = min(grid, W * B * RB * S)
        units = []
        for r in range(W):
            for b in range(B):
                L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
                ln = max(local(L - ql + 1 + t, r) for t in range(ql))
                units += [-(-ln // 64) if rb * 64 < ql * H else 0 for rb in range(RB)]
        parts = _balanced_parts(units, S, grid)
        for r in range(W):
            for b in range(B):
                L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
                for t in range(ql):
                    w = local(L - ql + 1 + t, r)
                    for h in range(H):
                        pl = parts[(r * B + b) * RB + (t * H + h) // 64]
                        active += sum(1 for lo, _ in pl if lo * 64 < w)
    else:
        for r in range(W):
            for b in range(B):
                L, ql = int(wl.seq_lens[b]), int(wl.qlens[b])
                tps_tok = max(1, -(-local(L, r) // (S * P))) * P
                for t in range(ql):
                    active += -(-local(L - ql + 1 + t, r) // tps_tok) * H
    kv = kv_bytes(wl)
    q = W * wl.num_rows * H * 1152  # each shard view reads the queries
    partial = (W * wl.num_rows * H * S * 8 + active * 1024) if S > 1 else \
        W * wl.num_rows * H * (1024 + 4)
    return {"kv": kv, "q": q, "partials": partial, "total": kv + q + partial}


class ClockSampler:
    """nvidia-smi sampled every 20 ms in the background; samples are kept with
    host timestamps so the timed region can be selected afterwards."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
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


def oracle_cpu_baseline(wl, target_s: float):
    """Times the float64 oracle (as it stands) on a prefix of whole requests
    sized to about target_s seconds of host CPU work."""
    import oracle
    oracle.build()
    q = wl.q_bits()
    kv = wl.kv_host()
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)

    def run(nreq):
        ind = wl.qo_indptr[:nreq + 1]
        t0 = time.perf_counter()
        oracle.attention(ind, row_len[:ind[-1]], q[:ind[-1]], kv, wl.kv_scale, wl.sm_scale,
                         wl.block_tables[0], wl.block_size)
        return time.perf_counter() - t0

    t1 = run(1)
    per_tok = 576 if wl.kv_dtype == "fp8" else 1152
    L0 = int(wl.seq_lens[0])
    est = t1 / max(L0, 1)  # seconds per visible token-request
    n, acc = 1, L0
    while n < wl.num_reqs and (acc + int(wl.seq_lens[n])) * est <= target_s:
        acc += int(wl.seq_lens[n])
        n += 1
    t = run(n)
    nb = int(wl.seq_lens[:n].astype(np.int64).sum()) * per_tok
    rows = int(wl.qo_indptr[n])
    return {"value": nb / t / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {n} of {wl.num_reqs} requests ({rows} verify rows x "
                      f"{wl.num_heads} heads, {nb / 1e6:.1f} MB of visible KV), {t:.2f} s",
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
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    H = wl.num_heads
    per_tok = 576 if wl.kv_dtype == "fp8" else 1152
    # each (row, head) item is charged its request's unique KV bytes / (rows x heads)
    items = [(r, h) for r in range(wl.num_rows) for h in range(H)]
    req = np.searchsorted(wl.qo_indptr, np.arange(wl.num_rows), side="right") - 1
    charge = np.array([wl.seq_lens[req[r]] * per_tok / (wl.qlens[req[r]] * H) for r, _ in items])
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    # calibrate items per step
    probe = np.array(items[:16], np.int32)
    t0 = time.perf_counter()
    oracle.attention(wl.qo_indptr, row_len, q, kv, wl.kv_scale, wl.sm_scale, wl.block_tables[0],
                     wl.block_size, sel=probe)
    per_item = (time.perf_counter() - t0) / len(probe)
    k = max(1, min(len(items), int(budget / max(per_item, 1e-9))))
    rng = np.random.default_rng(0)
    order = rng.permutation(len(items))
    pos = 0
    tot_t, tot_b, tot_rows = 0.0, 0.0, 0.0
    for step in range(args.warmup + args.steps):
        idx = order[np.arange(pos, pos + k) % len(items)]
        pos += k
        sel = np.array([items[i] for i in idx], np.int32)
        t0 = time.perf_counter()
        oracle.attention(wl.qo_indptr, row_len, q, kv, wl.kv_scale, wl.sm_scale,
                         wl.block_tables[0], wl.block_size, sel=sel)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            tot_t += dt
            tot_b += float(charge[idx].sum())
            tot_rows += k / H
    value = tot_b / tot_t / 1e9
    cpu = {"kind": "oracle", "cores": oracle.num_threads(), "value": value, "unit": "GB/s",
           "sample": f"{k} (row, head) items per step drawn from the workload, each charged its "
                     f"request's visible KV bytes / (rows x heads)"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, **wl.describe()},
            "query_rows_per_s": tot_rows / tot_t, "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def source_hash() -> str:
    h = hashlib.sha256()
    for f in ("mla_decode.cu", "mla_ptx.cuh"):
        with open(os.path.join(ROOT, "mla_decode_speculative_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


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

    from mla_decode_speculative_gb300 import build, mla, runner
    build.build()
    dev = torch.device("cuda", local)
    wl = make_workload(args.workload, seed=rank, device=dev if args.workload == "dcp8" else None)
    step = runner.step_for_workload(wl, dev)
    q, kv, seq, ind, bt = runner.device_inputs(wl, dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def one_step():
        step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            one_step()
    torch.cuda.synchronize()
    code = mla.get_device_error()
    if code:
        raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} during warm-up")

    # the whole step as one CUDA graph
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        one_step()
    torch.cuda.synchronize()

    # decode kernel alone (partials only), for the roofline
    dgraph = None
    if wl.num_segments > 1:
        # the row plan / shard views of the warm-up steps stay in the step's buffers
        W = wl.world_size
        dgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(dgraph, stream=stream):
            if W == 1:
                mla.decode_verify(q, kv, ind, step.row_len, step.subpage[0], step.P, step.S,
                                  step.max_qlen, wl.sm_scale, wl.kv_scale, out=step.out,
                                  lse=step.lse, workspace=step.workspace, skip_merge=True)
            else:
                mla.decode_verify(q, kv, ind, step.row_len_local, step.subpage, step.P, step.S,
                                  step.max_qlen, wl.sm_scale, wl.kv_scale, out=step.part_out,
                                  lse=step.part_lse, workspace=step.workspace, skip_merge=True,
                                  num_views=W)
        torch.cuda.synchronize()

    def timed(g, n):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        with torch.cuda.stream(stream):
            for k in range(n):
                # a ~50 us device spin ahead of the flush keeps the launch queue
                # ahead of the GPU, so no host-side delay falls inside a bracket
                torch.cuda._sleep(100000)
                flush.zero_()
                starts[k].record(stream)
                g.replay()
                ends[k].record(stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):  # graph warm-up under the same load
            flush.zero_()
            graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    step_ms = timed(graph, args.steps)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    mean_ms = max_over_ranks(float(np.mean(step_ms)), dist, dev)
    dec_ms = None
    if dgraph is not None:
        dec_ms = float(np.mean(timed(dgraph, max(20, min(args.steps, 500)))))
    clocks = sampler.summary(t_wall0, t_wall1)
    sampler.stop()
    code = mla.get_device_error()
    if code:
        raise RuntimeError(f"device error {mla.DEVICE_ERRORS.get(code, code)} while timing")

    # end to end through the public API: pinned host inputs in, results out
    e2e = None
    if not args.no_e2e:
        h_q = wl.q.pin_memory()
        h_seq = torch.as_tensor(wl.seq_lens, dtype=torch.int32).pin_memory()
        h_ind = torch.as_tensor(wl.qo_indptr, dtype=torch.int32).pin_memory()
        h_bt = torch.as_tensor(wl.block_tables, dtype=torch.int32).pin_memory()
        h_out = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
        h_lse = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
        d_q, d_seq, d_ind, d_bt = (torch.empty_like(x, device=dev) for x in (h_q, h_seq, h_ind, h_bt))
        n_e2e = max(20, min(args.steps, 300))
        s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        with torch.cuda.stream(stream):
            for k in range(n_e2e + 3):
                flush.zero_()
                if k >= 3:
                    s_ev[k - 3].record(stream)
                d_q.copy_(h_q, non_blocking=True)
                d_seq.copy_(h_seq, non_blocking=True)
                d_ind.copy_(h_ind, non_blocking=True)
                d_bt.copy_(h_bt, non_blocking=True)
                o, l = step(d_q, kv, d_seq, d_ind, d_bt, wl.sm_scale, wl.kv_scale)
                h_out.copy_(o, non_blocking=True)
                h_lse.copy_(l, non_blocking=True)
                if k >= 3:
                    e_ev[k - 3].record(stream)
                stream.synchronize()
        e2e_ms = max_over_ranks(float(np.mean([s.elapsed_time(e) for s, e in zip(s_ev, e_ev)])),
                                dist, dev)
        bi = sum(x.numel() * x.element_size() for x in (h_q, h_seq, h_ind, h_bt))
        bo = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
        e2e = {"value": world * kv_bytes(wl) / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "path": "runner.VerifyStep (C ABI, eager) with pinned host buffers; KV cache "
                       "resident on the device"}

    peaks, peak_kind = measured_peaks()
    roofline = None
    if dec_ms is not None:
        ub = decode_unit_bytes(wl)
        achieved = ub["total"] / (dec_ms * 1e-3) / 1e9
        traffic = None
        try:
            with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
                tr = json.load(f)
            for ent in tr.get("entries", [tr]):
                if ent.get("kernel_source_sha256") == source_hash() and ent.get("workload") == wl.name:
                    traffic = ent.get("bytes_per_launch")
        except (OSError, ValueError, AttributeError):
            pass
        roofline = {"kernel": "mla_decode_kernel<bf16>" if wl.kv_dtype == "bf16" else
                    "mla_decode_kernel<fp8>", "bound": "hbm", "achieved": achieved,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                    "traffic": traffic, "algorithmic_bytes": ub,
                    "avg_launch_ms": dec_ms,
                    "kv_only_gbs": ub["kv"] / (dec_ms * 1e-3) / 1e9}

    kvb = kv_bytes(wl)
    value = world * kvb / (mean_ms * 1e-3) / 1e9
    # plan (1) + decode (1) + segment merge (1 if S > 1); sharded: plan + W
    # shard views + one decode over the W views + segment merge + state merge
    per_decode = 2 if wl.num_segments > 1 else 1
    launches_per_step = (1 + per_decode if wl.world_size == 1 else
                         1 + wl.world_size + per_decode + 1)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.kv_dtype == "bf16" else "fp8_e4m3 cache, bf16 MMA",
            "data": "synthetic",
            "config": {**wl.describe(), "parallelism": f"replicas x{world}" if world > 1 else "1 gpu",
                       "l2": "flushed (256 MiB write) before every step, outside the timed bracket",
                       "launch": "one CUDA graph per step", "seed": "rank"},
            "hbm_frac_of_measured": value / world / peaks["hbm_gbs"],
            "query_rows_per_s": world * wl.num_rows / (mean_ms * 1e-3),
            "head_rows_per_s": world * wl.num_rows * wl.num_heads / (mean_ms * 1e-3),
            "roofline": roofline, "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks, "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
