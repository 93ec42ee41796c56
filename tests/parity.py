"""Shared parity machinery: run a workload through the C ABI, compute the
oracle on the same host bytes, compare with the stated tolerances.

Tolerances (the stated bar for this path): per (row, head) the output error
normalised by the row's scale, max_d |out - ref| / max_d |ref|, must be
<= 1e-2, and the natural-log LSE must agree to 1e-3 absolute.  Indexing
(row plan, shard view, sub-page tables) must be bit-exact.
"""
import numpy as np
import torch

import oracle

OUT_TOL = 1e-2
LSE_TOL = 1e-3


def rowwise_errors(out_gpu, lse_gpu, out_ref, lse_ref):
    """out_* [..., 512], lse_* [...] -> (normalised output error [...], lse error [...])."""
    og = out_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(out_gpu) else out_gpu
    lg = lse_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(lse_gpu) else lse_gpu
    scale = np.maximum(np.abs(out_ref).max(axis=-1), 1e-30)
    err = np.abs(og - out_ref).max(axis=-1) / scale
    both_inf = np.isneginf(lg) & np.isneginf(lse_ref)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(lg - lse_ref))
    # an empty row must be exactly zero with lse = -inf
    empty = np.isneginf(lse_ref)
    err = np.where(empty, np.abs(og).max(axis=-1), err)
    return err, lerr


def assert_close(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    err, lerr = rowwise_errors(out_gpu, lse_gpu, out_ref, lse_ref)
    assert np.isfinite(err).all() and np.isfinite(lerr).all(), f"{what}: non-finite result"
    assert err.max() <= OUT_TOL, f"{what}: normalised output error {err.max():.3e} > {OUT_TOL}"
    assert lerr.max() <= LSE_TOL, f"{what}: lse error {lerr.max():.3e} > {LSE_TOL}"
    return float(err.max()), float(lerr.max())


def oracle_reference(wl, sel=None):
    """Oracle (out, lse) of a workload; sel = [n, 2] (row, head) pairs or None."""
    q = wl.q_bits()
    kv = wl.kv_host()
    row_len, _, _ = oracle.plan_rows(wl.seq_lens, wl.qo_indptr)
    if wl.world_size == 1:
        return oracle.attention(wl.qo_indptr, row_len, q, kv, wl.kv_scale, wl.sm_scale,
                                wl.block_tables[0], wl.block_size, sel=sel)
    out, lse, _, _ = oracle.sharded_attention(wl.qo_indptr, row_len, q, kv, wl.kv_scale,
                                              wl.sm_scale, wl.block_tables, wl.block_size,
                                              wl.world_size, sel=sel, interleave=wl.interleave)
    return out, lse


def sample_pairs(wl, n, seed=0):
    """n (row, head) pairs: every request's last row and first row, plus random ones."""
    rng = np.random.default_rng(seed)
    ind = wl.qo_indptr
    rows = []
    for b in range(wl.num_reqs):
        rows += [ind[b], ind[b + 1] - 1]
    rows = np.array(rows)
    pick = rng.choice(rows, size=min(n // 2, rows.size), replace=False)
    extra = rng.integers(0, wl.num_rows, n - pick.size)
    r = np.concatenate([pick, extra])
    h = rng.integers(0, wl.num_heads, r.size)
    return np.stack([r, h], axis=1).astype(np.int32)


def run_gpu(wl, num_segments=None, device="cuda", uniform_segments=False):
    from mla_decode_speculative_gb300 import runner
    step = runner.step_for_workload(wl, device, num_segments, uniform_segments)
    q, kv, seq, ind, bt = runner.device_inputs(wl, device)
    out, lse = step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)
    torch.cuda.synchronize()
    return out, lse, step


def run_gpu_partials(wl, device="cuda"):
    """The workload's step (row plan + sub-page tables), then the decode alone
    with MLA_DECODE_SKIP_MERGE into the step's workspace: every unit's
    split-K partials and statistics stay there (the pages' two-step form),
    whatever the default path merges in-kernel.  Returns the step."""
    from mla_decode_speculative_gb300 import mla, runner
    step = runner.step_for_workload(wl, device)
    q, kv, seq, ind, bt = runner.device_inputs(wl, device)
    step(q, kv, seq, ind, bt, wl.sm_scale, wl.kv_scale)
    mla.decode_verify(q, kv, ind, step.row_len, step.subpage[0], step.P, step.S, step.max_qlen,
                      wl.sm_scale, wl.kv_scale, out=step.out, lse=step.lse, workspace=step.workspace,
                      skip_merge=True)
    torch.cuda.synchronize()
    return step


def rows_to_blocks(x, qo_indptr, num_heads, row_blocks):
    """[T, H, S, 512] per-(row, head) partials -> the decode workspace's block
    layout [B, RB, S, 8, 512, 8] (a request's rows t * H + h, 64 per block;
    block row i sits in row octet i // 8 at position i % 8 of each dim; unused
    rows left as NaN so that reading one would show)."""
    T, H, S, D = x.shape
    B = len(qo_indptr) - 1
    out = np.full((B, row_blocks, S, 8, D, 8), np.nan, dtype=x.dtype)
    flat = x.reshape(T * H, S, D)
    for b in range(B):
        r0, r1 = int(qo_indptr[b]) * H, int(qo_indptr[b + 1]) * H
        for i in range(r1 - r0):
            out[b, i // 64, :, (i % 64) // 8, :, i % 8] = flat[r0 + i]
    return out


def blocks_to_rows(blocks, qo_indptr, num_heads, num_rows):
    """Inverse of rows_to_blocks: [B, RB, S, 8, 512, 8] -> [T, H, S, 512]."""
    B, RB, S, _, D, _ = blocks.shape
    out = np.zeros((num_rows * num_heads, S, D), dtype=blocks.dtype)
    for b in range(B):
        r0, r1 = int(qo_indptr[b]) * num_heads, int(qo_indptr[b + 1]) * num_heads
        for i in range(r1 - r0):
            out[r0 + i] = blocks[b, i // 64, :, (i % 64) // 8, :, i % 8]
    return out.reshape(num_rows, num_heads, S, D)


def balanced_parts(unit_tiles, S, grid):
    """The balanced split as the header states it, restated for the test: a
    unit with t > 0 tiles is one overhead position followed by its t tiles;
    the V positions end to end are cut into n chunks [floor(cV/n),
    floor((c+1)V/n)) with n = min(grid, V // need), need = ceil(tmax / (S-1))
    (so no unit meets more than S chunks); unit u's part in chunk c is its
    segment c - (chunk of its first tile).  Returns {u: [(tile_lo, tile_hi)
    per segment]}."""
    V = sum(t + 1 for t in unit_tiles if t > 0)
    tmax = max(unit_tiles)
    need = max(-(-tmax // (S - 1)), 1)
    n = min(grid, max(V // need, 1)) if V else 1
    bounds = [c * V // n for c in range(n + 1)]
    parts, pos = {}, 0
    for u, t in enumerate(unit_tiles):
        start = pos + 1 if t else pos
        parts[u] = [(max(bounds[c], start) - start, min(bounds[c + 1], start + t) - start)
                    for c in range(n) if t and bounds[c] < start + t and bounds[c + 1] > start]
        pos = start + t
    return parts
