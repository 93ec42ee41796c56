"""The whole decode / verify step through the C ABI, with buffers allocated once.

``VerifyStep`` owns every device buffer one step needs (row plan, sub-page
tables, split-K workspace, shard partial states, outputs), sized by static
bounds, so a step issues only library launches and can be captured in a CUDA
graph.  Unsharded step: mla_plan_rows (+ sub-page expansion) ->
mla_decode_verify (decode + segment merge).  Context-sharded step (W round-robin
shards simulated on one device): mla_plan_rows (global windows) -> the W shard
row views in one mla_shard_row_views launch -> one mla_decode_verify over the
W row views (num_views = W)
into a [W, T, H, .] state buffer -> mla_merge_segments (state mode).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import mla


class VerifyStep:
    def __init__(self, *, num_reqs: int, num_rows: int, num_heads: int, max_qlen: int,
                 block_size: int, num_blocks: int, block_table_width: int, max_kv_len: int,
                 num_segments: int = 1, world_size: int = 1, kv_fp8: bool = False,
                 interleave: int = 1, uniform_segments: bool = False, fused_merge: bool = False,
                 device="cuda"):
        self.B, self.T, self.H = num_reqs, num_rows, num_heads
        self.max_qlen = max_qlen
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.W = world_size
        self.interleave = interleave
        self.S = num_segments
        self.uniform = uniform_segments  # the pages' equal split instead of the balanced one
        self.fused = fused_merge         # merge the balanced split's parts inside the decode kernel
        self.P = mla.page_size(block_size)
        self.sp_stride = max(1, -(-max_kv_len // self.P))
        self.kv_fp8 = kv_fp8
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.row_len = torch.empty(num_rows, **i32)
        self.row_req = torch.empty(num_rows, **i32)
        self.subpage = torch.empty((world_size, num_reqs, self.sp_stride), **i32)
        self.row_len_local = torch.empty((world_size, num_rows), **i32)
        # out and lse share one allocation (lse 256-byte aligned after out), so
        # a caller reads a step's result back in one copy (``StepIO``)
        out_bytes = num_rows * num_heads * mla.D_V * 2
        self.lse_offset = (out_bytes + 255) & ~255
        self.result = torch.empty(self.lse_offset + num_rows * num_heads * 4, dtype=torch.uint8, device=dev)
        self.out = self.result[:out_bytes].view(torch.bfloat16).view(num_rows, num_heads, mla.D_V)
        self.lse = self.result[self.lse_offset:].view(torch.float32).view(num_rows, num_heads)
        if world_size > 1:
            self.part_out = torch.empty((world_size, num_rows, num_heads, mla.D_V),
                                        dtype=torch.bfloat16, device=dev)
            self.part_lse = torch.empty((world_size, num_rows, num_heads), dtype=torch.float32,
                                        device=dev)
        a256 = lambda x: (x + 255) & ~255
        ws = 256  # work counter
        if num_segments > 1:
            items = world_size * num_rows * num_heads * num_segments
            units = world_size * num_reqs * mla.row_blocks(max_qlen, num_heads)
            blocks = units * num_segments
            ws += a256(blocks * 512 * 64 * 2) + 2 * a256(items * 4) + a256(units * 4)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def __call__(self, q: torch.Tensor, kv_cache: torch.Tensor, seq_lens: torch.Tensor,
                 qo_indptr: torch.Tensor, block_tables: torch.Tensor, sm_scale: float,
                 kv_scale: float = 1.0, stream=None):
        """block_tables: [W, B, width] int32 (W = 1 unsharded).  Returns (out, lse)."""
        if self.W == 1:
            mla.plan_rows(seq_lens, qo_indptr, self.T, block_tables[0], self.num_blocks,
                          self.block_size, self.sp_stride, row_len=self.row_len,
                          row_req=self.row_req, subpage_table=self.subpage[0], stream=stream)
            mla.decode_verify(q, kv_cache, qo_indptr, self.row_len, self.subpage[0], self.P,
                              self.S, self.max_qlen, sm_scale, kv_scale, out=self.out,
                              lse=self.lse, workspace=self.workspace, stream=stream,
                              uniform_segments=self.uniform, fused_merge=self.fused)
            return self.out, self.lse
        mla.plan_rows(seq_lens, qo_indptr, self.T, row_len=self.row_len, row_req=self.row_req,
                      stream=stream)
        # the W shard row views (one per simulated rank) in one launch
        mla.shard_row_views(qo_indptr, self.row_len, self.W, self.interleave, block_tables,
                            self.num_blocks, self.block_size, self.sp_stride,
                            row_len_local=self.row_len_local, subpage_tables=self.subpage,
                            stream=stream)
        # all W shard views in one decode launch, straight into the shard states
        mla.decode_verify(q, kv_cache, qo_indptr, self.row_len_local, self.subpage, self.P, self.S,
                          self.max_qlen, sm_scale, kv_scale, out=self.part_out, lse=self.part_lse,
                          workspace=self.workspace, stream=stream, num_views=self.W,
                          uniform_segments=self.uniform, fused_merge=self.fused)
        mla.merge_states(self.part_out, self.part_lse, out=self.out, lse=self.lse, stream=stream)
        return self.out, self.lse


class StepIO:
    """One step's host <-> device traffic in two copies.  The inputs (q,
    seq_lens, qo_indptr, block tables) live in one pinned host block and one
    device block at 256-byte aligned offsets; ``upload`` is a single
    host-to-device copy, after which ``device_inputs`` are views of the device
    block of the dtypes and shapes ``VerifyStep`` takes.  ``download`` copies the
    step's ``result`` block (out + lse) back in one device-to-host copy;
    ``out`` / ``lse`` are views of the pinned result block."""

    def __init__(self, step: VerifyStep, q_shape, num_reqs: int, block_tables_shape, device="cuda"):
        dev = torch.device(device)
        a256 = lambda x: (x + 255) & ~255
        specs = [("q", torch.bfloat16, tuple(q_shape)), ("seq_lens", torch.int32, (num_reqs,)),
                 ("qo_indptr", torch.int32, (num_reqs + 1,)),
                 ("block_tables", torch.int32, tuple(block_tables_shape))]
        self._layout, off = [], 0
        for name, dt, shape in specs:
            n = 1
            for d in shape:
                n *= int(d)
            nbytes = n * torch.tensor([], dtype=dt).element_size()
            self._layout.append((name, dt, shape, off, nbytes))
            off = a256(off + nbytes)
        self.in_bytes = off
        self.host_in = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev_in = torch.empty(off, dtype=torch.uint8, device=dev)
        self.step = step
        self.host_result = torch.empty(step.result.numel(), dtype=torch.uint8).pin_memory()
        out_bytes = step.out.numel() * 2
        self.out = self.host_result[:out_bytes].view(torch.bfloat16).view(step.out.shape)
        self.lse = self.host_result[step.lse_offset:].view(torch.float32).view(step.lse.shape)

    def _view(self, buf, name):
        for n, dt, shape, off, nbytes in self._layout:
            if n == name:
                return buf[off:off + nbytes].view(dt).view(shape)
        raise KeyError(name)

    def stage(self, q, seq_lens, qo_indptr, block_tables):
        """Packs a step's host inputs into the pinned block (host memory only)."""
        for name, x in (("q", q), ("seq_lens", seq_lens), ("qo_indptr", qo_indptr),
                        ("block_tables", block_tables)):
            self._view(self.host_in, name).copy_(torch.as_tensor(x).to(self._view(self.host_in, name).dtype))

    def upload(self):
        self.dev_in.copy_(self.host_in, non_blocking=True)

    def device_inputs(self):
        """(q, seq_lens, qo_indptr, block_tables) views of the device block."""
        return tuple(self._view(self.dev_in, n) for n in ("q", "seq_lens", "qo_indptr", "block_tables"))

    def download(self):
        self.host_result.copy_(self.step.result, non_blocking=True)


def step_for_workload(wl, device="cuda", num_segments: Optional[int] = None,
                      uniform_segments: bool = False, fused_merge: bool = False) -> VerifyStep:
    """A VerifyStep sized for a ``workloads.Workload``."""
    return VerifyStep(num_reqs=wl.num_reqs, num_rows=wl.num_rows, num_heads=wl.num_heads,
                      max_qlen=int(wl.qlens.max()), block_size=wl.block_size,
                      num_blocks=wl.num_blocks, block_table_width=wl.block_tables.shape[2],
                      max_kv_len=wl.max_kv_len,
                      num_segments=wl.num_segments if num_segments is None else num_segments,
                      world_size=wl.world_size, kv_fp8=(wl.kv_dtype == "fp8"),
                      interleave=wl.interleave, uniform_segments=uniform_segments,
                      fused_merge=fused_merge, device=device)


def device_inputs(wl, device="cuda"):
    """Copies a workload's inputs to the device: (q, kv, seq_lens, qo_indptr, block_tables)."""
    dev = torch.device(device)
    q = wl.q.to(dev, non_blocking=True)
    kv = wl.kv.to(dev, non_blocking=True)
    seq = torch.as_tensor(wl.seq_lens, dtype=torch.int32).to(dev)
    ind = torch.as_tensor(wl.qo_indptr, dtype=torch.int32).to(dev)
    bt = torch.as_tensor(wl.block_tables, dtype=torch.int32).to(dev)
    return q, kv, seq, ind, bt
