"""Seeded synthetic workloads for MLA decode / causal verify.

This module only draws inputs: request lengths, verify-row counts, shuffled
physical block tables, queries and cached latent rows (bf16, or fp8 e4m3 codes
with a per-tensor scale).  It holds none of the method's arithmetic (no
windows, no shard counts, no attention), so both the CUDA path and the float64
oracle can consume exactly the same bytes.

Recipe (shared by every config):
  * one ``torch.Generator`` seeded per workload (seed 0 unless stated);
  * q and the cached rows are N(0, 1) float32 rounded to bf16;
  * fp8 caches: N(0, 1) float32, per-tensor scale = amax / 448 over the whole
    pool, codes = RNE e4m3 ("fn") of x / scale (torch's float8_e4m3fn cast);
  * block tables are consecutive slices of a random permutation of a pool with
    10% slack blocks, so physical ids are non-contiguous;
  * sharded (context-parallel) workloads give every shard its own block table
    into one shared pool; each request gets ceil(L / W) slots per shard,
    enough for any round-robin split, and unused slots are never visible.
Large caches can be drawn on a CUDA device (``device=...``) with torch's own
generator; the host copy is then made on demand.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

D_K = 576
D_V = 512
SM_SCALE = 1.0 / math.sqrt(192.0)   # softmax scale of every configured workload
FP8_MAX = 448.0


@dataclasses.dataclass
class Workload:
    name: str
    num_heads: int
    seq_lens: np.ndarray          # [B] int32, tokens of each request incl. its qlen new ones
    qlens: np.ndarray             # [B] int32, verify rows of each request
    block_size: int
    kv_dtype: str                 # "bf16" or "fp8"
    world_size: int               # 1, or the number of round-robin context shards
    num_segments: int             # split-K segments the workload is run with
    q: torch.Tensor               # [T, H, 576] bf16
    kv: torch.Tensor              # [pool_blocks * block_size, 576] bf16, or uint8 e4m3 codes
    kv_scale: float               # 1.0 for bf16
    block_tables: np.ndarray      # [W, B, max_blocks] int32 (W = 1 when unsharded)
    num_blocks: int               # physical blocks in the pool
    sm_scale: float = SM_SCALE
    seed: int = 0
    max_kv_len: int = 0           # static bound on a row's tokens in one table's address space
    interleave: int = 1           # round-robin run length of the context shards

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def qo_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.qlens)]).astype(np.int32)

    @property
    def num_rows(self) -> int:
        return int(self.qlens.sum())

    @property
    def kv_rows(self) -> int:
        return int(self.kv.shape[0])

    def q_bits(self) -> np.ndarray:
        return self.q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    def kv_host(self) -> np.ndarray:
        kv = self.kv.cpu().contiguous()
        if self.kv_dtype == "bf16":
            return kv.view(torch.int16).numpy().view(np.uint16)
        return kv.numpy()

    def describe(self) -> dict:
        return {"workload": self.name, "batch": self.num_reqs, "heads": self.num_heads,
                "qlen": sorted(set(int(x) for x in self.qlens)),
                "seq_len_min": int(self.seq_lens.min()), "seq_len_max": int(self.seq_lens.max()),
                "block_size": self.block_size, "kv_dtype": self.kv_dtype,
                "world_size": self.world_size, "num_segments": self.num_segments,
                **({"interleave": self.interleave} if self.interleave != 1 else {})}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g: torch.Generator, device=None, chunk_rows=1 << 20) -> torch.Tensor:
    """N(0,1) float32 rounded to bf16, drawn in row chunks to bound host memory."""
    if device is not None and torch.device(device).type == "cuda":
        dg = torch.Generator(device=device)
        dg.manual_seed(int(torch.randint(0, 2**62, (1,), generator=g)))
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for s in range(0, shape[0], chunk_rows):
            e = min(shape[0], s + chunk_rows)
            out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=dg, device=device)
        return out
    out = torch.empty(shape, dtype=torch.bfloat16)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=g)
    return out


def _randn_fp8(shape, g: torch.Generator, device=None, chunk_rows=1 << 20):
    """N(0,1) float32 -> per-tensor scale amax/448 -> RNE e4m3 codes (uint8)."""
    if device is not None and torch.device(device).type == "cuda":
        # two passes over the same Philox stream: amax first, then the codes
        dseed = int(torch.randint(0, 2**62, (1,), generator=g))
        dg = torch.Generator(device=device)
        amax = 0.0
        dg.manual_seed(dseed)
        for s in range(0, shape[0], chunk_rows):
            e = min(shape[0], s + chunk_rows)
            x = torch.randn((e - s,) + tuple(shape[1:]), generator=dg, device=device)
            amax = max(amax, float(x.abs().max()))
        scale = amax / FP8_MAX
        codes = torch.empty(shape, dtype=torch.uint8, device=device)
        dg.manual_seed(dseed)
        for s in range(0, shape[0], chunk_rows):
            e = min(shape[0], s + chunk_rows)
            x = torch.randn((e - s,) + tuple(shape[1:]), generator=dg, device=device)
            codes[s:e] = (x / scale).clamp_(-FP8_MAX, FP8_MAX).to(
                torch.float8_e4m3fn).view(torch.uint8)
        return codes, scale
    x = torch.randn(shape, generator=g)
    scale = float(x.abs().max()) / FP8_MAX
    codes = (x / scale).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def make_workload(name: str, seq_lens, qlens, num_heads: int, block_size: int,
                  kv_dtype: str = "bf16", world_size: int = 1, num_segments: int = 1,
                  seed: int = 0, slack: float = 0.10, device=None,
                  max_kv_len: Optional[int] = None, interleave: int = 1) -> Workload:
    """Draw a workload.  seq_lens / qlens: per-request ints (qlen <= seq_len)."""
    g = _gen(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    qlens = np.asarray(qlens, dtype=np.int32)
    B = seq_lens.shape[0]
    W = int(world_size)
    # slots each request needs in one table's address space: at most I per
    # started cycle of I * W positions on any shard (ceil(L/W) for I = 1)
    I = int(interleave)
    slots = [int(-(-int(L) // (I * W))) * I for L in seq_lens]
    blocks_per_req = [-(-s // block_size) for s in slots]
    max_blocks = max(1, max(blocks_per_req))
    used = W * sum(blocks_per_req)
    num_blocks = max(1, int(math.ceil(used * (1.0 + slack))))
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    tables = np.full((W, B, max_blocks), -1, np.int32)
    pos = 0
    for r in range(W):
        for b in range(B):
            n = blocks_per_req[b]
            tables[r, b, :n] = perm[pos:pos + n]
            pos += n
    T = int(qlens.sum())
    q = _randn_bf16((T, num_heads, D_K), g)
    rows = num_blocks * block_size
    if kv_dtype == "bf16":
        kv = _randn_bf16((rows, D_K), g, device)
        kv_scale = 1.0
    elif kv_dtype == "fp8":
        kv, kv_scale = _randn_fp8((rows, D_K), g, device)
    else:
        raise ValueError(kv_dtype)
    if max_kv_len is None:
        max_kv_len = max(slots)
    return Workload(name=name, num_heads=num_heads, seq_lens=seq_lens, qlens=qlens,
                    block_size=block_size, kv_dtype=kv_dtype, world_size=W,
                    num_segments=num_segments, q=q, kv=kv, kv_scale=float(kv_scale),
                    block_tables=tables, num_blocks=num_blocks, seed=seed,
                    max_kv_len=int(max_kv_len), interleave=I)


# ---------------------------------------------------------------------------
# The configured workloads.

def decode_qlen1_bf16(seed: int = 0) -> Workload:
    """qlen=1 bf16 decode: batch 2, 16 heads, seq_len 256 each, block 16."""
    return make_workload("decode_qlen1_bf16_b2_h16_L256_bs16", [256, 256], [1, 1], 16, 16,
                         "bf16", 1, 1, seed)


def verify_mtp4_bf16(seed: int = 0, batch: int = 32, lo: int = 1024, hi: int = 8192,
                     num_segments: int = 16, device=None) -> Workload:
    """Causal MTP verify qlen=4 bf16: batch 32, 16 heads, seq_len U{1k..8k},
    block 64, 16 split-K segments."""
    g = _gen(seed + 1000)
    L = torch.randint(lo, hi + 1, (batch,), generator=g).numpy()
    return make_workload(f"verify_mtp4_bf16_b{batch}_h16_L{lo}-{hi}_bs64_s{num_segments}",
                         L, [4] * batch, 16, 64, "bf16", 1, num_segments, seed, device=device)


def fp8_mixed_qlen(seed: int = 0, batch: int = 64, lo: int = 512, hi: int = 32768,
                   num_segments: int = 16, device=None) -> Workload:
    """fp8_e4m3 cache: batch 64, 12 heads, qlen U{1,2,3}, seq_len log-uniform
    [512, 32k], block 64.  16 split-K segments: the longest request then
    splits into items of <= 2048 tokens, below the per-SM share of the batch
    (~3.3k tokens on 152 SMs), so no single item sets the step time."""
    g = _gen(seed + 2000)
    u = torch.rand(batch, generator=g, dtype=torch.float64).numpy()
    L = np.floor(np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))).astype(np.int32)
    L = np.clip(L, lo, hi)
    ql = torch.randint(1, 4, (batch,), generator=g).numpy()
    return make_workload(f"fp8_e4m3_b{batch}_h12_qlen1-3_L{lo}-{hi}_bs64_s{num_segments}",
                         L, ql, 12, 64, "fp8", 1, num_segments, seed, device=device)


def dcp8_verify_bf16(seed: int = 0, batch: int = 16, context: int = 131072,
                     world_size: int = 8, num_segments: int = 10, device=None) -> Workload:
    """Simulated 8-way round-robin context-sharded verify: batch 16, 16 heads,
    qlen 4, context 128k, bf16, block 64.  The 8 shard views are decoded in one
    launch; 10 split-K segments give 16 x 8 x 10 = 1280 work items of ~26
    tiles (about 8.4 per SM on 152 SMs), the fastest of 5/10/19/38 measured."""
    return make_workload(f"dcp{world_size}_verify_bf16_b{batch}_h16_qlen4_L{context}_bs64_s{num_segments}",
                         [context] * batch, [4] * batch, 16, 64, "bf16", world_size,
                         num_segments, seed, device=device,
                         max_kv_len=-(-context // world_size))


@dataclasses.dataclass
class SweepPoint:
    heads: int
    batch: int
    context: int
    qlen: int
    kv_dtype: str
    block_size: int
    seed: int

    def name(self) -> str:
        return (f"sweep_h{self.heads}_b{self.batch}_C{self.context}_q{self.qlen}_"
                f"{self.kv_dtype}_bs{self.block_size}")


def sweep_points(n: int = 100, seed: int = 0) -> List[SweepPoint]:
    """Seeded grid sample over heads {16,64,128} x batch 1..256 x context
    4k..132k x qlen {1,2,4,8} x {bf16, fp8} x block {16,64,256}."""
    g = _gen(seed + 3000)
    heads = [16, 64, 128]
    qlens = [1, 2, 4, 8]
    dts = ["bf16", "fp8"]
    bss = [16, 64, 256]
    pts = []
    for i in range(n):
        r = torch.randint(0, 1 << 30, (6,), generator=g).tolist()
        ctx = int(4096 * (132 * 1024 / 4096) ** (r[2] / float(1 << 30)))
        pts.append(SweepPoint(heads[r[0] % 3], 1 + r[1] % 256, ctx, qlens[r[3] % 4],
                              dts[r[4] % 2], bss[r[5] % 3], seed + i))
    return pts


def sweep_workload(p: SweepPoint, device=None, max_tokens: Optional[int] = None,
                   num_segments: int = 1) -> Workload:
    """Per-request seq_len U{qlen .. context}; optional cap on total tokens."""
    g = _gen(p.seed + 4000)
    L = torch.randint(p.qlen, p.context + 1, (p.batch,), generator=g).numpy()
    if max_tokens is not None and L.sum() > max_tokens:
        L = np.maximum(p.qlen, (L * (max_tokens / float(L.sum())))).astype(np.int32)
    name = p.name() + (f"_s{num_segments}" if num_segments > 1 else "")
    return make_workload(name, L, [p.qlen] * p.batch, p.heads, p.block_size,
                         p.kv_dtype, 1, num_segments, p.seed, device=device)
