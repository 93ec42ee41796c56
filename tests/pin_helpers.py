"""Test-side constructions used to pin the oracle to something other than itself.

* ``paged_from_dense`` lays logical per-request KV rows out in a shuffled
  physical block pool (the inverse direction of the oracle's table walk), so a
  brute force on the dense rows checks the oracle's paging.
* ``brute_attention`` is a dense numpy softmax with an explicit boolean mask
  matrix built from "row t sees positions [0, L - qlen + t]" -- no paging, no
  lengths, no loops over tokens.
"""
import numpy as np
import torch

D_K, D_V = 576, 512


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def e4m3_values_torch() -> np.ndarray:
    """All 256 e4m3fn codes decoded by torch's float8_e4m3fn dtype."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def paged_from_dense(dense, block_size, rng, slack_blocks=3, fill=None):
    """dense: list of [L_b, 576] arrays (uint16 bf16 bits or uint8 codes).
    Returns (pool [nblk*bs, 576], block_table [B, max_blocks] int32)."""
    dtype = dense[0].dtype
    nb = [-(-d.shape[0] // block_size) for d in dense]
    total = sum(nb) + slack_blocks
    perm = rng.permutation(total).astype(np.int32)
    pool = np.empty((total * block_size, D_K), dtype)
    if fill is None:
        if dtype == np.uint16:
            pool[:] = f32_to_bf16_bits(rng.standard_normal(pool.shape))
        else:
            pool[:] = rng.integers(0, 256, pool.shape, dtype=np.uint8) & 0x77
    else:
        pool[:] = fill
    table = np.full((len(dense), max(nb)), -1, np.int32)
    pos = 0
    for b, d in enumerate(dense):
        for p in range(nb[b]):
            blk = perm[pos]
            pos += 1
            table[b, p] = blk
            rows = d[p * block_size:(p + 1) * block_size]
            pool[blk * block_size: blk * block_size + rows.shape[0]] = rows
    return pool, table


def brute_attention(q_bits, dense, seq_lens, qlens, sm_scale, kv_scale=1.0, fp8=False):
    """Dense reference: out [T, H, 512], lse [T, H] in float64."""
    table = e4m3_values_torch() if fp8 else None
    outs, lses = [], []
    r0 = 0
    for b, d in enumerate(dense):
        L, ql = int(seq_lens[b]), int(qlens[b])
        K = (table[d] * kv_scale) if fp8 else bf16_bits_to_f64(d)
        K = K[:L]
        Q = bf16_bits_to_f64(q_bits[r0:r0 + ql])                # [ql, H, 576]
        S = sm_scale * np.einsum("thd,jd->thj", Q, K)            # [ql, H, L]
        pos = np.arange(L)[None, :]
        last = (L - ql + np.arange(ql))[:, None]
        mask = pos <= last                                       # [ql, L]
        S = np.where(mask[:, None, :], S, -np.inf)
        m = S.max(axis=-1, keepdims=True)
        E = np.exp(S - m)
        den = E.sum(axis=-1, keepdims=True)
        outs.append(np.einsum("thj,jd->thd", E / den, K[:, :D_V]))
        lses.append((m + np.log(den))[..., 0])
        r0 += ql
    return np.concatenate(outs), np.concatenate(lses)
