"""Owner-filtered paged KV write (mla_write_kv) on the GPU: the written cache
is bit-exact against the oracle's, for every rank of a round-robin split and
for bf16 and fp8 caches; untouched rows stay untouched."""
import numpy as np
import pytest
import torch

import oracle
from mla_decode_speculative_gb300 import mla, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("W,dtype", [(1, "bf16"), (8, "bf16"), (1, "fp8"), (4, "fp8")])
def test_write_kv_bit_exact(W, dtype):
    wl = workloads.make_workload("kvw", [300, 41, 1000, 7, 64], [4, 1, 3, 2, 8], 16, 16,
                                 kv_dtype=dtype, world_size=W, seed=W)
    rng = np.random.default_rng(W)
    kv_new = torch.tensor(rng.standard_normal((wl.num_rows, 576)) * 2, dtype=torch.float32).to(torch.bfloat16)
    kv_new_bits = kv_new.view(torch.int16).numpy().view(np.uint16)
    seq = torch.tensor(wl.seq_lens, dtype=torch.int32, device="cuda")
    ind = torch.tensor(wl.qo_indptr, dtype=torch.int32, device="cuda")
    for r in range(W):
        host = wl.kv_host().copy()
        oracle.write_kv(wl.seq_lens, wl.qo_indptr, kv_new_bits, W, r, wl.block_tables[r], wl.block_size,
                        host, kv_scale=wl.kv_scale)
        cache = wl.kv.clone().cuda()
        bt = torch.tensor(wl.block_tables[r], dtype=torch.int32, device="cuda")
        mla.write_kv(seq, ind, kv_new.cuda(), cache, bt, wl.num_blocks, wl.block_size, W, r, wl.kv_scale)
        torch.cuda.synchronize()
        assert mla.get_device_error() == 0
        got = cache.cpu()
        got = got.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else got.numpy()
        assert (got == host).all(), f"rank {r}: {(got != host).any(axis=1).sum()} rows differ"
        assert (host != wl.kv_host()).any() or wl.num_rows < W  # something was written


def test_write_kv_rejects_bad_interleave_and_bad_blocks():
    seq = torch.tensor([10], dtype=torch.int32, device="cuda")
    ind = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    kv_new = torch.zeros((2, 576), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((64, 576), dtype=torch.bfloat16, device="cuda")
    bt = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.write_kv(seq, ind, kv_new, cache, bt, 4, 16, 2, 0, interleave=0)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    bt = torch.tensor([[99]], dtype=torch.int32, device="cuda")
    mla.write_kv(seq, ind, kv_new, cache, bt, 4, 16)
    assert mla.get_device_error() == 3   # MLA_DEV_BAD_BLOCK_ID, nothing written
    assert (cache.float() == 0).all()


@pytest.mark.parametrize("W,I", [(3, 2), (8, 4), (2, 16)])
def test_write_kv_interleaved_bit_exact(W, I):
    """Interleave I > 1: runs of I positions dealt to the ranks in turn; every
    rank's cache after the GPU write equals the oracle's, byte for byte."""
    rng = np.random.default_rng(90 + W * I)
    seq = np.array([37, 5, 64, 9, 130], np.int32)
    ql = np.array([4, 2, 3, 1, 8], np.int32)
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    B, T, bs = len(seq), int(ind[-1]), 8
    kv_new = torch.randn((T, 576), generator=torch.Generator().manual_seed(W * I)).to(torch.bfloat16)
    bits = kv_new.view(torch.int16).numpy().view(np.uint16)
    cap = [max(oracle.il_local_len(int(L), W, r, I) for r in range(W)) for L in seq]
    nb = [-(-c // bs) for c in cap]
    for r in range(W):
        num_blocks = sum(nb) + 3
        perm = rng.permutation(num_blocks).astype(np.int32)
        bt = np.full((B, max(nb)), -1, np.int32)
        pos = 0
        for b in range(B):
            bt[b, :nb[b]] = perm[pos:pos + nb[b]]
            pos += nb[b]
        host = np.zeros((num_blocks * bs, 576), np.uint16)
        oracle.write_kv(seq, ind, bits, W, r, bt, bs, host, interleave=I)
        cache = torch.zeros((num_blocks * bs, 576), dtype=torch.bfloat16, device="cuda")
        mla.write_kv(torch.tensor(seq, device="cuda"), torch.tensor(ind, device="cuda"),
                     kv_new.to("cuda"), cache, torch.tensor(bt, device="cuda"), num_blocks, bs,
                     W, r, interleave=I)
        torch.cuda.synchronize()
        assert mla.get_device_error() == 0
        got = cache.cpu().view(torch.int16).numpy().view(np.uint16)
        assert (got == host).all(), f"rank {r}"
