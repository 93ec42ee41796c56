"""Pins of the float64 oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something that is not the oracle: golden
values worked by hand from the pages' formulas (tests/golden/), brute force
enumeration, a dense numpy softmax with an explicit mask matrix, torch's own
float8_e4m3fn decoding, closed forms and invariants.
"""
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden
from pin_helpers import (D_K, D_V, brute_attention, e4m3_values_torch, f32_to_bf16_bits,
                         paged_from_dense)

SM = 1.0 / math.sqrt(192.0)


# --------------------------------------------------------------------------- indexing

def test_page_size_golden():
    n = 0
    for line in read_golden("page_size.txt"):
        bs, p = map(int, line.split())
        assert oracle.page_size(bs) == p, bs
        n += 1
    assert n >= 20


def test_page_size_bit_identity():
    # largest power-of-two divisor is the lowest set bit: bs & -bs
    for bs in range(1, 5000):
        assert oracle.page_size(bs) == min(128, bs & -bs)


def test_verify_windows_golden():
    for line in read_golden("verify_windows.txt"):
        lhs, rhs = line.split(":")
        L, ql = map(int, lhs.split())
        want = list(map(int, rhs.split()))
        row_len, row_req, row_t = oracle.plan_rows([L], [0, ql])
        assert row_len.tolist() == want
        assert row_req.tolist() == [0] * ql
        assert row_t.tolist() == list(range(ql))


def test_plan_rows_multi_request_and_errors():
    seq = [10, 5, 300]
    ql = [4, 1, 3]
    ind = np.concatenate([[0], np.cumsum(ql)])
    row_len, row_req, row_t = oracle.plan_rows(seq, ind)
    assert row_len.tolist() == [7, 8, 9, 10, 5, 298, 299, 300]
    assert row_req.tolist() == [0, 0, 0, 0, 1, 2, 2, 2]
    with pytest.raises(oracle.OracleError):
        oracle.plan_rows([3], [0, 4])          # qlen > seq_len
    with pytest.raises(oracle.OracleError):
        oracle.plan_rows([3, 3], [0, 0, 1])    # qlen 0


def test_round_robin_golden():
    for line in read_golden("round_robin.txt"):
        lhs, rhs = line.split(":")
        w, W = map(int, lhs.split())
        want = list(map(int, rhs.split()))
        assert [oracle.rr_local_len(w, W, r) for r in range(W)] == want


def test_round_robin_brute_force_and_invariants():
    for W in range(1, 10):
        for w in range(0, 120):
            counts = [oracle.rr_local_len(w, W, r) for r in range(W)]
            brute = [sum(1 for g in range(w) if g % W == r) for r in range(W)]
            assert counts == brute, (w, W)
            assert sum(counts) == w
            assert all(c in (w // W, -(-w // W)) for c in counts)


def test_shard_row_view_per_row_causality():
    # consecutive verify rows: each shard gains 0 or 1 token and exactly one
    # shard (the owner of the newly visible position) gains one
    for W in (2, 3, 8):
        for L, ql in ((50, 4), (17, 8), (9, 9), (1000, 3)):
            row_len, _, _ = oracle.plan_rows([L], [0, ql])
            views = np.stack([oracle.shard_row_view(row_len, W, r) for r in range(W)])
            assert (views.sum(axis=0) == row_len).all()
            for t in range(ql - 1):
                gain = views[:, t + 1] - views[:, t]
                assert set(gain.tolist()) <= {0, 1}
                assert gain.sum() == 1
                assert gain[row_len[t] % W] == 1     # position row_len[t] is new


def test_negative_control_subtraction_breaks_the_sum():
    # "local length minus the causal offset" subtracts one token from EVERY
    # rank; the dropped tokens sit on different ranks, so the shard windows no
    # longer add up to the global window (vLLM #51705, 实现拆解 2).
    L, ql, W = 1000, 4, 8
    row_len, _, _ = oracle.plan_rows([L], [0, ql])
    bad = 0
    for t in range(ql):
        wrong = [max(0, oracle.rr_local_len(L, W, r) - (ql - 1 - t)) for r in range(W)]
        right = oracle.shard_row_view(row_len, W, 0)  # sanity on one rank
        assert right[t] == oracle.rr_local_len(row_len[t], W, 0)
        if sum(wrong) != row_len[t]:
            bad += 1
    assert bad == ql - 1      # every row but the last is wrong


def test_shard_row_view_rejects_bad_interleave_and_rank():
    with pytest.raises(oracle.OracleError):
        oracle.shard_row_view([10, 11], 4, 0, interleave=0)
    with pytest.raises(oracle.OracleError):
        oracle.shard_row_view([10], 4, 4)


# --------------------------------------------------------------------------- interleave > 1
# Runs of I consecutive positions are dealt to the ranks in turn (I = 1 is the
# pages' g(j) = j * W + r).  Pinned by enumeration, not by the closed forms.

def _deal(w, W, I):
    """Enumerate positions 0 .. w-1 run by run: per rank, its positions in order."""
    held = [[] for _ in range(W)]
    for run_start in range(0, w, I):
        held[(run_start // I) % W].extend(range(run_start, min(run_start + I, w)))
    return held


def test_interleave_counts_brute_force():
    for W in range(1, 7):
        for I in range(1, 6):
            for w in range(0, 140):
                held = _deal(w, W, I)
                counts = [oracle.il_local_len(w, W, r, I) for r in range(W)]
                assert counts == [len(h) for h in held], (w, W, I)
                assert sum(counts) == w
                if I == 1:
                    assert counts == [oracle.rr_local_len(w, W, r) for r in range(W)]


def test_interleave_owner_and_local_index_enumerated():
    # each rank's positions, in increasing order, sit at local indices 0, 1, 2, ...
    # (so every row's shard window is a prefix of the shard's local sequence)
    for W in (1, 2, 3, 8):
        for I in (1, 2, 4, 16):
            held = _deal(300, W, I)
            for r in range(W):
                for j, g in enumerate(held[r]):
                    assert oracle.il_owner(g, W, I) == r
                    assert oracle.il_local_index(g, W, I) == j


def test_interleave_row_view_per_row_causality():
    for W, I in ((2, 2), (3, 4), (8, 16), (4, 1)):
        for L, ql in ((50, 4), (17, 8), (1000, 3), (64, 64)):
            row_len, _, _ = oracle.plan_rows([L], [0, ql])
            views = np.stack([oracle.shard_row_view(row_len, W, r, I) for r in range(W)])
            assert (views.sum(axis=0) == row_len).all()
            for t in range(ql - 1):
                gain = views[:, t + 1] - views[:, t]
                assert set(gain.tolist()) <= {0, 1} and gain.sum() == 1
                assert gain[oracle.il_owner(int(row_len[t]), W, I)] == 1


def test_subpage_golden():
    for line in read_golden("subpages.txt"):
        lhs, rhs = line.split(":")
        bs, kv_len, width = map(int, lhs.split())
        bt_s, want_s = rhs.split("|")
        bt = np.array([list(map(int, bt_s.split()))], np.int32)
        want = list(map(int, want_s.split()))
        got = oracle.subpage_table([kv_len], bt, 100, bs, width)
        assert got[0].tolist() == want


def test_subpage_two_way_mapping():
    rng = np.random.default_rng(5)
    for bs in (16, 48, 64, 96, 256, 512):
        P = oracle.page_size(bs)
        L = [int(x) for x in rng.integers(1, 1500, 6)]
        nb = [-(-x // bs) for x in L]
        nblk = sum(nb) + 4
        perm = rng.permutation(nblk).astype(np.int32)
        bt = np.full((6, max(nb)), -1, np.int32)
        pos = 0
        for b in range(6):
            bt[b, :nb[b]] = perm[pos:pos + nb[b]]
            pos += nb[b]
        width = max(-(-x // P) for x in L) + 2
        sp = oracle.subpage_table(L, bt, nblk, bs, width)
        for b in range(6):
            for j in range(L[b]):
                direct = bt[b, j // bs] * bs + j % bs
                via_sp = sp[b, j // P] * P + j % P
                assert direct == via_sp
            assert (sp[b, -(-L[b] // P):] == -1).all()
    with pytest.raises(oracle.OracleError):
        oracle.subpage_table([10], np.array([[7]], np.int32), 5, 16, 1)  # block id 7 >= 5


# --------------------------------------------------------------------------- fp8

def test_e4m3_matches_torch_for_all_codes():
    ours = oracle.e4m3_table()
    ref = e4m3_values_torch()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.isnan(ours[nan]).all()
    assert (ours[~nan] == ref[~nan]).all()


def test_e4m3_spot_values():
    assert oracle.e4m3_to_double(0x00) == 0.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9       # smallest subnormal
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6       # smallest normal
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert oracle.e4m3_to_double(0x7E) == 448.0           # largest finite
    assert oracle.e4m3_to_double(0xBE) == -1.75


# --------------------------------------------------------------------------- attention

def _rand_case(rng, seq, ql, H, bs, fp8=False, slack=3):
    dense = []
    for L in seq:
        if fp8:
            dense.append((rng.integers(0, 256, (L, D_K), dtype=np.uint8) & 0x77)
                         | (rng.integers(0, 2, (L, D_K), dtype=np.uint8) << 7))
        else:
            dense.append(f32_to_bf16_bits(rng.standard_normal((L, D_K))))
    pool, bt = paged_from_dense(dense, bs, rng, slack)
    T = int(sum(ql))
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_K)))
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    return dense, pool, bt, q, ind


@pytest.mark.parametrize("bs", [1, 3, 16, 64])
def test_attention_matches_dense_brute_force(bs):
    rng = np.random.default_rng(bs)
    seq, ql, H = [9, 1, 16, 5], [3, 1, 4, 5], 2
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, bs)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    out, lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, bs)
    ref_out, ref_lse = brute_attention(q, dense, seq, ql, SM)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attention_fp8_matches_dense_brute_force():
    rng = np.random.default_rng(11)
    seq, ql, H = [12, 7], [2, 3], 2
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, 4, fp8=True)
    scale = 0.0123
    row_len, _, _ = oracle.plan_rows(seq, ind)
    out, lse = oracle.attention(ind, row_len, q, pool, scale, SM, bt, 4)
    ref_out, ref_lse = brute_attention(q, dense, seq, ql, SM, kv_scale=scale, fp8=True)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attention_selected_pairs_match_full():
    rng = np.random.default_rng(3)
    seq, ql, H = [40, 33], [4, 2], 3
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, 8)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    out, lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, 8)
    sel = np.array([[5, 2], [0, 0], [3, 1]])
    o2, l2 = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, 8, sel=sel)
    for k, (r, h) in enumerate(sel):
        assert (o2[k] == out[r, h]).all() and l2[k] == lse[r, h]


def test_closed_form_zero_query():
    # q = 0: every score is 0 -> out = mean of the visible V rows, lse = ln w
    rng = np.random.default_rng(1)
    seq, ql, H = [20], [4], 2
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, 16)
    q[:] = 0
    row_len, _, _ = oracle.plan_rows(seq, ind)
    out, lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, 16)
    V = (dense[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)[:, :D_V]
    for t in range(4):
        w = 17 + t
        np.testing.assert_allclose(out[t, 0], V[:w].mean(axis=0), atol=1e-13)
        assert abs(lse[t, 1] - math.log(w)) < 1e-13


def test_closed_form_identical_keys_and_single_token():
    rng = np.random.default_rng(2)
    L, ql, H = 6, 6, 1
    row = f32_to_bf16_bits(rng.standard_normal(D_K))
    dense = [np.tile(row, (L, 1))]
    pool, bt = paged_from_dense(dense, 4, rng)
    q = f32_to_bf16_bits(rng.standard_normal((ql, H, D_K)))
    ind = np.array([0, ql], np.int32)
    row_len, _, _ = oracle.plan_rows([L], ind)
    out, lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, 4)
    k = (row.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(ql):
        qd = (q[t, 0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        s = SM * float(qd @ k)
        np.testing.assert_allclose(out[t, 0], k[:D_V], atol=1e-14)
        assert abs(lse[t, 0] - (s + math.log(t + 1))) < 1e-12
    # row 0 of a block whose seq_len == qlen sees exactly one token
    assert row_len[0] == 1


def test_closed_form_one_hot_score():
    rng = np.random.default_rng(4)
    L = 30
    dense = [f32_to_bf16_bits(rng.standard_normal((L, D_K)) * 0.01)]
    star = 13
    dense[0][star] = f32_to_bf16_bits(np.full(D_K, 1.0))
    pool, bt = paged_from_dense(dense, 8, rng)
    q = f32_to_bf16_bits(np.full((1, 1, D_K), 4.0))   # score(star) ~ 166, others ~ 0
    ind = np.array([0, 1], np.int32)
    out, lse = oracle.attention(ind, [L], q, pool, 1.0, SM, bt, 8)
    np.testing.assert_allclose(out[0, 0], np.ones(D_V), atol=1e-12)
    assert abs(lse[0, 0] - SM * 4.0 * D_K) < 1e-9


def test_empty_row_gives_zero_and_minus_inf():
    rng = np.random.default_rng(6)
    dense, pool, bt, q, ind = _rand_case(rng, [8], [2], 2, 4)
    out, lse = oracle.attention(ind, [0, 3], q, pool, 1.0, SM, bt, 4)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1]).all()


def test_invariance_block_layout_and_page_size():
    # same logical cache, three different physical layouts / block sizes
    rng = np.random.default_rng(7)
    seq, ql, H = [70, 41, 128], [2, 4, 1], 2
    dense = [f32_to_bf16_bits(rng.standard_normal((L, D_K))) for L in seq]
    q = f32_to_bf16_bits(rng.standard_normal((sum(ql), H, D_K)))
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    results = []
    for bs in (16, 32, 96):
        pool, bt = paged_from_dense(dense, bs, rng)
        results.append(oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, bs))
    for o, l in results[1:]:
        np.testing.assert_allclose(o, results[0][0], atol=1e-13)
        np.testing.assert_allclose(l, results[0][1], atol=1e-13)


@pytest.mark.parametrize("S", [1, 2, 5, 16])
def test_segment_partials_merge_to_attention(S):
    rng = np.random.default_rng(8 + S)
    seq, ql, H, bs = [300, 64, 129], [4, 1, 3], 2, 16
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, bs)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    acc, mx, sm = oracle.segment_partials(ind, row_len, q, pool, 1.0, SM, bt, bs, S, 16)
    out, lse = oracle.merge_segments(acc, mx, sm)
    ref_out, ref_lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, bs)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
    # the pages' partition: segment s covers tps tiles, tps = cdiv(len, S*TILE)
    L = 300
    tps = -(-L // (S * 16))
    active = -(-L // (tps * 16))
    assert np.isneginf(mx[0, 0, active:]).all() and np.isfinite(mx[3, 0, :active]).all()


@pytest.mark.parametrize("seed", [0, 1])
def test_range_partials_over_any_partition_merge_to_attention(seed):
    """Partials over arbitrary contiguous cuts of each 64-row group's tokens
    (some slots empty, some past the rows' windows) merge to the attention."""
    rng = np.random.default_rng(40 + seed)
    seq, ql, H, bs = [300, 70, 129, 5], [4, 1, 3, 2], 40, 16  # 40 heads: groups of 64 rows split tokens
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, bs)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    B, S = len(seq), 6
    G = -(-max(ql) * H // 64)
    ranges = np.zeros((B, G, S, 2), np.int64)
    for b in range(B):
        for g in range(G):
            cuts = np.sort(rng.integers(0, seq[b] + 1, S - 1))
            edges = np.concatenate([[0], cuts, [seq[b] + int(rng.integers(0, 40))]])
            ranges[b, g, :, 0], ranges[b, g, :, 1] = edges[:-1], edges[1:]
    acc, mx, sm = oracle.range_partials(ind, row_len, q, pool, 1.0, SM, bt, bs, ranges)
    out, lse = oracle.merge_segments(acc, mx, sm)
    ref_out, ref_lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, bs)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
    # a slot is empty exactly when its range holds none of the row's visible tokens
    for t in range(int(ind[-1])):
        b = int(np.searchsorted(ind, t, side="right") - 1)
        for h in range(H):
            g = ((t - ind[b]) * H + h) // 64
            for s_ in range(S):
                lo, hi = ranges[b, g, s_]
                assert np.isneginf(mx[t, h, s_]) == (min(hi, row_len[t]) <= lo)


def test_range_partials_single_token_and_pages_split():
    """A one-token range holds that token's V row with l = 1; the pages'
    ranges reproduce oracle_segment_partials exactly."""
    rng = np.random.default_rng(44)
    seq, ql, H, bs = [90, 33], [3, 1], 2, 16
    dense, pool, bt, q, ind = _rand_case(rng, seq, ql, H, bs)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    ranges = np.zeros((2, 1, 2, 2), np.int64)
    ranges[:, 0, 0] = [7, 8]          # token 7 alone
    ranges[:, 0, 1] = [200, 300]      # past every window: empty
    acc, mx, sm = oracle.range_partials(ind, row_len, q, pool, 1.0, SM, bt, bs, ranges)
    for t in range(4):
        b = 0 if t < 3 else 1
        v7 = (dense[b][7, :D_V].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        for h in range(H):
            assert sm[t, h, 0] == 1.0 and np.array_equal(acc[t, h, 0], v7)
            assert np.isneginf(mx[t, h, 1]) and sm[t, h, 1] == 0.0 and not acc[t, h, 1].any()
    S, tile = 3, 16
    seg_acc, seg_mx, seg_sm = oracle.segment_partials(ind, row_len, q, pool, 1.0, SM, bt, bs, S, tile)
    pr = np.zeros((2, 1, S, 2), np.int64)
    for b in range(2):
        gl = int(max(row_len[ind[b]:ind[b + 1]]))
        tps = -(-gl // (S * tile))
        for s_ in range(S):
            pr[b, 0, s_] = [s_ * tps * tile, (s_ + 1) * tps * tile]
    acc2, mx2, sm2 = oracle.range_partials(ind, row_len, q, pool, 1.0, SM, bt, bs, pr)
    assert np.array_equal(acc2, seg_acc) and np.array_equal(mx2, seg_mx) and np.array_equal(sm2, seg_sm)


def test_merge_identity_and_arbitrary_split():
    rng = np.random.default_rng(9)
    L = 57
    K = f32_to_bf16_bits(rng.standard_normal((L, D_K)))
    Kd = (K.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qd = rng.standard_normal(D_K)
    s = SM * (Kd @ qd)
    # whole attention
    m = s.max()
    e = np.exp(s - m)
    whole = (e @ Kd[:, :D_V]) / e.sum()
    whole_lse = m + math.log(e.sum())
    # arbitrary split into 4 key subsets, each its own (out, lse) state
    lab = rng.integers(0, 4, L)
    outs, lses = [], []
    for k in range(4):
        idx = lab == k
        mk = s[idx].max()
        ek = np.exp(s[idx] - mk)
        outs.append((ek @ Kd[idx, :D_V]) / ek.sum())
        lses.append(mk + math.log(ek.sum()))
    o, l = oracle.merge_states(np.array(outs)[:, None], np.array(lses)[:, None])
    np.testing.assert_allclose(o[0], whole, atol=1e-13)
    assert abs(l[0] - whole_lse) < 1e-13
    # a single part is the identity; an empty part (-inf) is ignored
    o1, l1 = oracle.merge_states(np.array(outs[:1])[:, None], np.array(lses[:1])[:, None])
    assert (o1[0] == outs[0]).all() and l1[0] == lses[0]
    o2, l2 = oracle.merge_states(np.array([outs[0], np.zeros(D_V)])[:, None],
                                 np.array([lses[0], -np.inf])[:, None])
    np.testing.assert_allclose(o2[0], outs[0], atol=1e-15)
    # same split in the base-2 segment convention
    acc = np.array([np.exp2((s[lab == k] - s[lab == k].max()) / math.log(2)) @ Kd[lab == k, :D_V]
                    for k in range(4)])
    mx = np.array([s[lab == k].max() / math.log(2) for k in range(4)])
    sm = np.array([np.exp2((s[lab == k] - s[lab == k].max()) / math.log(2)).sum() for k in range(4)])
    o3, l3 = oracle.merge_segments(acc[None], mx[None], sm[None])
    np.testing.assert_allclose(o3[0], whole, atol=1e-13)
    assert abs(l3[0] - whole_lse) < 1e-13
    # all empty
    o4, l4 = oracle.merge_segments(np.zeros((1, 2, D_V)), np.full((1, 2), -np.inf), np.zeros((1, 2)))
    assert (o4 == 0).all() and np.isneginf(l4).all()


def _shard_layout(dense, W, bs, rng, I=1):
    """Round-robin layout built by enumeration: runs of I positions of request b
    dealt to the shards in turn, each shard keeping its positions in order (for
    I = 1: position g at shard g % W, local index g // W).  Returns per-shard
    block tables over one shared pool."""
    shard_dense = [[d[np.array(_deal(d.shape[0], W, I)[r], dtype=np.int64)] for d in dense]
                   for r in range(W)]
    pools, tables = [], []
    offset = 0
    for r in range(W):
        sd = [x if x.shape[0] > 0 else x.reshape(0, D_K) for x in shard_dense[r]]
        sd = [x if x.shape[0] > 0 else np.zeros((1, D_K), dense[0].dtype) for x in sd]
        pool, bt = paged_from_dense(sd, bs, rng, slack_blocks=1)
        bt = np.where(bt >= 0, bt + offset, -1)
        offset += pool.shape[0] // bs
        pools.append(pool)
        tables.append(bt)
    mb = max(t.shape[1] for t in tables)
    tables = [np.pad(t, ((0, 0), (0, mb - t.shape[1])), constant_values=-1) for t in tables]
    return np.concatenate(pools), np.stack(tables)


@pytest.mark.parametrize("W,I", [(3, 2), (8, 4), (2, 16)])
def test_sharded_merge_equals_unsharded_interleaved(W, I):
    rng = np.random.default_rng(60 + W)
    seq, ql, H, bs = [37, 5, 64], [4, 3, 2], 2, 4
    dense = [f32_to_bf16_bits(rng.standard_normal((L, D_K))) for L in seq]
    q = f32_to_bf16_bits(rng.standard_normal((sum(ql), H, D_K)))
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    pool, bt = paged_from_dense(dense, bs, rng)
    ref_out, ref_lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, bs)
    spool, sbt = _shard_layout(dense, W, bs, rng, I)
    out, lse, _, _ = oracle.sharded_attention(ind, row_len, q, spool, 1.0, SM, sbt, bs, W,
                                              interleave=I)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


@pytest.mark.parametrize("W", [2, 3, 8])
def test_sharded_merge_equals_unsharded(W):
    rng = np.random.default_rng(20 + W)
    seq, ql, H, bs = [37, 5, 64], [4, 3, 2], 2, 4
    dense = [f32_to_bf16_bits(rng.standard_normal((L, D_K))) for L in seq]
    q = f32_to_bf16_bits(rng.standard_normal((sum(ql), H, D_K)))
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    row_len, _, _ = oracle.plan_rows(seq, ind)
    pool, bt = paged_from_dense(dense, bs, rng)
    ref_out, ref_lse = oracle.attention(ind, row_len, q, pool, 1.0, SM, bt, bs)
    spool, sbt = _shard_layout(dense, W, bs, rng)
    out, lse, parts_o, parts_l = oracle.sharded_attention(ind, row_len, q, spool, 1.0, SM,
                                                           sbt, bs, W)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
    # the subtraction row view gives a different (wrong) answer
    wrong_parts_o, wrong_parts_l = [], []
    for r in range(W):
        local = np.array([max(0, oracle.rr_local_len(seq[b], W, r) - (ql[b] - 1 - t))
                          for b in range(len(seq)) for t in range(ql[b])], np.int32)
        o, l = oracle.attention(ind, local, q, spool, 1.0, SM, sbt[r], bs)
        wrong_parts_o.append(o)
        wrong_parts_l.append(l)
    wo, wl = oracle.merge_states(np.stack(wrong_parts_o), np.stack(wrong_parts_l))
    assert np.abs(wo - ref_out).max() > 1e-2


# --------------------------------------------------------------------------- KV write

def test_e4m3_encode_matches_torch_in_range():
    import torch
    rng = np.random.default_rng(30)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 1e-3,
                        [0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 1.0625, 0.5]]).astype(np.float32)
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert (ref == ours).all()


def test_e4m3_encode_ties_saturation_and_sign():
    # exact midpoints between neighbouring codes go to the even code
    for c in range(0, 0x7D):
        lo, hi = oracle.e4m3_to_double(c), oracle.e4m3_to_double(c + 1)
        mid = np.float32((lo + hi) / 2)
        if float(mid) == (lo + hi) / 2:
            want = c if c % 2 == 0 else c + 1
            assert oracle.e4m3_encode(mid) == want, c
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE  # saturate
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(-0.0) == 0x80 and oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(float("nan")) == 0x7F


@pytest.mark.parametrize("W,I", [(1, 1), (3, 1), (8, 1), (3, 2), (8, 4)])
def test_write_kv_places_tokens_by_round_robin(W, I):
    rng = np.random.default_rng(40 + W + 7 * I)
    seq, ql, bs = [37, 5, 64, 9], [4, 2, 3, 1], 8
    B = len(seq)
    T = sum(ql)
    ind = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    kv_new = f32_to_bf16_bits(rng.standard_normal((T, D_K)))
    cap = [max(1, max(len(h) for h in _deal(L, W, I))) for L in seq]
    nb = [-(-c // bs) for c in cap]
    for r in range(W):
        perm = rng.permutation(sum(nb) + 2).astype(np.int32)
        bt = np.full((B, max(nb)), -1, np.int32)
        pos = 0
        for b in range(B):
            bt[b, :nb[b]] = perm[pos:pos + nb[b]]
            pos += nb[b]
        cache = np.zeros(((sum(nb) + 2) * bs, D_K), np.uint16)
        oracle.write_kv(seq, ind, kv_new, W, r, bt, bs, cache, interleave=I)
        # expected, by enumerating positions: token t of b at g = L - qlen + t,
        # at the rank's local index = its rank among the positions that rank holds
        want = np.zeros_like(cache)
        for b in range(B):
            held = _deal(seq[b], W, I)[r]
            for t in range(ql[b]):
                g = seq[b] - ql[b] + t
                if g in held:
                    j = held.index(g)
                    want[bt[b, j // bs] * bs + j % bs] = kv_new[ind[b] + t]
        assert (cache == want).all()


def test_write_kv_fp8_codes():
    rng = np.random.default_rng(50)
    seq, ql, bs = [20, 6], [3, 2], 4
    ind = np.array([0, 3, 5], np.int32)
    kv_new = f32_to_bf16_bits(rng.standard_normal((5, D_K)) * 3)
    bt = np.array([[3, 0, 1, 2, 4], [5, 6, -1, -1, -1]], np.int32)
    cache = np.zeros((7 * bs, D_K), np.uint8)
    scale = 0.01171875
    oracle.write_kv(seq, ind, kv_new, 1, 0, bt, bs, cache, kv_scale=scale)
    import torch
    vals = (kv_new.astype(np.uint32) << 16).view(np.float32)
    q = torch.tensor(vals / np.float32(scale)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for b in range(2):
        for t in range(ql[b]):
            g = seq[b] - ql[b] + t
            assert (cache[bt[b, g // bs] * bs + g % bs] == q[ind[b] + t]).all()
