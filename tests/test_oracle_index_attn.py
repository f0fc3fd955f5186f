"""Pins for the oracle's RoPE, indexer, selection and attention (CPU only).

Checks: closed forms of RoPE (pair 0 rotates by p radians, pair D/4 by p/100
at theta=10000, the group law, norm preservation); a hand-worked indexer
score; brute-force top-k by repeated extraction; the pool constants; the
Full-top-k-inside-pool and Reindex/Reuse invariants; and attention special
cases that reduce to torch's scaled_dot_product_attention.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O


# ----------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity_and_quantizes_like_plain():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, 512))
    assert np.array_equal(O.rope(x, np.zeros(5)), x)
    a = O.append_main_latent(x, np.zeros(5, dtype=np.int64))
    b = O.append_plain_fp4(x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rope_closed_forms():
    p = 1234.0
    e0 = np.zeros((1, 512)); e0[0, 0] = 1.0
    y = O.rope(e0, np.array([p]))
    # pair 0 has frequency theta^0 = 1: rotation by p radians, in channels 0 and 1 only
    assert y[0, 0] == pytest.approx(np.cos(p), abs=1e-12)
    assert y[0, 1] == pytest.approx(np.sin(p), abs=1e-12)
    assert np.count_nonzero(y[0, 2:]) == 0
    # pair 128 (channels 256, 257): 10000^(-256/512) = 1/100
    e = np.zeros((1, 512)); e[0, 257] = 1.0
    y = O.rope(e, np.array([p]))
    assert y[0, 256] == pytest.approx(-np.sin(p / 100), abs=1e-12)
    assert y[0, 257] == pytest.approx(np.cos(p / 100), abs=1e-12)
    assert np.count_nonzero(np.delete(y[0], [256, 257])) == 0


def test_rope_group_law_and_norms():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(4, 512))
    p1 = np.array([3, 1000, 77777, 1 << 20])
    p2 = np.array([5, 24, 3, 12345])
    a = O.rope(O.rope(x, p1), p2)
    b = O.rope(x, p1 + p2)
    assert np.max(np.abs(a - b)) < 1e-9
    n0 = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    y = O.rope(x, p1)
    n1 = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    assert np.max(np.abs(n0 - n1)) < 1e-12


# --------------------------------------------------------------- indexer
def test_index_score_hand_worked():
    # 2 heads of dim 16: q0 = e0, q1 = e1, w = (1, 0.5)
    q = np.zeros((2, 16)); q[0, 0] = 1; q[1, 1] = 1
    w = np.array([1.0, 0.5])
    k = np.zeros((4, 16))
    k[0, :2] = (2, 3)     # 1*2 + 0.5*3 = 3.5
    k[1, :2] = (-1, 4)    # ReLU(-1) = 0; 0.5*4 = 2
    k[2, :2] = (3, -2)    # 3 + 0 = 3
    k[3, :2] = (-1, -1)   # 0
    assert O.index_scores(q, w, k).tolist() == [3.5, 2.0, 3.0, 0.0]


def test_index_scores_exact_against_rationals():
    """On FP4-dequantized data, the fp64 scores agree with exact rational
    arithmetic to 1e-15 relative (the per-head dots are exact in fp64)."""
    rng = np.random.default_rng(2)
    qc, qs = O.quantize_fp4(rng.normal(size=(32, 128)))
    kc, ks = O.quantize_fp4(rng.normal(size=(6, 128)))
    q, k = O.dequantize_fp4(qc, qs), O.dequantize_fp4(kc, ks)
    w = rng.uniform(size=32).astype(np.float32).astype(np.float64)
    got = O.index_scores(q, w, k)
    for s in range(6):
        exact = Fraction(0)
        for h in range(32):
            dot = sum(Fraction(q[h, d]) * Fraction(k[s, d]) for d in range(128))
            exact += Fraction(w[h]) * max(dot, Fraction(0))
        assert abs(Fraction(got[s]) - exact) <= abs(exact) * Fraction(1, 10 ** 15)


def _brute_top(values, count):
    """Repeated extraction: take the largest remaining, lowest index on ties."""
    vals = list(values)
    taken = []
    for _ in range(min(count, len(vals))):
        best = None
        for i, v in enumerate(vals):
            if i in taken:
                continue
            if best is None or v > vals[best]:
                best = i
        taken.append(best)
    return sorted(taken)


@pytest.mark.parametrize("seed", range(8))
def test_select_top_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 60))
    vals = rng.integers(0, 6, n).astype(float)  # many ties
    count = int(rng.integers(1, 70))
    assert O.select_top(vals, count).tolist() == _brute_top(vals, count)


def test_block_max_partial_last_block():
    s = np.arange(21, dtype=float)[::-1]  # 20 .. 0
    b = O.block_max(s)
    assert b.tolist() == [20, 12, 4]  # last block holds positions 16..20 only


def test_pool_constants():
    assert O.POOL_BLOCKS * O.BLOCK == 16384
    rng = np.random.default_rng(3)
    n = 20000
    s = rng.normal(size=n)
    pool = O.select_top(O.block_max(s), O.POOL_BLOCKS)
    assert len(pool) == min(O.POOL_BLOCKS, -(-n // 8))
    assert len(O.pool_positions(pool, n)) == 16384
    small = O.select_top(O.block_max(s[:100]), O.POOL_BLOCKS)
    assert len(small) == 13  # ceil(100/8): fewer blocks than the pool holds


def test_visibility_m2_edges():
    assert [O.visible_entries(p, 2) for p in range(5)] == [0, 1, 1, 2, 2]
    assert O.visible_entries(524287, 2) == 262144
    assert O.visible_entries(520192, 2) == 260096
    assert [O.visible_entries(p, 1) for p in range(3)] == [1, 2, 3]


def _random_index_case(seed, n, hot=8):
    rng = np.random.default_rng(seed)
    qc, qs = O.quantize_fp4(rng.normal(size=(32, 128)))
    q = O.dequantize_fp4(qc, qs)
    k_real = rng.normal(size=(n, 128))
    u = q.sum(axis=0) / np.sqrt(32)
    for b in rng.choice(-(-n // 8), size=min(hot, -(-n // 8)), replace=False):
        k_real[b * 8: b * 8 + 8] += 0.5 * u
    kc, ks = O.quantize_fp4(k_real)
    return q, rng.uniform(size=32), O.dequantize_fp4(kc, ks), rng


@pytest.mark.parametrize("n,P,K", [(3000, 64, 512), (8191, 256, 512), (517, 256, 512),
                                   (40, 3, 20), (30000, 2048, 512), (6000, 512, 512)])
def test_full_topk_lies_in_top_blocks_and_reindex_reproduces_it(n, P, K):
    """The global top-K positions lie in the top-max(P, K) blocks by block
    maximum (ties to the lower block).  So for K <= P they lie in the pool and
    a Reindex layer given the Full layer's own q, w reproduces the Full top-K."""
    q, w, k, rng = _random_index_case(4, n)
    pool, top, scores, bmax = O.index_full(q, w, k, n, P, K)
    top = top[top >= 0]
    assert len(top) == min(K, n)
    wide = O.select_top(bmax, max(P, K))
    assert set((top // 8).tolist()) <= set(wide.tolist())
    if K <= P:
        assert set((top // 8).tolist()) <= set(pool[pool >= 0].tolist())
        re, cand, _ = O.index_reindex(q, w, k, n, pool, K)
        assert np.array_equal(re[re >= 0], top)
    # Reuse layers take the indices unchanged
    assert O.index_reuse(top) is top


def test_full_topk_can_leave_a_pool_smaller_than_k():
    """With fewer pool blocks than K (the tiny 256-block pool with K = 512)
    the global top-K need not fit in the pool: a case that shows it."""
    q, w, k, rng = _random_index_case(4, 3000)
    pool, top, *_ = O.index_full(q, w, k, 3000, 64, 512)
    top = top[top >= 0]
    assert not set((top // 8).tolist()) <= set(pool.tolist())


def test_reindex_selects_only_pool_positions():
    q, w, k, rng = _random_index_case(5, 4000)
    pool, top, *_ = O.index_full(q, w, k, 4000, 32, 512)
    q2 = rng.normal(size=(32, 128))
    re, cand, _ = O.index_reindex(q2, rng.uniform(size=32), k, 4000, pool, 512)
    re = re[re >= 0]
    assert len(re) == 256  # 32 blocks x 8 positions < 512: all of the pool
    assert set((re // 8).tolist()) <= set(pool.tolist())


# ------------------------------------------------------------- attention
def _sdpa(q, keys, scale):
    qt = torch.from_numpy(q)[None, :, None, :]        # [1, H, 1, D]
    kt = torch.from_numpy(keys)[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=scale)
    return o[0, :, 0, :].numpy()


def test_attention_dense_when_k_covers_context_and_no_window():
    rng = np.random.default_rng(6)
    n = 300
    c = rng.normal(size=(n, 512))
    q = rng.normal(size=(64, 512))
    o, lse = O.sparse_attention(q, c, np.zeros((0, 512)))
    assert np.max(np.abs(o - _sdpa(q, c, O.SM_SCALE))) < 1e-12
    ref_lse = np.log(np.exp(O.SM_SCALE * q @ c.T).sum(axis=1))
    assert np.max(np.abs(lse - ref_lse)) < 1e-10


def test_attention_window_only_and_merged_softmax():
    rng = np.random.default_rng(7)
    q = rng.normal(size=(64, 512))
    win = rng.normal(size=(128, 512))
    o, _ = O.sparse_attention(q, np.zeros((0, 512)), win)
    assert np.max(np.abs(o - _sdpa(q, win, O.SM_SCALE))) < 1e-12
    sel = rng.normal(size=(37, 512))
    sel[3] = win[5]  # the same latent in both sets is counted twice (no dedup)
    o, _ = O.sparse_attention(q, sel, win)
    both = np.concatenate([sel, win])
    assert np.max(np.abs(o - _sdpa(q, both, O.SM_SCALE))) < 1e-12


def test_attention_single_entry_returns_it():
    rng = np.random.default_rng(8)
    c = rng.normal(size=(1, 512))
    q = rng.normal(size=(64, 512))
    o, lse = O.sparse_attention(q, c, np.zeros((0, 512)))
    assert np.max(np.abs(o - c)) < 1e-12
    assert np.max(np.abs(lse - O.SM_SCALE * (q @ c[0]))) < 1e-12


def test_attention_inputs_window_ring_and_pads():
    rng = np.random.default_rng(9)
    n = 300
    codes = rng.integers(0, 16, (n, 512))
    scales = rng.integers(0x20, 0x40, (n, 32)).astype(np.uint8)
    ring = rng.integers(0, 0x7E, (128, 512)).astype(np.uint8)
    ids = np.array([5, 17, 299, -1, -1])
    sel, win = O.attention_inputs(ids, codes, scales, ring, n)
    assert sel.shape == (3, 512) and win.shape == (128, 512)
    assert np.array_equal(sel[1], O.dequantize_fp4(codes[17], scales[17]))
    # positions 172..299: position p sits in slot p mod 128
    assert np.array_equal(win[0], O.e4m3_decode(ring[172 % 128]))
    assert np.array_equal(win[-1], O.e4m3_decode(ring[299 % 128]))
    # short context: only slots 0..n-1 exist
    _, win = O.attention_inputs(ids[:1], codes, scales, ring, 10)
    assert win.shape == (10, 512)
    assert np.array_equal(win[9], O.e4m3_decode(ring[9]))


def test_decode_group_reuse_layers_share_indices():
    rng = np.random.default_rng(10)
    n = 1500
    layers = ("F", "R", "X", "R")
    iq = {0: rng.normal(size=(32, 128)), 2: rng.normal(size=(32, 128))}
    iw = {0: rng.uniform(size=32), 2: rng.uniform(size=32)}
    swa = {i: rng.normal(size=(128, 512)) for i in range(4)}
    aq = {i: rng.normal(size=(64, 512)) for i in range(4)}
    out = O.decode_group_query(layers, iq, iw, rng.normal(size=(n, 128)), rng.normal(size=(n, 512)),
                               np.arange(n), swa, aq, n, pool_blocks=64, topk=100)
    assert out["topk"][1] is out["topk"][0]
    assert out["topk"][3] is out["topk"][2]
    assert not np.array_equal(out["topk"][0], out["topk"][2])
    assert set((out["topk"][2] // 8).tolist()) <= set(out["pool"].tolist())
    for i in range(4):
        assert out["o"][i].shape == (64, 512) and np.all(np.isfinite(out["o"][i]))


def test_shared_sequence_window_is_the_ring_window_of_the_same_positions():
    """The prefill window (rows of the shared sequence) selects exactly the
    latents a decode ring holding the same last positions selects, so the
    prefill attention reduces to the pinned ring definition; a context
    shorter than the window takes all of its positions."""
    rng = np.random.default_rng(17)
    W_ = 128
    for n in (1, 77, 128, 129, 1000):
        win_rows = rng.integers(0, 0x7F, (n, 512)).astype(np.uint8)  # finite E4M3 bytes
        win_rows[:, ::3] |= 0x80
        ring = np.zeros((W_, 512), dtype=np.uint8)
        for p in range(max(0, n - W_), n):
            ring[p % W_] = win_rows[p]
        codes = rng.integers(0, 16, (n, 512))
        scales = rng.integers(0x30, 0x40, (n, 32)).astype(np.uint8)
        topk = np.array([0, n - 1, -1, n // 2])
        sel_a, win_a = O.attention_inputs(topk, codes, scales, ring, n, W_)
        sel_b, win_b = O.attention_inputs_shared_window(topk, codes, scales, win_rows, n, W_)
        assert np.array_equal(sel_a, sel_b) and np.array_equal(win_a, win_b)
        assert win_b.shape[0] == min(n, W_)
        assert np.array_equal(win_b, O.e4m3_decode(win_rows[max(0, n - W_):n]))
