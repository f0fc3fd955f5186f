"""Index + attention on the GPU against the oracle, through the C ABI.

Each case builds a LayerGroup (caches written by the library's own append
kernels from seeded bf16 inputs), runs one step, and checks every sampled
query: cache bytes bit-exact; Full-layer pool and top-k against the oracle's
global definitions; Reindex top-k against the oracle run on the GPU's pool;
attention of every layer against the oracle run on the GPU's index set.
"""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import bf16_to_f64, check_attention, check_status, run_group, verify_query

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("records", [True, False])
def test_tiny_group_8k(records):
    """8192 entries, Full + Reindex + Reuse, pool 256 x 8 (smaller than
    top-512: the Full top-k comes from the top-512 blocks); indexer K as
    576-byte records or as BLOCK8 codes with a scale plane."""
    from csa2_sparse_attention_gb300 import abi
    wl = W.tiny()
    g = run_group(wl, ik_layout=abi.LAYOUT_BLOCK8R if records else abi.LAYOUT_BLOCK8)
    check_status(g)
    verify_query(g, wl, 0)
    # the Reuse layer attends over the Reindex layer's own top-k buffer (the
    # same device memory, not a copy); only Full/Reindex layers own one
    assert sorted(g.topk) == [0, 1]
    assert g.attn_index[2] is g.topk[1] and g.attn_index[2].data_ptr() == g.topk[1].data_ptr()
    assert g.attn_index[1] is g.topk[1] and g.attn_index[0] is g.topk[0]


@pytest.mark.parametrize("pool,topk", [(2048, 512), (256, 512), (64, 100)])
def test_ragged_small_contexts(pool, topk):
    """Partial last blocks, contexts below the window, below one block,
    and fewer blocks than the pool."""
    ctx = [20000, 8191, 1000, 333, 129, 100, 17, 8, 5, 1]
    wl = W.small_variant(W.group_128k(), ctx, name="ragged-small",
                         layers=("F", "R", "X", "R"), pool_blocks=pool, topk=topk, hot_blocks=4)
    g = run_group(wl)
    check_status(g)
    for q in range(len(ctx)):
        verify_query(g, wl, q)


def test_many_query_shared_cache_m2():
    """Queries at consecutive raw positions over one shared m=2 cache."""
    wl = W.many_query(queries=48, entries=6000, m=2)
    g = run_group(wl)
    check_status(g)
    for q in (0, 1, 23, 47):
        verify_query(g, wl, q, check_cache=(q == 0))


# The batch size picks the attention launch form (8 + 128 entries per query,
# so 2 splits of 128 or 1 of 160).  On a 152-SM GB300: reps 1 (4 queries)
# four head groups per query, reps 5 (20) two head groups, reps 10 (40) two
# head groups over one 160-entry split, reps 33 (132) one CTA per query with
# an online softmax over 128-entry chunks.
@pytest.mark.parametrize("reps", [1, 5, 10, 33])
def test_attention_direct_edge_cases(reps):
    """Direct csa2_sparse_attn calls: -1 pads, empty selection, window 0,
    single entry, and an out-of-range index that is skipped and recorded;
    the bf16 output is the fp32 output rounded once."""
    from csa2_sparse_attention_gb300 import abi
    rng = np.random.default_rng(11)
    n_rows, B, K, Wn = 64, 4 * reps, 8, 128
    codes = rng.integers(0, 256, (n_rows, 256)).astype(np.uint8)
    scales = rng.integers(0x28, 0x38, (n_rows, 32)).astype(np.uint8)
    swa = rng.integers(0, 0x7E, (B, Wn, 512)).astype(np.uint8)
    q = torch.randn((B, 64, 512), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    kv_start = np.tile(np.array([0, 16, 32, 48], dtype=np.int64), reps)
    n_vis = np.tile(np.array([16, 1, 16, 12], dtype=np.int32), reps)
    top = np.full((B, K), -1, dtype=np.int32)
    top[0::4, :5] = [0, 3, 7, 8, 15]
    top[1::4, 0] = 0
    top[2::4, :3] = [1, 2, 99]       # 99 >= n: skipped and recorded
    cases_window = 0
    d = "cuda"
    t = lambda a: torch.from_numpy(a).to(d)
    out = torch.zeros((B, 64, 512), dtype=torch.float32, device=d)
    lse = torch.zeros((B, 64), dtype=torch.float32, device=d)
    for window in (Wn, cases_window):
        ws = torch.zeros(abi.csa2_workspace_bytes(abi.OP_SPARSE_ATTN, B, 16, 1, K), dtype=torch.uint8, device=d)
        abi.csa2_sparse_attn(q.to(d), B, t(codes), t(scales), n_rows, t(kv_start), t(n_vis), t(top), K,
                             t(swa), None, window, 1 / np.sqrt(512), out, abi.OUT_F32, lse, ws, ws.numel())
        torch.cuda.synchronize()
        st = abi.csa2_status_fetch(ws)
        assert st[0] == abi.ERR_DEVICE_BOUNDS and st[1] == 7 and st[2] % 4 == 2 and st[3] == 99
        out16 = torch.zeros((B, 64, 512), dtype=torch.bfloat16, device=d)
        ws16 = torch.zeros_like(ws)
        abi.csa2_sparse_attn(q.to(d), B, t(codes), t(scales), n_rows, t(kv_start), t(n_vis), t(top), K,
                             t(swa), None, window, 1 / np.sqrt(512), out16, abi.OUT_BF16, None, ws16, ws16.numel())
        torch.cuda.synchronize()
        assert torch.equal(out16, out.to(torch.bfloat16))
        qn = bf16_to_f64(q)
        for b in range(B):
            rows = codes[kv_start[b]:kv_start[b] + n_vis[b]]
            cu = O.unpack_codes(rows)
            sc = scales[kv_start[b]:kv_start[b] + n_vis[b]]
            ids = top[b].copy()
            ids[ids >= n_vis[b]] = -1
            sel, win = O.attention_inputs(ids, cu, sc, swa[b], int(n_vis[b]), Wn)
            if window == 0:
                win = win[:0]
            o_ref, lse_ref = O.sparse_attention(qn[b], sel, win)
            if sel.shape[0] + win.shape[0] == 0:
                assert np.all(bf16_to_f64(out[b]) == 0)
                assert np.all(np.isneginf(lse[b].cpu().numpy()))
            else:
                check_attention(bf16_to_f64(out[b]), o_ref, f"b{b} window {window}")
                # fp32 logits over 512 terms: error <= 512 * 2^-24 * sigma * sum|q_i c_i|
                allc = np.concatenate([sel, win])
                bound = 512 * 2.0 ** -24 * (np.abs(qn[b]) @ np.abs(allc).T).max(axis=1) / np.sqrt(512)
                assert np.all(np.abs(lse[b].cpu().numpy() - lse_ref) <= bound + 1e-5 * np.abs(lse_ref))


def test_attention_bf16_output_within_its_rounding():
    """The bf16 output is the fp32 result rounded once: within bf16's unit
    roundoff (2^-8) of the oracle plus the fp32 path's own error."""
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    wl = W.tiny()
    g = LayerGroup(wl, out_dtype=torch.bfloat16)
    g.fill()
    g.step()
    torch.cuda.synchronize()
    inp_check = verify_query.__globals__["oracle_query"](wl, 0)
    from oracle import csa2_oracle as Orc
    lc, ls = Orc.quantize_fp4(Orc.rope(inp_check["latent_real"], inp_check["positions"]))
    for li in range(len(wl.layers)):
        src = W.index_source(wl, li)
        ring = Orc.append_swa_fp8(inp_check["swa_real"][li])
        sel, win = Orc.attention_inputs(g.topk[src][0].cpu().numpy(), lc, ls, ring, wl.contexts[0], wl.window)
        o_ref, _ = Orc.sparse_attention(inp_check["attn_q"][li], sel, win)
        o = bf16_to_f64(g.out[li][0])
        err = np.abs(o - o_ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(o_ref) + 1e-5 * np.abs(o_ref).max(axis=-1, keepdims=True))


# 3 queries (four head groups), 42 (two head groups over one 160-entry split)
# or 129 (one CTA per query)
@pytest.mark.parametrize("reps", [1, 14, 43])
def test_attention_subnormal_window_bytes_and_scales(reps):
    """Window bytes that are all E4M3 subnormals (|x| <= 7 * 2^-9) and FP4
    rows whose scales are all subnormal: the output is made of those values
    only, so a decode that flushed them to zero fails the relative check."""
    from csa2_sparse_attention_gb300 import abi
    rng = np.random.default_rng(12)
    n_rows, B, K, Wn = 64, 3 * reps, 16, 128
    codes = rng.integers(0, 256, (n_rows, 256)).astype(np.uint8)
    scales = rng.integers(0x01, 0x08, (n_rows, 32)).astype(np.uint8)          # subnormal scales
    sub = np.concatenate([np.arange(0x01, 0x08), np.arange(0x81, 0x88)]).astype(np.uint8)
    swa = rng.choice(sub, (B, Wn, 512)).astype(np.uint8)                     # subnormal window
    q = torch.randn((B, 64, 512), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    kv_start = np.tile(np.array([0, 16, 32], dtype=np.int64), reps)
    n_vis = np.tile(np.array([16, 16, 30], dtype=np.int32), reps)
    top = np.full((B, K), -1, dtype=np.int32)
    top[1::3, :6] = [0, 2, 4, 6, 8, 10]  # query 0: window only; 1: both; 2: top-k only (window 0)
    top[2::3, :16] = np.arange(16)
    d = "cuda"
    t = lambda a: torch.from_numpy(a).to(d)
    out = torch.zeros((B, 64, 512), dtype=torch.float32, device=d)
    lse = torch.zeros((B, 64), dtype=torch.float32, device=d)
    qn = bf16_to_f64(q)
    for window in (Wn, 0):
        ws = torch.zeros(abi.csa2_workspace_bytes(abi.OP_SPARSE_ATTN, B, 16, 1, K), dtype=torch.uint8, device=d)
        abi.csa2_sparse_attn(q.to(d), B, t(codes), t(scales), n_rows, t(kv_start), t(n_vis), t(top), K,
                             t(swa), None, window, 1 / np.sqrt(512), out, abi.OUT_F32, lse, ws, ws.numel())
        torch.cuda.synchronize()
        assert abi.csa2_status_fetch(ws)[0] == 0
        for b in range(B):
            rows = codes[kv_start[b]:kv_start[b] + n_vis[b]]
            sel, win = O.attention_inputs(top[b], O.unpack_codes(rows), scales[kv_start[b]:kv_start[b] + n_vis[b]],
                                          swa[b], int(n_vis[b]), Wn)
            if window == 0:
                win = win[:0]
            if sel.shape[0] + win.shape[0] == 0:
                continue
            o_ref, _ = O.sparse_attention(qn[b], sel, win)
            assert np.abs(o_ref).max() < 2.0 ** -3 * 6  # built from subnormal-scale values only
            check_attention(bf16_to_f64(out[b]), o_ref, f"subnormal b{b} window {window}")


def test_many_queries_each_with_its_own_cache():
    """256 queries (the many-query scan's batch size) whose caches all
    differ: every query is its own run inside a group of four."""
    ctx = [1000 + 7 * i for i in range(256)]
    wl = W.small_variant(W.group_128k(), ctx, name="many-own-caches", layers=("F", "X", "R"),
                         pool_blocks=128, topk=512, hot_blocks=2)
    g = run_group(wl)
    check_status(g)
    for q in (0, 1, 130, 255):
        verify_query(g, wl, q, check_cache=(q == 0))


def test_step_with_pipelined_host_io_matches_plain_step():
    """LayerGroup.step_io (inputs in and outputs out on two copy streams,
    captured with the step in one graph) reads back exactly what a plain
    step computes, for every layer."""
    wl = W.tiny()
    g = run_group(wl)
    plain = [(o.clone(), l.clone()) for o, l in zip(g.out, g.lse)]
    host = g.host_buffers()
    for hl in host[2]:  # poison the host outputs
        for h in hl:
            h.fill_(float("nan"))
    stream = torch.cuda.Stream()
    g.capture_io(stream, (torch.cuda.Stream(), torch.cuda.Stream()), host)
    g.replay_io()
    torch.cuda.synchronize()
    check_status(g)
    for li, (o, l) in enumerate(plain):
        assert torch.equal(host[2][li][0], o.cpu()), f"layer {li} output"
        assert torch.equal(host[2][li][1], l.cpu()), f"layer {li} lse"


def test_index_calls_with_a_query_that_sees_nothing():
    """csa2_index_full and csa2_index_reindex where one query of three has no
    visible position: its pool and top-k are all -1 pads, the other queries
    match the oracle, and nothing is recorded as an error."""
    from csa2_sparse_attention_gb300 import abi
    from tests.helpers import check_selection, kth_value, rows_to_block8
    contexts = (5000, 0, 300)
    n_q, P, K = len(contexts), 256, 128
    rng = np.random.default_rng(31)
    rows_of = [max(8, ((n + 7) // 8) * 8) for n in contexts]
    kv_start = np.concatenate([[0], np.cumsum(rows_of)[:-1]]).astype(np.int64)
    n_rows = int(sum(rows_of))
    k_real = torch.randn((n_rows, 128), generator=torch.Generator().manual_seed(32)).to(torch.bfloat16)
    kc, ks = O.quantize_fp4(k_real.float().numpy().astype(np.float64))
    kdq = O.dequantize_fp4(kc, ks)
    q_real = torch.randn((n_q * 32, 128), generator=torch.Generator().manual_seed(33)).to(torch.bfloat16)
    qc, qs = O.quantize_fp4(q_real.float().numpy().astype(np.float64))
    qdq = O.dequantize_fp4(qc, qs).reshape(n_q, 32, 128)
    w = rng.uniform(0, 1, (n_q, 32)).astype(np.float32)
    d = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(d)
    args = (t(rows_to_block8(O.pack_codes(qc))), t(qs), t(w), n_q, t(rows_to_block8(O.pack_codes(kc))), t(ks),
            n_rows, t(kv_start), t(np.asarray(contexts, dtype=np.int32)), max(contexts))
    ws = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_FULL, n_q, max(contexts), P, K), dtype=torch.uint8,
                     device=d)
    pool = torch.full((n_q, P), -7, dtype=torch.int32, device=d)
    topk = torch.full((n_q, K), -7, dtype=torch.int32, device=d)
    abi.csa2_index_full(*args, P, K, pool, topk, ws, ws.numel())
    ws_re = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_REINDEX, n_q, max(contexts), P, K),
                        dtype=torch.uint8, device=d)
    topk_re = torch.full((n_q, K), -7, dtype=torch.int32, device=d)
    abi.csa2_index_reindex(*args, pool, P, K, topk_re, ws_re, ws_re.numel())
    torch.cuda.synchronize()
    assert abi.csa2_status_fetch(ws)[0] == 0 and abi.csa2_status_fetch(ws_re)[0] == 0
    assert torch.all(pool[1] == -1) and torch.all(topk[1] == -1) and torch.all(topk_re[1] == -1)
    for q in (0, 2):
        n = contexts[q]
        scores = O.index_scores(qdq[q], w[q].astype(np.float64), kdq[kv_start[q]:kv_start[q] + n])
        bmax = O.block_max(scores)
        check_selection(pool[q].cpu().numpy(), O.select_top(bmax, P), lambda b: bmax[b], kth_value(bmax, P),
                        f"q{q} pool")
        top_o = O.select_top(scores, K)
        check_selection(topk[q].cpu().numpy(), top_o, lambda p: scores[p], kth_value(scores, K), f"q{q} top-k")
        re_o, cand, sc = O.index_reindex(qdq[q], w[q].astype(np.float64), kdq[kv_start[q]:kv_start[q] + n], n,
                                         pool[q].cpu().numpy(), K)
        smap = dict(zip(cand.tolist(), sc.tolist()))
        check_selection(topk_re[q].cpu().numpy(), re_o, lambda p: smap[p], kth_value(sc, K), f"q{q} reindex")
