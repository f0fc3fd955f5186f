"""Test infrastructure: oracle inputs for a workload query, the BLOCK8 layout
permutation, and the acceptance rules.

Acceptance (floating-point results are compared with the fp64 oracle):
  * FP4/FP8 bytes: bit-exact when both sides quantize the same values; after
    RoPE (device fp32 vs oracle fp64) a byte may differ only where the
    oracle's value lies within 2^-20 relative of a rounding threshold.
  * top-k / pool sets: identical except members whose oracle score lies
    within 1e-5 relative of the K-th (P-th block) oracle score.
  * attention: max|o - o*| / max|o*| <= 2e-3 per (query, head) with o* the
    oracle run on the GPU's index set.  bf16 rounding of the output alone
    contributes up to 2^-9 ~ 1.95e-3, so the kernels keep their own error
    near fp32 level.
"""
from __future__ import annotations

import numpy as np

from csa2_sparse_attention_gb300 import workloads as W
from oracle import csa2_oracle as O

TOPK_REL = 1e-5
ATTN_REL = 2e-3


def block8_to_rows(plane, n_rows):
    """BLOCK8 code plane (bytes) -> row-major [n_rows][64]."""
    a = np.asarray(plane, dtype=np.uint8).reshape(n_rows // 8, 4, 8, 16)
    return a.transpose(0, 2, 1, 3).reshape(n_rows, 64)


def rows_to_block8(rows):
    n = rows.shape[0]
    return np.ascontiguousarray(rows.reshape(n // 8, 8, 4, 16).transpose(0, 2, 1, 3)).reshape(-1)


def rows_to_records(code_rows, scale_rows):
    """Row-major codes [n][64] and scales [n][8] (n a multiple of 8) ->
    BLOCK8R records (576 bytes per 8 rows)."""
    n = code_rows.shape[0]
    blk = rows_to_block8(code_rows).reshape(n // 8, 512)
    return np.ascontiguousarray(np.concatenate([blk, np.asarray(scale_rows, np.uint8).reshape(n // 8, 64)],
                                               axis=1)).reshape(-1)


def records_to_rows(plane, n_rows):
    """BLOCK8R records (576 bytes per 8 rows: codes as BLOCK8, then the 8
    rows' 8 scale bytes) -> (codes [n_rows][64], scales [n_rows][8])."""
    a = np.asarray(plane, dtype=np.uint8).reshape(n_rows // 8, 576)
    codes = block8_to_rows(a[:, :512].reshape(-1), n_rows)
    return codes, a[:, 512:].reshape(n_rows, 8)


def indexer_k_planes(g, r0, r1):
    """Rows [r0, r1) (r0 a multiple of 8) of a LayerGroup's indexer K as
    (codes [rows][64], scales [rows][8]), whichever layout it uses."""
    from csa2_sparse_attention_gb300 import abi
    r1_8 = (r1 + 7) // 8 * 8
    if g.ik_layout == abi.LAYOUT_BLOCK8R:
        codes, scales = records_to_rows(g.ik_codes[r0 // 8 * 576:r1_8 // 8 * 576].cpu().numpy(), r1_8 - r0)
    else:
        codes = block8_to_rows(g.ik_codes[r0 * 64:r1_8 * 64].cpu().numpy(), r1_8 - r0)
        scales = g.ik_scales[r0:r1_8].cpu().numpy()
    return codes[:r1 - r0], scales[:r1 - r0]


def check_selection(gpu_ids, oracle_ids, score_of, kth, label="", strict=False):
    """Sets equal except members whose score is within TOPK_REL of kth.
    gpu_ids must be ascending then -1 padded.  strict: the sets must be
    exactly equal (no waiver), for inputs whose scores are exact on both
    sides, so that equal scores are genuine ties the rule breaks toward the
    lower index."""
    g = np.asarray(gpu_ids)
    valid = g[g >= 0]
    assert np.all(g[len(valid):] == -1), f"{label}: pads not at the end"
    assert np.all(np.diff(valid) > 0), f"{label}: not strictly ascending"
    o = np.asarray(oracle_ids)
    o = o[o >= 0]
    assert len(valid) == len(o), f"{label}: {len(valid)} vs {len(o)} selected"
    diff = set(valid.tolist()) ^ set(o.tolist())
    if strict:
        assert not diff, f"{label}: {len(diff)} members differ (strict), e.g. {sorted(diff)[:5]}"
        return 0
    tol = TOPK_REL * max(abs(kth), 1e-30)
    bad = [p for p in diff if abs(score_of(p) - kth) > tol]
    assert not bad, f"{label}: {len(bad)} members differ beyond tolerance, e.g. {bad[:5]}"
    return len(diff)


def kth_value(values, k):
    v = np.sort(np.asarray(values))[::-1]
    return v[min(k, len(v)) - 1]


def check_attention(o_gpu, o_ref, label=""):
    """Per head row: max|o - o*| / max|o*| <= ATTN_REL."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.max(np.abs(o_gpu - o_ref), axis=-1)
    den = np.max(np.abs(o_ref), axis=-1)
    rel = np.where(den > 0, err / np.where(den > 0, den, 1), err)
    worst = float(rel.max())
    assert worst <= ATTN_REL, f"{label}: attention rel error {worst:.3g} > {ATTN_REL}"
    return worst


def oracle_query(wl: W.Workload, q, n=None):
    """Inputs of query q in the form oracle.decode_group_query takes."""
    r = W.request_of(wl, q)
    n = wl.contexts[q] if n is None else n
    idx = [i for i, m in enumerate(wl.layers) if m in (W.FULL, W.REINDEX)]
    return dict(
        layers=wl.layers,
        index_q={i: W.indexer_q(wl, q, i) for i in idx},
        index_w={i: W.indexer_w(wl, q, i).astype(np.float64) for i in idx},
        k_real=W.indexer_k_rows(wl, r, 0, n),
        latent_real=W.main_latent_rows(wl, r, 0, n),
        positions=W.latent_positions(wl, r)[:n],
        swa_real={i: (W.swa_seq_rows(wl, i, 0, n) if wl.shared_window else W.swa_ring(wl, q, i))
                  for i in range(len(wl.layers))},
        attn_q={i: W.attn_q(wl, q, i) for i in range(len(wl.layers))},
        n=n, pool_blocks=wl.pool_blocks, topk=wl.topk, window=wl.window)


def bf16_to_f64(t):
    """A torch bf16 tensor (any device) as float64 numpy."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def run_group(wl, **kw):
    import torch
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    g = LayerGroup(wl, **kw)
    for ws in (g.ws_app, g.ws_full, g.ws_re, g.ws_attn):
        ws.zero_()
    g.fill()
    g.step()
    torch.cuda.synchronize()
    return g


def verify_query(g, wl, q, check_cache=True):
    inp = oracle_query(wl, q)
    n, P, K = inp["n"], wl.pool_blocks, wl.topk
    r = W.request_of(wl, q)
    base = g.row_base[r] if not wl.shared_cache else 0
    kc, ks = O.quantize_fp4(inp["k_real"])
    kdq = O.dequantize_fp4(kc, ks)
    lc, ls = O.quantize_fp4(O.rope(inp["latent_real"], inp["positions"]))
    if check_cache:
        gk, gs = indexer_k_planes(g, base, base + n)
        assert np.array_equal(gk, O.pack_codes(kc)), "indexer K bytes"
        assert np.array_equal(gs, ks), "indexer K scales"
        gl = g.kv_codes[base:base + n].cpu().numpy()
        assert np.array_equal(gl, O.pack_codes(lc)), "main latent bytes"
        assert np.array_equal(g.kv_scales[base:base + n].cpu().numpy(), ls), "main latent scales"
    topk_of = {}
    for li, mode in enumerate(wl.layers):
        if mode in (W.FULL, W.REINDEX):
            qc, qs = O.quantize_fp4(inp["index_q"][li])
            qdq = O.dequantize_fp4(qc, qs)
            gt = g.topk[li][q].cpu().numpy()
            if mode == W.FULL:
                pool_o, top_o, scores, bmax = O.index_full(qdq, inp["index_w"][li], kdq, n, P, K)
                gp = g.pools[li][q].cpu().numpy()
                check_selection(gp, pool_o, lambda b: bmax[b], kth_value(bmax, P), f"q{q} pool")
                check_selection(gt, top_o, lambda p: scores[p], kth_value(scores, K), f"q{q} L{li} top-k")
                gpu_pool = gp
            else:
                re_o, cand, sc = O.index_reindex(qdq, inp["index_w"][li], kdq, n, gpu_pool, K)
                smap = dict(zip(cand.tolist(), sc.tolist()))
                check_selection(gt, re_o, lambda p: smap[p], kth_value(sc, K), f"q{q} L{li} reindex")
            topk_of[li] = gt
        else:
            topk_of[li] = topk_of[W.index_source(wl, li)]
        ring = O.append_swa_fp8(inp["swa_real"][li])
        if wl.shared_window:  # the window over the shared sequence: rows [0, n) of the layer's array
            assert np.array_equal(g.swa[li][:n].cpu().numpy(), ring), "window bytes"
            sel, win = O.attention_inputs_shared_window(topk_of[li], lc, ls, ring, n, wl.window)
        else:
            assert np.array_equal(g.swa[li][q].cpu().numpy(), ring), "window bytes"
            sel, win = O.attention_inputs(topk_of[li], lc, ls, ring, n, wl.window)
        o_ref, lse_ref = O.sparse_attention(inp["attn_q"][li], sel, win)
        check_attention(bf16_to_f64(g.out[li][q]), o_ref, f"q{q} L{li} attention")
        lse = g.lse[li][q].cpu().numpy()
        assert np.allclose(lse, lse_ref, rtol=1e-5, atol=1e-5), f"q{q} L{li} lse"


def check_status(g):
    for name, st in g.status().items():
        assert st[0] == 0, (name, st)




def run_group_graph(wl):
    """A group stepped the way the bench times it: one eager step (kernel
    attributes), then one CUDA-graph replay of the step."""
    import torch
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    g = LayerGroup(wl)
    for ws in (g.ws_app, g.ws_full, g.ws_re, g.ws_attn):
        ws.zero_()
    g.fill()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        g.step(stream)
    stream.synchronize()
    g.capture(stream)
    g.replay()
    stream.synchronize()
    return g


def verify_query_at_scale(g, wl, q, cache_sample=2048, seed=7):
    """One query of a full-size group against the oracle.

    The indexer K cache is compared bit-exact on every row (the Full index
    scores all of them); the main-latent cache on `cache_sample` random rows,
    the last row and every row the attention layers read; the Full pool and
    top-k against the oracle's definitions over the whole context; each
    Reindex top-k against the oracle on the GPU's pool; each attention layer
    against the oracle on the GPU's index set."""
    r = W.request_of(wl, q)
    n = int(wl.contexts[q])
    P, K = wl.pool_blocks, wl.topk
    base = 0 if wl.shared_cache else g.row_base[r]
    assert base % 8 == 0
    rows = W.cache_rows(wl, r)
    # indexer K: every row of the query's view
    kc, ks = O.quantize_fp4(W.indexer_k_rows(wl, r, 0, n))
    gk, gs = indexer_k_planes(g, base, base + n)
    assert np.array_equal(gk, O.pack_codes(kc)), f"q{q} indexer K bytes"
    assert np.array_equal(gs, ks), f"q{q} indexer K scales"
    kdq = O.dequantize_fp4(kc, ks)
    del kc
    # indices: Full against the global definitions, Reindex on the GPU's pool
    topk_of = {}
    for li, mode in enumerate(wl.layers):
        if mode not in (W.FULL, W.REINDEX):
            topk_of[li] = topk_of[W.index_source(wl, li)]
            continue
        qc, qs = O.quantize_fp4(W.indexer_q(wl, q, li).astype(np.float64))
        qdq = O.dequantize_fp4(qc, qs)
        wv = W.indexer_w(wl, q, li).astype(np.float64)
        gt = g.topk[li][q].cpu().numpy()
        if mode == W.FULL:
            pool_o, top_o, scores, bmax = O.index_full(qdq, wv, kdq, n, P, K)
            gp = g.pools[li][q].cpu().numpy()
            check_selection(gp, pool_o, lambda b: bmax[b], kth_value(bmax, P), f"q{q} pool")
            check_selection(gt, top_o, lambda p: scores[p], kth_value(scores, K), f"q{q} L{li} top-k")
            gpu_pool = gp
        else:
            re_o, cand, sc = O.index_reindex(qdq, wv, kdq, n, gpu_pool, K)
            smap = dict(zip(cand.tolist(), sc.tolist()))
            check_selection(gt, re_o, lambda p: smap[p], kth_value(sc, K), f"q{q} L{li} reindex")
        topk_of[li] = gt
    del kdq
    # main latents: the sampled rows and every row the attention reads
    rng = np.random.default_rng(seed + q)
    used = np.concatenate([t[t >= 0] for t in topk_of.values()])
    need = np.unique(np.concatenate([rng.integers(0, n, cache_sample), used, [n - 1]])).astype(np.int64)
    lat = W.main_latent_rows(wl, r, 0, rows)[need].astype(np.float64)
    lc, ls = O.quantize_fp4(O.rope(lat, W.latent_positions(wl, r)[need]))
    del lat
    import torch
    idx = torch.as_tensor(base + need, device=g.kv_codes.device)
    assert np.array_equal(g.kv_codes[idx].cpu().numpy(), O.pack_codes(lc)), f"q{q} main latent bytes"
    assert np.array_equal(g.kv_scales[idx].cpu().numpy(), ls), f"q{q} main latent scales"
    row_of = np.full(n, -1, dtype=np.int64)
    row_of[need] = np.arange(need.size)
    for li in range(len(wl.layers)):
        t = topk_of[li]
        ids = np.where(t >= 0, row_of[np.maximum(t, 0)], -1)
        if wl.shared_window:  # only the window's rows of the shared sequence are drawn and compared
            w0 = max(0, n - wl.window)
            rows = O.append_swa_fp8(W.swa_seq_rows(wl, li, w0, n))
            assert np.array_equal(g.swa[li][w0:n].cpu().numpy(), rows), f"q{q} L{li} window bytes"
            seq = np.zeros((n, 512), dtype=np.uint8)
            seq[w0:n] = rows
            sel, win = O.attention_inputs_shared_window(ids, lc, ls, seq, n, wl.window)
        else:
            ring = O.append_swa_fp8(W.swa_ring(wl, q, li))
            assert np.array_equal(g.swa[li][q].cpu().numpy(), ring), f"q{q} L{li} window bytes"
            sel, win = O.attention_inputs(ids, lc, ls, ring, n, wl.window)
        o_ref, lse_ref = O.sparse_attention(W.attn_q(wl, q, li), sel, win)
        check_attention(bf16_to_f64(g.out[li][q]), o_ref, f"q{q} L{li} attention")
        lse = g.lse[li][q].cpu().numpy()
        assert np.allclose(lse, lse_ref, rtol=1e-5, atol=1e-5), f"q{q} L{li} lse"
