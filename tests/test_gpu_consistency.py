"""Prefill-vs-decode index consistency and index-buffer ownership.

[T4] ic.work analysis of V4.1-Flash KV-cache compression, "614GB显存门槛与框架落地
的暗礁": runtimes met KV-index ownership bugs across layers and index
invalidation; [T1] §二 mode table: Full layers make the indices (and the
shared pool), Reindex layers their own top-k inside that pool, Reuse layers
only read.

1. Prefill vs decode.  A prefill chunk of Q >= 256 queries over one shared
   cache runs as the many-query contraction (query groups share K tiles);
   the same queries decoded one token at a time (each appending its own
   indexer-key row first, then indexing with a batch of one) run the decode
   scan.  The pools and top-K sets must agree (the many-query scan sums the
   heads in another order, so a member may differ only where scores tie
   within the acceptance tolerance, and nearly all queries agree bit for
   bit), Reindex on the same pool must agree exactly, and the incrementally
   appended key rows must equal the bulk-appended ones.
2. Ownership.  Stepping a layer group one layer at a time, every Full /
   Reindex layer's top-k buffer and the shared pool must keep their bytes
   (hashed) through all later layers of the group.
"""
import hashlib

import numpy as np
import pytest
import torch

from csa2_sparse_attention_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import check_selection, kth_value, records_to_rows

pytestmark = pytest.mark.gpu


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).cuda()


def test_prefill_chunk_and_token_by_token_decode_give_identical_indices():
    from csa2_sparse_attention_gb300 import abi
    rng = np.random.default_rng(2026)
    n0, nq, P, K = 8192, 288, 256, 512  # 288 queries: the many-query path (>= 256)
    n_all = n0 + nq
    n_rows = (n_all + 7) // 8 * 8
    keys = W.to_bf16_exact(rng.standard_normal((n_all, 128), dtype=np.float32))
    # a few hot blocks so the pools are not decided by noise alone
    hot = rng.choice(n_all // 8, 24, replace=False)
    keys.reshape(-1, 8, 128)[hot] += np.float32(0.75)
    keys = W.to_bf16_exact(keys)
    iq = W.to_bf16_exact(rng.standard_normal((nq * 32, 128), dtype=np.float32))
    iw = rng.uniform(0, 1, (nq, 32)).astype(np.float32)
    ws_app = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    rec = abi.LAYOUT_BLOCK8R

    def empty_keys():
        return torch.zeros(n_rows // 8 * 576, dtype=torch.uint8, device="cuda")

    # indexer queries (shared by both paths): BLOCK8 codes + scales
    q_codes = torch.zeros(nq * 32 * 64, dtype=torch.uint8, device="cuda")
    q_scales = torch.zeros((nq * 32, 8), dtype=torch.uint8, device="cuda")
    abi.csa2_quantize_append(_bf16(iq), nq * 32, 128, abi.FMT_FP4, abi.LAYOUT_BLOCK8, None, None, 0, None,
                             nq * 32, q_codes, q_scales, ws_app, ws_app.numel())
    w = torch.from_numpy(iw).cuda()

    # ---- prefill: every key appended at once, one index call over the chunk
    k_pre = empty_keys()
    abi.csa2_quantize_append(_bf16(keys), n_all, 128, abi.FMT_FP4, rec, None, None, 0, None, n_rows,
                             k_pre, None, ws_app, ws_app.numel())
    vis = np.arange(n0 + 1, n_all + 1, dtype=np.int32)  # query t sees positions [0, n0 + t]
    ws = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_FULL, nq, n_all, P, K), dtype=torch.uint8,
                     device="cuda")
    pool_pre = torch.full((nq, P), -7, dtype=torch.int32, device="cuda")
    top_pre = torch.full((nq, K), -7, dtype=torch.int32, device="cuda")
    abi.csa2_index_full(q_codes, q_scales, w, nq, k_pre, None, n_rows,
                        torch.zeros(nq, dtype=torch.int64, device="cuda"), torch.from_numpy(vis).cuda(), n_all,
                        P, K, pool_pre, top_pre, ws, ws.numel())
    re_pre = torch.full((nq, K), -7, dtype=torch.int32, device="cuda")
    ws_re = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_REINDEX, nq, n_all, P, K), dtype=torch.uint8,
                        device="cuda")
    # a Reindex layer with its own indexer queries
    q_codes_r = torch.zeros_like(q_codes)
    q_scales_r = torch.zeros_like(q_scales)
    iq_r = W.to_bf16_exact(rng.standard_normal((nq * 32, 128), dtype=np.float32))
    abi.csa2_quantize_append(_bf16(iq_r), nq * 32, 128, abi.FMT_FP4, abi.LAYOUT_BLOCK8, None, None, 0, None,
                             nq * 32, q_codes_r, q_scales_r, ws_app, ws_app.numel())
    abi.csa2_index_reindex(q_codes_r, q_scales_r, w, nq, k_pre, None, n_rows,
                           torch.zeros(nq, dtype=torch.int64, device="cuda"), torch.from_numpy(vis).cuda(), n_all,
                           pool_pre, P, K, re_pre, ws_re, ws_re.numel())
    torch.cuda.synchronize()
    assert abi.csa2_status_fetch(ws)[0] == 0 and abi.csa2_status_fetch(ws_re)[0] == 0

    # ---- decode: the prefix, then one token appended and indexed at a time
    k_dec = empty_keys()
    abi.csa2_quantize_append(_bf16(keys[:n0]), n0, 128, abi.FMT_FP4, rec, None, None, 0, None, n_rows,
                             k_dec, None, ws_app, ws_app.numel())
    ws1 = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_FULL, 1, n_all, P, K), dtype=torch.uint8,
                      device="cuda")
    ws1r = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_REINDEX, 1, n_all, P, K), dtype=torch.uint8,
                       device="cuda")
    pool_dec = torch.full((nq, P), -7, dtype=torch.int32, device="cuda")
    top_dec = torch.full((nq, K), -7, dtype=torch.int32, device="cuda")
    re_dec = torch.full((nq, K), -7, dtype=torch.int32, device="cuda")
    zero = torch.zeros(1, dtype=torch.int64, device="cuda")
    tok = _bf16(keys[n0:])
    for t in range(nq):
        row = torch.tensor([n0 + t], dtype=torch.int64, device="cuda")
        abi.csa2_quantize_append(tok[t:t + 1], 1, 128, abi.FMT_FP4, rec, None, None, 0, row, n_rows,
                                 k_dec, None, ws_app, ws_app.numel())
        nvis = torch.tensor([n0 + t + 1], dtype=torch.int32, device="cuda")
        qc = q_codes[t * 32 * 64:(t + 1) * 32 * 64]
        abi.csa2_index_full(qc, q_scales[t * 32:(t + 1) * 32], w[t:t + 1], 1, k_dec, None, n_rows, zero, nvis,
                            n_all, P, K, pool_dec[t:t + 1], top_dec[t:t + 1], ws1, ws1.numel())
        abi.csa2_index_reindex(q_codes_r[t * 32 * 64:(t + 1) * 32 * 64], q_scales_r[t * 32:(t + 1) * 32],
                               w[t:t + 1], 1, k_dec, None, n_rows, zero, nvis, n_all, pool_dec[t:t + 1], P, K,
                               re_dec[t:t + 1], ws1r, ws1r.numel())
    torch.cuda.synchronize()
    assert abi.csa2_status_fetch(ws1)[0] == 0 and abi.csa2_status_fetch(ws1r)[0] == 0
    assert abi.csa2_status_fetch(ws_app)[0] == 0

    # the same key bytes, appended at once or one token at a time
    assert torch.equal(k_pre, k_dec)
    # the same indices, query by query.  The many-query scan sums the heads
    # in another order than the decode scan, so a member may differ only
    # where the scores tie within the acceptance tolerance at the K-th
    # (P-th block) score; the Reindex scorer is the same kernel on both
    # sides, so where the pools agree its top-k must agree exactly.
    kc, ks = records_to_rows(k_pre.cpu().numpy(), n_rows)
    kdq = O.dequantize_fp4(O.unpack_codes(kc), ks)
    qdq = O.dequantize_fp4(*O.quantize_fp4(iq.astype(np.float64))).reshape(nq, 32, 128)
    qdq_r = O.dequantize_fp4(*O.quantize_fp4(iq_r.astype(np.float64))).reshape(nq, 32, 128)
    pp, tp, rp = pool_pre.cpu().numpy(), top_pre.cpu().numpy(), re_pre.cpu().numpy()
    pd, td, rd = pool_dec.cpu().numpy(), top_dec.cpu().numpy(), re_dec.cpu().numpy()
    exact = 0
    for t in range(nq):
        n = n0 + t + 1
        pool_o, top_o, scores, bmax = O.index_full(qdq[t], iw[t].astype(np.float64), kdq, n, P, K)
        for name, a_, b_ in (("prefill", pp[t], tp[t]), ("decode", pd[t], td[t])):
            check_selection(a_, pool_o, lambda x: bmax[x], kth_value(bmax, P), f"t{t} {name} pool")
            check_selection(b_, top_o, lambda x: scores[x], kth_value(scores, K), f"t{t} {name} top-k")
        check_selection(pd[t], pp[t], lambda x: bmax[x], kth_value(bmax, P), f"t{t} pool prefill/decode")
        check_selection(td[t], tp[t], lambda x: scores[x], kth_value(scores, K), f"t{t} top-k prefill/decode")
        if np.array_equal(pp[t], pd[t]):
            exact += np.array_equal(tp[t], td[t])
            assert np.array_equal(rp[t], rd[t]), f"t{t}: Reindex top-k differs on the same pool"
        else:
            for name, pool_g, re_g in (("prefill", pp[t], rp[t]), ("decode", pd[t], rd[t])):
                re_o, cand, sc = O.index_reindex(qdq_r[t], iw[t].astype(np.float64), kdq, n, pool_g, K)
                smap = dict(zip(cand.tolist(), sc.tolist()))
                check_selection(re_g, re_o, lambda x: smap[x], kth_value(sc, K), f"t{t} {name} reindex")
    assert exact >= nq * 0.9, f"only {exact} of {nq} queries give bit-identical indices"


def _digest(t):
    return hashlib.sha256(t.contiguous().cpu().numpy().tobytes()).hexdigest()


@pytest.mark.parametrize("encoder", [False, True])
def test_index_buffers_keep_their_bytes_through_later_layers(encoder):
    """A 20-layer decoder group ([Full + 3 Reuse] + 4 x [Reindex + 3 Reuse])
    or an 18-layer encoder group ([Full + 5 Reuse] x 3, m = 2, prefill
    attention) stepped one layer at a time: each Full layer's pool is written
    only by that layer, each Full / Reindex top-k buffer only by its own
    layer, and none of them changes while the later layers (their Reuse
    layers' attention, the other Full and Reindex layers) run."""
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    if encoder:
        wl = W.encoder_m2(queries=64, entries=40000)
    else:
        wl = W.small_variant(W.group_128k(), (12000, 9000, 16384, 20000), name="ownership", hot_blocks=8)
    g = LayerGroup(wl)
    g.fill()
    for ws in (g.ws_app, g.ws_full, g.ws_re, g.ws_attn):
        ws.zero_()
    s = torch.cuda.current_stream()
    if not wl.shared_cache:
        g.append_token(s)
    buffers = [(f"topk{i}", g.topk[i]) for i in g.index_layers] + [(f"pool{i}", t) for i, t in g.pools.items()]
    owned = {}  # buffer name -> digest when its owning layer finished
    for li, mode in enumerate(wl.layers):
        before = {name: _digest(t) for name, t in buffers}
        g.layer(li, s, swa_append=not wl.shared_cache)
        torch.cuda.synchronize()
        after = {name: _digest(t) for name, t in buffers}
        changed = {name for name in after if after[name] != before[name]}
        # only the layer's own buffers may change
        allowed = set()
        if mode == W.FULL:
            allowed = {f"topk{li}", f"pool{li}"}
        elif mode == W.REINDEX:
            allowed = {f"topk{li}"}
        assert changed <= allowed, f"layer {li} ({mode}) wrote {sorted(changed - allowed)}"
        for name in allowed:
            assert name in changed, f"layer {li} left {name} unwritten"
            owned[name] = after[name]
        # every buffer owned by an earlier layer still has its bytes
        for name, d in owned.items():
            assert after[name] == d, f"{name} changed during layer {li}"
        # the attention of this layer read its index source's buffer
        assert g.attn_index[li] is g.topk[W.index_source(wl, li)]
    for name, st in g.status().items():
        assert st[0] == 0, (name, st)
