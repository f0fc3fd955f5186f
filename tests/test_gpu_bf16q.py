"""The bf16-query index calls (csa2_index_full_bf16, csa2_index_reindex_bf16).

They quantize the indexer query to FP4 inside the call (in the scorers'
prologue for decode batches and Reindex layers, into the workspace for a
many-query Full layer), exactly as csa2_quantize_append with CSA2_FMT_FP4
does, so a layer group stepped with them must give the same bytes as one
that quantizes each query with its own append launch first: pools, top-k,
attention outputs and log-sum-exps, bit for bit.
"""
from dataclasses import replace

import pytest
import torch

from csa2_sparse_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(g):
    return {"pool": g.pool, **{f"pool{i}": p for i, p in g.pools.items()},
            **{f"topk{i}": t for i, t in g.topk.items()},
            **{f"out{i}": o for i, o in enumerate(g.out)}, **{f"lse{i}": x for i, x in enumerate(g.lse)}}


def _cases():
    return [
        ("tiny-K-above-P", W.tiny(), None),  # the Full layer re-scores its top-512 blocks (pool scorer)
        ("decode-records", W.small_variant(W.group_128k(), (40000, 9001, 20000), name="q16", layers=("F", "X", "R", "X"),
                                           hot_blocks=8), "rec"),
        ("decode-split", W.small_variant(W.group_128k(), (40000, 9001, 20000), name="q16s", layers=("F", "X", "R", "X"),
                                         hot_blocks=8), "split"),
        ("many-query", W.many_query(queries=288, entries=20000, m=1), None),  # >= 256 queries: quantized into ws
        # a Reindex layer over many queries quantizes in the pool scorer's prologue
        ("many-query-FXR", replace(W.many_query(queries=288, entries=20000, m=1), name="q16mq", layers=("F", "X", "R")),
         None),
    ]


@pytest.mark.parametrize("name,wl,layout", _cases(), ids=[c[0] for c in _cases()])
def test_bf16_query_calls_match_quantize_then_index(name, wl, layout):
    from csa2_sparse_attention_gb300 import abi
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    kw = {}
    if layout is not None:
        kw["ik_layout"] = abi.LAYOUT_BLOCK8R if layout == "rec" else abi.LAYOUT_BLOCK8
    groups = []
    for fused in (False, True):
        g = LayerGroup(wl, fused_q=fused, **kw)
        g.fill()
        g.step()
        torch.cuda.synchronize()
        for k, st in g.status().items():
            assert st[0] == 0, (fused, k, st)
        groups.append(g)
    a, b = (_outputs(g) for g in groups)
    assert a.keys() == b.keys()
    for k in a:
        assert torch.equal(a[k], b[k]), f"{name}: {k} differs between the bf16-query and FP4-query calls"
