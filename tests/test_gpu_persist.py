"""FP4 global-KV persistence: save a request's main latent and indexer K,
restore them into a group whose caches were never filled, and step again.

[T1] "持久缓存为什么能降到 1/8" and [T3] 第三刀: the persistent cache is the FP4
global KV; the window KV is not persisted.  The restored group refills only
its per-layer inputs (queries, window rings, current-token latents), as a
server rebuilding the window would, and must then produce bit-identical
pools, top-K and attention outputs.
"""
import io

import numpy as np
import pytest
import torch

from csa2_sparse_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _snapshot(g):
    return {"pool": g.pool.clone(), **{f"topk{i}": t.clone() for i, t in g.topk.items()},
            **{f"out{li}": o.clone() for li, o in enumerate(g.out)},
            **{f"lse{li}": x.clone() for li, x in enumerate(g.lse)}}


@pytest.mark.parametrize("records", [True, False])
def test_restored_global_kv_gives_identical_indices_and_outputs(records):
    from csa2_sparse_attention_gb300 import abi, persist
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    layout = abi.LAYOUT_BLOCK8R if records else abi.LAYOUT_BLOCK8
    wl = W.small_variant(W.group_128k(), (9000, 20001, 4096), name="persist", layers=("F", "R", "X", "R"),
                         hot_blocks=8)
    g1 = LayerGroup(wl, ik_layout=layout)
    g1.fill()
    g1.step()
    torch.cuda.synchronize()
    ref = _snapshot(g1)
    files = []
    for r in range(wl.batch):
        f = io.BytesIO()
        size = persist.save_request(g1, r, f)
        n = wl.contexts[r]
        assert size >= n * 288 + n * 72  # main latent + indexer K, no window
        files.append(f.getvalue())

    g2 = LayerGroup(wl, ik_layout=layout)  # caches never filled
    g2.fill_layer_inputs()
    for r in range(wl.batch):
        persist.load_request(g2, r, io.BytesIO(files[r]))
    assert torch.equal(g1.kv_codes, g2.kv_codes) and torch.equal(g1.kv_scales, g2.kv_scales)
    assert torch.equal(g1.ik_codes, g2.ik_codes)
    if not records:
        assert torch.equal(g1.ik_scales, g2.ik_scales)
    g2.step()
    torch.cuda.synchronize()
    got = _snapshot(g2)
    for name, t in ref.items():
        assert torch.equal(t, got[name]), f"{name} differs after the restore"
    for name, st in g2.status().items():
        assert st[0] == 0, (name, st)

    # a damaged file, or one for another request, is refused without touching the cache
    bad = bytearray(files[0])
    bad[100] ^= 1
    before = g2.kv_codes.clone()
    with pytest.raises(ValueError, match="checksum"):
        persist.load_request(g2, 0, io.BytesIO(bytes(bad)))
    with pytest.raises(ValueError, match="rows"):
        persist.load_request(g2, 1, io.BytesIO(files[0]))
    assert torch.equal(before, g2.kv_codes)
