"""The allocation-free Reindex entry point (csa2_index_reindex_noalloc).

Callers without a device allocator cannot provide a workspace, so this
variant keeps its score scratch in a fixed library-owned device array.  It
must select exactly what csa2_index_reindex selects, call after call, and
must refuse problems larger than its array before launching anything.
"""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_noalloc_reindex_matches_reindex_on_two_calls():
    from csa2_sparse_attention_gb300 import abi
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    wl = W.small_variant(W.group_128k(), [20000, 8191, 1000, 333, 17, 5], name="noalloc",
                         layers=("F", "X"), pool_blocks=256, topk=512, hot_blocks=4)
    g = LayerGroup(wl, fused_q=False)  # the step quantizes the indexer queries into iq_codes / iq_scales
    g.fill()
    g.step()
    torch.cuda.synchronize()
    li = 1
    args = (g.iq_codes[li], g.iq_scales[li], g.iw[li], g.B, g.ik_codes, g.ik_scales, g.n_rows,
            g.kv_start, g.n_visible, g.max_visible, g.pool, g.P, g.K)
    ref = torch.full((g.B, g.K), -3, dtype=torch.int32, device="cuda")
    ws = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_REINDEX, g.B, g.max_visible, g.P, g.K),
                     dtype=torch.uint8, device="cuda")
    abi.csa2_index_reindex(*args, ref, ws, ws.numel())
    torch.cuda.synchronize()
    assert torch.equal(ref, g.topk[li])
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full((g.B, g.K), -7, dtype=torch.int32, device="cuda")
        abi.csa2_index_reindex_noalloc(*args, out, status)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert torch.count_nonzero(status).item() == 0
    assert abi.csa2_status_fetch(ws)[0] == 0


def test_noalloc_reindex_rejects_problems_beyond_its_array():
    from csa2_sparse_attention_gb300 import abi
    fake = 1 << 20  # never dereferenced: the size check comes before any launch
    st = abi.lib.csa2_index_reindex_noalloc(fake, fake, fake, 33, fake, fake, 64, fake, fake, 8, fake,
                                            2048, 512, fake, None, None)
    assert st == abi.ERR_UNSUPPORTED
    assert np.int64(33) * 8 * 2048 > 512 * 1024
