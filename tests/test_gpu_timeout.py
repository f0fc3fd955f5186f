"""The device give-up paths: a bounded wait that runs out records
CSA2_ERR_TIMEOUT, the kernel waits for the copies and MMAs it already
started, and the next normal call is correct.

The test sets the library's wait limit to 1 ns (csa2_debug_wait_limit; any
limit under 1 ms makes every bounded wait give up at once), so the waits on
copies and MMAs in flight give up in the decode scan, the pool scoring, the
many-query scan and the attention kernel; nothing is left waiting on a flag
that no one sets, and no device fault is involved.  With the limit restored,
the same step gives the same bytes as before.
"""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(g):
    return [t.clone() for t in [g.pool, *g.topk.values(), *g.out, *g.lse]]


def _reset_status(g):
    from csa2_sparse_attention_gb300 import abi
    for ws in (g.ws_app, g.ws_full, g.ws_re, g.ws_attn):
        abi.csa2_status_reset(ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("batch", [3, 288])  # decode scan, and the many-query scan (>= 256 queries)
def test_short_wait_limit_times_out_then_next_call_is_correct(batch):
    from csa2_sparse_attention_gb300 import abi
    from csa2_sparse_attention_gb300.layer_group import LayerGroup
    if batch == 3:
        wl = W.small_variant(W.group_128k(), (40000, 20000, 33333), name="timeout", layers=("F", "X", "R"),
                             hot_blocks=8)
    else:
        wl = W.many_query(queries=batch, entries=20000, m=1)
    g = LayerGroup(wl)
    g.fill()
    _reset_status(g)
    g.step()
    torch.cuda.synchronize()
    for name, st in g.status().items():
        assert st[0] == 0, (name, st)
    ref = _outputs(g)

    abi.csa2_debug_wait_limit(1)
    try:
        _reset_status(g)
        g.step()
        torch.cuda.synchronize()
        st = g.status()
    finally:
        abi.csa2_debug_wait_limit(0)
    assert st["full"][0] == abi.ERR_TIMEOUT, st
    assert st["attn"][0] == abi.ERR_TIMEOUT, st

    # the context is intact and the next normal step reproduces the outputs
    _reset_status(g)
    g.step()
    torch.cuda.synchronize()
    for name, s in g.status().items():
        assert s[0] == 0, (name, s)
    for a, b in zip(ref, _outputs(g)):
        assert torch.equal(a, b)
