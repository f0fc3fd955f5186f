"""Encoder-side CSA2 at m = 2: [Full + 5 Reuse] x 3 over a prefill chunk.

[T1] §二 layout paragraph: the encoder's CSA2 layers run at m = 2 in three
groups of one Full and five Reuse layers.  Every query of the chunk sees the
entries its raw position has completed (n = floor((p + 1) / 2)), takes its
Full layer's pool and top-512, and attends to them plus its own causal
window of 128 entries over the shared sequence (csa2_sparse_attn_prefill).
Checked against the oracle: the Full index over the whole visible context,
and every one of the 18 attention layers on the GPU's index set.
"""
import pytest

from csa2_sparse_attention_gb300 import workloads as W
from tests.helpers import check_status, run_group, run_group_graph, verify_query, verify_query_at_scale

pytestmark = pytest.mark.gpu


def test_encoder_group_small():
    wl = W.encoder_m2(queries=300, entries=6000)
    assert wl.layers == W.ENCODER_LAYOUT and len(wl.layers) == 18
    g = run_group(wl)
    check_status(g)
    for q in (0, 150, 299):
        verify_query(g, wl, q, check_cache=(q == 0))
    # a query's window is the last 128 entries before it: queries at the
    # chunk's start and end see different windows over the same rows
    assert wl.contexts[0] < wl.contexts[-1]


def test_encoder_group_full_size_sampled():
    """4096 queries over 262,144 m=2 entries (the many-query index size),
    one eager step then one CUDA-graph replay; sampled queries."""
    wl = W.encoder_m2()
    g = run_group_graph(wl)
    check_status(g)
    for q in (0, 2047, 4095):
        verify_query_at_scale(g, wl, q)
