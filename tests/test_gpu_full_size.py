"""Parity at the bench's full sizes, in the launch configuration the bench
times (one CUDA-graph replay of the whole step), on sampled queries.

For each sampled query the oracle recomputes the Full index over the whole
context, every Reindex layer on the GPU's pool and every attention layer on
the GPU's index set; the caches are compared bit-exact (every indexer K row,
a sample of the main-latent rows plus every row the attention reads)."""
import numpy as np
import pytest

from csa2_sparse_attention_gb300 import workloads as W
from tests.helpers import check_status, run_group_graph, verify_query_at_scale

pytestmark = pytest.mark.gpu


def test_group_128k_batch16_sampled():
    wl = W.group_128k()
    g = run_group_graph(wl)
    check_status(g)
    for q in (0, 15):
        verify_query_at_scale(g, wl, q)


def test_group_1m_batch4_sampled():
    wl = W.group_1m()
    g = run_group_graph(wl)
    check_status(g)
    verify_query_at_scale(g, wl, 3)


def test_many_query_4096x262144_sampled():
    wl = W.many_query()
    g = run_group_graph(wl)
    check_status(g)
    for q in (0, 2047, 4095):
        verify_query_at_scale(g, wl, q, cache_sample=512)


def test_ragged_64_requests_sampled():
    wl = W.ragged()
    g = run_group_graph(wl)
    check_status(g)
    ctx = np.asarray(wl.contexts)
    for q in (int(np.argmin(ctx)), int(np.argmax(ctx))):
        verify_query_at_scale(g, wl, q)
