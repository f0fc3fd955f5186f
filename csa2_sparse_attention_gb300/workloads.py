"""Seeded synthetic inputs for the CSA2 decode step.

This module only draws inputs: bf16 vectors, weights, positions and the
planted "hot" structure of the indexer keys.  It holds none of the method's
arithmetic (no quantization, RoPE, scoring, selection or attention), so the
CUDA path and the CPU oracle can both consume exactly the same bytes.

Every array is a pure function of (seed, workload index, stream kind,
request, layer, chunk): chunks are drawn from independent PCG64 streams, so
the result does not depend on how many threads generate it.  bf16 values are
returned as float32 arrays whose values are exactly representable in bf16
(rounded to nearest-even by torch's bf16 conversion).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

SEED = 20260910

# stream kinds
_K_INDEX_Q, _K_INDEX_W, _K_INDEX_K, _K_HOT, _K_LATENT, _K_SWA, _K_ATTN_Q, _K_CTX, _K_SWA_SEQ = range(9)
_CHUNK_ROWS = 8192

FULL, REINDEX, REUSE = "F", "X", "R"
GROUP_LAYOUT = (FULL, REUSE, REUSE, REUSE) + (REINDEX, REUSE, REUSE, REUSE) * 4
# [T1] §二 layout paragraph: the encoder's CSA2 layers run at m = 2 in three
# groups of one Full and five Reuse layers
ENCODER_LAYOUT = (FULL, REUSE, REUSE, REUSE, REUSE, REUSE) * 3


@dataclass(frozen=True)
class Workload:
    """One synthetic CSA2 workload.

    contexts: visible compressed entries per query (n); queries of one
    request share a cache when `shared_cache` is set (prefill-style many-query
    indexing), otherwise every query has its own cache of `capacity(q)` rows.
    """
    name: str
    index: int
    contexts: tuple
    layers: tuple
    pool_blocks: int = 2048
    topk: int = 512
    window: int = 128
    hot_blocks: int = 0            # planted hot blocks per query (0 = none)
    shared_cache: bool = False
    cache_entries: int = 0         # rows of the shared cache (shared_cache only)
    m: int = 1                     # raw tokens per compressed entry
    raw_positions: tuple = ()      # per-query raw position (shared_cache only)
    shared_window: bool = False    # window over the shared sequence (prefill) instead of a ring per query
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def batch(self):
        return len(self.contexts)

    def describe(self):
        return {"workload": self.name, "queries": self.batch,
                "context": (self.contexts[0] if len(set(self.contexts)) == 1
                            else f"ragged {min(self.contexts)}..{max(self.contexts)}"),
                "layers": "".join(self.layers), "pool_blocks": self.pool_blocks,
                "topk": self.topk, "window": self.window}


def _ragged_contexts(count=64, lo=4096, hi=1 << 20):
    rng = np.random.Generator(np.random.PCG64([SEED, 4, _K_CTX]))
    u = rng.uniform(math.log(lo), math.log(hi), size=count)
    return tuple(int(v) for v in np.floor(np.exp(u)).astype(np.int64))


def tiny():
    """Single decode step, 8192 entries, one Full + one Reindex + one Reuse
    layer, pool 256 x 8, 16 hot blocks."""
    return Workload("decode-8k-b1-FXR", 0, (8192,), (FULL, REINDEX, REUSE),
                    pool_blocks=256, hot_blocks=16)


def group_128k(batch=16):
    """20-layer decoder group at 131072 entries, batch 16, 64 hot blocks."""
    return Workload(f"decode-128k-b{batch}-group20", 1, (131072,) * batch, GROUP_LAYOUT,
                    hot_blocks=64)


def group_1m(batch=4):
    """20-layer decoder group at 1,048,576 entries, batch 4, ~1% hot blocks."""
    n = 1 << 20
    return Workload(f"decode-1m-b{batch}-group20", 2, (n,) * batch, GROUP_LAYOUT,
                    hot_blocks=round(0.01 * n / 8))


def many_query(queries=4096, entries=262144, m=2):
    """Prefill-chunk indexing: `queries` consecutive raw positions ending at
    the last raw token, against one shared cache of `entries` m=2 entries."""
    raw_end = entries * m  # exclusive
    raw = tuple(range(raw_end - queries, raw_end))
    ctx = tuple((p + 1) // m for p in raw)
    return Workload(f"manyq-{queries}x{entries}-m{m}", 3, ctx, (FULL,),
                    shared_cache=True, cache_entries=entries, m=m, raw_positions=raw)


def encoder_m2(queries=4096, entries=262144, m=2):
    """Encoder-side CSA2 over a prefill chunk: `queries` consecutive raw
    positions ending at the last raw token, one shared cache of `entries`
    m=2 entries, layers [Full + 5 Reuse] x 3; each query attends to its
    top-512 and its own causal window over the shared sequence."""
    raw_end = entries * m
    raw = tuple(range(raw_end - queries, raw_end))
    ctx = tuple((p + 1) // m for p in raw)
    return Workload(f"encoder-{queries}x{entries}-m{m}-FRRRRRx3", 5, ctx, ENCODER_LAYOUT,
                    shared_cache=True, cache_entries=entries, m=m, raw_positions=raw, shared_window=True)


def ragged(count=64):
    """64 concurrent decode requests, contexts log-uniform in [4096, 2^20],
    one Full + one Reindex layer each."""
    return Workload(f"ragged-{count}req", 4, _ragged_contexts(count), (FULL, REINDEX))


def small_variant(w: Workload, contexts, name=None, **kw):
    """Same layer layout and shapes with other context lengths (tests)."""
    from dataclasses import replace
    return replace(w, name=name or f"{w.name}-small", contexts=tuple(contexts), **kw)


# ---------------------------------------------------------------------------
def _rng(w: Workload, kind, *key):
    return np.random.Generator(np.random.PCG64([SEED, w.index, kind, *key]))


def to_bf16_exact(x):
    """Round float32 values to bf16 (nearest-even) and return them as float32."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_bits(x):
    """uint16 bit patterns of bf16-exact float32 values."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _normal_rows(w, kind, key, rows, dim, r0=0, r1=None, threads=16):
    """Rows [r0, r1) of an N(0,1) float32 [rows][dim] array drawn chunk by
    chunk (8192 rows per independent stream)."""
    r1 = rows if r1 is None else min(r1, rows)
    c_lo, c_hi = r0 // _CHUNK_ROWS, -(-r1 // _CHUNK_ROWS)
    out = np.empty((r1 - r0, dim), dtype=np.float32)

    def fill(c):
        a = c * _CHUNK_ROWS
        b = min(rows, a + _CHUNK_ROWS)
        blk = _rng(w, kind, *key, c).standard_normal((b - a, dim), dtype=np.float32)
        lo, hi = max(a, r0), min(b, r1)
        out[lo - r0:hi - r0] = blk[lo - a:hi - a]

    chunks = range(c_lo, c_hi)
    if len(chunks) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, chunks))
    else:
        for c in chunks:
            fill(c)
    return out


def cache_rows(w: Workload, q):
    """Rows of query q's cache (its own cache, or the shared one)."""
    return w.cache_entries if w.shared_cache else w.contexts[q]


def request_of(w: Workload, q):
    return 0 if w.shared_cache else q


def indexer_q(w: Workload, q, layer):
    """Indexer query of query q at layer `layer`: bf16 [32][128] N(0,1)."""
    x = _rng(w, _K_INDEX_Q, q, layer).standard_normal((32, 128), dtype=np.float32)
    return to_bf16_exact(x)


def indexer_w(w: Workload, q, layer):
    """Head weights w[32] ~ U(0,1) (fp32, used as given)."""
    return _rng(w, _K_INDEX_W, q, layer).uniform(0.0, 1.0, size=32).astype(np.float32)


def hot_blocks(w: Workload, req):
    """Distinct planted hot blocks of request `req`'s cache, ascending."""
    if w.hot_blocks <= 0:
        return np.zeros(0, dtype=np.int64)
    nb = -(-cache_rows(w, req) // 8)
    rng = _rng(w, _K_HOT, req)
    return np.sort(rng.choice(nb, size=min(w.hot_blocks, nb), replace=False)).astype(np.int64)


def indexer_k_rows(w: Workload, req, r0=0, r1=None):
    """Rows [r0, r1) of request `req`'s indexer keys: bf16 [rows][128] N(0,1);
    every position of a hot block is shifted by 0.5 * u with
    u = sum_h q[h] / sqrt(32), q the request's layer-0 indexer query."""
    rows = cache_rows(w, req)
    r1 = rows if r1 is None else min(r1, rows)
    k = _normal_rows(w, _K_INDEX_K, (req,), rows, 128, r0, r1)
    hb = hot_blocks(w, req)
    if hb.size:
        u = indexer_q(w, req, 0).sum(axis=0) / np.float32(math.sqrt(32.0))
        pos = (hb[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
        pos = pos[(pos >= r0) & (pos < r1)]
        k[pos - r0] += np.float32(0.5) * u[None, :]
    return to_bf16_exact(k)


def indexer_k(w: Workload, req):
    return indexer_k_rows(w, req)


def main_latent_rows(w: Workload, req, r0=0, r1=None):
    """Rows [r0, r1) of request `req`'s main latents (pre-RoPE): bf16
    [rows][512] N(0,1)."""
    return to_bf16_exact(_normal_rows(w, _K_LATENT, (req,), cache_rows(w, req), 512, r0, r1))


def main_latent(w: Workload, req):
    return main_latent_rows(w, req)


def latent_positions(w: Workload, req):
    """RoPE position of every cache row: the last raw token of the entry."""
    rows = cache_rows(w, req)
    return (np.arange(rows, dtype=np.int64) * w.m + (w.m - 1)).astype(np.int64)


def swa_ring(w: Workload, q, layer):
    """Sliding-window latents of query q at `layer`, by ring slot: bf16
    [window][512] N(0,1)."""
    x = _rng(w, _K_SWA, q, layer).standard_normal((w.window, 512), dtype=np.float32)
    return to_bf16_exact(x)


def swa_seq_rows(w: Workload, layer, r0=0, r1=None):
    """Rows [r0, r1) of a layer's window latents over the shared sequence
    (one per compressed position): bf16 [entries][512] N(0,1)."""
    return to_bf16_exact(_normal_rows(w, _K_SWA_SEQ, (layer,), w.cache_entries, 512, r0, r1))


def attn_q(w: Workload, q, layer):
    """Main attention query of query q at `layer`: bf16 [64][512] N(0,1)."""
    x = _rng(w, _K_ATTN_Q, q, layer).standard_normal((64, 512), dtype=np.float32)
    return to_bf16_exact(x)


def reindex_layers(w: Workload):
    return [i for i, m in enumerate(w.layers) if m == REINDEX]


def index_source(w: Workload, layer):
    """The Full/Reindex layer whose top-k a layer uses (itself for F/X)."""
    for i in range(layer, -1, -1):
        if w.layers[i] in (FULL, REINDEX):
            return i
    raise ValueError("layer group must start with a Full layer")
