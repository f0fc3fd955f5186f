"""csa2_index_full at the size boundaries of the selection paths, with exact
ties everywhere: the indexer keys repeat 16 distinct rows, so the oracle's
scores come from a 16-entry table.

- Contexts whose block maxima do not fit one CTA's shared memory: the pool
  selection splits each query's blocks over a cluster of CTAs (16K or 32K
  keys each), and the ties run across the cluster's segments.
- 8192 / 8193 and 16,384 / 16,385 blocks: 8 or 16 keys per thread held in
  registers, or staged in shared memory.
- A context of fewer than P blocks: every block is taken, and the pool is
  padded with -1, so the top-K candidates include missing positions.

Identical key rows give bit-identical scores on the GPU (fp32) and in the
oracle (fp64), and the 16 distinct scores of every query are checked to lie
far apart relative to fp32 rounding, so the two sides rank every position the
same way and every equal score is a genuine tie.  The pool and top-K sets must
therefore be exactly equal: that pins the rule that ties go to the lower
block and the lower position."""
import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O
from tests.helpers import check_selection, kth_value, rows_to_block8, rows_to_records

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("contexts,records", [((300_000, 50_000, 262_143), False), ((1_600_000, 1_000_003), True),
                                              ((65_536, 65_537, 131_072, 131_073, 8_000), True)])
def test_pool_and_topk_at_selection_path_boundaries(contexts, records):
    """(Indexer K as BLOCK8 codes with a scale plane, or as 576-byte records.)"""
    from csa2_sparse_attention_gb300 import abi
    rng = np.random.default_rng(sum(contexts))
    n_q, P, K = len(contexts), 2048, 512
    distinct = torch.randn((16, 128), generator=torch.Generator().manual_seed(21)).to(torch.bfloat16)
    kc16, ks16 = O.quantize_fp4(distinct.float().numpy().astype(np.float64))
    k16 = O.dequantize_fp4(kc16, ks16)
    pk16 = O.pack_codes(kc16)
    rows_of = [((n + 7) // 8) * 8 for n in contexts]
    kv_start = np.concatenate([[0], np.cumsum(rows_of)[:-1]]).astype(np.int64)
    n_rows = int(sum(rows_of))
    row_id = rng.integers(0, 16, n_rows)
    if records:
        k_codes = torch.from_numpy(rows_to_records(pk16[row_id], ks16[row_id])).cuda()
        k_scales = None
    else:
        k_codes = torch.from_numpy(rows_to_block8(pk16[row_id])).cuda()
        k_scales = torch.from_numpy(np.ascontiguousarray(ks16[row_id])).cuda()
    q_real = torch.randn((n_q * 32, 128), generator=torch.Generator().manual_seed(22)).to(torch.bfloat16)
    qc, qs = O.quantize_fp4(q_real.float().numpy().astype(np.float64))
    q_codes = torch.from_numpy(rows_to_block8(O.pack_codes(qc))).cuda()
    q_scales = torch.from_numpy(np.ascontiguousarray(qs)).cuda()
    w = rng.uniform(0, 1, (n_q, 32)).astype(np.float32)
    n_vis = np.asarray(contexts, dtype=np.int32)
    max_visible = int(n_vis.max())
    ws = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_FULL, n_q, max_visible, P, K), dtype=torch.uint8,
                     device="cuda")
    pool = torch.full((n_q, P), -7, dtype=torch.int32, device="cuda")
    topk = torch.full((n_q, K), -7, dtype=torch.int32, device="cuda")
    abi.csa2_index_full(q_codes, q_scales, torch.from_numpy(w).cuda(), n_q, k_codes, k_scales, n_rows,
                        torch.from_numpy(kv_start).cuda(), torch.from_numpy(n_vis).cuda(), max_visible, P, K,
                        pool, topk, ws, ws.numel())
    torch.cuda.synchronize()
    assert abi.csa2_status_fetch(ws)[0] == 0
    qdq = O.dequantize_fp4(qc, qs).reshape(n_q, 32, 128)
    for q, n in enumerate(contexts):
        table = O.index_scores(qdq[q], w[q].astype(np.float64), k16)  # score of each distinct row
        ts = np.sort(table)
        assert ts[0] > 0 and np.min(np.diff(ts) / ts[1:]) > 1e-4, "distinct scores too close for a strict check"
        scores = table[row_id[kv_start[q]:kv_start[q] + n]]
        bmax = O.block_max(scores)
        check_selection(pool[q].cpu().numpy(), O.select_top(bmax, P), lambda b: bmax[b], kth_value(bmax, P),
                        f"q{q} pool (n={n})", strict=True)
        check_selection(topk[q].cpu().numpy(), O.select_top(scores, K), lambda p: scores[p],
                        kth_value(scores, K), f"q{q} top-k (n={n})", strict=True)
