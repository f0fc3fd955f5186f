"""KV append on the GPU (csa2_quantize_append) against the oracle, bit-exact."""
import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O
from tests.helpers import block8_to_rows, records_to_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from csa2_sparse_attention_gb300 import abi
    return abi


def _all_bf16_positive_finite():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32) << 16
    return bits.view(np.float32)


def run_fp4(A, x, dim=128, layout=0, pos=None, dst=None, n_rows=None, table_pos=None):
    n = x.shape[0]
    n_rows = n if n_rows is None else n_rows
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).cuda()
    rec = layout == A.LAYOUT_BLOCK8R
    codes = torch.zeros(n_rows // 8 * 576 if rec else n_rows * dim // 2, dtype=torch.uint8, device="cuda")
    scales = None if rec else torch.zeros((n_rows, dim // 16), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    table, max_pos, pos_t = None, 0, None
    if pos is not None:
        max_pos = int(table_pos or (int(np.max(pos)) + 1))
        table = torch.zeros(A.csa2_rope_table_bytes(dim, max_pos), dtype=torch.uint8, device="cuda")
        A.csa2_rope_table_init(10000.0, dim, max_pos, table)
        pos_t = torch.from_numpy(np.asarray(pos, dtype=np.int64)).cuda()
    dst_t = None if dst is None else torch.from_numpy(np.asarray(dst, dtype=np.int64)).cuda()
    A.csa2_quantize_append(xt, n, dim, A.FMT_FP4, layout, pos_t, table, max_pos, dst_t, n_rows,
                           codes, scales, ws, ws.numel())
    torch.cuda.synchronize()
    st = A.csa2_status_fetch(ws)
    c = codes.cpu().numpy()
    if rec:
        c, sc = records_to_rows(c, n_rows)
        return c, sc, st
    c = block8_to_rows(c, n_rows) if layout == A.LAYOUT_BLOCK8 else c.reshape(n_rows, dim // 2)
    return c, scales.cpu().numpy(), st


def test_fp4_scale_of_every_bf16_amax(A):
    a = _all_bf16_positive_finite()
    a = np.concatenate([a, -a])
    n_groups = a.size
    pad = (-n_groups) % 8
    g = np.zeros((n_groups + pad, 16), dtype=np.float32)
    g[:n_groups, 0] = a
    g[:n_groups, 7] = a / 3  # a second element with its own rounding
    x = torch.from_numpy(g.reshape(-1, 128)).to(torch.bfloat16).to(torch.float32).numpy()
    codes, scales, st = run_fp4(A, x)
    assert st[0] == 0
    ref_codes, ref_scales = O.quantize_fp4(x.astype(np.float64))
    assert np.array_equal(scales, ref_scales)
    assert np.array_equal(codes, O.pack_codes(ref_codes))


def test_fp4_codes_for_every_scale_and_every_bf16_below_amax(A):
    """For every finite positive E4M3 scale s, every bf16 |x| <= 6s (both
    signs) is coded in groups whose amax is exactly 6s."""
    allx = _all_bf16_positive_finite()
    rows = []
    for sb in range(0x01, 0x7F):
        s = float(O.e4m3_decode(sb))
        a = np.float32(6.0 * s)
        xs = allx[allx <= a]
        xs = np.concatenate([xs, -xs, [0.0, -0.0]]).astype(np.float32)
        m = (-xs.size) % 15
        xs = np.concatenate([xs, np.zeros(m, dtype=np.float32)]).reshape(-1, 15)
        grp = np.concatenate([np.full((xs.shape[0], 1), a, dtype=np.float32), xs], axis=1)
        rows.append(grp)
    g = np.concatenate(rows)
    pad = (-g.shape[0]) % 8
    g = np.concatenate([g, np.zeros((pad, 16), dtype=np.float32)])
    x = g.reshape(-1, 128)
    codes, scales, st = run_fp4(A, x)
    assert st[0] == 0
    ref_codes, ref_scales = O.quantize_fp4(x.astype(np.float64))
    assert np.array_equal(scales, ref_scales)
    bad = np.nonzero(codes != O.pack_codes(ref_codes))
    assert bad[0].size == 0, (x.reshape(-1)[bad[0][:3] * 2], codes[bad][:3])


def test_fp8_every_bf16(A):
    bits = np.concatenate([np.arange(0x0000, 0x7F80), np.arange(0x8000, 0xFF80)]).astype(np.uint32) << 16
    x = bits.view(np.float32)
    pad = (-x.size) % 512
    x = np.concatenate([x, np.zeros(pad, dtype=np.float32)]).reshape(-1, 512)
    n = x.shape[0]
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    out = torch.zeros((n, 512), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    A.csa2_quantize_append(xt, n, 512, A.FMT_FP8, A.LAYOUT_ROWS, None, None, 0, None, n, out, None, ws, 256)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), O.e4m3_encode(x.astype(np.float64)))


@pytest.mark.parametrize("records", [False, True])
def test_block8_layout_with_destination_rows(A, records):
    """BLOCK8 codes with a scale plane, and BLOCK8R 576-byte records."""
    rng = np.random.default_rng(5)
    n_rows = 1000
    x = rng.normal(size=(600, 128)).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    dst = rng.permutation(n_rows)[:600]
    codes, scales, st = run_fp4(A, x, layout=A.LAYOUT_BLOCK8R if records else A.LAYOUT_BLOCK8, dst=dst,
                                n_rows=n_rows)
    assert st[0] == 0
    rc, rs = O.quantize_fp4(x.astype(np.float64))
    assert np.array_equal(codes[dst], O.pack_codes(rc))
    assert np.array_equal(scales[dst], rs)
    untouched = np.setdiff1d(np.arange(n_rows), dst)
    assert np.all(codes[untouched] == 0) and np.all(scales[untouched] == 0)


def _near_threshold(y, rel=2.0 ** -20):
    """Groups of real rows y[..., 16] whose amax/6 is near an E4M3 tie or
    whose elements are near an E2M1 tie of the oracle's scale."""
    g = y.reshape(-1, 16)
    amax = np.abs(g).max(axis=1)
    vals = O.e4m3_decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2
    q = amax / 6
    near_s = np.min(np.abs(q[:, None] - mids[None, :]), axis=1) <= rel * np.maximum(q, 1e-30)
    _, sb = O.quantize_fp4(g)
    s = O.e4m3_decode(sb[:, 0])[:, None]
    t = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    r = np.abs(g) / np.where(s > 0, s, 1)
    near_c = np.any(np.min(np.abs(r[..., None] - t), axis=-1) <= rel * 6, axis=1)
    return near_s | near_c


def test_rope_append_matches_oracle(A):
    rng = np.random.default_rng(6)
    n = 4096
    x = rng.normal(size=(n, 512)).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    pos = np.concatenate([np.arange(2048), rng.integers(0, 1 << 20, 2048)]).astype(np.int64)
    codes, scales, st = run_fp4(A, x, dim=512, pos=pos, table_pos=1 << 20)
    assert st[0] == 0
    y = O.rope(x.astype(np.float64), pos)
    rc, rs = O.quantize_fp4(y)
    rp = O.pack_codes(rc)
    bad_groups = (np.any(codes.reshape(n, 32, 8) != rp.reshape(n, 32, 8), axis=2) | (scales != rs)).reshape(-1)
    # the device resolves groups near a rounding tie in fp64, so only ties
    # within fp64 rounding of the angle (~1e-10 relative) could differ
    ok = _near_threshold(y, rel=2.0 ** -30)
    assert np.all(ok[bad_groups]), f"{bad_groups.sum()} groups differ, {np.sum(bad_groups & ~ok)} not near a tie"
    # position 0 rotates nothing: the bytes equal the plain quantizer's
    pc, ps = O.quantize_fp4(x[:1].astype(np.float64))
    assert np.array_equal(codes[0], O.pack_codes(pc)[0]) and np.array_equal(scales[0], ps[0])


def test_append_out_of_range_row_is_skipped_and_recorded(A):
    x = np.ones((16, 128), dtype=np.float32)
    dst = np.arange(16)
    dst[5] = 40  # plane has 16 rows
    codes, scales, st = run_fp4(A, x, dst=dst, n_rows=16)
    assert st[0] == A.ERR_DEVICE_BOUNDS and st[1] == 1 and st[2] == 5 and st[3] == 40
    rc, rs = O.quantize_fp4(np.ones((1, 128)))
    assert np.all(scales[dst[dst < 16]] == rs[0])
    assert np.all(scales[5] == 0)
