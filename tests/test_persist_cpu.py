"""The global-KV file format on the host: round trip, damage, mismatch.
(Host tensors stand in for a layer group's device planes.)"""
import io
from types import SimpleNamespace

import pytest
import torch


def _group(contexts, layout, seed):
    from csa2_sparse_attention_gb300 import abi
    g = torch.Generator().manual_seed(seed)
    caps = [(n + 7) // 8 * 8 for n in contexts]
    rows = sum(caps)
    base = [sum(caps[:i]) for i in range(len(caps))]
    rnd = lambda *shape: torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    ik = rnd(rows // 8 * 576) if layout == abi.LAYOUT_BLOCK8R else rnd(rows * 64)
    return SimpleNamespace(wl=SimpleNamespace(shared_cache=False), row_base=base, contexts=list(contexts),
                           kv_codes=rnd(rows, 256), kv_scales=rnd(rows, 32), ik_layout=layout, ik_codes=ik,
                           ik_scales=None if layout == abi.LAYOUT_BLOCK8R else rnd(rows, 8), dev="cpu")


@pytest.mark.parametrize("records", [True, False])
def test_round_trip_damage_and_mismatch(records):
    from csa2_sparse_attention_gb300 import abi, persist
    layout = abi.LAYOUT_BLOCK8R if records else abi.LAYOUT_BLOCK8
    src = _group((100, 37, 64), layout, 1)
    dst = _group((100, 37, 64), layout, 2)
    f = io.BytesIO()
    persist.save_request(src, 1, f)
    blob = f.getvalue()
    persist.load_request(dst, 1, io.BytesIO(blob))
    ks, n = src.row_base[1], src.contexts[1]
    assert torch.equal(dst.kv_codes[ks:ks + n], src.kv_codes[ks:ks + n])
    assert torch.equal(dst.kv_scales[ks:ks + n], src.kv_scales[ks:ks + n])
    b0, b1 = ks // 8, (ks + n + 7) // 8
    if records:
        assert torch.equal(dst.ik_codes[b0 * 576:b1 * 576], src.ik_codes[b0 * 576:b1 * 576])
    else:
        assert torch.equal(dst.ik_codes[b0 * 512:b1 * 512], src.ik_codes[b0 * 512:b1 * 512])
        assert torch.equal(dst.ik_scales[b0 * 8:b1 * 8], src.ik_scales[b0 * 8:b1 * 8])
    # the other requests' rows are untouched
    other = _group((100, 37, 64), layout, 2)
    assert torch.equal(dst.kv_codes[:ks], other.kv_codes[:ks])
    assert torch.equal(dst.kv_codes[ks + n:], other.kv_codes[ks + n:])
    # damage anywhere is caught by the checksum; wrong request / layout by the header
    for pos in (9, len(blob) // 2, len(blob) - 1):
        bad = bytearray(blob)
        bad[pos] ^= 0x10
        with pytest.raises(ValueError):
            persist.load_request(dst, 1, io.BytesIO(bytes(bad)))
    with pytest.raises(ValueError, match="rows"):
        persist.load_request(dst, 0, io.BytesIO(blob))
    with pytest.raises(ValueError):
        persist.load_request(_group((100, 37, 64), abi.LAYOUT_BLOCK8 if records else abi.LAYOUT_BLOCK8R, 3), 1,
                             io.BytesIO(blob))
    with pytest.raises(ValueError, match="not a CSA2"):
        persist.load_request(dst, 1, io.BytesIO(b"XXXXXXXX" + blob[8:]))
