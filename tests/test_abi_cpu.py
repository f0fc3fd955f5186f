"""The C-ABI library loads and exports every entry point include/csa2.h
declares; host-side argument checks return before any launch (no GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def abi():
    from csa2_sparse_attention_gb300 import build
    build.build()
    from csa2_sparse_attention_gb300 import abi as A
    return A


def _declared():
    with open(os.path.join(ROOT, "include", "csa2.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(csa2_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("csa2_quantize_append", "csa2_index_full", "csa2_index_reindex", "csa2_sparse_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(abi):
    names = _declared()
    assert names
    for n in names:
        assert hasattr(abi.lib, n), n
        assert n in abi.EXPORTS, n


def test_status_strings_and_version(abi):
    assert abi.csa2_abi_version() == 1
    assert abi.csa2_status_string(0) == "ok"
    for s in range(1, 7):
        assert abi.csa2_status_string(s) != "unknown status"
    assert abi.csa2_status_string(99) == "unknown status"


def test_workspace_sizes(abi):
    A = abi
    assert A.csa2_workspace_bytes(A.OP_APPEND, 1, 0, 1, 1) == A.STATUS_BYTES
    full = A.csa2_workspace_bytes(A.OP_INDEX_FULL, 16, 131072, 2048, 512)
    # block maxima 16 x 16384 + scores 16 x 16384 positions, fp32
    assert full >= 16 * 16384 * 4 * 2
    assert A.csa2_workspace_bytes(A.OP_INDEX_FULL, 1, 100, 0, 512) == 0
    # 512 + 128 entries in splits of 128: 5 partial outputs per query
    assert A.csa2_workspace_bytes(A.OP_SPARSE_ATTN, 2, 1000, 2048, 512) >= 2 * 5 * 64 * 512 * 4
    assert A.csa2_workspace_bytes(99, 1, 1, 1, 1) == 0
    assert A.csa2_rope_table_bytes(512, 1 << 20) == (1024 + 1024) * 256 * (8 + 16)


def test_host_argument_errors_return_before_launch(abi):
    A = abi
    st = A.lib.csa2_quantize_append(None, 4, 512, A.FMT_FP4, A.LAYOUT_ROWS, None, None, 0, None, 4,
                                    None, None, None, 0, None)
    assert st == A.ERR_WORKSPACE
    fake = 1 << 20  # never dereferenced: every check below fails first
    st = A.lib.csa2_quantize_append(None, 4, 512, A.FMT_FP4, A.LAYOUT_ROWS, None, None, 0, None, 4,
                                    fake, fake, fake, 256, None)
    assert st == A.ERR_INVALID_ARG
    st = A.lib.csa2_quantize_append(fake, 4, 96, A.FMT_FP4, A.LAYOUT_ROWS, None, None, 0, None, 4,
                                    fake, fake, fake, 256, None)
    assert st == A.ERR_UNSUPPORTED
    assert A.lib.csa2_debug_wait_limit(-1) == A.ERR_INVALID_ARG  # checked before any device call
    # 576-byte records: scales live in the records (dst_scales must be NULL), dim 128 only
    st = A.lib.csa2_quantize_append(fake, 4, 128, A.FMT_FP4, A.LAYOUT_BLOCK8R, None, None, 0, None, 8,
                                    fake, fake, fake, 256, None)
    assert st == A.ERR_INVALID_ARG
    st = A.lib.csa2_quantize_append(fake, 4, 512, A.FMT_FP4, A.LAYOUT_BLOCK8R, None, None, 0, None, 8,
                                    fake, None, fake, 256, None)
    assert st == A.ERR_UNSUPPORTED
    st = A.lib.csa2_quantize_append(fake, 4, 128, A.FMT_FP4, A.LAYOUT_BLOCK8, None, None, 0, None, 8,
                                    fake, None, fake, 256, None)
    assert st == A.ERR_INVALID_ARG  # BLOCK8 needs its scale plane
    st = A.lib.csa2_index_full(fake, fake, fake, 1, fake, fake, 12, fake, fake, 100, 2048, 512,
                               fake, fake, fake, 1 << 30, None)
    assert st == A.ERR_UNSUPPORTED  # n_rows not a multiple of 8
    st = A.lib.csa2_index_full(fake, fake, fake, 1, fake, fake, 16, fake, fake, 100, 2048, 4096,
                               fake, fake, fake, 1 << 30, None)
    assert st == A.ERR_UNSUPPORTED  # topk above 2048
    st = A.lib.csa2_index_full(fake, fake, fake, 1, fake, fake, 16, fake, fake, 100, 2048, 512,
                               fake, fake, fake, 64, None)
    assert st == A.ERR_WORKSPACE
    # the bf16-query forms: the query pointer is required and 16-byte aligned
    st = A.lib.csa2_index_full_bf16(None, fake, 1, fake, fake, 16, fake, fake, 100, 2048, 512,
                                    fake, fake, fake, 1 << 30, None)
    assert st == A.ERR_INVALID_ARG
    st = A.lib.csa2_index_full_bf16(fake + 2, fake, 1, fake, fake, 16, fake, fake, 100, 2048, 512,
                                    fake, fake, fake, 1 << 30, None)
    assert st == A.ERR_INVALID_ARG
    st = A.lib.csa2_index_reindex_bf16(None, fake, 1, fake, fake, 16, fake, fake, 100, fake, 2048, 512,
                                       fake, fake, 1 << 30, None)
    assert st == A.ERR_INVALID_ARG
    st = A.lib.csa2_index_reindex_bf16(fake, fake, 1, fake, fake, 12, fake, fake, 100, fake, 2048, 512,
                                       fake, fake, 1 << 30, None)
    assert st == A.ERR_UNSUPPORTED  # n_rows not a multiple of 8
    st = A.lib.csa2_sparse_attn(fake, 1, fake, fake, 16, fake, fake, fake, 512, fake, None, 129, 0.04,
                                fake, A.OUT_F32, None, fake, 1 << 30, None)
    assert st == A.ERR_INVALID_ARG  # window above 128
    st = A.lib.csa2_sparse_attn(fake, 1, fake, fake, 16, fake, fake, fake, 512, fake, None, 128, -1.0,
                                fake, A.OUT_F32, None, fake, 1 << 30, None)
    assert st == A.ERR_INVALID_ARG
    st = A.lib.csa2_sparse_attn(fake, 1, fake, fake, 16, fake, fake, fake, 512, fake, None, 128, 0.04,
                                fake, 7, None, fake, 1 << 30, None)
    assert st == A.ERR_INVALID_ARG  # unknown output type
    with pytest.raises(A.Csa2Error):
        A.csa2_rope_table_init(10000.0, 512, 0, fake, None)


def test_empty_batches_return_ok_and_launch_nothing(abi):
    """Every call with zero rows or queries returns OK after its argument and
    workspace checks, touching no memory (the pointers are never valid) and
    launching nothing."""
    A = abi
    fake = 1 << 20
    c0 = A.csa2_launch_count()
    assert A.lib.csa2_quantize_append(fake, 0, 512, A.FMT_FP4, A.LAYOUT_ROWS, None, None, 0, None, 4,
                                      fake, fake, fake, 256, None) == A.OK
    assert A.lib.csa2_index_full(fake, fake, fake, 0, fake, fake, 16, fake, fake, 100, 2048, 512,
                                 fake, fake, fake, 1 << 30, None) == A.OK
    assert A.lib.csa2_index_reindex(fake, fake, fake, 0, fake, fake, 16, fake, fake, 100, fake, 2048, 512,
                                    fake, fake, 1 << 30, None) == A.OK
    assert A.lib.csa2_index_full_bf16(fake, fake, 0, fake, fake, 16, fake, fake, 100, 2048, 512,
                                      fake, fake, fake, 1 << 30, None) == A.OK
    assert A.lib.csa2_index_reindex_bf16(fake, fake, 0, fake, fake, 16, fake, fake, 100, fake, 2048, 512,
                                         fake, fake, 1 << 30, None) == A.OK
    assert A.lib.csa2_sparse_attn(fake, 0, fake, fake, 16, fake, fake, fake, 512, fake, None, 128, 0.04,
                                  fake, A.OUT_F32, None, fake, 1 << 30, None) == A.OK
    assert A.csa2_launch_count() == c0
