"""ctypes binding of the CSA2 C ABI (include/csa2.h): same names, argument
marshalling only.  Every computation runs in the CUDA library.

Pointer arguments accept an int (a device or host address), None (NULL) or
any object with ``data_ptr()`` (a torch tensor); stream arguments accept an
int, None or a torch stream.  A non-zero status raises Csa2Error.  Importing
this module loads libcsa2.so and raises ImportError if it has not been built
(run ``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa2.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"CSA2 CUDA library not built: {_LIB_PATH} is missing")
lib = ctypes.CDLL(_LIB_PATH)
LIB_PATH = _LIB_PATH

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_BOUNDS, ERR_WORKSPACE = range(7)
FMT_FP4, FMT_FP8 = 0, 1
LAYOUT_ROWS, LAYOUT_BLOCK8, LAYOUT_BLOCK8R = 0, 1, 2
OP_APPEND, OP_INDEX_FULL, OP_INDEX_REINDEX, OP_SPARSE_ATTN = range(4)
OUT_BF16, OUT_F32 = 0, 1
INDEX_HEADS, INDEX_DIM, ATTN_HEADS, LATENT_DIM, BLOCK, STATUS_BYTES = 32, 128, 64, 512, 8, 256

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_int = ctypes.c_int
_sz = ctypes.c_size_t

EXPORTS = {
    "csa2_abi_version": (_int, []),
    "csa2_status_string": (ctypes.c_char_p, [_int]),
    "csa2_workspace_bytes": (_sz, [_int, _i64, _i32, _int, _int]),
    "csa2_status_reset": (_int, [_p, _p]),
    "csa2_status_fetch": (_int, [_p, ctypes.POINTER(_i32), _p]),
    "csa2_rope_table_bytes": (_sz, [_int, _i64]),
    "csa2_rope_table_init": (_int, [ctypes.c_float, _int, _i64, _p, _p]),
    "csa2_quantize_append": (_int, [_p, _i64, _int, _int, _int, _p, _p, _i64, _p, _i64, _p, _p, _p, _sz, _p]),
    "csa2_index_full": (_int, [_p, _p, _p, _i64, _p, _p, _i64, _p, _p, _i32, _int, _int, _p, _p, _p, _sz, _p]),
    "csa2_index_reindex": (_int, [_p, _p, _p, _i64, _p, _p, _i64, _p, _p, _i32, _p, _int, _int, _p, _p, _sz, _p]),
    "csa2_index_full_bf16": (_int, [_p, _p, _i64, _p, _p, _i64, _p, _p, _i32, _int, _int, _p, _p, _p, _sz, _p]),
    "csa2_index_reindex_bf16": (_int, [_p, _p, _i64, _p, _p, _i64, _p, _p, _i32, _p, _int, _int, _p, _p, _sz, _p]),
    "csa2_sparse_attn": (_int, [_p, _i64, _p, _p, _i64, _p, _p, _p, _int, _p, _p, _int, ctypes.c_float,
                                _p, _int, _p, _p, _sz, _p]),
    "csa2_sparse_attn_prefill": (_int, [_p, _i64, _p, _p, _i64, _p, _p, _p, _int, _p, _int, ctypes.c_float,
                                        _p, _int, _p, _p, _sz, _p]),
    "csa2_index_reindex_noalloc": (_int, [_p, _p, _p, _i64, _p, _p, _i64, _p, _p, _i32, _p, _int, _int, _p,
                                          _p, _p]),
    "csa2_launch_count": (_i64, []),
    "csa2_debug_wait_limit": (_int, [_i64]),
    "csa2_kernel_name": (ctypes.c_char_p, [_int]),
    "csa2_timer_enable": (_int, [_int, _int]),
    "csa2_timer_read": (_int, [_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i32)]),
}
for _name, (_res, _args) in EXPORTS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class Csa2Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {csa2_status_string(status)} (status {status})")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, status):
    if status != OK:
        raise Csa2Error(fn, status)
    return status


def csa2_abi_version():
    return lib.csa2_abi_version()


def csa2_status_string(status):
    return lib.csa2_status_string(status).decode()


def csa2_workspace_bytes(op, n_q, max_visible, pool_blocks, topk):
    return lib.csa2_workspace_bytes(op, n_q, max_visible, pool_blocks, topk)


def csa2_status_reset(ws, stream=None):
    return _check("csa2_status_reset", lib.csa2_status_reset(_ptr(ws), _stream(stream)))


def csa2_status_fetch(ws, stream=None):
    out = (_i32 * 4)()
    _check("csa2_status_fetch", lib.csa2_status_fetch(_ptr(ws), out, _stream(stream)))
    return list(out)


def csa2_rope_table_bytes(dim, max_pos):
    return lib.csa2_rope_table_bytes(dim, max_pos)


def csa2_rope_table_init(theta, dim, max_pos, table, stream=None):
    return _check("csa2_rope_table_init",
                  lib.csa2_rope_table_init(theta, dim, max_pos, _ptr(table), _stream(stream)))


def csa2_quantize_append(x_bf16, n, dim, fmt, layout, pos, rope_table, rope_max_pos, dst_row, n_rows,
                         dst_codes, dst_scales, ws, ws_bytes, stream=None):
    return _check("csa2_quantize_append", lib.csa2_quantize_append(
        _ptr(x_bf16), n, dim, fmt, layout, _ptr(pos), _ptr(rope_table), rope_max_pos, _ptr(dst_row),
        n_rows, _ptr(dst_codes), _ptr(dst_scales), _ptr(ws), ws_bytes, _stream(stream)))


def csa2_index_full(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible,
                    max_visible, pool_blocks, topk, out_pool, out_topk, ws, ws_bytes, stream=None):
    return _check("csa2_index_full", lib.csa2_index_full(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), n_q, _ptr(k_codes), _ptr(k_scales), n_rows,
        _ptr(kv_start), _ptr(n_visible), max_visible, pool_blocks, topk, _ptr(out_pool),
        _ptr(out_topk), _ptr(ws), ws_bytes, _stream(stream)))


def csa2_index_reindex(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible,
                       max_visible, pool, pool_blocks, topk, out_topk, ws, ws_bytes, stream=None):
    return _check("csa2_index_reindex", lib.csa2_index_reindex(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), n_q, _ptr(k_codes), _ptr(k_scales), n_rows,
        _ptr(kv_start), _ptr(n_visible), max_visible, _ptr(pool), pool_blocks, topk, _ptr(out_topk),
        _ptr(ws), ws_bytes, _stream(stream)))


def csa2_index_full_bf16(q_bf16, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible,
                         pool_blocks, topk, out_pool, out_topk, ws, ws_bytes, stream=None):
    """csa2_index_full with the indexer query as bf16 rows [n_q * 32][128]."""
    return _check("csa2_index_full_bf16", lib.csa2_index_full_bf16(
        _ptr(q_bf16), _ptr(w), n_q, _ptr(k_codes), _ptr(k_scales), n_rows, _ptr(kv_start), _ptr(n_visible),
        max_visible, pool_blocks, topk, _ptr(out_pool), _ptr(out_topk), _ptr(ws), ws_bytes, _stream(stream)))


def csa2_index_reindex_bf16(q_bf16, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible,
                            pool, pool_blocks, topk, out_topk, ws, ws_bytes, stream=None):
    """csa2_index_reindex with the indexer query as bf16 rows [n_q * 32][128]."""
    return _check("csa2_index_reindex_bf16", lib.csa2_index_reindex_bf16(
        _ptr(q_bf16), _ptr(w), n_q, _ptr(k_codes), _ptr(k_scales), n_rows, _ptr(kv_start), _ptr(n_visible),
        max_visible, _ptr(pool), pool_blocks, topk, _ptr(out_topk), _ptr(ws), ws_bytes, _stream(stream)))


def csa2_index_reindex_noalloc(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible,
                               max_visible, pool, pool_blocks, topk, out_topk, status, stream=None):
    """csa2_index_reindex with the library's own fixed device scratch, for
    callers that cannot allocate device memory; `status` is a device int32[4]
    or None."""
    return _check("csa2_index_reindex_noalloc", lib.csa2_index_reindex_noalloc(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), n_q, _ptr(k_codes), _ptr(k_scales), n_rows,
        _ptr(kv_start), _ptr(n_visible), max_visible, _ptr(pool), pool_blocks, topk, _ptr(out_topk),
        _ptr(status), _stream(stream)))


def csa2_sparse_attn(q_bf16, n_q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa,
                     swa_new_bf16, window, sm_scale, out, out_dtype, out_lse, ws, ws_bytes, stream=None):
    return _check("csa2_sparse_attn", lib.csa2_sparse_attn(
        _ptr(q_bf16), n_q, _ptr(kv_codes), _ptr(kv_scales), n_rows, _ptr(kv_start), _ptr(n_visible),
        _ptr(topk), k, _ptr(swa), _ptr(swa_new_bf16), window, sm_scale, _ptr(out), out_dtype,
        _ptr(out_lse), _ptr(ws), ws_bytes, _stream(stream)))


def csa2_sparse_attn_prefill(q_bf16, n_q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa_rows,
                             window, sm_scale, out, out_dtype, out_lse, ws, ws_bytes, stream=None):
    return _check("csa2_sparse_attn_prefill", lib.csa2_sparse_attn_prefill(
        _ptr(q_bf16), n_q, _ptr(kv_codes), _ptr(kv_scales), n_rows, _ptr(kv_start), _ptr(n_visible),
        _ptr(topk), k, _ptr(swa_rows), window, sm_scale, _ptr(out), out_dtype, _ptr(out_lse), _ptr(ws),
        ws_bytes, _stream(stream)))


KERNELS = ("scan_blockmax", "select_blocks", "pool_score", "select_topk", "attn_split",
           "attn_merge", "quantize_fp4", "quantize_fp8", "rope_table")


def csa2_launch_count():
    return lib.csa2_launch_count()


def csa2_debug_wait_limit(ns):
    """Test hook: the bounded device waits' limit in ns for later launches (0: 2 s)."""
    return _check("csa2_debug_wait_limit", lib.csa2_debug_wait_limit(ns))


def csa2_kernel_name(kernel_id):
    return lib.csa2_kernel_name(kernel_id).decode()


def csa2_timer_enable(kernel_id, max_launches):
    return _check("csa2_timer_enable", lib.csa2_timer_enable(kernel_id, max_launches))


def csa2_timer_read(kernel_id):
    """(total milliseconds, launches timed) since csa2_timer_enable."""
    ms = ctypes.c_double()
    n = _i32()
    _check("csa2_timer_read", lib.csa2_timer_read(kernel_id, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value
