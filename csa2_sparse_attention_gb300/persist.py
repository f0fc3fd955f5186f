"""Save and restore a request's FP4 global KV cache, without the window.

[T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", "持久缓存为什么能降到
1/8", and [T3] "DeepSeek-V4.1-Flash：全局 KV 仅 890 B/token，百万上下文怎么做成的？",
第三刀: the persistent (global) cache keeps the FP4 main latent and the
indexer keys; the sliding-window KV is not persisted (it is rebuilt from the
last tokens).  A request's global KV is its rows of three planes:

  main latent codes   rows x 256 B  (E2M1, two per byte)
  main latent scales  rows x 32 B   (E4M3, one per 16 channels)
  indexer K           the request's 8-row blocks: 576-byte records (codes
                      then scales), or BLOCK8 codes and row-major scales

The bytes are copied as they are stored (no re-quantization), so a restored
request indexes and attends exactly as before.  Format: the magic
b"CSA2KV01", a little-endian header (rows, indexer-K layout, byte counts of
each plane), the planes in the order above, and the SHA-256 of everything
before it.  This is device-to-host plumbing: the planes move with torch
copies; no arithmetic of the method runs here.
"""
from __future__ import annotations

import hashlib
import struct

import torch

from . import abi

MAGIC = b"CSA2KV01"
_HEADER = struct.Struct("<8sqiqqqq")  # magic, rows, ik layout, bytes: codes, scales, ik codes, ik scales


def _request_planes(g, r):
    """(rows, views of the request's bytes in each plane) of LayerGroup g."""
    if g.wl.shared_cache:
        ks, n = 0, int(g.wl.cache_entries)
    else:
        ks, n = int(g.row_base[r]), int(g.contexts[r])
    b0, b1 = ks // 8, (ks + n + 7) // 8
    planes = [g.kv_codes[ks:ks + n], g.kv_scales[ks:ks + n]]
    if g.ik_layout == abi.LAYOUT_BLOCK8R:
        planes += [g.ik_codes[b0 * 576:b1 * 576], None]
    else:
        planes += [g.ik_codes[b0 * 512:b1 * 512], g.ik_scales[b0 * 8:b1 * 8]]
    return n, planes


def save_request(g, r, f):
    """Write request r's global KV (as stored in LayerGroup g) to the binary
    file object f.  Returns the number of bytes written."""
    n, planes = _request_planes(g, r)
    blobs = [p.contiguous().cpu().numpy().tobytes() if p is not None else b"" for p in planes]
    head = _HEADER.pack(MAGIC, n, g.ik_layout, *(len(b) for b in blobs))
    h = hashlib.sha256(head)
    for b in blobs:
        h.update(b)
    data = head + b"".join(blobs) + h.digest()
    f.write(data)
    return len(data)


def load_request(g, r, f):
    """Restore request r of LayerGroup g from a file written by save_request.
    The request's context length and g's indexer-K layout must match the
    file's; a damaged or mismatched file raises ValueError and leaves g's
    cache untouched."""
    data = f.read()
    if len(data) < _HEADER.size + 32:
        raise ValueError("KV file too short")
    magic, n, layout, *sizes = _HEADER.unpack_from(data)
    if magic != MAGIC:
        raise ValueError("not a CSA2 KV file")
    body_end = _HEADER.size + sum(sizes)
    if len(data) != body_end + 32 or hashlib.sha256(data[:body_end]).digest() != data[body_end:]:
        raise ValueError("KV file damaged (checksum)")
    n_here, planes = _request_planes(g, r)
    if n != n_here or layout != g.ik_layout:
        raise ValueError(f"KV file holds {n} rows in layout {layout}; the request has {n_here} in {g.ik_layout}")
    off = _HEADER.size
    staged = []
    for p, size in zip(planes, sizes):
        if (p is None) != (size == 0) or (p is not None and p.numel() * p.element_size() != size):
            raise ValueError("KV file plane sizes do not match the request")
        if p is not None:
            src = torch.frombuffer(bytearray(data[off:off + size]), dtype=torch.uint8).view(p.shape)
            staged.append((p, src))
        off += size
    for p, src in staged:
        p.copy_(src.to(p.device))
    if torch.device(g.dev).type == "cuda":
        torch.cuda.synchronize(g.dev)
