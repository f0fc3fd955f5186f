"""CPU oracle for the CSA2 attention step (test infrastructure, not product code).

This module is a plain, slow, fp64 restatement of what the CSA2 decode step
computes.  It exists only to check the CUDA library: the tests, the smoke
check and the benchmark's CPU-baseline leg may import it; the product path
(the C-ABI library and its Python binding) never does, and shares no code,
table or helper with it.  Nothing here is blocked, fused or reordered beyond
the definitions below; numpy matmul and sorting are used as library steps.

Sources (four secondary web pages about DeepSeek-V4.1-Flash):
  [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解"
  [T2] the blog post "DeepSeek V4.1 Flash vs V4 Pro" (my-blog pages.dev)
  [T3] "DeepSeek-V4.1-Flash：全局 KV 仅 890 B/token，百万上下文怎么做成的？"
  [T4] the ic.work analysis "DeepSeek-V4.1-Flash KV cache compression architecture"

The pages fix the formats, shapes and modes but no formula.  Where they are
silent this module takes the plainest reading, marked READING below:
  * E2M1 is the OCP MX element format; the scale is OCP FP8 E4M3 "FN".
  * A group's scale is RNE_E4M3(amax / 6) (satfinite); elements are rounded to
    the nearest E2M1 value with ties to the even code, saturating at 6; the
    IEEE sign is kept (so -0.1 with a large scale gives code 8, i.e. -0).
  * Two codes per byte, the even channel in the low nibble.
  * RoPE pairs channels (2i, 2i+1) with angle p * theta^(-2i/D), theta=10000,
    over all D channels, p the 0-based absolute position.
  * Indexer score I(t,s) = sum_h w[t,h] * ReLU(q~[t,h] . k~[s]) with q~, k~
    dequantized FP4 and w in fp32 as given; no RoPE on indexer Q/K.
  * Ties in every top-k are broken toward the lower index; outputs are sorted
    ascending and padded with -1.
  * Attention: softmax scale 1/sqrt(512); the selected entries and the window
    entries are not deduplicated (they come from different caches); no sink;
    the value vector is the same latent as the key (K = V = latent).

Parity is pinned by tests that do not re-type these formulas: format tables
against torch's float8_e4m3fn, hand-worked golden groups, nearest-point
properties, brute-force selection on tiny inputs, RoPE group laws, and
attention special cases that reduce to torch's scaled_dot_product_attention.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# Constants fixed by the pages.
# [T1] §二 (CSA2 layout paragraph): 32 index heads of dim 128, top-512 per
# query; main attention 64 heads of dim 512.  [T1] 层级化稀疏索引器: the pool
# holds 2048 blocks of 8 positions.  [T2] 黑科技之一 / [T4]: window 128.
# ---------------------------------------------------------------------------
INDEX_HEADS = 32
INDEX_DIM = 128
TOPK = 512
POOL_BLOCKS = 2048
BLOCK = 8
ATTN_HEADS = 64
LATENT_DIM = 512
WINDOW = 128
GROUP = 16  # channels per E4M3 scale, [T1] §三 / [T2] 黑科技之三 / [T3] 第三刀
ROPE_THETA = 10000.0
SM_SCALE = 1.0 / math.sqrt(LATENT_DIM)  # READING: 1/sqrt(head dim)

# ---------------------------------------------------------------------------
# FP4 element format E2M1, the MXFP4-family element ([T1] §三).
# Bits s e1 e0 m; exponent bias 1; e=0 is subnormal (m * 0.5).
# ---------------------------------------------------------------------------
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(code):
    """Value of 4-bit E2M1 code(s): sign bit 3, magnitude from bits 0-2."""
    code = np.asarray(code, dtype=np.int64)
    mag = E2M1_MAGNITUDES[code & 7]
    return np.where(code & 8, -mag, mag)


# ---------------------------------------------------------------------------
# FP8 E4M3 ("FN" variant: no infinities, 0x7F / 0xFF are NaN, max 448).
# Used for the per-16 scales ([T1] §三) and for the sliding-window KV
# ([T1] §三 and [T3] 第三刀: the window KV is kept in FP8).
# ---------------------------------------------------------------------------
def e4m3_decode(byte):
    """Value of E4M3FN byte(s): bias 7, subnormals m/8 * 2^-6, 0x7F/0xFF NaN."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    normal = (1.0 + m / 8.0) * np.power(2.0, e - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = sign * np.where(e == 0, sub, normal)
    return np.where((b & 0x7F) == 0x7F, np.nan, val)


# The 127 finite non-negative E4M3 values, ascending, with their bytes.
_E4M3_POS_BYTES = np.arange(0x00, 0x7F, dtype=np.int64)
_E4M3_POS_VALUES = e4m3_decode(_E4M3_POS_BYTES)
E4M3_MAX = 448.0


def e4m3_encode(x):
    """Round real(s) to E4M3FN bytes: nearest value, ties to even mantissa,
    saturating to +-448 (satfinite).  The sign of the input is kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    vals = _E4M3_POS_VALUES
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_hi = np.abs(vals[hi] - a)
    d_lo = np.abs(a - vals[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((_E4M3_POS_BYTES[lo] & 1) == 0))
    idx = np.where(pick_lo, lo, hi)
    idx = np.where(a >= E4M3_MAX, len(vals) - 1, idx)
    byte = _E4M3_POS_BYTES[idx]
    return np.where(np.signbit(x), byte | 0x80, byte).astype(np.uint8)


# ---------------------------------------------------------------------------
# Block-scaled FP4 quantization of groups of 16 channels.
# [T1] §三 and [T2] 黑科技之三: E2M1 data, one E4M3 scale per 16 channels,
# like NVFP4 without its second-level global scale.
# ---------------------------------------------------------------------------
def quantize_fp4(x):
    """Quantize real rows x[..., D] (D % 16 == 0) to (codes, scales).

    codes: int array [..., D] of 4-bit codes (one per channel, unpacked).
    scales: uint8 array [..., D/16] of E4M3 scale bytes.
    READING: s = RNE_E4M3(amax/6) (satfinite); s == 0 gives all-zero codes;
    else code = sign(x) | nearest E2M1 magnitude of |x|/s, ties to the even
    code, saturating at 6.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    assert d % GROUP == 0
    if x.size > (1 << 20):  # same definition, row chunks bound the memory
        flat = x.reshape(-1, d)
        parts = [quantize_fp4(flat[i:i + (1 << 20) // d]) for i in range(0, flat.shape[0], (1 << 20) // d)]
        return (np.concatenate([p[0] for p in parts]).reshape(x.shape),
                np.concatenate([p[1] for p in parts]).reshape(x.shape[:-1] + (d // GROUP,)))
    g = x.reshape(x.shape[:-1] + (d // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)
    sbyte = e4m3_encode(amax / 6.0)
    s = e4m3_decode(sbyte)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, np.abs(g) / np.where(s > 0, s, 1.0), 0.0)
    # nearest magnitude; among equal distances prefer the even code
    dist = np.abs(q[..., None] - E2M1_MAGNITUDES)
    best = np.min(dist, axis=-1, keepdims=True)
    is_best = dist == best
    even_best = is_best & (np.arange(8) % 2 == 0)
    mag_code = np.where(np.any(even_best, axis=-1),
                        np.argmax(even_best, axis=-1),
                        np.argmax(is_best, axis=-1))
    mag_code = np.where(q > 6.0, 7, mag_code)  # saturate at 6
    sign = np.where(np.signbit(g), 8, 0)
    codes = np.where(s > 0, sign | mag_code, 0)
    return codes.reshape(x.shape).astype(np.int64), sbyte


def dequantize_fp4(codes, scales):
    """Real values of (codes[..., D], scales[..., D/16]): code value * scale."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    v = e2m1_decode(codes).reshape(codes.shape[:-1] + (d // GROUP, GROUP))
    s = e4m3_decode(scales)[..., None]
    return (v * s).reshape(codes.shape)


def pack_codes(codes):
    """Two codes per byte, even channel in the low nibble (READING)."""
    codes = np.asarray(codes, dtype=np.int64)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed):
    packed = np.asarray(packed, dtype=np.int64)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


# ---------------------------------------------------------------------------
# RoPE on the main latent, applied before quantization.
# [T1] §三 and [T3] 第三刀: the main KV is quantized after RoPE.
# ---------------------------------------------------------------------------
def rope(x, pos, theta=ROPE_THETA):
    """Rotate channel pairs (2i, 2i+1) of x[N][D] by pos[N] * theta^(-2i/D)."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64)
    d = x.shape[-1]
    i = np.arange(d // 2, dtype=np.float64)
    freq = np.power(float(theta), -2.0 * i / d)
    ang = pos[:, None] * freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    xe, xo = x[:, 0::2], x[:, 1::2]
    y = np.empty_like(x)
    y[:, 0::2] = xe * c - xo * s
    y[:, 1::2] = xe * s + xo * c
    return y


def append_main_latent(x_bf16_as_f64, pos, theta=ROPE_THETA):
    """KV append for the main latent: RoPE, then FP4 (packed codes, scales)."""
    codes, scales = quantize_fp4(rope(x_bf16_as_f64, pos, theta))
    return pack_codes(codes), scales


def append_plain_fp4(x):
    """KV append for indexer K / indexer Q rows: FP4 without RoPE (READING)."""
    codes, scales = quantize_fp4(x)
    return pack_codes(codes), scales


def append_swa_fp8(x):
    """Sliding-window latent: plain E4M3 per element, no scale (READING)."""
    return e4m3_encode(x)


# ---------------------------------------------------------------------------
# Hierarchical sparse indexer.
# [T1] 层级化稀疏索引器 and [T3] 第二刀 / Fig. 5: the first Full layer scores
# every visible position, keeps the blocks (8 positions) with the highest
# in-block maximum as a shared pool of 2048 blocks, and later Reindex layers
# score only inside that pool and pick their own top-512.
# ---------------------------------------------------------------------------
def index_scores(q, w, k):
    """I(s) = sum_h w[h] * max(0, q[h] . k[s]) for real q[H][d], w[H], k[n][d].

    The pages give no score formula; this library fixes it as stated here.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dots = k @ q.T  # [n][H]
    return np.maximum(dots, 0.0) @ w


def block_max(scores, block=BLOCK):
    """B[b] = max of scores over positions [8b, 8b+8) that exist (a partial
    last block uses its visible positions only)."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    nb = -(-n // block)
    out = np.full(nb, -np.inf)
    for b in range(nb):
        out[b] = np.max(scores[b * block: min(n, (b + 1) * block)])
    return out


def select_top(values, count):
    """Indices of the `count` largest values, ties toward the lower index,
    returned ascending; fewer values than count returns them all."""
    values = np.asarray(values, dtype=np.float64)
    idx = np.arange(values.shape[0])
    order = np.lexsort((idx, -values))  # by value desc, then index asc
    return np.sort(order[:count])


def pad(ids, length):
    out = np.full(length, -1, dtype=np.int64)
    out[: len(ids)] = ids
    return out


def visible_entries(raw_pos, m):
    """Number of compressed entries (one per m raw tokens) a query at 0-based
    raw position raw_pos may see.  [T1] §二 gives m=1 (decoder) and m=2
    (encoder).  READING: an entry is visible once all its m tokens are at or
    before the query."""
    return (raw_pos + 1) // m


def index_full(q, w, k, n, pool_blocks=POOL_BLOCKS, topk=TOPK):
    """Full-layer index for one query over its first n cache entries.

    Returns (pool, topk_ids): pool = the top-min(P, ceil(n/8)) blocks by block
    maximum; topk_ids = the top-min(K, n) positions by score over ALL visible
    positions (the global definition), both ascending and padded with -1.
    Also returns the fp64 scores for tolerance checks.
    """
    scores = index_scores(q, w, np.asarray(k)[:n])
    bmax = block_max(scores)
    pool = select_top(bmax, pool_blocks)
    top = select_top(scores, topk)
    return pad(pool, pool_blocks), pad(top, topk), scores, bmax


def pool_positions(pool, n, block=BLOCK):
    """Positions covered by the pool blocks (ascending), clipped to n."""
    pool = np.asarray(pool)
    pool = pool[pool >= 0]
    pos = (pool[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return pos[pos < n]


def index_reindex(q, w, k, n, pool, topk=TOPK):
    """Reindex layer: score only the pool's positions with this layer's own
    q, w against the shared indexer K; top-min(K, |pool positions|).
    [T1] §二 mode table; [T2] 黑科技之二; [T3] 第二刀."""
    cand = pool_positions(pool, n)
    scores = index_scores(q, w, np.asarray(k)[cand])
    top = cand[select_top(scores, topk)]
    return pad(np.sort(top), topk), cand, scores


def index_reuse(prev_topk):
    """Reuse layer: indices inherited unchanged ([T1] §二 mode table)."""
    return prev_topk


# ---------------------------------------------------------------------------
# Sparse attention with one merged softmax.
# [T1] §二: 64 heads over a 512-dim latent, each layer keeps its own Q and
# sliding-window KV; [T3] 第三刀: FP4 main KV is dequantized before attention;
# the window stays FP8.
# ---------------------------------------------------------------------------
def window_positions(n, window=WINDOW):
    """The last min(W, n) positions, ascending."""
    return np.arange(max(0, n - window), n)


def sparse_attention(q, sel_latents, win_latents, sm_scale=SM_SCALE):
    """o[h] = sum_j p[h,j] c[j] with p = softmax_j(sm_scale * q[h] . c[j]) over
    the union E of selected and window entries (no dedup), K = V = latent.

    q: [H][D]; sel_latents: [ns][D]; win_latents: [nw][D] (real values).
    Returns (o [H][D], lse [H]) with lse = log sum_j exp(sm_scale * q.c_j).
    """
    q = np.asarray(q, dtype=np.float64)
    c = np.concatenate([np.asarray(sel_latents, dtype=np.float64).reshape(-1, q.shape[1]),
                        np.asarray(win_latents, dtype=np.float64).reshape(-1, q.shape[1])], axis=0)
    if c.shape[0] == 0:
        return np.zeros_like(q), np.full(q.shape[0], -np.inf)
    logits = sm_scale * (q @ c.T)  # [H][E]
    m = np.max(logits, axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = np.sum(p, axis=1, keepdims=True)
    o = (p / l) @ c
    return o, (m + np.log(l))[:, 0]


def attention_inputs(topk_ids, main_codes, main_scales, swa_ring, n, window=WINDOW):
    """Gather the real latents one attention call sees.

    topk_ids: [K] positions (-1 pads skipped); main_codes/main_scales: the
    query's main-KV rows (codes unpacked [n][512], scales [n][32]);
    swa_ring: E4M3 bytes [window][512] with slot = position mod window.
    """
    ids = np.asarray(topk_ids)
    ids = ids[ids >= 0]
    sel = dequantize_fp4(np.asarray(main_codes)[ids], np.asarray(main_scales)[ids])
    wpos = window_positions(n, window)
    win = e4m3_decode(np.asarray(swa_ring)[wpos % window])
    return sel, win


def attention_inputs_shared_window(topk_ids, main_codes, main_scales, win_rows, n, window=WINDOW):
    """The latents one prefill attention call sees: as attention_inputs, but
    the window is the query's own causal window over the shared sequence,
    the rows of the last min(W, n) positions of win_rows [positions][512]
    (E4M3 bytes, one row per compressed position).  READING of [T1] §二 (the
    encoder's layers at m = 2 keep a 128-entry window like the decoder's):
    each prefill query's window holds the entries just before it in the
    sequence all the chunk's queries share."""
    ids = np.asarray(topk_ids)
    ids = ids[ids >= 0]
    sel = dequantize_fp4(np.asarray(main_codes)[ids], np.asarray(main_scales)[ids])
    win = e4m3_decode(np.asarray(win_rows)[window_positions(n, window)])
    return sel, win


# ---------------------------------------------------------------------------
# One query through a layer group.
# [T1] §二: decoder layout [Full + 3 Reuse] + 4 x [Reindex + 3 Reuse]; every
# layer keeps its own attention Q and sliding-window KV.
# ---------------------------------------------------------------------------
def decode_group_query(layers, index_q, index_w, k_real, latent_real, positions,
                       swa_real, attn_q, n, pool_blocks=POOL_BLOCKS, topk=TOPK,
                       window=WINDOW, sm_scale=SM_SCALE, theta=ROPE_THETA):
    """Run one query through `layers` (a sequence of "F", "X", "R").

    index_q / index_w: dict layer -> real (bf16-valued) indexer q [32][128] and
    w [32] for Full/Reindex layers; k_real [n][128] and latent_real [n][512]
    the bf16 cache inputs (pre-quantization; latents pre-RoPE) with their
    RoPE positions; swa_real / attn_q: dict layer -> [window][512] ring (by
    slot) and [64][512].  Returns dict with per-layer topk, the pool, and the
    attention outputs and lse.
    """
    k_codes, k_scales = quantize_fp4(np.asarray(k_real)[:n])
    lat_codes, lat_scales = quantize_fp4(rope(np.asarray(latent_real)[:n], np.asarray(positions)[:n], theta))
    rings = {li: append_swa_fp8(swa_real[li]) for li in range(len(layers))}
    return decode_group_step(layers, index_q, index_w, dequantize_fp4(k_codes, k_scales),
                             lat_codes, lat_scales, rings, attn_q, n, pool_blocks, topk,
                             window, sm_scale)


def decode_group_step(layers, index_q, index_w, k_dequant, lat_codes, lat_scales, rings,
                      attn_q, n, pool_blocks=POOL_BLOCKS, topk=TOPK, window=WINDOW,
                      sm_scale=SM_SCALE):
    """The per-step part of decode_group_query, given caches already in their
    stored formats: k_dequant [n][128] real indexer keys, the main latent's
    codes [n][512] and scales [n][32], and E4M3 window rings per layer."""
    out = {"topk": {}, "pool": None, "o": {}, "lse": {}, "scores": {}}
    cur = None
    for li, mode in enumerate(layers):
        if mode == "F":
            qc, qs = quantize_fp4(index_q[li])
            pool, cur, scores, _ = index_full(dequantize_fp4(qc, qs), index_w[li], k_dequant, n,
                                              pool_blocks, topk)
            out["pool"] = pool
            out["scores"][li] = scores
        elif mode == "X":
            qc, qs = quantize_fp4(index_q[li])
            cur, _, scores = index_reindex(dequantize_fp4(qc, qs), index_w[li], k_dequant, n,
                                           out["pool"], topk)
            out["scores"][li] = scores
        elif mode == "R":
            cur = index_reuse(cur)
        else:
            raise ValueError(mode)
        out["topk"][li] = cur
        sel, win = attention_inputs(cur, lat_codes, lat_scales, rings[li], n, window)
        out["o"][li], out["lse"][li] = sparse_attention(attn_q[li], sel, win, sm_scale)
    return out
