// Workspace layouts of the index and attention calls (host + device).
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kMaxWindow = 128;
constexpr int kMaxPoolBlocks = 4096;
constexpr int kMaxTopk = 2048;

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// csa2_index_full: block maxima, the wide candidate list (only when
// topk > pool_blocks), and per-candidate-position scores.
// Batches of at least this many queries run the full scan as the many-query
// contraction (groups of queries share each K tile).
constexpr int64_t kMqMinQueries = 256;
// Smaller batches whose candidate pool has at most this many blocks keep the
// scan's per-position scores, and the Full layer's top-K reads them instead
// of scoring the pool again.
constexpr int64_t kPosScoreMaxCand = 2048;

struct IndexFullWs {
    size_t blockmax, cand, scores, pos, qcodes, qscales, total;
    int64_t nb_stride, cand_stride, score_stride, pos_stride;  // pos_stride 0: no per-position scores
};
__host__ __device__ inline IndexFullWs index_full_ws(int64_t n_q, int64_t max_visible, int P, int K) {
    IndexFullWs w{};
    w.nb_stride = ((max_visible + 7) / 8 + 3) / 4 * 4;
    const int64_t C = P > K ? P : K;
    w.cand_stride = C;
    w.score_stride = 8 * C;
    w.pos_stride = (n_q < kMqMinQueries && C <= kPosScoreMaxCand) ? 8 * w.nb_stride : 0;
    size_t off = CSA2_STATUS_BYTES;
    w.blockmax = off;
    off = align256(off + size_t(n_q) * size_t(w.nb_stride) * 4);
    w.cand = off;
    if (K > P) off = align256(off + size_t(n_q) * size_t(C) * 4);
    w.scores = off;
    if (w.pos_stride == 0) off = align256(off + size_t(n_q) * size_t(w.score_stride) * 4);
    w.pos = off;
    off = align256(off + size_t(n_q) * size_t(w.pos_stride) * 4);
    // csa2_index_full_bf16 with many queries: the query quantized to FP4
    // (BLOCK8 codes, scales) for the many-query scan
    const size_t qrows = n_q >= kMqMinQueries ? size_t(n_q) * 32 : 0;
    w.qcodes = off;
    off = align256(off + qrows * 64);
    w.qscales = off;
    off = align256(off + qrows * 8);
    w.total = off;
    return w;
}

struct ReindexWs {
    size_t scores, total;
    int64_t score_stride;
};
__host__ __device__ inline ReindexWs reindex_ws(int64_t n_q, int P) {
    ReindexWs w{};
    w.score_stride = 8 * int64_t(P);
    w.scores = CSA2_STATUS_BYTES;
    w.total = align256(w.scores + size_t(n_q) * size_t(w.score_stride) * 4);
    return w;
}

// csa2_sparse_attn: 128 entries per CTA (the M of the tensor-core tile).
constexpr int kAttnEntries = 128;

// split partials: O fp32 [64][512] and (m, l) per head per split
struct AttnWs {
    size_t part_o, part_ml, total;
    int splits, entries;
};
__host__ __device__ inline AttnWs attn_ws(int64_t n_q, int k, int window) {
    AttnWs w{};
    const int total = k + window;
    w.entries = kAttnEntries;
    w.splits = (total + w.entries - 1) / w.entries;
    if (w.splits < 1) w.splits = 1;
    w.part_o = CSA2_STATUS_BYTES;
    size_t off = align256(w.part_o + size_t(n_q) * w.splits * CSA2_ATTN_HEADS * CSA2_LATENT_DIM * 4);
    w.part_ml = off;
    off = align256(off + size_t(n_q) * w.splits * CSA2_ATTN_HEADS * 2 * 4);
    w.total = off;
    return w;
}

}  // namespace csa2
