// Hierarchical sparse indexer: full scan with per-8 block maxima, top pool
// blocks, in-pool re-scoring and top-k.
//
// [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", 层级化稀疏索引器,
// and [T3] "DeepSeek-V4.1-Flash：全局 KV 仅 890 B/token，百万上下文怎么做成的？",
// 第二刀 / Fig. 5: the first Full layer scores every visible position, keeps
// the blocks of 8 with the highest in-block maximum as a shared pool (2048 x
// 8 = 16,384 candidates) and the Reindex layers score only inside the pool.
//
// Score (the pages give none; this library's definition):
//   I(t,s) = sum_h w[t][h] * max(0, q~[t][h] . k~[s]),  32 heads x 128 dims.
//
// Scoring core (scan and pool): a warp scores 16 positions against all 32
// heads with 32 m16n8k16 f16 MMAs.  Operands are FP4 dequantized in
// registers: an E2M1 pair converts to f16x2 and is multiplied by its group's
// E4M3 scale, both exact in f16 (at most 6 significant bits, magnitudes in
// [2^-10, 2688]); products are exact and accumulate in fp32.  The reduction
// index of each MMA is a permutation of channels shared by both operands, so
// each thread reads one contiguous 16-byte chunk (32 channels) per row.
#include "csa2_common.cuh"
#include "csa2_timer.cuh"
#include "csa2_layout.cuh"

namespace csa2 {

// ------------------------------------------------------------ scoring core
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t byte_of(const uint4& v, int b) {
    const uint32_t w = b < 4 ? v.x : b < 8 ? v.y : b < 12 ? v.z : v.w;
    return (w >> (8 * (b & 3))) & 0xFF;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t s) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&s));
    return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t scale_h2(uint32_t sbyte) {
    __half2 h = __float2half2_rn(e4m3_value(sbyte));
    return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of the 16-byte chunk c (channels 32c..32c+31) of row r in the
// BLOCK8 layout.
__device__ __forceinline__ int64_t block8_chunk(int64_t r, int c) {
    return (r >> 3) * 512 + c * 128 + (r & 7) * 16;
}

// Indexer query of one query as MMA B fragments: [n-tile j][k-step kk][2].
struct QFrag {
    uint32_t b[4][8][2];
    float w[4][2];
};

__device__ __forceinline__ void load_qfrag(QFrag& f, const uint8_t* __restrict__ q_codes,
                                           const uint8_t* __restrict__ q_scales,
                                           const float* __restrict__ w, int64_t q) {
    const int lane = lane_id(), t = lane & 3, hn = lane >> 2;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t r = q * 32 + 8 * j + hn;
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(q_codes + block8_chunk(r, t)));
        const uint32_t s0 = scale_h2(__ldg(q_scales + r * 8 + 2 * t));
        const uint32_t s1 = scale_h2(__ldg(q_scales + r * 8 + 2 * t + 1));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t s = kk < 4 ? s0 : s1;
            f.b[j][kk][0] = hmul2_u32(e2m1x2_to_f16x2(byte_of(c, 2 * kk)), s);
            f.b[j][kk][1] = hmul2_u32(e2m1x2_to_f16x2(byte_of(c, 2 * kk + 1)), s);
        }
        f.w[j][0] = __ldg(w + q * 32 + 8 * j + 2 * t);
        f.w[j][1] = __ldg(w + q * 32 + 8 * j + 2 * t + 1);
    }
}

// Raw FP4 data of the two rows a thread feeds into one 16-position tile.
struct KRaw {
    uint4 c0, c1;
    uint32_t s0, s1;  // two scale bytes (groups 2t, 2t+1) of each row
};

__device__ __forceinline__ void load_kraw(KRaw& k, const uint8_t* __restrict__ k_codes,
                                          const uint8_t* __restrict__ k_scales, int64_t r0,
                                          bool v0, int64_t r1, bool v1) {
    const int t = lane_id() & 3;
    k.c0 = v0 ? __ldg(reinterpret_cast<const uint4*>(k_codes + block8_chunk(r0, t))) : make_uint4(0, 0, 0, 0);
    k.c1 = v1 ? __ldg(reinterpret_cast<const uint4*>(k_codes + block8_chunk(r1, t))) : make_uint4(0, 0, 0, 0);
    k.s0 = v0 ? __ldg(reinterpret_cast<const uint16_t*>(k_scales + r0 * 8 + 2 * t)) : 0u;
    k.s1 = v1 ? __ldg(reinterpret_cast<const uint16_t*>(k_scales + r1 * 8 + 2 * t)) : 0u;
}

// Scores of the tile's rows lane/4 (out0) and lane/4 + 8 (out1), full sums
// over the 32 heads in every lane of the quad.
__device__ __forceinline__ void score_tile(const QFrag& f, const KRaw& k, float& out0, float& out1) {
    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    const uint32_t sa0 = scale_h2(k.s0 & 0xFF), sa1 = scale_h2((k.s0 >> 8) & 0xFF);
    const uint32_t sb0 = scale_h2(k.s1 & 0xFF), sb1 = scale_h2((k.s1 >> 8) & 0xFF);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t s0 = kk < 4 ? sa0 : sa1, s1 = kk < 4 ? sb0 : sb1;
        uint32_t a[4];
        a[0] = hmul2_u32(e2m1x2_to_f16x2(byte_of(k.c0, 2 * kk)), s0);
        a[1] = hmul2_u32(e2m1x2_to_f16x2(byte_of(k.c1, 2 * kk)), s1);
        a[2] = hmul2_u32(e2m1x2_to_f16x2(byte_of(k.c0, 2 * kk + 1)), s0);
        a[3] = hmul2_u32(e2m1x2_to_f16x2(byte_of(k.c1, 2 * kk + 1)), s1);
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(acc[j], a, f.b[j][kk][0], f.b[j][kk][1]);
    }
    float x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x0 = fmaf(f.w[j][0], fmaxf(acc[j][0], 0.f), x0);
        x0 = fmaf(f.w[j][1], fmaxf(acc[j][1], 0.f), x0);
        x1 = fmaf(f.w[j][0], fmaxf(acc[j][2], 0.f), x1);
        x1 = fmaf(f.w[j][1], fmaxf(acc[j][3], 0.f), x1);
    }
    x0 += __shfl_xor_sync(0xffffffffu, x0, 1);
    x1 += __shfl_xor_sync(0xffffffffu, x1, 1);
    x0 += __shfl_xor_sync(0xffffffffu, x0, 2);
    x1 += __shfl_xor_sync(0xffffffffu, x1, 2);
    out0 = x0;
    out1 = x1;
}

// Per-query validity shared by every index/attention kernel.
__device__ __forceinline__ int32_t checked_visible(const int64_t* kv_start, const int32_t* n_visible,
                                                   int64_t q, int32_t max_visible, int64_t n_rows,
                                                   Status* st, bool report) {
    const int64_t ks = kv_start[q];
    const int32_t n = n_visible[q];
    if (ks < 0 || (ks & 7)) {
        if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_KV_START, int32_t(q), int32_t(ks));
        return 0;
    }
    if (n < 0 || n > max_visible) {
        if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_VISIBLE, int32_t(q), n);
        return 0;
    }
    if (ks + n > n_rows) {
        if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_ROWS, int32_t(q), n);
        return 0;
    }
    return n;
}

// ------------------------------------------------------------ full scan
constexpr int kScanWarps = 8;
constexpr int kScanChunk = 2048;  // positions per CTA

// grid (ceil(max_visible / 2048), n_q); block maxima of blocks [256x, 256x+256).
__global__ void __launch_bounds__(kScanWarps * 32) scan_blockmax_kernel(
    const uint8_t* __restrict__ q_codes, const uint8_t* __restrict__ q_scales,
    const float* __restrict__ w, const uint8_t* __restrict__ k_codes,
    const uint8_t* __restrict__ k_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, float* __restrict__ blockmax,
    int64_t nb_stride, Status* st) {
    const int64_t q = blockIdx.y;
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, st,
                                      blockIdx.x == 0 && threadIdx.x == 0);
    const int64_t base = int64_t(blockIdx.x) * kScanChunk;
    if (base >= n) return;
    const int64_t ks = kv_start[q];
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    QFrag f;
    load_qfrag(f, q_codes, q_scales, w, q);
    const int64_t end = base + kScanChunk < n ? base + kScanChunk : n;
    const int64_t nblk_vis = (n + 7) >> 3;  // blocks holding visible positions
    float* out = blockmax + q * nb_stride;
    KRaw cur, nxt;
    int64_t p = base + 16 * warp;
    auto fetch = [&](KRaw& k, int64_t p0) {
        const int64_t b0 = p0 >> 3;
        load_kraw(k, k_codes, k_scales, ks + p0 + (lane >> 2), b0 < nblk_vis,
                  ks + p0 + 8 + (lane >> 2), b0 + 1 < nblk_vis);
    };
    if (p < end) fetch(cur, p);
    for (; p < end; p += 16 * kScanWarps) {
        const int64_t pn = p + 16 * kScanWarps;
        if (pn < end) fetch(nxt, pn);
        float s0, s1;
        score_tile(f, cur, s0, s1);
        const int64_t pos0 = p + (lane >> 2), pos1 = pos0 + 8;
        float m0 = pos0 < n ? s0 : -INFINITY;
        float m1 = pos1 < n ? s1 : -INFINITY;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
        }
        const int64_t b = p >> 3;
        if (lane == 0) {
            out[b] = m0;
            if (b + 1 < nblk_vis) out[b + 1] = m1;
        }
        cur = nxt;
    }
}

// ------------------------------------------------------------ pool scoring
constexpr int kPoolWarps = 8;
constexpr int kPoolBlocksPerCta = 128;

// grid (ceil(C / 128), n_q).  scores[q][8*i + r] = I(t, 8*cand[q][i] + r), or
// -inf for a pad, an out-of-range block or a position >= n.
__global__ void __launch_bounds__(kPoolWarps * 32) pool_score_kernel(
    const uint8_t* __restrict__ q_codes, const uint8_t* __restrict__ q_scales,
    const float* __restrict__ w, const uint8_t* __restrict__ k_codes,
    const uint8_t* __restrict__ k_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, const int32_t* __restrict__ cand,
    int64_t cand_stride, int C, float* __restrict__ scores, int64_t score_stride, Status* st,
    bool check_cand) {
    const int64_t q = blockIdx.y;
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, st, false);
    const int64_t ks = kv_start[q];
    const int64_t nb = (int64_t(n) + 7) >> 3;
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int i_begin = blockIdx.x * kPoolBlocksPerCta;
    const int i_end = min(C, i_begin + kPoolBlocksPerCta);
    float* out = scores + q * score_stride;
    const int32_t* cq = cand + q * cand_stride;
    QFrag f;
    bool have_q = false;
    for (int i = i_begin + 2 * warp; i < i_end; i += 2 * kPoolWarps) {
        int64_t b0 = cq[i];
        int64_t b1 = i + 1 < i_end ? cq[i + 1] : -1;
        if (check_cand && lane == 0) {
            if (b0 < -1 || b0 >= nb)
                record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_POOL, int32_t(q), int32_t(b0));
            if (i + 1 < i_end && (b1 < -1 || b1 >= nb))
                record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_POOL, int32_t(q), int32_t(b1));
        }
        const bool v0 = b0 >= 0 && b0 < nb, v1 = b1 >= 0 && b1 < nb;
        float s0 = -INFINITY, s1 = -INFINITY;
        if (v0 || v1) {
            if (!have_q) {
                load_qfrag(f, q_codes, q_scales, w, q);
                have_q = true;
            }
            KRaw k;
            load_kraw(k, k_codes, k_scales, ks + 8 * b0 + (lane >> 2), v0, ks + 8 * b1 + (lane >> 2), v1);
            score_tile(f, k, s0, s1);
        }
        const int r = lane >> 2;
        if ((lane & 3) == 0) {
            out[8 * int64_t(i) + r] = (v0 && 8 * b0 + r < n) ? s0 : -INFINITY;
            if (i + 1 < i_end) out[8 * int64_t(i + 1) + r] = (v1 && 8 * b1 + r < n) ? s1 : -INFINITY;
        }
    }
}

// ------------------------------------------------------------ selection
constexpr int kSelThreads = 1024;
constexpr int kSelSmemKeys = 16384;  // keys staged in shared memory (64 KB)

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int& total, int* sh /*>= 33*/) {
    const int lane = lane_id(), warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < nw ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) sh[lane] = s;  // inclusive warp prefix
    }
    __syncthreads();
    total = sh[nw - 1];
    const int before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
    __syncthreads();
    return before;
}

// Key of element i (float scores/maxima, larger first).
struct KeySrc {
    const float* g;   // global values
    const uint32_t* s;  // staged keys in shared memory, or null
    __device__ __forceinline__ uint32_t operator()(int i) const {
        return s ? s[i] : float_key(g[i]);
    }
};

// Threshold key T and how many keys equal to T to take so that exactly
// `count` of the n keys are selected (keys > T plus the first ones == T in
// index order).  8-bit radix passes, warp-aggregated histogram.
__device__ void radix_threshold(const KeySrc& key, int n, int count, uint32_t& thr, int& take_eq,
                                int* hist /*[256]*/, int* sh) {
    const int tid = threadIdx.x, lane = lane_id();
    uint32_t prefix = 0, mask = 0;
    int remaining = count;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int b = 0; b < n; b += blockDim.x) {
            const int i = b + tid;
            bool m = false;
            uint32_t d = 0;
            if (i < n) {
                const uint32_t k = key(i);
                m = (k & mask) == prefix;
                d = (k >> shift) & 0xFF;
            }
            const unsigned mm = __ballot_sync(0xffffffffu, m);
            if (m) {
                const unsigned peers = __match_any_sync(mm, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
            }
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns bins 255-8l .. 248-8l (descending)
            int c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
                sum += c[j];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - sum;  // keys in higher bins than this lane's
            const bool here = excl < remaining && remaining <= incl;
            if (here) {
                int acc = excl, dsel = 255 - 8 * lane - 7;
                for (int j = 0; j < 8; ++j) {
                    if (acc + c[j] >= remaining) {
                        dsel = 255 - 8 * lane - j;
                        break;
                    }
                    acc += c[j];
                }
                sh[0] = dsel;
                sh[1] = remaining - acc;
            }
        }
        __syncthreads();
        prefix |= uint32_t(sh[0]) << shift;
        mask |= 0xFFu << shift;
        remaining = sh[1];
        __syncthreads();
    }
    thr = prefix;
    take_eq = remaining;
}

// Select `count` of n keys (see radix_threshold) and write out[j] = map(i) for
// the selected i in increasing i; pads out[count..pad_to) with -1.
template <class Map>
__device__ void select_compact(const KeySrc& key, int n, int count, int pad_to, int32_t* out,
                               Map map, int* hist, int* sh) {
    const int tid = threadIdx.x;
    if (count > n) count = n;
    if (count <= 0) {
        for (int i = tid; i < pad_to; i += blockDim.x) out[i] = -1;
        return;
    }
    uint32_t thr = 0;
    int take_eq = 0;
    if (count < n) {
        radix_threshold(key, n, count, thr, take_eq, hist, sh);
    } else {
        thr = 0;  // every key is >= 0: take all keys equal to 0 too
        take_eq = n;
    }
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int gt = 0, eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = key(i);
        gt += k > thr;
        eq += k == thr;
    }
    int tot;
    const int eq_before = block_exclusive_scan(eq, tot, sh + 2);
    int take = take_eq - eq_before;
    take = take < 0 ? 0 : (take > eq ? eq : take);
    const int out_before = block_exclusive_scan(gt + take, tot, sh + 2);
    int o = out_before, e = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = key(i);
        if (k > thr || (k == thr && e++ < take)) out[o++] = map(i);
    }
    for (int i = count + tid; i < pad_to; i += blockDim.x) out[i] = -1;
}

struct IdentityMap {
    __device__ __forceinline__ int32_t operator()(int i) const { return i; }
};
struct CandPosMap {
    const int32_t* cand;
    __device__ __forceinline__ int32_t operator()(int i) const { return 8 * cand[i >> 3] + (i & 7); }
};

// Top-`count` blocks by block maximum.  grid n_q, 1024 threads.
__global__ void __launch_bounds__(kSelThreads) select_blocks_kernel(
    const float* __restrict__ blockmax, int64_t nb_stride, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, int64_t n_rows, int count,
    int32_t* __restrict__ out, int64_t out_stride, int smem_keys_cap) {
    extern __shared__ uint32_t smem_keys[];
    __shared__ int hist[256];
    __shared__ int sh[40];
    const int64_t q = blockIdx.x;
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, nullptr, false);
    const int nb = (n + 7) >> 3;
    const float* v = blockmax + q * nb_stride;
    KeySrc key{v, nullptr};
    if (nb <= smem_keys_cap) {
        for (int i = threadIdx.x; i < nb; i += blockDim.x) smem_keys[i] = float_key(v[i]);
        key.s = smem_keys;
        __syncthreads();
    }
    select_compact(key, nb, count, count, out + q * out_stride, IdentityMap{}, hist, sh);
}

// Top-`count` positions among the scored candidates.  grid n_q, 1024 threads.
__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ cand,
    int64_t cand_stride, int C, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, int64_t n_rows, int count,
    int32_t* __restrict__ out, int64_t out_stride, int smem_keys_cap) {
    extern __shared__ uint32_t smem_keys[];
    __shared__ int hist[256];
    __shared__ int sh[40];
    const int64_t q = blockIdx.x;
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, nullptr, false);
    const int32_t* cq = cand + q * cand_stride;
    const int nb = (n + 7) >> 3;
    // positions that exist among the candidates
    int valid = 0;
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        const int32_t b = cq[i];
        if (b >= 0 && b < nb) valid += min(8, n - 8 * b);
    }
    int total;
    block_exclusive_scan(valid, total, sh + 2);
    const int m = 8 * C;
    const float* v = scores + q * score_stride;
    KeySrc key{v, nullptr};
    if (m <= smem_keys_cap) {
        for (int i = threadIdx.x; i < m; i += blockDim.x) smem_keys[i] = float_key(v[i]);
        key.s = smem_keys;
        __syncthreads();
    }
    select_compact(key, m, min(count, total), count, out + q * out_stride, CandPosMap{cq}, hist, sh);
}

// ------------------------------------------------------------ launches
static csa2_status check_index_args(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                    int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                    int64_t n_rows, const int64_t* kv_start,
                                    const int32_t* n_visible, int32_t max_visible,
                                    int pool_blocks, int topk) {
    if (n_q < 0 || n_rows < 0 || max_visible < 0) return CSA2_ERR_INVALID_ARG;
    if (!q_codes || !q_scales || !w || !k_codes || !k_scales || !kv_start || !n_visible)
        return CSA2_ERR_INVALID_ARG;
    if (!aligned16(q_codes) || !aligned16(k_codes) || !aligned16(k_scales) || !aligned16(q_scales))
        return CSA2_ERR_INVALID_ARG;
    if (n_rows % 8) return CSA2_ERR_UNSUPPORTED;
    if (pool_blocks < 1 || pool_blocks > kMaxPoolBlocks || topk < 1 || topk > kMaxTopk)
        return CSA2_ERR_UNSUPPORTED;
    if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;  // grid.y / grid.x limits of the launches
    return CSA2_OK;
}

// Keys a selection launch stages in shared memory (all n, or none).
static int sel_cap(int64_t n) { return n <= kSelSmemKeys ? int(n) : 0; }

// Opt the selection kernels into 64 KB of dynamic shared memory, once per device.
static csa2_status prepare_select_kernels() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
    if (done[dev]) return CSA2_OK;
    const int bytes = kSelSmemKeys * 4;
    if (cudaFuncSetAttribute(select_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return CSA2_ERR_CUDA;
    done[dev] = true;
    return CSA2_OK;
}

}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_index_full(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                       int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                       int64_t n_rows, const int64_t* kv_start,
                                       const int32_t* n_visible, int32_t max_visible,
                                       int pool_blocks, int topk, int32_t* out_pool,
                                       int32_t* out_topk, void* ws, size_t ws_bytes,
                                       csa2_stream_t stream) {
    csa2_status e = check_index_args(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start,
                                     n_visible, max_visible, pool_blocks, topk);
    if (e != CSA2_OK) return e;
    if (!out_pool || !out_topk) return CSA2_ERR_INVALID_ARG;
    const IndexFullWs L = index_full_ws(n_q, max_visible, pool_blocks, topk);
    if (!ws || !aligned16(ws) || ws_bytes < L.total) return CSA2_ERR_WORKSPACE;
    if (n_q == 0) return CSA2_OK;
    if ((e = prepare_select_kernels()) != CSA2_OK) return e;
    cudaStream_t s = cudaStream_t(stream);
    char* base = static_cast<char*>(ws);
    Status* st = reinterpret_cast<Status*>(base);
    float* blockmax = reinterpret_cast<float*>(base + L.blockmax);
    float* scores = reinterpret_cast<float*>(base + L.scores);
    const int C = pool_blocks > topk ? pool_blocks : topk;
    if (max_visible > 0) {
        dim3 grid(unsigned(ceil_div<int64_t>(max_visible, kScanChunk)), unsigned(n_q));
        timer_begin(K_SCAN, s);
        scan_blockmax_kernel<<<grid, kScanWarps * 32, 0, s>>>(q_codes, q_scales, w, k_codes, k_scales,
                                                              n_rows, kv_start, n_visible, max_visible,
                                                              blockmax, L.nb_stride, st);
        timer_end(K_SCAN, s);
    }
    const int cap_b = sel_cap(L.nb_stride);
    timer_begin(K_SELECT_BLOCKS, s);
    select_blocks_kernel<<<unsigned(n_q), kSelThreads, size_t(cap_b) * 4, s>>>(
        blockmax, L.nb_stride, kv_start, n_visible, max_visible, n_rows, pool_blocks, out_pool,
        pool_blocks, cap_b);
    timer_end(K_SELECT_BLOCKS, s);
    const int32_t* cand = out_pool;
    int64_t cand_stride = pool_blocks;
    if (topk > pool_blocks) {
        // the top-k positions lie in the top-max(P, K) blocks
        int32_t* wide = reinterpret_cast<int32_t*>(base + L.cand);
        timer_begin(K_SELECT_BLOCKS, s);
        select_blocks_kernel<<<unsigned(n_q), kSelThreads, size_t(cap_b) * 4, s>>>(
            blockmax, L.nb_stride, kv_start, n_visible, max_visible, n_rows, topk, wide, topk, cap_b);
        timer_end(K_SELECT_BLOCKS, s);
        cand = wide;
        cand_stride = topk;
    }
    dim3 pgrid(unsigned(ceil_div(C, kPoolBlocksPerCta)), unsigned(n_q));
    timer_begin(K_POOL_SCORE, s);
    pool_score_kernel<<<pgrid, kPoolWarps * 32, 0, s>>>(q_codes, q_scales, w, k_codes, k_scales, n_rows,
                                                        kv_start, n_visible, max_visible, cand,
                                                        cand_stride, C, scores, L.score_stride, st,
                                                        false);
    timer_end(K_POOL_SCORE, s);
    const int cap_t = sel_cap(8 * int64_t(C));
    timer_begin(K_SELECT_TOPK, s);
    select_topk_kernel<<<unsigned(n_q), kSelThreads, size_t(cap_t) * 4, s>>>(
        scores, L.score_stride, cand, cand_stride, C, kv_start, n_visible, max_visible, n_rows, topk,
        out_topk, topk, cap_t);
    timer_end(K_SELECT_TOPK, s);
    return launch_status();
}

extern "C" csa2_status csa2_index_reindex(const uint8_t* q_codes, const uint8_t* q_scales,
                                          const float* w, int64_t n_q, const uint8_t* k_codes,
                                          const uint8_t* k_scales, int64_t n_rows,
                                          const int64_t* kv_start, const int32_t* n_visible,
                                          int32_t max_visible, const int32_t* pool, int pool_blocks,
                                          int topk, int32_t* out_topk, void* ws, size_t ws_bytes,
                                          csa2_stream_t stream) {
    csa2_status e = check_index_args(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start,
                                     n_visible, max_visible, pool_blocks, topk);
    if (e != CSA2_OK) return e;
    if (!pool || !out_topk) return CSA2_ERR_INVALID_ARG;
    const ReindexWs L = reindex_ws(n_q, pool_blocks);
    if (!ws || !aligned16(ws) || ws_bytes < L.total) return CSA2_ERR_WORKSPACE;
    if (n_q == 0) return CSA2_OK;
    if ((e = prepare_select_kernels()) != CSA2_OK) return e;
    cudaStream_t s = cudaStream_t(stream);
    char* base = static_cast<char*>(ws);
    Status* st = reinterpret_cast<Status*>(base);
    float* scores = reinterpret_cast<float*>(base + L.scores);
    dim3 pgrid(unsigned(ceil_div(pool_blocks, kPoolBlocksPerCta)), unsigned(n_q));
    timer_begin(K_POOL_SCORE, s);
    pool_score_kernel<<<pgrid, kPoolWarps * 32, 0, s>>>(q_codes, q_scales, w, k_codes, k_scales, n_rows,
                                                        kv_start, n_visible, max_visible, pool,
                                                        pool_blocks, pool_blocks, scores,
                                                        L.score_stride, st, true);
    timer_end(K_POOL_SCORE, s);
    const int cap_t = sel_cap(8 * int64_t(pool_blocks));
    timer_begin(K_SELECT_TOPK, s);
    select_topk_kernel<<<unsigned(n_q), kSelThreads, size_t(cap_t) * 4, s>>>(
        scores, L.score_stride, pool, pool_blocks, pool_blocks, kv_start, n_visible, max_visible,
        n_rows, topk, out_topk, topk, cap_t);
    timer_end(K_SELECT_TOPK, s);
    return launch_status();
}
