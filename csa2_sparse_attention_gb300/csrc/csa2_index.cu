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
// Scoring (scan and pool) runs on the 5th-generation tensor cores as block-
// scaled FP4 MMAs (E2M1 operands, one E4M3 scale per 16 channels, fp32
// accumulate in TMEM); the ReLU, head weights, head sum and block maximum
// are applied to the accumulator in registers.
#include "csa2_common.cuh"
#include "csa2_timer.cuh"
#include "csa2_layout.cuh"
#include "csa2_pipe.cuh"
#include "csa2_tc.cuh"

#include <climits>
#include <cooperative_groups.h>
#include <cuda.h>  // CUtensorMap and the tensor-map encoder's types (the encoder is fetched from the driver at run time)

namespace csa2 {

// Per-query validity shared by every index/attention kernel.
__device__ __forceinline__ int32_t checked_visible_values(int64_t ks, int32_t n, int64_t q, int32_t max_visible,
                                                          int64_t n_rows, Status* st, bool report);
__device__ __forceinline__ int32_t checked_visible(const int64_t* kv_start, const int32_t* n_visible,
                                                   int64_t q, int32_t max_visible, int64_t n_rows,
                                                   Status* st, bool report) {
    return checked_visible_values(kv_start[q], n_visible[q], q, max_visible, n_rows, st, report);
}
// The same checks on values already loaded.
__device__ __forceinline__ int32_t checked_visible_values(int64_t ks, int32_t n, int64_t q, int32_t max_visible,
                                                          int64_t n_rows, Status* st, bool report) {
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

constexpr int kTile = 128;  // positions per tensor-core tile (16 blocks of 8)

// ------------------------------------------------------------ tensor-core scorer
// Block-scaled FP4 tcgen05 scorer shared by the full scan and the in-pool
// scoring, on a (CTAs per query, queries) grid of about two CTAs per SM.  For
// the scan, C carries the query count (0: never rebalance); when the
// queries' visible counts differ, the CTAs are reassigned so that every CTA
// gets about the same number of tiles (scan_map).  A tile is 16 blocks = 128 positions (M); N = 32 index heads;
// K = 128 channels as two kind::mxf4nvf4 MMAs of 64 with one E4M3 scale per
// 16 channels, so the FP4 codes go from shared memory to the tensor core
// without dequantization.  Warp 0 streams tiles (contiguous blocks for the
// scan, the candidate blocks for the pool) into a ring of shared-memory
// stages with bulk copies (the pool's records four at a time with TMA
// gathers); warp 1 issues the MMAs; warps 2..9, two groups of four taking
// alternate tiles, copy each tile's scales into TMEM and reduce the 32 head
// scores of every position: the block maxima (scan) or per-position scores
// (pool).  One group alone could not keep up with the scan's tile rate.
constexpr int kTcThreads = 320;     // producer, MMA, two epilogue groups of 4 warps
constexpr int kTcStages = 8;
constexpr int kTcAcc = 4;            // accumulator stages (32 TMEM columns each)
constexpr int kTcSf = 4;             // scale-factor slots (8 columns each)
constexpr uint32_t kTcCols = 256;
constexpr uint32_t kColAcc = 0, kColSfa = 128, kColSfb = 160;
constexpr int kTcSfLead = 3;         // tiles whose scales are staged ahead (< kTcSf)
constexpr int kTcMaxCandPerCta = 4096;
static_assert(kTcMaxCandPerCta >= kMaxPoolBlocks, "a CTA stages at most all candidate blocks");

// Indexer K arrives either as BLOCK8 code blocks of 512 bytes with the
// scales in their own row-major plane, or as 576-byte records (a block's 512
// code bytes, then its 8 rows x 8 scale bytes).  A stage of the ring holds
// one tile in the same form: 16 records, or 16 x 512 code bytes then 16 x 64
// scale bytes.  The MMA reads the codes in place (8-row groups 576 or 512
// bytes apart).
constexpr int kStageBytes = kTile * 72;
template <bool REC>
__device__ __forceinline__ uint8_t* stage_codes(uint8_t* ring, int s) {
    return ring + s * kStageBytes;
}
template <bool REC>
__device__ __forceinline__ uint8_t* stage_scales(uint8_t* ring, int s, int row) {
    return ring + s * kStageBytes + (REC ? (row >> 3) * 576 + 512 + (row & 7) * 8 : kTile * 64 + row * 8);
}

struct TcScanSmem {
    uint8_t ring[kTcStages * kStageBytes];
    uint8_t qcodes[32 * 64];          // the query's 32 heads, BLOCK8 = canonical K-major
    uint8_t qsc[32 * 8];              // their scales, when the query arrives as bf16
    int32_t cand[kTcMaxCandPerCta];   // this CTA's candidate blocks (pool scoring)
    uint64_t full[kTcStages], empty[kTcStages];
    uint64_t sfa_ready[kTcSf];
    uint64_t acc_full[kTcAcc], acc_empty[kTcAcc];
    uint64_t qbar;
    uint32_t tmem;
    int abort_flag;
};

// Queries the balanced scan mapping handles (its per-lane register arrays);
// it runs only when the batch also fits the device's SM count, so that one
// wave of two CTAs per SM holds a CTA of every active query.
constexpr int kScanMaxQ = 152;


// The balanced scan mapping over a grid of G CTAs (b = this CTA's linear
// index): query q gets ceil(tiles_q G / T) CTAs (T = all visible tiles; G
// is replaced by G - active queries when rounding up would need more than G)
// and each of them a contiguous slice of that query's tiles.  Warp 0 does
// it with shuffles (lane l holds queries l QPL .. l QPL + QPL - 1) and
// publishes this CTA's slice.  Returns whether the CTA has tiles.
__device__ bool scan_map(const int64_t* kv_start, const int32_t* n_visible, int32_t max_visible, int64_t n_rows,
                         int nq, uint32_t G, uint32_t b, Status* st, int64_t* slice, int64_t& q, int64_t& t0,
                         int64_t& t1, int32_t& n) {
    constexpr int QPL = (kScanMaxQ + 31) / 32;
    // slice (shared memory): q (or -1), t0, t1, n
    if (threadIdx.x < 32) {
        const int lane = lane_id();
        uint32_t tq[QPL];
        int32_t nv[QPL];
        uint32_t run = 0;
#pragma unroll
        for (int j = 0; j < QPL; ++j) {
            const int i = lane * QPL + j;
            nv[j] = i < nq ? checked_visible(kv_start, n_visible, i, max_visible, n_rows, st,
                                             st != nullptr && blockIdx.x == 0)
                           : 0;
            tq[j] = uint32_t((((int64_t(nv[j]) + 7) >> 3) + 15) >> 4);
            run += tq[j];
        }
        auto incl_scan = [&](uint32_t x) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            return x;
        };
        const uint32_t T = __shfl_sync(0xffffffffu, incl_scan(run), 31);
        uint32_t c[QPL], csum = 0, cbase = 0;
        int found = -1;
        if (T > 0) {
            auto ctas = [&](uint64_t G) {
                uint32_t sum = 0;
#pragma unroll
                for (int j = 0; j < QPL; ++j) {
                    const uint64_t v = (uint64_t(tq[j]) * G + T - 1) / T;
                    c[j] = uint32_t(v < tq[j] ? v : tq[j]);
                    sum += c[j];
                }
                return sum;
            };
            csum = ctas(G);
            uint32_t cin = incl_scan(csum);
            if (__shfl_sync(0xffffffffu, cin, 31) > G) {
                uint32_t act = 0;
#pragma unroll
                for (int j = 0; j < QPL; ++j) act += tq[j] > 0;
                act = __reduce_add_sync(0xffffffffu, act);
                csum = ctas(G > act ? G - act : 1u);
                cin = incl_scan(csum);
            }
            cbase = cin - csum;
            if (b >= cbase && b < cin) {  // this lane holds the CTA's query
                uint32_t lo = cbase;
#pragma unroll
                for (int j = 0; j < QPL; ++j) {
                    if (found < 0 && b < lo + c[j]) {
                        found = j;
                        const int64_t jj = b - lo;
                        slice[0] = int64_t(lane) * QPL + j;
                        slice[1] = jj * tq[j] / c[j];
                        slice[2] = (jj + 1) * tq[j] / c[j];
                        slice[3] = nv[j];
                    }
                    lo += c[j];
                }
            }
        }
        if (!__any_sync(0xffffffffu, found >= 0) && lane == 0) slice[0] = -1;
    }
    __syncthreads();
    q = slice[0];
    t0 = slice[1];
    t1 = slice[2];
    n = int32_t(slice[3]);
    __syncthreads();  // every thread has read the slice before it is written again
    return q >= 0;
}

template <bool GATHER, bool REC>
__global__ void __launch_bounds__(kTcThreads, 2) score_tc_kernel(
    const uint8_t* __restrict__ q_codes, const uint8_t* __restrict__ q_scales,
    const float* __restrict__ w, const uint8_t* __restrict__ k_codes,
    const uint8_t* __restrict__ k_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, const int32_t* __restrict__ cand,
    int64_t cand_stride, int C, float* __restrict__ out, int64_t out_stride, int ctas_per_query,
    bool check_cand, Status* st, float* __restrict__ pos_scores, int64_t pos_stride, uint64_t wlim,
    const __grid_constant__ CUtensorMap kmap, bool use_map, const uint16_t* __restrict__ q_bf16) {
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    TcScanSmem& S = *reinterpret_cast<TcScanSmem*>(tc_smem_raw);
    constexpr bool rec = REC;  // indexer K as 576-byte records (k_scales unused)
    grid_dep_wait();
    grid_dep_launch();
    int64_t q = blockIdx.y, t0, t1;
    int32_t n;
    const int64_t ks_row = kv_start[q];  // this grid row's query, loaded alongside the checks below
    const int32_t n_row = n_visible[q];
    // the scan of a batch whose contexts differ (C = its query count, at most
    // kScanMaxQ) spreads all visible tiles over the grid; equal contexts (and
    // the pool scoring) split each query over its row of the grid
    bool skewed = false;
    if (!GATHER && C > 0) {  // every warp checks (no block barrier)
        const int32_t n0 = n_visible[0];
        bool diff = false;
        for (int i = int(lane_id()); i < C; i += 32) diff |= n_visible[i] != n0;
        skewed = __any_sync(0xffffffffu, diff);
    }
    if (skewed) {
        if (!scan_map(kv_start, n_visible, max_visible, n_rows, int(C), gridDim.x * gridDim.y,
                      blockIdx.x + gridDim.x * blockIdx.y, st, reinterpret_cast<int64_t*>(S.cand), q, t0, t1, n))
            return;
    } else {
        n = checked_visible_values(ks_row, n_row, q, max_visible, n_rows, GATHER ? nullptr : st,
                                   !GATHER && blockIdx.x == 0 && threadIdx.x == 0);
        const int64_t tiles_q = GATHER ? (C + 15) / 16 : ((int64_t(n) + 7) / 8 + 15) / 16;
        const int64_t per = (tiles_q + ctas_per_query - 1) / ctas_per_query;
        t0 = int64_t(blockIdx.x) * per;
        t1 = t0 + per < tiles_q ? t0 + per : tiles_q;
    }
    const int64_t nblk_vis = (int64_t(n) + 7) >> 3;
    if (n <= 0 || t0 >= t1) {
        if (GATHER) {  // nothing visible: every score of this range is -inf
            const int64_t end = t1 * 128 < 8 * int64_t(C) ? t1 * 128 : 8 * int64_t(C);
            for (int64_t i = t0 * 128 + threadIdx.x; i < end; i += blockDim.x) out[q * out_stride + i] = -INFINITY;
        }
        return;
    }
    const int64_t ks = kv_start[q];
    const int32_t* cq = GATHER ? cand + q * cand_stride : nullptr;
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int ntiles = int(t1 - t0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int f = 0; f < kTcSf; ++f) mbar_init(&S.sfa_ready[f], 128);
        for (int a = 0; a < kTcAcc; ++a) {
            mbar_init(&S.acc_full[a], 1);
            mbar_init(&S.acc_empty[a], 128);
        }
        mbar_init(&S.qbar, 1);
        S.abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&S.tmem, kTcCols);
    if (GATHER) {  // this CTA's candidate ids, once, by every thread
        const int64_t c_lo = t0 * 16, c_hi = t1 * 16 < C ? t1 * 16 : C;
        for (int64_t ci = c_lo + threadIdx.x; ci < c_hi; ci += blockDim.x) S.cand[ci - c_lo] = cq[ci];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    // (warp 0 lane 0) tiles whose copies were issued; (warp 1 lane 0) tiles
    // whose MMAs were issued: what a give-up must wait for before TMEM and
    // shared memory are released
    int issued = 0, mma_n = 0;
    if (q_bf16 != nullptr && warp > 0) {
        // the query as bf16: warps 1..9 quantize its 32 heads (256 groups of
        // 16 channels) into the MMA's B operand and its scales, exactly as
        // the FP4 append does, while warp 0 already streams K tiles
        for (int grp = int(threadIdx.x) - 32; grp < 256; grp += kTcThreads - 32) {
            const int h = grp >> 3, g = grp & 7;
            const uint4* src = reinterpret_cast<const uint4*>(q_bf16 + (q * 32 + h) * 128 + 16 * g);
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float v[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[2 * j] = bf16_lo(wv[j]);
                v[2 * j + 1] = bf16_hi(wv[j]);
            }
            uint32_t cw[2];
            S.qsc[h * 8 + g] = uint8_t(quantize_group16(v, cw));
            *reinterpret_cast<uint2*>(S.qcodes + (h >> 3) * 512 + (g >> 1) * 128 + (h & 7) * 16 + (g & 1) * 8) =
                make_uint2(cw[0], cw[1]);
        }
        fence_async_smem();  // the codes are the MMA's operand
        asm volatile("bar.sync 1, %0;" ::"n"(kTcThreads - 32) : "memory");
    }

    if (warp == 0) {  // ------------------------------------------ producer
        // the scan copies a tile with one bulk copy from lane 0 (two in the
        // split layout); the gather takes a tile's 16 blocks with four TMA
        // gathers (records) or spreads 32 copies (codes, scales) over the lanes
        if (lane == 0 && q_bf16 == nullptr) {
            mbar_arrive_expect_tx(&S.qbar, 32 * 64);
            bulk_g2s(S.qcodes, q_codes + (q * 32 / 8) * 512, 32 * 64, &S.qbar);
        }
        for (int i = 0; i < ntiles; ++i) {
            const int s = i % kTcStages, r = i / kTcStages;
            int ok = 1;
            if (lane == 0 && r > 0 && !mbar_wait(&S.empty[s], (r - 1) & 1, wlim)) {
                record(st, CSA2_ERR_TIMEOUT, 10, int32_t(q), i);
                S.abort_flag = 1;
                ok = 0;
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const int64_t t = t0 + i;
            if (!GATHER) {
                if (lane == 0) {
                    const int64_t nvb64 = nblk_vis - t * 16;
                    const uint32_t nvb = uint32_t(nvb64 < 16 ? nvb64 : 16);
                    mbar_arrive_expect_tx(&S.full[s], nvb * (512 + 64));
                    if (rec) {
                        bulk_g2s(stage_codes<rec>(S.ring, s), k_codes + ((ks >> 3) + t * 16) * 576, nvb * 576,
                                 &S.full[s]);
                    } else {
                        bulk_g2s(stage_codes<rec>(S.ring, s), k_codes + ((ks >> 3) + t * 16) * 512, nvb * 512,
                                 &S.full[s]);
                        bulk_g2s(stage_scales<rec>(S.ring, s, 0), k_scales + (ks + t * kTile) * 8, nvb * 64,
                                 &S.full[s]);
                    }
                }
                issued = i + 1;
            } else {
                // block j of the tile: lane j its record (or its codes, and
                // lane 16 + j its scales)
                const int j = lane & 15;
                const int64_t ci = t * 16 + j;
                const int32_t bl = ci < C ? S.cand[ci - t0 * 16] : -1;
                const bool live = bl >= 0 && bl < nblk_vis && (lane < 16 || !rec);
                if (lane < 16 && !live && check_cand && (bl < -1 || bl >= nblk_vis))
                    record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_POOL, int32_t(q), bl);
                if (rec && use_map) {
                    // four TMA gathers of four records each (lanes 0..3); a
                    // slot without a valid block re-reads the query's first
                    // block, whose scores the epilogue discards
                    const int32_t row = int32_t((ks >> 3) + (live ? bl : 0));
                    const int g4 = 4 * (lane & 3);
                    const int32_t r0 = __shfl_sync(0xffffffffu, row, g4), r1 = __shfl_sync(0xffffffffu, row, g4 + 1);
                    const int32_t r2 = __shfl_sync(0xffffffffu, row, g4 + 2), r3 = __shfl_sync(0xffffffffu, row, g4 + 3);
                    if (lane == 0) mbar_arrive_expect_tx(&S.full[s], 16 * 576);
                    __syncwarp();
                    if (lane < 4) tma_gather4(stage_codes<rec>(S.ring, s) + g4 * 576, &kmap, r0, r1, r2, r3, &S.full[s]);
                    issued = i + 1;
                    continue;
                }
                const uint32_t bytes = __reduce_add_sync(0xffffffffu, live ? (lane < 16 ? (rec ? 576u : 512u) : 64u) : 0u);
                if (lane == 0) mbar_arrive_expect_tx(&S.full[s], bytes);  // 0 bytes: the phase completes at once
                __syncwarp();
                if (live) {
                    if (rec)
                        bulk_g2s(stage_codes<rec>(S.ring, s) + j * 576, k_codes + ((ks >> 3) + bl) * 576, 576,
                                 &S.full[s]);
                    else if (lane < 16)
                        bulk_g2s(stage_codes<rec>(S.ring, s) + j * 512, k_codes + ((ks >> 3) + bl) * 512, 512,
                                 &S.full[s]);
                    else
                        bulk_g2s(stage_scales<rec>(S.ring, s, 8 * j), k_scales + (ks + 8 * int64_t(bl)) * 8, 64,
                                 &S.full[s]);
                }
                issued = i + 1;
            }
        }
    } else if (warp == 1) {  // ----------------------------------- MMA issue
        if (lane == 0) {
            bool ok = q_bf16 != nullptr || mbar_wait(&S.qbar, 0, wlim);
            constexpr uint32_t id = idesc_mxf4nvf4(128, 32);
            const uint32_t qa = smem_u32(S.qcodes);
            for (int i = 0; ok && i < ntiles; ++i) {
                const int s = i % kTcStages, f = i % kTcSf, a = i % kTcAcc;
                ok = mbar_wait(&S.full[s], (i / kTcStages) & 1, wlim) && mbar_wait(&S.sfa_ready[f], (i / kTcSf) & 1, wlim) &&
                     (i < kTcAcc || mbar_wait(&S.acc_empty[a], ((i / kTcAcc) - 1) & 1, wlim));
                if (!ok) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(stage_codes<rec>(S.ring, s)), sbo = rec ? 576 : 512;
                const uint32_t d = tmem + kColAcc + 32 * a;
                const uint32_t sfa = tmem + kColSfa + 8 * f, sfb = tmem + kColSfb;
                mma_mxf4_ss(d, umma_desc(ka, 128, sbo), umma_desc(qa, 128, 512), id, sfa, sfb, false);
                mma_mxf4_ss(d, umma_desc(ka + 256, 128, sbo), umma_desc(qa + 256, 128, 512), id, sfa + 4, sfb + 4, true);
                tc_commit(&S.acc_full[a]);
                tc_commit(&S.empty[s]);
                mma_n = i + 1;
            }
            if (!ok) {
                record(st, CSA2_ERR_TIMEOUT, 11, int32_t(q), 0);
                S.abort_flag = 1;
            }
        }
    } else {  // --------------------------------------------------- epilogue
        // two groups of 4 warps (one per TMEM lane quadrant) take alternate
        // tiles: group eg reads the accumulators of tiles eg, eg + 2, ...
        // and stages those tiles' scales
        const int eg = (warp - 2) >> 2;         // epilogue group
        const int quad = warp & 3;              // TMEM lane quadrant of this warp
        const int row = 32 * quad + lane;       // position within a tile
        const uint32_t lane_base = tmem + (uint32_t(32 * quad) << 16);
        float wv[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) wv[h] = __ldg(w + q * 32 + h);
        if (eg == 0) {  // the query's scales (B), replicated in every quadrant
            const uint2 qs = q_bf16 != nullptr ? *reinterpret_cast<const uint2*>(S.qsc + lane * 8)
                                               : __ldg(reinterpret_cast<const uint2*>(q_scales + (q * 32 + lane) * 8));
            tmem_st4(lane_base + kColSfb, qs.x, 0u, 0u, 0u);
            tmem_st4(lane_base + kColSfb + 4, qs.y, 0u, 0u, 0u);
        }
        auto stage_sf = [&](int i) -> bool {  // tile i's scales (A) into slot i % kTcSf
            const int s = i % kTcStages, f = i % kTcSf;
            if (!mbar_wait(&S.full[s], (i / kTcStages) & 1, wlim)) return false;
            uint2 r4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                r4[j] = *reinterpret_cast<const uint2*>(stage_scales<rec>(S.ring, s, lane + 32 * j));
            tmem_st4(lane_base + kColSfa + 8 * f, r4[0].x, r4[1].x, r4[2].x, r4[3].x);
            tmem_st4(lane_base + kColSfa + 8 * f + 4, r4[0].y, r4[1].y, r4[2].y, r4[3].y);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&S.sfa_ready[f]);
            return true;
        };
        bool ok = true;
        // the four scale slots start free: tiles eg and eg + 2
        for (int i = eg; ok && i < kTcSf && i < ntiles; i += 2) ok = stage_sf(i);
        for (int i = eg; ok && i < ntiles; i += 2) {
            const int a = i % kTcAcc;
            if (!mbar_wait(&S.acc_full[a], (i / kTcAcc) & 1, wlim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // tile i's MMA is done, so the slot of tile i + kTcSf is free
            if (i + kTcSf < ntiles && !stage_sf(i + kTcSf)) {
                ok = false;
                break;
            }
            uint32_t r[32];
            tmem_ld32(lane_base + kColAcc + 32 * a, r);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&S.acc_empty[a]);
            float x = 0.f;
#pragma unroll
            for (int h = 0; h < 32; ++h) x = fmaf(wv[h], fmaxf(__uint_as_float(r[h]), 0.f), x);
            const int64_t t = t0 + i;
            if (!GATHER) {
                const int64_t pos = t * kTile + row;
                if (pos_scores != nullptr && pos < n) pos_scores[q * pos_stride + pos] = x;
                float m = pos < n ? x : -INFINITY;
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                const int64_t b = pos >> 3;
                if ((lane & 7) == 0 && b < nblk_vis) out[q * out_stride + b] = m;
            } else {
                const int64_t ci = t * 16 + (row >> 3);
                if (ci < C) {
                    const int32_t b = S.cand[ci - t0 * 16];
                    const bool v = b >= 0 && b < nblk_vis && 8 * int64_t(b) + (row & 7) < n;
                    out[q * out_stride + 8 * ci + (row & 7)] = v ? x : -INFINITY;
                }
            }
        }
        if (!ok && lane == 0) {
            record(st, CSA2_ERR_TIMEOUT, 12, int32_t(q), 0);
            S.abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (S.abort_flag) {  // (uniform: nothing writes the flag after the barrier)
        // a wait gave up: wait for the copies and MMAs already issued (the
        // last commit covers every earlier MMA) before anything is released
        if (lane == 0 && warp == 0) {
            if (q_bf16 == nullptr) mbar_wait(&S.qbar, 0, kDrainNs);
            for (int i = issued > kTcStages ? issued - kTcStages : 0; i < issued; ++i)
                mbar_wait(&S.full[i % kTcStages], (i / kTcStages) & 1, kDrainNs);
        } else if (lane == 0 && warp == 1 && mma_n > 0) {
            mbar_wait(&S.empty[(mma_n - 1) % kTcStages], ((mma_n - 1) / kTcStages) & 1, kDrainNs);
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) tmem_dealloc(tmem, kTcCols);
}

// ------------------------------------------------------------ selection
// One 1024-thread CTA per query selects `count` of n keys (larger first,
// ties to the lower index) and writes the selected indices in increasing
// order.  Keys are uint32 images of the floats (float_key), staged in shared
// memory when they fit.  An 8-bit radix pass over all keys picks the top
// digit of the threshold; the keys sharing that digit are collected into a
// short candidate list and the three remaining passes run on it.  The output
// is compacted over warp-contiguous segments (coalesced reads, two block
// scans) so it comes out in index order.
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeys = 32768;  // keys staged in shared memory (128 KB)
constexpr int kCandCap = 4096;       // candidates kept after the first pass

struct SelShared {
    int hist[256];
    int wsum[3][kSelWarps];
    int misc[kSelWarps];
    int bins[kSelWarps][32];
    int tbins[kSelWarps][33];  // register selection: bucket counts per warp (padded rows)
    int ttot[2][32];           // register selection: bucket totals of a round (by round parity)
    uint32_t cand_key[kCandCap];
    // cluster selection: this CTA's contribution, read by its peers
    int cl_hist[2][32];    // bucket counts of a round (double-buffered by round parity)
    uint32_t cl_minmax[2];
    int cl_cnt[2];         // keys above / equal to the threshold in this CTA's segment
};

// Key of element i (float scores/maxima, larger first).
struct KeySrc {
    const float* g;     // global values
    const uint32_t* s;  // staged keys in shared memory, or null
    __device__ __forceinline__ uint32_t operator()(int i) const {
        return s ? s[i] : float_key(g[i]);
    }
};

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Histogram of the 8-bit digit at `shift` of the keys produced by get(i) for
// i < n that match (k & mask) == prefix; warp-aggregated with match_any.
template <class Get>
__device__ __forceinline__ void radix_hist(Get get, int n, uint32_t prefix, uint32_t mask, int shift,
                                           int* hist) {
    const int lane = lane_id();
    for (int b = 0; b < n; b += blockDim.x) {
        const int i = b + threadIdx.x;
        bool m = false;
        uint32_t d = 0;
        if (i < n) {
            const uint32_t k = get(i);
            m = (k & mask) == prefix;
            d = (k >> shift) & 0xFF;
        }
        const unsigned mm = __ballot_sync(0xffffffffu, m);
        if (m) {
            const unsigned peers = __match_any_sync(mm, d);
            if (lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
        }
    }
}

// Warp 0 finds the digit holding the `remaining`-th largest key; writes
// misc[0] = digit, misc[1] = how many keys of that digit are still needed.
__device__ __forceinline__ void radix_pick(const int* hist, int remaining, int* misc) {
    const int lane = lane_id();
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
    const int excl = incl - sum;
    if (excl < remaining && remaining <= incl) {
        int acc = excl, dsel = 255 - 8 * lane - 7;
        for (int j = 0; j < 8; ++j) {
            if (acc + c[j] >= remaining) {
                dsel = 255 - 8 * lane - j;
                break;
            }
            acc += c[j];
        }
        misc[0] = dsel;
        misc[1] = remaining - acc;
    }
}

// Threshold key T and the number of keys equal to T to take so that exactly
// `count` (< n) keys are selected: keys > T plus the first keys == T.
__device__ void radix_threshold(const KeySrc& key, int n, int count, uint32_t& thr, int& take_eq,
                                SelShared& sm) {
    const int tid = threadIdx.x;
    for (int i = tid; i < 256; i += blockDim.x) sm.hist[i] = 0;
    if (tid == 0) {
        sm.misc[0] = 0;  // always a valid digit, even if no lane claims one
        sm.misc[1] = 1;
        sm.misc[2] = 0;
    }
    __syncthreads();
    radix_hist(key, n, 0u, 0u, 24, sm.hist);
    __syncthreads();
    if (tid < 32) radix_pick(sm.hist, count, sm.misc);
    __syncthreads();
    uint32_t prefix = uint32_t(sm.misc[0]) << 24, mask = 0xFF000000u;
    int remaining = sm.misc[1];
    const int ncand = sm.hist[sm.misc[0]];
    const bool use_cand = ncand <= kCandCap;
    if (use_cand) {  // keys sharing the top digit
        const int lane = lane_id();
        for (int b = 0; b < n; b += blockDim.x) {
            const int i = b + tid;
            uint32_t k = 0;
            bool m = false;
            if (i < n) {
                k = key(i);
                m = (k & mask) == prefix;
            }
            const unsigned mm = __ballot_sync(0xffffffffu, m);
            int base = 0;
            if (lane == 0 && mm) base = atomicAdd(&sm.misc[2], __popc(mm));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (m) sm.cand_key[base + __popc(mm & lanemask_lt())] = k;
        }
    }
    __syncthreads();
    for (int shift = 16; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) sm.hist[i] = 0;
        __syncthreads();
        if (use_cand)
            radix_hist([&](int i) { return sm.cand_key[i]; }, ncand, prefix, mask, shift, sm.hist);
        else
            radix_hist(key, n, prefix, mask, shift, sm.hist);
        __syncthreads();
        if (tid < 32) radix_pick(sm.hist, remaining, sm.misc);
        __syncthreads();
        prefix |= uint32_t(sm.misc[0]) << shift;
        mask |= 0xFFu << shift;
        remaining = sm.misc[1];
        __syncthreads();
    }
    thr = prefix;
    take_eq = remaining;
}

// Threshold by a 32-way search over the key range with the keys held in
// registers (KPT per thread, n <= KPT * 1024).  Each round splits the live
// range [lo, hi] into 32 buckets of 2^shift keys, counts the keys per bucket
// (per-warp histograms), and keeps the bucket holding the count-th largest
// key; `above` counts the keys beyond the live range.  At most 7 rounds of
// two barriers end with lo == hi == T, take_eq = count - above.
template <int KPT, bool CL>
__device__ void kary_threshold(const uint32_t* keys, int n, int count, uint32_t& thr, int& take_eq,
                               SelShared& sm) {
    namespace cg = cooperative_groups;
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    uint32_t k[KPT];
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int i = tid + j * kSelThreads;
        k[j] = i < n ? keys[i] : 0u;  // 0 sorts below every real key
        if (i < n) {
            kmin = min(kmin, k[j]);
            kmax = max(kmax, k[j]);
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
        sm.wsum[0][warp] = int(kmin ^ 0x80000000u);
        sm.wsum[1][warp] = int(kmax ^ 0x80000000u);
    }
    __syncthreads();
    uint32_t lo = uint32_t(__reduce_min_sync(0xffffffffu, sm.wsum[0][lane])) ^ 0x80000000u;
    uint32_t hi = uint32_t(__reduce_max_sync(0xffffffffu, sm.wsum[1][lane])) ^ 0x80000000u;
    if constexpr (CL) {  // the range over the whole cluster
        cg::cluster_group cluster = cg::this_cluster();
        if (tid == 0) {
            sm.cl_minmax[0] = lo;
            sm.cl_minmax[1] = hi;
        }
        cluster.sync();
        const int nb = int(cluster.num_blocks());
        for (int p = 0; p < nb; ++p) {
            const uint32_t* mm = cluster.map_shared_rank(sm.cl_minmax, p);
            lo = min(lo, mm[0]);
            hi = max(hi, mm[1]);
        }
    }
    int above = 0;
    // per-warp 32-bin histograms: sm.bins[warp][bin]
    for (int i = tid; i < kSelWarps * 32; i += blockDim.x) sm.bins[i >> 5][i & 31] = 0;
    __syncthreads();
    for (int round = 0; lo < hi; ++round) {
        const uint32_t width = hi - lo;
        const int bits = 32 - __clz(width);           // width < 2^bits
        const int shift = bits > 5 ? bits - 5 : 0;    // (width >> shift) < 32
#pragma unroll
        for (int j = 0; j < KPT; ++j)
            if (k[j] >= lo && k[j] <= hi) atomicAdd(&sm.bins[warp][(k[j] - lo) >> shift], 1);
        __syncthreads();
        int c = 0;
        if (warp == 0) {
            for (int w = 0; w < kSelWarps; ++w) {
                c += sm.bins[w][lane];
                sm.bins[w][lane] = 0;  // ready for the next round
            }
            if constexpr (CL) sm.cl_hist[round & 1][lane] = c;
        }
        if constexpr (CL) {  // bucket counts over the whole cluster; the peers decide identically
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            if (warp == 0) {
                c = 0;
                const int nb = int(cluster.num_blocks());
                for (int p = 0; p < nb; ++p) c += cluster.map_shared_rank(&sm.cl_hist[round & 1][0], p)[lane];
            }
        }
        if (warp == 0) {
            // suffix sums from the top bucket down
            int suf = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += y;
            }
            const unsigned ok = __ballot_sync(0xffffffffu, above + suf >= count);
            const int bsel = 31 - __clz(ok);  // highest bucket still holding the threshold
            const int suf_next = __shfl_sync(0xffffffffu, suf, (bsel + 1) & 31);
            if (lane == 0) {
                sm.misc[0] = bsel;
                sm.misc[1] = above + (bsel < 31 ? suf_next : 0);
            }
        }
        __syncthreads();
        const uint32_t b = uint32_t(sm.misc[0]);
        above = sm.misc[1];
        const uint32_t nlo = lo + (b << shift);
        const uint32_t nhi = nlo + ((1u << shift) - 1u);
        lo = nlo;
        hi = nhi < hi ? nhi : hi;
        __syncthreads();
    }
    thr = lo;
    take_eq = count - above;
}

// Keys above / equal to thr per warp-contiguous segment of whole 32-key
// chunks (sm.wsum[0] / [1] per warp); returns after a block barrier.
__device__ void segment_counts(const KeySrc& key, int n, uint32_t thr, SelShared& sm) {
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int seg = ((n + kSelWarps - 1) / kSelWarps + 31) & ~31;
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    int gt = 0, eq = 0;
    for (int i = lo + lane; i < hi; i += 32) {
        const uint32_t k = key(i);
        gt += k > thr;
        eq += k == thr;
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0) {
        sm.wsum[0][warp] = gt;
        sm.wsum[1][warp] = eq;
    }
    __syncthreads();
}

// With segment_counts done: writes out[out_base + j] = map(i) for the keys
// above thr and the first take_eq keys equal to it, in increasing i.
template <class Map>
__device__ void segment_emit(const KeySrc& key, int n, uint32_t thr, int take_eq, int out_base, int32_t* out,
                             Map map, SelShared& sm) {
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int seg = ((n + kSelWarps - 1) / kSelWarps + 31) & ~31;
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    if (warp == 0) {
        // exclusive scans over warps: equal keys before, then selections before
        const int e = sm.wsum[1][lane];
        int ie = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ie, o);
            if (lane >= o) ie += y;
        }
        const int eq_before = ie - e;
        int take = take_eq - eq_before;
        take = take < 0 ? 0 : (take > e ? e : take);
        const int sel = sm.wsum[0][lane] + take;
        int is = sel;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, is, o);
            if (lane >= o) is += y;
        }
        sm.wsum[1][lane] = eq_before;
        sm.wsum[2][lane] = is - sel;
    }
    __syncthreads();
    int eq_run = sm.wsum[1][warp], out_run = out_base + sm.wsum[2][warp];
    const unsigned lt = lanemask_lt();
    constexpr int U = 4;  // chunks whose ballots are in flight together
    for (int b = lo; b < hi; b += 32 * U) {
        uint32_t kk[U];
        bool in[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = b + 32 * u + lane;
            in[u] = i < hi;
            kk[u] = in[u] ? key(i) : 0u;
        }
        unsigned eqm[U];
#pragma unroll
        for (int u = 0; u < U; ++u) eqm[u] = __ballot_sync(0xffffffffu, in[u] && kk[u] == thr);
        unsigned selm[U];
        int er = eq_run;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool is_eq = (eqm[u] >> lane) & 1u;
            const bool sel = (in[u] && kk[u] > thr) || (is_eq && er + __popc(eqm[u] & lt) < take_eq);
            selm[u] = __ballot_sync(0xffffffffu, sel);
            er += __popc(eqm[u]);
        }
        eq_run = er;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if ((selm[u] >> lane) & 1u) out[out_run + __popc(selm[u] & lt)] = map(b + 32 * u + lane);
            out_run += __popc(selm[u]);
        }
    }
}

// Select `count` of n keys and write out[j] = map(i) for the selected i in
// increasing i; pads out[count..pad_to) with -1.
template <class Map>
__device__ void select_compact(const KeySrc& key, int n, int count, int pad_to, int32_t* out,
                               Map map, SelShared& sm) {
    const int tid = threadIdx.x;
    if (count > n) count = n;
    if (count <= 0) {
        for (int i = tid; i < pad_to; i += blockDim.x) out[i] = -1;
        return;
    }
    uint32_t thr = 0;
    int take_eq = n;  // count == n: every key (all are >= 0) is taken
    if (count < n) {
        if (key.s && n <= 8 * kSelThreads)
            kary_threshold<8, false>(key.s, n, count, thr, take_eq, sm);
        else if (key.s && n <= 16 * kSelThreads)
            kary_threshold<16, false>(key.s, n, count, thr, take_eq, sm);
        else if (key.s && n <= 32 * kSelThreads)
            kary_threshold<32, false>(key.s, n, count, thr, take_eq, sm);
        else
            radix_threshold(key, n, count, thr, take_eq, sm);
    }
    segment_counts(key, n, thr, sm);
    segment_emit(key, n, thr, take_eq, 0, out, map, sm);
    for (int i = count + tid; i < pad_to; i += blockDim.x) out[i] = -1;
}

// ---- selection with the keys in registers (n <= KPT * 1024): thread t
// holds keys KPT t .. KPT t + KPT - 1, so warp w holds one contiguous
// segment and the ordered output needs no pass over shared memory.

// Keys of v[KPT t + j] (float_key), 0 past n (below every real key).
template <int KPT>
__device__ __forceinline__ void load_keys(const float* __restrict__ v, int n, uint32_t (&k)[KPT]) {
    static_assert(KPT % 4 == 0, "whole float4s");
    const int base = KPT * int(threadIdx.x);
    if (base + KPT <= n) {  // rows start 16-byte aligned and KPT t is a multiple of 4
        const float4* v4 = reinterpret_cast<const float4*>(v + base);
#pragma unroll
        for (int j = 0; j < KPT / 4; ++j) {
            const float4 x = v4[j];
            k[4 * j] = float_key(x.x);
            k[4 * j + 1] = float_key(x.y);
            k[4 * j + 2] = float_key(x.z);
            k[4 * j + 3] = float_key(x.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < KPT; ++j) k[j] = base + j < n ? float_key(v[base + j]) : 0u;
    }
}

// Threshold rounds of kary_threshold over register-held keys, starting
// from the key range [lo, hi] of the n keys.  Each round the per-warp
// bucket counts are summed by a transposed read (warp w totals bucket w
// over all warps) and every warp takes the bucket decision from the 32
// totals itself: two block barriers per round.  Once the live bucket holds
// at most kSelList keys they are compacted into shared memory and the later
// rounds scan only that list.  sm.tbins must be zero on entry; it is zero
// again on return.
constexpr int kSelList = kCandCap;  // compacted live keys (sm.cand_key)
template <int KPT>
__device__ void kary_regs(const uint32_t (&k)[KPT], uint32_t lo, uint32_t hi, int count, uint32_t& thr,
                          int& take_eq, SelShared& sm) {
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    int above = 0;
    int listed = -1;  // keys in sm.cand_key once compacted
    for (int round = 0; lo < hi; ++round) {
        const uint32_t width = hi - lo;
        const int bits = 32 - __clz(width);
        const int shift = bits > 5 ? bits - 5 : 0;
        if (listed < 0) {
#pragma unroll
            for (int j = 0; j < KPT; ++j)
                if (k[j] >= lo && k[j] <= hi) atomicAdd(&sm.tbins[warp][(k[j] - lo) >> shift], 1);
        } else {
            for (int i = tid; i < listed; i += blockDim.x) {
                const uint32_t x = sm.cand_key[i];
                if (x >= lo && x <= hi) atomicAdd(&sm.tbins[warp][(x - lo) >> shift], 1);
            }
        }
        __syncthreads();
        int c = sm.tbins[lane][warp];  // bucket `warp` of warp `lane`
        sm.tbins[lane][warp] = 0;
        c = __reduce_add_sync(0xffffffffu, c);
        if (lane == 0) sm.ttot[round & 1][warp] = c;
        __syncthreads();
        c = sm.ttot[round & 1][lane];
        int suf = c;  // keys in buckets lane .. 31
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf += y;
        }
        const unsigned ok = __ballot_sync(0xffffffffu, above + suf >= count);
        const int bsel = 31 - __clz(ok);
        const int suf_next = __shfl_sync(0xffffffffu, suf, (bsel + 1) & 31);
        const int live = __shfl_sync(0xffffffffu, c, bsel);
        above += bsel < 31 ? suf_next : 0;
        const uint32_t nlo = lo + (uint32_t(bsel) << shift);
        const uint32_t nhi = nlo + ((1u << shift) - 1u);
        lo = nlo;
        hi = nhi < hi ? nhi : hi;
        if (listed < 0 && lo < hi && live <= kSelList) {  // compact the live keys
            int mine = 0;
#pragma unroll
            for (int j = 0; j < KPT; ++j) mine += k[j] >= lo && k[j] <= hi;
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sm.misc[warp] = incl;
            __syncthreads();
            const int wt = sm.misc[lane];
            int wi = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += y;
            }
            int pos = __shfl_sync(0xffffffffu, wi - wt, warp) + incl - mine;
#pragma unroll
            for (int j = 0; j < KPT; ++j)
                if (k[j] >= lo && k[j] <= hi) sm.cand_key[pos++] = k[j];
            listed = live;
            __syncthreads();
        }
    }
    thr = lo;
    take_eq = count - above;
}

// Select `count` of the n register-held keys (larger first, ties to the
// lower index) and write out[j] = map(i) for the selected i in increasing
// i; pads out[count..pad_to) with -1.  CAP: count is first capped at the
// number of keys above float_key(-inf) (positions that exist score above
// -inf).  before_emit() runs before the block barrier that precedes the
// output (the place to stage what map() reads).  sm.tbins must be zero on
// entry.
template <int KPT, bool CAP, class Map, class Pre>
__device__ void select_regs(const uint32_t (&k)[KPT], int n, int count, int pad_to, int32_t* out, Map map,
                            SelShared& sm, Pre before_emit) {
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const uint32_t neg_inf = float_key(-INFINITY);
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    int nvalid = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        if (KPT * tid + j < n) {
            kmin = min(kmin, k[j]);
            kmax = max(kmax, k[j]);
            nvalid += k[j] > neg_inf;
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    nvalid = __reduce_add_sync(0xffffffffu, nvalid);
    if (lane == 0) {
        sm.wsum[0][warp] = int(kmin ^ 0x80000000u);
        sm.wsum[1][warp] = int(kmax ^ 0x80000000u);
        sm.wsum[2][warp] = nvalid;
    }
    __syncthreads();
    const uint32_t lo = uint32_t(__reduce_min_sync(0xffffffffu, sm.wsum[0][lane])) ^ 0x80000000u;
    const uint32_t hi = uint32_t(__reduce_max_sync(0xffffffffu, sm.wsum[1][lane])) ^ 0x80000000u;
    if (CAP) count = min(count, __reduce_add_sync(0xffffffffu, sm.wsum[2][lane]));
    if (count > n) count = n;
    __syncthreads();  // sm.wsum is reused below
    if (count <= 0) {
        for (int i = tid; i < pad_to; i += blockDim.x) out[i] = -1;
        return;
    }
    uint32_t thr = 0;
    int take_eq = n;  // count == n: every key is taken
    if (count < n) kary_regs<KPT>(k, lo, hi, count, thr, take_eq, sm);
    static_assert(KPT <= 32, "one bit per key");
    uint32_t gt_m = 0, eq_m = 0;  // this thread's keys above / equal to thr
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const bool in = KPT * tid + j < n;
        gt_m |= uint32_t(in && k[j] > thr) << j;
        eq_m |= uint32_t(in && k[j] == thr) << j;
    }
    const int gt = __popc(gt_m), eq = __popc(eq_m);
    int gi = gt, ei = eq;  // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y1 = __shfl_up_sync(0xffffffffu, gi, o);
        const int y2 = __shfl_up_sync(0xffffffffu, ei, o);
        if (lane >= o) {
            gi += y1;
            ei += y2;
        }
    }
    if (lane == 31) {
        sm.wsum[0][warp] = gi;
        sm.wsum[1][warp] = ei;
    }
    before_emit();
    __syncthreads();
    // every warp scans the warp totals: equal keys before each warp, then
    // selections before each warp
    const int e = sm.wsum[1][lane];
    int ie = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) ie += y;
    }
    int tw = take_eq - (ie - e);
    tw = tw < 0 ? 0 : (tw > e ? e : tw);
    const int sw = sm.wsum[0][lane] + tw;
    int is = sw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, is, o);
        if (lane >= o) is += y;
    }
    const int eq_before = __shfl_sync(0xffffffffu, ie - e, warp) + (ei - eq);
    int take = take_eq - eq_before;
    take = take < 0 ? 0 : (take > eq ? eq : take);
    const int sel = gt + take;
    int si = sel;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, si, o);
        if (lane >= o) si += y;
    }
    int pos = __shfl_sync(0xffffffffu, is - sw, warp) + si - sel;
    // the selected keys: all above thr and the first `take` equal to it
    uint32_t sel_m = gt_m;
    for (int t = 0; t < take; ++t) {
        sel_m |= eq_m & (0u - eq_m);  // lowest remaining equal key
        eq_m &= eq_m - 1u;
    }
    while (sel_m) {
        const int j = __ffs(sel_m) - 1;
        sel_m &= sel_m - 1u;
        out[pos++] = map(KPT * tid + j);
    }
    for (int i = count + tid; i < pad_to; i += blockDim.x) out[i] = -1;
}

struct NoStage {
    __device__ __forceinline__ void operator()() const {}
};

struct IdentityMap {
    __device__ __forceinline__ int32_t operator()(int i) const { return i; }
};
struct CandPosMap {
    const int32_t* cand;  // shared-memory copy of the candidate blocks
    __device__ __forceinline__ int32_t operator()(int i) const { return 8 * cand[i >> 3] + (i & 7); }
};

// Top-`count` blocks by block maximum.  grid n_q, 1024 threads; dynamic
// shared memory holds up to smem_keys_cap keys.
__global__ void __launch_bounds__(kSelThreads) select_blocks_kernel(
    const float* __restrict__ blockmax, int64_t nb_stride, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, int64_t n_rows, int count,
    int32_t* __restrict__ out, int64_t out_stride, int smem_keys_cap) {
    extern __shared__ uint32_t smem_keys[];
    __shared__ SelShared sm;
    const int64_t q = blockIdx.x;
    grid_dep_wait();
    grid_dep_launch();
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, nullptr, false);
    const int nb = (n + 7) >> 3;
    const float* v = blockmax + q * nb_stride;
    // up to 16 keys per thread: in registers (rows start 16-byte aligned, nb_stride % 4 == 0)
    for (int i = threadIdx.x; i < kSelWarps * 33; i += blockDim.x) (&sm.tbins[0][0])[i] = 0;
    if (nb <= 8 * kSelThreads) {
        uint32_t k[8];
        load_keys<8>(v, nb, k);
        select_regs<8, false>(k, nb, count, count, out + q * out_stride, IdentityMap{}, sm, NoStage{});
        return;
    }
    if (nb <= 16 * kSelThreads) {
        uint32_t k[16];
        load_keys<16>(v, nb, k);
        select_regs<16, false>(k, nb, count, count, out + q * out_stride, IdentityMap{}, sm, NoStage{});
        return;
    }
    KeySrc key{v, nullptr};
    if (nb <= smem_keys_cap) {  // rows start 16-byte aligned (nb_stride % 4 == 0)
        const float4* v4 = reinterpret_cast<const float4*>(v);
        for (int i = threadIdx.x; i < nb / 4; i += blockDim.x) {
            const float4 x = v4[i];
            smem_keys[4 * i] = float_key(x.x);
            smem_keys[4 * i + 1] = float_key(x.y);
            smem_keys[4 * i + 2] = float_key(x.z);
            smem_keys[4 * i + 3] = float_key(x.w);
        }
        for (int i = (nb & ~3) + threadIdx.x; i < nb; i += blockDim.x) smem_keys[i] = float_key(v[i]);
        key.s = smem_keys;
        __syncthreads();
    }
    select_compact(key, nb, count, count, out + q * out_stride, IdentityMap{}, sm);
}

struct OffsetMap {
    int32_t base;
    __device__ __forceinline__ int32_t operator()(int i) const { return base + i; }
};

// Top-`count` blocks by block maximum for queries with more blocks than one
// CTA stages.  The query's blocks are split over a cluster of G CTAs (rank r
// holds blocks [r S, r S + S), S = seg_keys = 1024 KPT, in shared memory);
// every threshold round sums its bucket counts over the cluster through
// distributed shared memory, and each segment's selections are offset by
// those of the lower ranks, so the output stays ascending.  grid (G, n_q),
// clusters of G along x, 1024 threads.
template <int KPT>
__global__ void __launch_bounds__(kSelThreads) select_blocks_cluster_kernel(
    const float* __restrict__ blockmax, int64_t nb_stride, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, int64_t n_rows, int count,
    int32_t* __restrict__ out, int64_t out_stride, int seg_keys) {
    namespace cg = cooperative_groups;
    extern __shared__ uint32_t smem_keys[];
    __shared__ SelShared sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int64_t q = blockIdx.y;
    const int rank = int(cluster.block_rank());
    grid_dep_wait();
    grid_dep_launch();
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, nullptr, false);
    const int nb = (n + 7) >> 3;
    const int s0 = min(nb, rank * seg_keys), s1 = min(nb, s0 + seg_keys), nl = s1 - s0;
    {  // this segment's keys; s0 is a multiple of 32 and rows start 16-byte aligned
        const float* v = blockmax + q * nb_stride + s0;
        const float4* v4 = reinterpret_cast<const float4*>(v);
        for (int i = tid; i < nl / 4; i += blockDim.x) {
            const float4 x = v4[i];
            smem_keys[4 * i] = float_key(x.x);
            smem_keys[4 * i + 1] = float_key(x.y);
            smem_keys[4 * i + 2] = float_key(x.z);
            smem_keys[4 * i + 3] = float_key(x.w);
        }
        for (int i = (nl & ~3) + tid; i < nl; i += blockDim.x) smem_keys[i] = float_key(v[i]);
    }
    __syncthreads();
    const int cnt = min(count, nb);  // uniform over the cluster (one query)
    int32_t* o = out + q * out_stride;
    if (cnt > 0) {
        uint32_t thr = 0;
        int take_eq = nb;  // cnt == nb: every key is taken
        if (cnt < nb) kary_threshold<KPT, true>(smem_keys, nl, cnt, thr, take_eq, sm);
        const KeySrc key{nullptr, smem_keys};
        segment_counts(key, nl, thr, sm);
        if (warp == 0) {
            const int gt = __reduce_add_sync(0xffffffffu, sm.wsum[0][lane]);
            const int eq = __reduce_add_sync(0xffffffffu, sm.wsum[1][lane]);
            if (lane == 0) {
                sm.cl_cnt[0] = gt;
                sm.cl_cnt[1] = eq;
            }
        }
        cluster.sync();
        if (tid == 0) {  // equal keys and selections in the lower ranks' segments
            int eq_before = 0, out_before = 0;
            for (int p = 0; p < rank; ++p) {
                const int* c = cluster.map_shared_rank(sm.cl_cnt, p);
                const int t = take_eq - eq_before;
                out_before += c[0] + (t < 0 ? 0 : (t > c[1] ? c[1] : t));
                eq_before += c[1];
            }
            sm.misc[2] = take_eq - eq_before;
            sm.misc[3] = out_before;
        }
        __syncthreads();
        segment_emit(key, nl, thr, sm.misc[2], sm.misc[3], o, OffsetMap{s0}, sm);
    }
    if (rank == 0)
        for (int i = cnt + tid; i < count; i += blockDim.x) o[i] = -1;
    cluster.sync();  // the peers have read this CTA's shared memory
}

// Top-`count` positions among the scored candidates.  grid n_q, 1024
// threads; dynamic shared memory: C candidate blocks, then the keys.
__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ cand,
    int64_t cand_stride, int C, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, int32_t max_visible, int64_t n_rows, int count,
    int32_t* __restrict__ out, int64_t out_stride, int smem_keys_cap, const float* __restrict__ pos_scores,
    int64_t pos_stride) {
    extern __shared__ uint32_t smem_dyn[];
    __shared__ SelShared sm;
    int32_t* cblk = reinterpret_cast<int32_t*>(smem_dyn);
    uint32_t* keys = smem_dyn + C;
    const int64_t q = blockIdx.x;
    grid_dep_wait();
    grid_dep_launch();
    const int m = 8 * C;
    const float* v = scores + q * score_stride;
    const int32_t* cq = cand + q * cand_stride;
    constexpr int KR = 16;
    if (m <= KR * kSelThreads) {
        // the candidates' scores in registers (16 per thread; m = 8C: whole
        // float4s, 16-byte aligned rows).  Positions that do not exist score
        // -inf, so the count is capped from the keys themselves, and the
        // candidate ids (at most 2 per thread) are only staged in shared
        // memory for the output
        uint32_t k[KR];
        int32_t cid[2];
        if (pos_scores == nullptr) {
            load_keys<KR>(v, m, k);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = int(threadIdx.x) + r * kSelThreads;
                cid[r] = i < C ? cq[i] : -1;
            }
        } else {
            // keys 16t .. 16t + 15 are the 8 positions of candidates 2t and
            // 2t + 1, read from the scan's per-position scores (rows 16-byte
            // aligned); missing positions score -inf as the pool scorer's do
            const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, nullptr, false);
            const int nb = (n + 7) >> 3;
            const float* ps = pos_scores + q * pos_stride;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int ci = 2 * int(threadIdx.x) + r;
                const int32_t b = ci < C ? cq[ci] : -1;
                float x[8];
                if (b >= 0 && b < nb) {
                    const float4 lo = reinterpret_cast<const float4*>(ps + 8 * int64_t(b))[0];
                    const float4 hi = reinterpret_cast<const float4*>(ps + 8 * int64_t(b))[1];
                    x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
                    x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = -INFINITY;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    k[8 * r + j] = float_key(b >= 0 && b < nb && 8 * b + j < n ? x[j] : -INFINITY);
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = int(threadIdx.x) + r * kSelThreads;
                cid[r] = i < C ? cq[i] : -1;
            }
        }
        for (int i = threadIdx.x; i < kSelWarps * 33; i += blockDim.x) (&sm.tbins[0][0])[i] = 0;
        select_regs<KR, true>(k, m, count, count, out + q * out_stride, CandPosMap{cblk}, sm, [&] {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = int(threadIdx.x) + r * kSelThreads;
                if (i < C) cblk[i] = cid[r];
            }
        });
        return;
    }
    const int32_t n = checked_visible(kv_start, n_visible, q, max_visible, n_rows, nullptr, false);
    const int nb = (n + 7) >> 3;
    int valid = 0;  // positions that exist among the candidates
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        const int32_t b = cq[i];
        cblk[i] = b;
        if (b >= 0 && b < nb) valid += min(8, n - 8 * b);
    }
    for (int o = 16; o > 0; o >>= 1) valid += __shfl_xor_sync(0xffffffffu, valid, o);
    if (lane_id() == 0) sm.misc[threadIdx.x >> 5] = valid;
    __syncthreads();
    int total = 0;
    for (int w = 0; w < kSelWarps; ++w) total += sm.misc[w];
    __syncthreads();
    KeySrc key{v, nullptr};
    if (m <= smem_keys_cap) {  // m = 8C: whole float4s, 16-byte aligned rows
        const float4* v4 = reinterpret_cast<const float4*>(v);
        for (int i = threadIdx.x; i < m / 4; i += blockDim.x) {
            const float4 x = v4[i];
            keys[4 * i] = float_key(x.x);
            keys[4 * i + 1] = float_key(x.y);
            keys[4 * i + 2] = float_key(x.z);
            keys[4 * i + 3] = float_key(x.w);
        }
        key.s = keys;
    }
    __syncthreads();
    select_compact(key, m, min(count, total), count, out + q * out_stride, CandPosMap{cblk}, sm);
}

// Full scan for many queries over shared caches (prefill chunks): a CTA
// takes a group of kMqQ = 4 consecutive queries and a range of 128-position
// K tiles; queries of the group with the same kv_start share each tile in
// one block-scaled MMA (M = 128 positions, N = 32 x queries <= 128), so the
// K tile is read once per group instead of once per query.  The accumulator
// holds one tile (TMEM columns 0..127); the epilogue applies w.ReLU and the
// 8-position block max per query, masking positions past each query's
// visible count.  Queries of a group whose kv_start differs are processed
// as separate runs (the pipeline drains between runs).  Warp 0 streams the
// tiles, warp 1 issues the MMAs, warps 2..17 are the epilogue: warp w reads
// TMEM lane quadrant w % 4 for query (w - 2) / 4 of the run, holding that
// query's w in registers; tile i's scales are staged by the four warps of
// query slot i % 4, which spreads that work over the epilogue (a fixed
// group of stagers had bounded the scan: 9.89 -> 8.26 ms at 4096 x 262,144).
// grid (chunks, ceil(n_q / 4)), 576 threads, one CTA per SM.
constexpr int kMqQ = 4;
constexpr int kMqThreads = 64 + kMqQ * 128;
constexpr int kMqAcc = 2;                         // accumulators (128 TMEM columns each)
constexpr uint32_t kMqCols = 512;
constexpr uint32_t kMqColSfa = 256, kMqColSfb = 288;  // scale slots (4 x 8 columns), query scales (8)

struct MqSmem {
    uint8_t ring[kTcStages * kStageBytes];
    uint8_t qcodes[kMqQ * 32 * 64];  // the run's query heads, BLOCK8 = canonical K-major
    float w[kMqQ * 32];
    int32_t n[kMqQ];
    int64_t ks[kMqQ];
    uint64_t full[kTcStages], empty[kTcStages];
    uint64_t sfa_ready[kTcSf];
    uint64_t acc_full[kMqAcc], acc_empty[kMqAcc], qbar;
    uint32_t tmem;
    int abort_flag;
};

template <bool REC>
__global__ void __launch_bounds__(kMqThreads, 1) scan_mq_kernel(
    const uint8_t* __restrict__ q_codes, const uint8_t* __restrict__ q_scales, const float* __restrict__ w,
    const uint8_t* __restrict__ k_codes, const uint8_t* __restrict__ k_scales, int64_t n_rows,
    const int64_t* __restrict__ kv_start, const int32_t* __restrict__ n_visible, int32_t max_visible, int64_t n_q,
    float* __restrict__ out, int64_t out_stride, Status* st, uint64_t wlim) {
    extern __shared__ __align__(1024) uint8_t mq_smem_raw[];
    MqSmem& S = *reinterpret_cast<MqSmem*>(mq_smem_raw);
    constexpr bool rec = REC;  // indexer K as 576-byte records (k_scales unused)
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int64_t q0 = int64_t(blockIdx.y) * kMqQ;
    const int nqg = int(n_q - q0 < kMqQ ? n_q - q0 : kMqQ);
    grid_dep_wait();
    grid_dep_launch();
    if (tid < kMqQ) {
        const int64_t q = q0 + tid;
        S.n[tid] = tid < nqg ? checked_visible(kv_start, n_visible, q, max_visible, n_rows, st,
                                               blockIdx.x == 0) : 0;
        S.ks[tid] = tid < nqg ? kv_start[q] : -1;
    }
    if (tid < kMqQ * 32) S.w[tid] = tid < nqg * 32 ? __ldg(w + q0 * 32 + tid) : 0.f;
    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int f = 0; f < kTcSf; ++f) mbar_init(&S.sfa_ready[f], 128);
        for (int a = 0; a < kMqAcc; ++a) {
            mbar_init(&S.acc_full[a], 1);
            mbar_init(&S.acc_empty[a], kMqThreads - 64);
        }
        mbar_init(&S.qbar, 1);
        S.abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&S.tmem, kMqCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    const int quad = warp & 3;
    const uint32_t lane_base = tmem + (uint32_t(32 * quad) << 16);
    int it = 0;   // tiles issued so far (ring, slot and accumulator phases)
    // (warp 0 lane 0) tiles whose copies were issued and Q copies; (warp 1
    // lane 0) tiles whose MMAs were issued: what a give-up must wait for
    int issued = 0, q_copies = 0, mma_n = 0;
    int run = 0;  // runs so far (Q phase)
    for (int r0 = 0; r0 < nqg;) {
        int r1 = r0 + 1;  // [r0, r1): queries with the same row range start, and something visible
        while (r1 < nqg && S.ks[r1] == S.ks[r0]) ++r1;
        int nmax = 0;
        for (int j = r0; j < r1; ++j) nmax = max(nmax, S.n[j]);
        const int64_t ks = S.ks[r0];
        const int64_t nblk = (int64_t(nmax) + 7) >> 3, tiles = (nblk + 15) >> 4;
        const int64_t per = (tiles + gridDim.x - 1) / gridDim.x;
        const int64_t t0 = int64_t(blockIdx.x) * per;
        const int64_t t1 = t0 + per < tiles ? t0 + per : tiles;
        const int nr = r1 - r0, ntiles = t0 < t1 ? int(t1 - t0) : 0;
        if (ntiles > 0) {
            if (run > 0) {
                tc_fence_before();
                __syncthreads();  // the previous run has drained (its MMAs and accumulator reads are done)
                tc_fence_after();
            }
            if (S.abort_flag) break;
            if (warp == 0) {  // ---------------------------------- producer
                if (lane == 0) {
                    mbar_arrive_expect_tx(&S.qbar, uint32_t(nr) * 32 * 64);
                    bulk_g2s(S.qcodes, q_codes + ((q0 + r0) * 32 / 8) * 512, uint32_t(nr) * 32 * 64, &S.qbar);
                    ++q_copies;
                    for (int i = 0; i < ntiles; ++i) {
                        const int g = it + i, s = g % kTcStages, rr = g / kTcStages;
                        if (rr > 0 && !mbar_wait(&S.empty[s], (rr - 1) & 1, wlim)) {
                            record(st, CSA2_ERR_TIMEOUT, 20, int32_t(q0 + r0), i);
                            S.abort_flag = 1;
                            break;
                        }
                        const int64_t t = t0 + i;
                        const int64_t nvb64 = nblk - t * 16;
                        const uint32_t nvb = uint32_t(nvb64 < 16 ? nvb64 : 16);
                        mbar_arrive_expect_tx(&S.full[s], nvb * (512 + 64));
                        if (rec) {
                            bulk_g2s(stage_codes<rec>(S.ring, s), k_codes + ((ks >> 3) + t * 16) * 576, nvb * 576,
                                     &S.full[s]);
                        } else {
                            bulk_g2s(stage_codes<rec>(S.ring, s), k_codes + ((ks >> 3) + t * 16) * 512, nvb * 512,
                                     &S.full[s]);
                            bulk_g2s(stage_scales<rec>(S.ring, s, 0), k_scales + (ks + t * kTile) * 8, nvb * 64,
                                     &S.full[s]);
                        }
                        issued = g + 1;
                    }
                }
            } else if (warp == 1) {  // --------------------------- MMA issue
                if (lane == 0) {
                    bool ok = mbar_wait(&S.qbar, run & 1, wlim);
                    const uint32_t id = idesc_mxf4nvf4(128, 32 * nr);
                    const uint32_t qa = smem_u32(S.qcodes);
                    for (int i = 0; ok && i < ntiles; ++i) {
                        const int g = it + i, s = g % kTcStages, f = g % kTcSf;
                        const int a = g % kMqAcc;
                        ok = mbar_wait(&S.full[s], (g / kTcStages) & 1, wlim) && mbar_wait(&S.sfa_ready[f], (g / kTcSf) & 1, wlim) &&
                             (g < kMqAcc || mbar_wait(&S.acc_empty[a], ((g / kMqAcc) - 1) & 1, wlim));
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t ka = smem_u32(stage_codes<rec>(S.ring, s)), sbo = rec ? 576 : 512;
                        const uint32_t d = tmem + 128 * a;
                        const uint32_t sfa = tmem + kMqColSfa + 8 * f, sfb = tmem + kMqColSfb;
                        mma_mxf4_ss(d, umma_desc(ka, 128, sbo), umma_desc(qa, 128, 512), id, sfa, sfb, false);
                        mma_mxf4_ss(d, umma_desc(ka + 256, 128, sbo), umma_desc(qa + 256, 128, 512), id, sfa + 4,
                                    sfb + 4, true);
                        tc_commit(&S.acc_full[a]);
                        tc_commit(&S.empty[s]);
                        mma_n = g + 1;
                    }
                    if (!ok) {
                        record(st, CSA2_ERR_TIMEOUT, 21, int32_t(q0 + r0), 0);
                        S.abort_flag = 1;
                    }
                }
            } else {  // ------------------------------------------ epilogue
                const int row = 32 * quad + lane;
                const int jq = (warp - 2) >> 2;  // this warp's query within the run
                const bool stager = jq == 0;     // warps 2..5 (one per lane quadrant) store the run's query scales
                float wh[32];                    // w / 2 of this warp's query (w relu(x) = w/2 (x + |x|))
#pragma unroll
                for (int h = 0; h < 32; ++h) wh[h] = jq < nr ? 0.5f * S.w[(r0 + jq) * 32 + h] : 0.f;
                if (stager) {  // the run's query scales (B): rows l + 32 i of the run in column i
                    uint2 qs[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int hr = lane + 32 * i;  // head row within the run
                        qs[i] = hr < nr * 32
                                    ? __ldg(reinterpret_cast<const uint2*>(q_scales + ((q0 + r0) * 32 + hr) * 8))
                                    : make_uint2(0u, 0u);
                    }
                    tmem_st4(lane_base + kMqColSfb, qs[0].x, qs[1].x, qs[2].x, qs[3].x);
                    tmem_st4(lane_base + kMqColSfb + 4, qs[0].y, qs[1].y, qs[2].y, qs[3].y);
                }
                auto stage_sf = [&](int i) -> bool {
                    const int g = it + i, s = g % kTcStages, f = g % kTcSf;
                    if (!mbar_wait(&S.full[s], (g / kTcStages) & 1, wlim)) return false;
                    uint2 r4[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        r4[j] = *reinterpret_cast<const uint2*>(stage_scales<rec>(S.ring, s, lane + 32 * j));
                    tmem_st4(lane_base + kMqColSfa + 8 * f, r4[0].x, r4[1].x, r4[2].x, r4[3].x);
                    tmem_st4(lane_base + kMqColSfa + 8 * f + 4, r4[0].y, r4[1].y, r4[2].y, r4[3].y);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&S.sfa_ready[f]);
                    return true;
                };
                bool ok = true;
                // tile i's scales are staged by the warps of query slot i % 4
                for (int i = 0; ok && i < kTcSfLead && i < ntiles; ++i)
                    if (jq == (i & 3)) ok = stage_sf(i);
                const int32_t nj = jq < nr ? S.n[r0 + jq] : 0;
                const int64_t nbj = (int64_t(nj) + 7) >> 3;
                float* outj = out + (q0 + r0 + jq) * out_stride;
                for (int i = 0; ok && i < ntiles; ++i) {
                    if (jq == ((i + kTcSfLead) & 3) && i + kTcSfLead < ntiles) ok = stage_sf(i + kTcSfLead);
                    const int g = it + i, a = g % kMqAcc;
                    if (!ok || !mbar_wait(&S.acc_full[a], (g / kMqAcc) & 1, wlim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t r[32];
                    if (jq < nr) {
                        tmem_ld32(lane_base + 128 * a + 32 * jq, r);
                        tmem_ld_wait();
                    }
                    tc_fence_before();
                    mbar_arrive(&S.acc_empty[a]);  // the accumulator may be overwritten
                    if (jq < nr) {
                        float x0 = 0.f, x1 = 0.f;
#pragma unroll
                        for (int h = 0; h < 32; h += 2) {
                            const float a0 = __uint_as_float(r[h]), a1 = __uint_as_float(r[h + 1]);
                            x0 = fmaf(wh[h], a0 + fabsf(a0), x0);
                            x1 = fmaf(wh[h + 1], a1 + fabsf(a1), x1);
                        }
                        const float x = x0 + x1;
                        const int64_t pos = (t0 + i) * kTile + row;
                        float m = pos < nj ? x : -INFINITY;
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                        const int64_t b = pos >> 3;
                        if ((lane & 7) == 0 && b < nbj) outj[b] = m;
                    }
                }
                if (!ok && lane == 0) {
                    record(st, CSA2_ERR_TIMEOUT, 22, int32_t(q0 + r0), 0);
                    S.abort_flag = 1;
                }
            }
            it += ntiles;
            ++run;
        }
        r0 = r1;
    }
    tc_fence_before();
    __syncthreads();
    if (S.abort_flag) {  // (uniform: nothing writes the flag after the barrier)
        // a wait gave up: wait for the copies and MMAs already issued (the
        // last commit covers every earlier MMA) before anything is released
        if (lane == 0 && warp == 0) {
            if (q_copies > 0) mbar_wait(&S.qbar, (q_copies - 1) & 1, kDrainNs);
            for (int g = issued > kTcStages ? issued - kTcStages : 0; g < issued; ++g)
                mbar_wait(&S.full[g % kTcStages], (g / kTcStages) & 1, kDrainNs);
        } else if (lane == 0 && warp == 1 && mma_n > 0) {
            mbar_wait(&S.empty[(mma_n - 1) % kTcStages], ((mma_n - 1) / kTcStages) & 1, kDrainNs);
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) tmem_dealloc(tmem, kMqCols);
}

// ------------------------------------------------------------ launches
// q_bf16 non-null: the query arrives as bf16 rows (q_codes, q_scales unused)
static csa2_status check_index_args(const uint8_t* q_codes, const uint8_t* q_scales, const void* q_bf16,
                                    const float* w, int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                    int64_t n_rows, const int64_t* kv_start,
                                    const int32_t* n_visible, int32_t max_visible,
                                    int pool_blocks, int topk) {
    if (n_q < 0 || n_rows < 0 || max_visible < 0) return CSA2_ERR_INVALID_ARG;
    // k_scales NULL: k_codes holds 576-byte records (CSA2_LAYOUT_BLOCK8R)
    if (!w || !k_codes || !kv_start || !n_visible) return CSA2_ERR_INVALID_ARG;
    if (q_bf16 != nullptr ? !aligned16(q_bf16)
                          : (!q_codes || !q_scales || !aligned16(q_codes) || !aligned16(q_scales)))
        return CSA2_ERR_INVALID_ARG;
    if (!aligned16(k_codes) || (k_scales && !aligned16(k_scales))) return CSA2_ERR_INVALID_ARG;
    if (n_rows % 8) return CSA2_ERR_UNSUPPORTED;
    if (pool_blocks < 1 || pool_blocks > kMaxPoolBlocks || topk < 1 || topk > kMaxTopk)
        return CSA2_ERR_UNSUPPORTED;
    if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;  // grid.y / grid.x limits of the launches
    return CSA2_OK;
}

// Keys a selection launch stages in shared memory (all n, or none).
static int sel_cap(int64_t n) { return n <= kSelSmemKeys ? int(n) : 0; }

// Opt the selection kernels into their dynamic shared memory (keys plus, for
// the top-k select, the candidate blocks), once per device.
static csa2_status prepare_select_kernels() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
    if (done[dev]) return CSA2_OK;
    const int bytes = (kSelSmemKeys + kMaxPoolBlocks) * 4;
    const int tc = int(sizeof(TcScanSmem)), mq = int(sizeof(MqSmem));
    const auto smem = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (cudaFuncSetAttribute(score_tc_kernel<false, false>, smem, tc) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<false, true>, smem, tc) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<true, false>, smem, tc) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<true, true>, smem, tc) != cudaSuccess ||
        cudaFuncSetAttribute(scan_mq_kernel<false>, smem, mq) != cudaSuccess ||
        cudaFuncSetAttribute(scan_mq_kernel<true>, smem, mq) != cudaSuccess ||
        cudaFuncSetAttribute(select_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(select_blocks_cluster_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             16 * kSelThreads * 4) != cudaSuccess ||
        cudaFuncSetAttribute(select_blocks_cluster_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             32 * kSelThreads * 4) != cudaSuccess)
        return CSA2_ERR_CUDA;
    done[dev] = true;
    return CSA2_OK;
}

// The driver's tensor-map encoder, fetched once (null when unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult res = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &res) !=
                cudaSuccess ||
            res != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return EncodeTiledFn(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// A tensor map over indexer-K records viewed as [n_rows / 8][144] 32-bit
// words with one-row boxes, for the pool gather's four-record TMA gathers.
// False when none can be made; the gather then copies record by record.
static bool records_map(CUtensorMap* m, const uint8_t* k_codes, int64_t n_rows) {
    const int64_t nb = n_rows / 8;
    const EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr || nb <= 0 || nb > INT32_MAX) return false;
    const cuuint64_t dim[2] = {144, cuuint64_t(nb)};
    const cuuint64_t stride[1] = {576};
    const cuuint32_t box[2] = {144, 1}, step[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(k_codes), dim, stride, box, step,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs per query for a tensor-core scorer launch: two resident CTAs per SM
// over the whole batch, at most one per tile.
static int64_t tc_ctas_per_query(int64_t n_q, int64_t tiles_max) {
    int64_t cpq = 2 * int64_t(sm_count()) / n_q;
    return cpq < 1 ? 1 : (cpq > tiles_max ? tiles_max : cpq);
}

// Top-`count` blocks of every query: one CTA per query while a query's
// blocks fit its shared memory, else a cluster of up to 8 CTAs per query
// splitting them (16K or 32K keys each), else one CTA selecting from global
// memory.
constexpr int kSelClusterMax = 8;
static void launch_select_blocks(const float* blockmax, int64_t nb_stride, int64_t n_q,
                                 const int64_t* kv_start, const int32_t* n_visible, int32_t max_visible,
                                 int64_t n_rows, int count, int32_t* out, int64_t out_stride, cudaStream_t s) {
    const int64_t nb_max = ceil_div<int64_t>(max_visible, 8);
    timer_begin(K_SELECT_BLOCKS, s);
    if (nb_max > kSelSmemKeys) {
        const int64_t g16 = ceil_div<int64_t>(nb_max, 16 * kSelThreads);
        const int64_t g32 = ceil_div<int64_t>(nb_max, 32 * kSelThreads);
        if (g16 <= kSelClusterMax) {
            launch(select_blocks_cluster_kernel<16>, dim3(unsigned(g16), unsigned(n_q)), kSelThreads,
                   size_t(16 * kSelThreads) * 4, s, unsigned(g16), blockmax, nb_stride, kv_start, n_visible,
                   max_visible, n_rows, count, out, out_stride, 16 * kSelThreads);
            timer_end(K_SELECT_BLOCKS, s);
            return;
        }
        if (g32 <= kSelClusterMax) {
            launch(select_blocks_cluster_kernel<32>, dim3(unsigned(g32), unsigned(n_q)), kSelThreads,
                   size_t(32 * kSelThreads) * 4, s, unsigned(g32), blockmax, nb_stride, kv_start, n_visible,
                   max_visible, n_rows, count, out, out_stride, 32 * kSelThreads);
            timer_end(K_SELECT_BLOCKS, s);
            return;
        }
    }
    const int cap_b = sel_cap(nb_stride);
    launch(select_blocks_kernel, unsigned(n_q), kSelThreads, size_t(cap_b) * 4, s, 1, blockmax, nb_stride,
           kv_start, n_visible, max_visible, n_rows, count, out, out_stride, cap_b);
    timer_end(K_SELECT_BLOCKS, s);
}

// Per-position scores of the candidate blocks, then their top-k (the pool
// scoring of csa2_index_full and all of csa2_index_reindex).
static void launch_pool_topk(const uint8_t* q_codes, const uint8_t* q_scales, const float* w, int64_t n_q,
                             const uint8_t* k_codes, const uint8_t* k_scales, int64_t n_rows,
                             const int64_t* kv_start, const int32_t* n_visible, int32_t max_visible,
                             const int32_t* cand, int64_t cand_stride, int C, int topk, int32_t* out_topk,
                             float* scores, int64_t score_stride, bool check_cand, Status* st, cudaStream_t s,
                             const float* pos_scores = nullptr, int64_t pos_stride = 0,
                             const uint16_t* q_bf16 = nullptr) {
    // with the scan's per-position scores at hand (pos_scores), the candidates
    // are not scored again: the selection reads their scores from there
    if (pos_scores == nullptr) {
        const int64_t cpq = tc_ctas_per_query(n_q, (C + 15) / 16);
        const dim3 grid(static_cast<unsigned>(cpq), static_cast<unsigned>(n_q));
        CUtensorMap kmap = {};
        const bool use_map = k_scales == nullptr && records_map(&kmap, k_codes, n_rows);
        timer_begin(K_POOL_SCORE, s);
        launch(k_scales == nullptr ? score_tc_kernel<true, true> : score_tc_kernel<true, false>, grid, kTcThreads,
            sizeof(TcScanSmem), s, 1, q_codes, q_scales, w, k_codes, k_scales, n_rows, kv_start, n_visible,
            max_visible, cand, cand_stride, C, scores, score_stride, int(cpq), check_cand, st, nullptr, int64_t(0),
            wait_limit_ns(), kmap, use_map, q_bf16);
        timer_end(K_POOL_SCORE, s);
    }
    const int cap_t = sel_cap(8 * int64_t(C));
    timer_begin(K_SELECT_TOPK, s);
    launch(select_topk_kernel, unsigned(n_q), kSelThreads, size_t(cap_t + C) * 4, s, 1,
        scores, score_stride, cand, cand_stride, C, kv_start, n_visible, max_visible, n_rows, topk, out_topk, topk,
        cap_t, pos_scores, pos_stride);
    timer_end(K_SELECT_TOPK, s);
}

}  // namespace csa2

using namespace csa2;

// csa2_index_full, with the query as FP4 (q_codes, q_scales) or as bf16
// rows (q_bf16): the decode scorers quantize a bf16 query in their
// prologue; the many-query scan reads it quantized into the workspace.
static csa2_status index_full(const uint8_t* q_codes, const uint8_t* q_scales, const uint16_t* q_bf16,
                              const float* w, int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                              int64_t n_rows, const int64_t* kv_start, const int32_t* n_visible,
                              int32_t max_visible, int pool_blocks, int topk, int32_t* out_pool, int32_t* out_topk,
                              void* ws, size_t ws_bytes, csa2_stream_t stream) {
    csa2_status e = check_index_args(q_codes, q_scales, q_bf16, w, n_q, k_codes, k_scales, n_rows, kv_start,
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
    if (q_bf16 != nullptr && n_q >= kMqMinQueries) {
        // the many-query scan shares each query's FP4 operand across CTAs:
        // quantize it once into the workspace, then index as from FP4
        uint8_t* qc = reinterpret_cast<uint8_t*>(base + L.qcodes);
        uint8_t* qs = reinterpret_cast<uint8_t*>(base + L.qscales);
        if ((e = csa2_quantize_append(q_bf16, n_q * 32, 128, CSA2_FMT_FP4, CSA2_LAYOUT_BLOCK8, nullptr, nullptr, 0,
                                      nullptr, n_q * 32, qc, qs, ws, ws_bytes, stream)) != CSA2_OK)
            return e;
        q_codes = qc;
        q_scales = qs;
        q_bf16 = nullptr;
    }
    if (max_visible > 0 && n_q >= kMqMinQueries) {
        // many queries: groups of 4 share each K tile; about 8 waves of one CTA per SM
        const int64_t groups = ceil_div<int64_t>(n_q, kMqQ);
        const int64_t tiles = ceil_div<int64_t>(max_visible, kTile);
        int64_t chunks = ceil_div<int64_t>(8 * int64_t(sm_count()), groups);
        chunks = chunks < 1 ? 1 : (chunks > tiles ? tiles : chunks);
        timer_begin(K_SCAN, s);
        launch(k_scales == nullptr ? scan_mq_kernel<true> : scan_mq_kernel<false>,
               dim3(unsigned(chunks), unsigned(groups)), kMqThreads, sizeof(MqSmem), s, 1, q_codes,
               q_scales, w, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible, n_q, blockmax, L.nb_stride,
               st, wait_limit_ns());
        timer_end(K_SCAN, s);
    } else if (max_visible > 0) {
        const int64_t cpq = tc_ctas_per_query(n_q, ceil_div<int64_t>(max_visible, kTile));
        const dim3 grid(static_cast<unsigned>(cpq), static_cast<unsigned>(n_q));
        timer_begin(K_SCAN, s);
        launch(k_scales == nullptr ? score_tc_kernel<false, true> : score_tc_kernel<false, false>, grid,
            kTcThreads, sizeof(TcScanSmem), s, 1,
            q_codes, q_scales, w, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible, nullptr, 0,
            (n_q <= kScanMaxQ && n_q <= sm_count()) ? int(n_q) : 0, blockmax, L.nb_stride, int(cpq), false, st,
            L.pos_stride ? reinterpret_cast<float*>(base + L.pos) : nullptr, L.pos_stride, wait_limit_ns(),
            CUtensorMap{}, false, q_bf16);
        timer_end(K_SCAN, s);
    }
    launch_select_blocks(blockmax, L.nb_stride, n_q, kv_start, n_visible, max_visible, n_rows, pool_blocks,
                         out_pool, pool_blocks, s);
    const int32_t* cand = out_pool;
    int64_t cand_stride = pool_blocks;
    if (topk > pool_blocks) {
        // the top-k positions lie in the top-max(P, K) blocks
        int32_t* wide = reinterpret_cast<int32_t*>(base + L.cand);
        launch_select_blocks(blockmax, L.nb_stride, n_q, kv_start, n_visible, max_visible, n_rows, topk, wide,
                             topk, s);
        cand = wide;
        cand_stride = topk;
    }
    launch_pool_topk(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible, cand,
                     cand_stride, C, topk, out_topk, scores, L.score_stride, false, st, s,
                     L.pos_stride && max_visible > 0 ? reinterpret_cast<const float*>(base + L.pos) : nullptr,
                     L.pos_stride, q_bf16);
    return launch_status();
}

extern "C" csa2_status csa2_index_full(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                       int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                       int64_t n_rows, const int64_t* kv_start,
                                       const int32_t* n_visible, int32_t max_visible,
                                       int pool_blocks, int topk, int32_t* out_pool,
                                       int32_t* out_topk, void* ws, size_t ws_bytes,
                                       csa2_stream_t stream) {
    return index_full(q_codes, q_scales, nullptr, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible,
                      max_visible, pool_blocks, topk, out_pool, out_topk, ws, ws_bytes, stream);
}

extern "C" csa2_status csa2_index_full_bf16(const void* q_bf16, const float* w, int64_t n_q,
                                            const uint8_t* k_codes, const uint8_t* k_scales, int64_t n_rows,
                                            const int64_t* kv_start, const int32_t* n_visible,
                                            int32_t max_visible, int pool_blocks, int topk, int32_t* out_pool,
                                            int32_t* out_topk, void* ws, size_t ws_bytes,
                                            csa2_stream_t stream) {
    if (!q_bf16) return CSA2_ERR_INVALID_ARG;
    return index_full(nullptr, nullptr, static_cast<const uint16_t*>(q_bf16), w, n_q, k_codes, k_scales, n_rows,
                      kv_start, n_visible, max_visible, pool_blocks, topk, out_pool, out_topk, ws, ws_bytes,
                      stream);
}

// csa2_index_reindex with the query as FP4 or (q_bf16) as bf16 rows,
// quantized by the pool scorer's prologue
static csa2_status index_reindex(const uint8_t* q_codes, const uint8_t* q_scales, const uint16_t* q_bf16,
                                 const float* w, int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                 int64_t n_rows, const int64_t* kv_start, const int32_t* n_visible,
                                 int32_t max_visible, const int32_t* pool, int pool_blocks, int topk,
                                 int32_t* out_topk, void* ws, size_t ws_bytes, csa2_stream_t stream) {
    csa2_status e = check_index_args(q_codes, q_scales, q_bf16, w, n_q, k_codes, k_scales, n_rows, kv_start,
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
    launch_pool_topk(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible, pool,
                     pool_blocks, pool_blocks, topk, out_topk, scores, L.score_stride, true, st, s, nullptr, 0,
                     q_bf16);
    return launch_status();
}

extern "C" csa2_status csa2_index_reindex(const uint8_t* q_codes, const uint8_t* q_scales,
                                          const float* w, int64_t n_q, const uint8_t* k_codes,
                                          const uint8_t* k_scales, int64_t n_rows,
                                          const int64_t* kv_start, const int32_t* n_visible,
                                          int32_t max_visible, const int32_t* pool, int pool_blocks,
                                          int topk, int32_t* out_topk, void* ws, size_t ws_bytes,
                                          csa2_stream_t stream) {
    return index_reindex(q_codes, q_scales, nullptr, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible,
                         max_visible, pool, pool_blocks, topk, out_topk, ws, ws_bytes, stream);
}

extern "C" csa2_status csa2_index_reindex_bf16(const void* q_bf16, const float* w, int64_t n_q,
                                               const uint8_t* k_codes, const uint8_t* k_scales, int64_t n_rows,
                                               const int64_t* kv_start, const int32_t* n_visible,
                                               int32_t max_visible, const int32_t* pool, int pool_blocks, int topk,
                                               int32_t* out_topk, void* ws, size_t ws_bytes,
                                               csa2_stream_t stream) {
    if (!q_bf16) return CSA2_ERR_INVALID_ARG;
    return index_reindex(nullptr, nullptr, static_cast<const uint16_t*>(q_bf16), w, n_q, k_codes, k_scales, n_rows,
                         kv_start, n_visible, max_visible, pool, pool_blocks, topk, out_topk, ws, ws_bytes, stream);
}

// ------------------------------------------------------------ no-allocation variant
// csa2_index_reindex for callers that cannot allocate device memory (an
// allocator-less runtime, a caller whose memory budget is fixed up front, or
// code running where cudaMalloc is not allowed).  The per-position score
// scratch lives in a fixed library-owned device array instead of a
// caller-provided workspace.
namespace csa2 {
constexpr int64_t kNoallocScoreFloats = int64_t(512) * 1024;  // 2 MiB of fp32 scores
static __device__ __align__(256) float g_noalloc_scores[kNoallocScoreFloats];
static float* g_noalloc_ptr[64] = {};  // device address of g_noalloc_scores, per device
}  // namespace csa2

extern "C" csa2_status csa2_index_reindex_noalloc(const uint8_t* q_codes, const uint8_t* q_scales,
                                                  const float* w, int64_t n_q, const uint8_t* k_codes,
                                                  const uint8_t* k_scales, int64_t n_rows,
                                                  const int64_t* kv_start, const int32_t* n_visible,
                                                  int32_t max_visible, const int32_t* pool,
                                                  int pool_blocks, int topk, int32_t* out_topk,
                                                  int32_t* status, csa2_stream_t stream) {
    csa2_status e = check_index_args(q_codes, q_scales, nullptr, w, n_q, k_codes, k_scales, n_rows, kv_start,
                                     n_visible, max_visible, pool_blocks, topk);
    if (e != CSA2_OK) return e;
    if (!pool || !out_topk) return CSA2_ERR_INVALID_ARG;
    if (status && (reinterpret_cast<uintptr_t>(status) & 3)) return CSA2_ERR_INVALID_ARG;
    if (n_q * 8 * int64_t(pool_blocks) > kNoallocScoreFloats) return CSA2_ERR_UNSUPPORTED;
    if (n_q == 0) return CSA2_OK;
    if ((e = prepare_select_kernels()) != CSA2_OK) return e;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
    if (g_noalloc_ptr[dev] == nullptr) {  // first call on this device: resolve the array's address
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scores) != cudaSuccess || p == nullptr) return CSA2_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    float* scores = g_noalloc_ptr[dev];
    const int64_t stride = 8 * int64_t(pool_blocks);
    Status* st = reinterpret_cast<Status*>(status);
    cudaStream_t s = cudaStream_t(stream);
    launch_pool_topk(q_codes, q_scales, w, n_q, k_codes, k_scales, n_rows, kv_start, n_visible, max_visible, pool,
                     pool_blocks, pool_blocks, topk, out_topk, scores, stride, true, st, s);
    return launch_status();
}
