// Sparse attention over the selected FP4 latents plus the FP8 window, with
// one merged softmax.
//
// [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", §二: main
// attention has 64 heads of dim 512 over one shared latent per entry, each
// layer keeps its own query and window KV; [T3] "DeepSeek-V4.1-Flash：全局 KV
// 仅 890 B/token，百万上下文怎么做成的？", 第三刀: the FP4 main KV is dequantized
// before attention and the window KV stays FP8.
//
// Split-K over entries: CTA (split, query) takes E entries (E in 16..80,
// chosen per launch so the grid fills whole waves of one CTA per SM), gathers
// and dequantizes them into shared memory (exact in bf16), computes
// S = Q C^T (bf16 MMA, fp32 accumulate), the split's softmax statistics
// (m, l), and O_s = P C with P split into f16 hi + lo parts (C converted in
// place to f16, still exact), so the partial output carries ~2^-22 relative
// error.  When a query's splits fit one thread-block cluster (<= 8 CTAs) the
// splits merge through distributed shared memory: each CTA keeps its partial
// for half the dims at a time in its own shared memory and reduces one slice
// of the dims over all peers.  Otherwise partials go to the workspace and a
// merge kernel combines them.  Either way the result is rounded once, to
// fp32 or bf16.
//
// Optionally the kernel also appends the current token's window latent: the
// bf16 row for position n-1 is rounded to E4M3 (as csa2_quantize_append FP8
// does), written to its ring slot, and used for that entry.
#include "csa2_common.cuh"
#include "csa2_timer.cuh"
#include "csa2_layout.cuh"

#include <cfloat>

#include <cooperative_groups.h>

namespace csa2 {

constexpr int kAttnThreads = 256;
constexpr int kH = CSA2_ATTN_HEADS;
constexpr int kD = CSA2_LATENT_DIM;

template <int E>
struct AttnSmem {
    static constexpr int kSStride = E + 4;   // fp32 S row stride
    static constexpr int kPStride = E + 8;   // f16 P row stride (16-byte multiple)
    uint4 q[kH * kD / 8];          // bf16 [64][512], 16-byte chunks swizzled
    uint4 c[E * kD / 8];           // bf16 then f16 [E][512], swizzled
    float s[kH * kSStride];
    __half p_hi[kH * kPStride];
    __half p_lo[kH * kPStride];
    uint32_t lut4[256];            // E2M1 pair -> bf16x2 (unscaled)
    uint16_t lut8[256];            // E4M3 byte -> bf16
    int ok[E];                     // entry valid
    float ml[kH][2];               // this split's (m, l) per head
    float wts[kH][16];             // merge weights a_s / L per head and split
};

// byte offset of 16-byte chunk c of row r in a [rows][512] 16-bit tile
__device__ __forceinline__ uint32_t swz(int r, int c) { return uint32_t(r * 1024 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint16_t bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// grid (splits, n_q), 256 threads.  Writes the split's unnormalized partial
// O_s = sum_j exp(l_j - m_s) c_j (fp32 [64][512]) and (m_s, l_s) per head.
template <int E, bool CLUSTER>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(
    const uint16_t* __restrict__ qg, const uint8_t* __restrict__ kv_codes,
    const uint8_t* __restrict__ kv_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, const int32_t* __restrict__ topk, int k,
    uint8_t* __restrict__ swa, const uint16_t* __restrict__ swa_new, int window, float sm_scale,
    float* __restrict__ part_o, float* __restrict__ part_ml, int splits, void* __restrict__ out,
    bool out_f32, float* __restrict__ out_lse, Status* st) {
    using Sm = AttnSmem<E>;
    constexpr int kSStride = Sm::kSStride, kPStride = Sm::kPStride;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Sm& S = *reinterpret_cast<Sm*>(smem_raw);
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int split = blockIdx.x;
    const int64_t q = blockIdx.y;

    // Q (bf16 [64][512]) into swizzled shared memory, asynchronously
    const uint16_t* qsrc = qg + q * (kH * kD);
    for (int i = tid; i < kH * kD / 8; i += kAttnThreads) {
        const int r = i >> 6, c = i & 63;
        cp_async16(smem_addr(reinterpret_cast<uint8_t*>(S.q) + swz(r, c)), qsrc + r * kD + c * 8);
    }
    // tables: E2M1 pair -> bf16x2, E4M3 -> bf16 (exact)
    {
        const int b = tid;
        const float e2m1[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        const float lo = (b & 8 ? -1.f : 1.f) * e2m1[b & 7];
        const float hi = (b & 128 ? -1.f : 1.f) * e2m1[(b >> 4) & 7];
        S.lut4[b] = uint32_t(bf16_bits(lo)) | (uint32_t(bf16_bits(hi)) << 16);
        S.lut8[b] = bf16_bits(e4m3_value(uint32_t(b)));
    }
    // per-query validity (reported once per query)
    int32_t n = 0;
    const int64_t ks = kv_start[q];
    {
        const int32_t nv = n_visible[q];
        const bool report = split == 0 && tid == 0;
        if (ks < 0) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_KV_START, int32_t(q), int32_t(ks));
        } else if (nv < 0 || ks + nv > n_rows) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_ROWS, int32_t(q), nv);
        } else {
            n = nv;
        }
    }
    const int nw = n < window ? n : window;
    __syncthreads();  // tables ready

    // gather + dequantize: item -> (entry e = item/4, quarter qq = item%4)
    uint8_t* crow = reinterpret_cast<uint8_t*>(S.c);
    for (int item = tid; item < E * 4; item += kAttnThreads) {
        const int e = item >> 2, qq = item & 3;
        const int ge = split * E + e;
        bool ok = false;
        if (ge < k) {
            const int32_t p = topk[q * k + ge];
            if (p >= 0 && p < n) {
                ok = true;
                const int64_t row = ks + p;
                const uint4* src = reinterpret_cast<const uint4*>(kv_codes + row * 256 + qq * 64);
                const uint2 sc = __ldg(reinterpret_cast<const uint2*>(kv_scales + row * 32 + qq * 8));
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = __ldg(src + j);
                const uint32_t scw[2] = {sc.x, sc.y};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // groups 2j, 2j+1 of this quarter
                        const uint32_t sb = (scw[(2 * j + h) >> 2] >> (8 * ((2 * j + h) & 3))) & 0xFF;
                        const uint32_t s16 = S.lut8[sb];
                        const uint32_t s2 = s16 | (s16 << 16);
                        uint32_t outw[8];
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const uint32_t w = wv[2 * h + m];
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb)
                                outw[4 * m + bb] = bf16x2_mul(S.lut4[(w >> (8 * bb)) & 0xFF], s2);
                        }
                        const int chunk = qq * 16 + 4 * j + 2 * h;
                        *reinterpret_cast<uint4*>(crow + swz(e, chunk)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
                        *reinterpret_cast<uint4*>(crow + swz(e, chunk + 1)) = make_uint4(outw[4], outw[5], outw[6], outw[7]);
                    }
                }
            } else if (p < -1 || p >= n) {
                if (qq == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_TOPK, int32_t(q), p);
            }
        } else if (ge - k < nw) {
            ok = true;
            const int64_t pos = int64_t(n - nw) + (ge - k);
            const int64_t slot = pos % window;
            uint8_t* ring = swa + (q * window + slot) * kD + qq * 128;
            uint4 v[8];
            if (swa_new != nullptr && pos == n - 1) {
                // current token: E4M3 of its bf16 latent, stored to the ring and used here
                const uint4* src = reinterpret_cast<const uint4*>(swa_new + q * kD + qq * 128);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 a = __ldg(src + 2 * j), b = __ldg(src + 2 * j + 1);
                    const uint32_t w8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                    uint32_t o4[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        o4[m] = e4m3x2_rn_sat(bf16_lo(w8[2 * m]), bf16_hi(w8[2 * m])) |
                                (e4m3x2_rn_sat(bf16_lo(w8[2 * m + 1]), bf16_hi(w8[2 * m + 1])) << 16);
                    v[j] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                    reinterpret_cast<uint4*>(ring)[j] = v[j];
                }
            } else {
                const uint4* src = reinterpret_cast<const uint4*>(ring);
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = src[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                uint32_t outw[8];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t w = wv[m];
                    outw[2 * m] = uint32_t(S.lut8[w & 0xFF]) | (uint32_t(S.lut8[(w >> 8) & 0xFF]) << 16);
                    outw[2 * m + 1] = uint32_t(S.lut8[(w >> 16) & 0xFF]) | (uint32_t(S.lut8[w >> 24]) << 16);
                }
                const int chunk = qq * 16 + 2 * j;
                *reinterpret_cast<uint4*>(crow + swz(e, chunk)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
                *reinterpret_cast<uint4*>(crow + swz(e, chunk + 1)) = make_uint4(outw[4], outw[5], outw[6], outw[7]);
            }
        }
        if (!ok) {
            for (int c = qq * 16; c < qq * 16 + 16; ++c)
                *reinterpret_cast<uint4*>(crow + swz(e, c)) = make_uint4(0, 0, 0, 0);
        }
        if (qq == 0) S.ok[e] = ok;
    }
    cp_async_wait_all();
    __syncthreads();

    // S = Q C^T: warp -> heads 16*(warp%4).., entry groups of 16: eh, eh+2, ...
    const int hg = warp & 3, eh = warp >> 2;
    {
        constexpr int G = E / 16;             // entry groups
        constexpr int GW = (G + 1) / 2;       // groups per warp (at most)
        float acc[GW][2][4];
#pragma unroll
        for (int g = 0; g < GW; ++g)
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[g][j][0] = acc[g][j][1] = acc[g][j][2] = acc[g][j][3] = 0.f;
        const uint32_t qb = smem_addr(S.q), cb = smem_addr(S.c);
        const int arow = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll 2
        for (int kk = 0; kk < kD / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(qb + swz(arow, 2 * kk + (lane >> 4)), a);
#pragma unroll
            for (int g = 0; g < GW; ++g) {
                const int grp = eh + 2 * g;
                if (grp < G) {
                    uint32_t b[4];
                    const int brow = 16 * grp + (lane & 7) + 8 * (lane >> 4);
                    ldsm_x4(cb + swz(brow, 2 * kk + ((lane >> 3) & 1)), b);
                    mma_bf16(acc[g][0], a, b[0], b[1]);
                    mma_bf16(acc[g][1], a, b[2], b[3]);
                }
            }
        }
        const int r = 16 * hg + (lane >> 2);
#pragma unroll
        for (int g = 0; g < GW; ++g) {
            const int grp = eh + 2 * g;
            if (grp < G) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = 16 * grp + 8 * j + 2 * (lane & 3);
                    S.s[r * kSStride + c] = acc[g][j][0];
                    S.s[r * kSStride + c + 1] = acc[g][j][1];
                    S.s[(r + 8) * kSStride + c] = acc[g][j][2];
                    S.s[(r + 8) * kSStride + c + 1] = acc[g][j][3];
                }
            }
        }
    }
    __syncthreads();

    // softmax statistics of this split: thread -> (head tid/4, entries c, c+4, ...)
    {
        constexpr int PER = E / 4;
        const int h = tid >> 2, c0 = tid & 3;
        float x[PER], m = -INFINITY;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int c = c0 + 4 * j;
            x[j] = S.ok[c] ? sm_scale * S.s[h * kSStride + c] : -INFINITY;
            m = fmaxf(m, x[j]);
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int c = c0 + 4 * j;
            const float p = x[j] == -INFINITY ? 0.f : expf(x[j] - m);
            l += p;
            const __half hi = __float2half_rn(p);
            S.p_hi[h * kPStride + c] = hi;
            S.p_lo[h * kPStride + c] = __float2half_rn(p - __half2float(hi));
        }
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (c0 == 0) {
            if (CLUSTER) {
                S.ml[h][0] = m;
                S.ml[h][1] = l;
            } else {
                float* ml = part_ml + ((q * splits + split) * kH + h) * 2;
                ml[0] = m;
                ml[1] = l;
            }
        }
    }
    // C from bf16 to f16 in place (exact for FP4 and E4M3 values)
    {
        uint32_t* cw = reinterpret_cast<uint32_t*>(S.c);
        for (int i = tid; i < E * kD / 2; i += kAttnThreads) {
            const uint32_t v = cw[i];
            const __half2 h = __floats2half2_rn(bf16_lo(v), bf16_hi(v));
            cw[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    __syncthreads();

    // O_s = P C in two halves of 256 dims: warp -> heads 16*hg.., dims
    // 256*half + 128*(warp/4) .. +128
    {
        const int dh = warp >> 2;
        const uint32_t ph = smem_addr(S.p_hi), pl = smem_addr(S.p_lo), cb = smem_addr(S.c);
        const int arow = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1);
        float* part = part_o + (q * splits + split) * int64_t(kH * kD);
        float* X = reinterpret_cast<float*>(S.q);  // [64][256] fp32 (Q is no longer needed)
        for (int half = 0; half < 2; ++half) {
            const int d0 = 256 * half + 128 * dh;  // first dim of this warp's slice
            float acc[16][4];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
            for (int kq = 0; kq < E / 16; ++kq) {
                uint32_t ahi[4], alo[4];
                const uint32_t aoff = uint32_t((arow * kPStride + 16 * kq + 8 * (lane >> 4)) * 2);
                ldsm_x4(ph + aoff, ahi);
                ldsm_x4(pl + aoff, alo);
                const int erow = 16 * kq + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    uint32_t b[4];
                    ldsm_x4_t(cb + swz(erow, (d0 >> 3) + j + (lane >> 4)), b);
                    mma_f16(acc[j], ahi, b[0], b[1]);
                    mma_f16(acc[j], alo, b[0], b[1]);
                    mma_f16(acc[j + 1], ahi, b[2], b[3]);
                    mma_f16(acc[j + 1], alo, b[2], b[3]);
                }
            }
            const int r = 16 * hg + (lane >> 2);
            if (!CLUSTER) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = d0 + 8 * j + 2 * (lane & 3);
                    *reinterpret_cast<float2*>(part + r * kD + c) = make_float2(acc[j][0], acc[j][1]);
                    *reinterpret_cast<float2*>(part + (r + 8) * kD + c) = make_float2(acc[j][2], acc[j][3]);
                }
                continue;
            }
            namespace cg = cooperative_groups;
            cg::cluster_group cluster = cg::this_cluster();
            if (half == 1) cluster.sync();  // peers finished reading the first half
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int c = d0 - 256 * half + 8 * j + 2 * (lane & 3);
                *reinterpret_cast<float2*>(X + r * 256 + c) = make_float2(acc[j][0], acc[j][1]);
                *reinterpret_cast<float2*>(X + (r + 8) * 256 + c) = make_float2(acc[j][2], acc[j][3]);
            }
            cluster.sync();  // every partial of this half (and every (m, l)) is visible
            const int rank = int(cluster.block_rank());
            if (half == 0 && tid < kH) {
                // merge weights of head tid over the splits
                float M = -INFINITY;
                for (int p = 0; p < splits; ++p) {
                    const float* pml = cluster.map_shared_rank(&S.ml[0][0], p);
                    M = fmaxf(M, pml[tid * 2]);
                }
                float L = 0.f, a[16];
                for (int p = 0; p < splits; ++p) {
                    const float* pml = cluster.map_shared_rank(&S.ml[0][0], p);
                    const float mp = pml[tid * 2];
                    a[p] = (M == -INFINITY || mp == -INFINITY) ? 0.f : expf(mp - M);
                    L = fmaf(a[p], pml[tid * 2 + 1], L);
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
                for (int p = 0; p < splits; ++p) S.wts[tid][p] = a[p] * inv;
                if (rank == 0 && out_lse) out_lse[q * kH + tid] = L > 0.f ? M + logf(L) : -INFINITY;
            }
            __syncthreads();
            // this CTA reduces dims [lo, hi) of the half over all peers
            const int per = (256 + splits - 1) / splits;
            const int lo = rank * per, hi = min(256, lo + per);
            const int width = hi - lo;
            for (int idx = tid; idx < kH * width; idx += kAttnThreads) {
                const int h = idx / width, d = lo + idx % width;
                float o = 0.f;
                for (int p = 0; p < splits; ++p) {
                    const float* px = cluster.map_shared_rank(X, p);
                    o = fmaf(S.wts[h][p], px[h * 256 + d], o);
                }
                const int64_t oi = (q * kH + h) * int64_t(kD) + 256 * half + d;
                if (out_f32) static_cast<float*>(out)[oi] = o;
                else static_cast<uint16_t*>(out)[oi] = bf16_bits(o);
            }
        }
        if (CLUSTER) cooperative_groups::this_cluster().sync();  // peers done with our shared memory
    }
}

// grid (n_q, 8): one warp per head (8 heads per CTA), 16 dims per lane.  The
// split statistics are loaded by the lanes in parallel and the partial rows
// of four splits are in flight at a time.
template <bool F32>
__global__ void __launch_bounds__(256) attn_merge_kernel(const float* __restrict__ part_o,
                                                         const float* __restrict__ part_ml, int splits,
                                                         void* __restrict__ out, float* __restrict__ lse) {
    const int64_t q = blockIdx.x;
    const int h = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int lane = lane_id();
    // lane s < splits holds split s's (m, l); at most 128 splits
    float M = -INFINITY, ms[4], ls[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int s = lane + 32 * r;
        ms[r] = -INFINITY;
        ls[r] = 0.f;
        if (s < splits) {
            const float2 v = *reinterpret_cast<const float2*>(part_ml + ((q * splits + s) * kH + h) * 2);
            ms[r] = v.x;
            ls[r] = v.y;
        }
        M = fmaxf(M, ms[r]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float a[4], L = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        a[r] = (M == -INFINITY || ms[r] == -INFINITY) ? 0.f : expf(ms[r] - M);
        L = fmaf(a[r], ls[r], L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    const int64_t sstride = int64_t(kH) * kD / 4;  // float4 per split
    const float4* base = reinterpret_cast<const float4*>(part_o) + (q * splits * kH + h) * int64_t(kD / 4);
    for (int s0 = 0; s0 < splits; s0 += 4) {
        float4 v[4][4];
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int s = s0 + u;
            const int r = (s >> 5) & 3;
            float wr = 0.f;
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float t = __shfl_sync(0xffffffffu, a[rr], s & 31);
                if (rr == r) wr = t;
            }
            w[u] = s < splits ? wr : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[u][j] = w[u] != 0.f ? base[s * sstride + lane + 32 * j] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[4 * j] = fmaf(w[u], v[u][j].x, acc[4 * j]);
                acc[4 * j + 1] = fmaf(w[u], v[u][j].y, acc[4 * j + 1]);
                acc[4 * j + 2] = fmaf(w[u], v[u][j].z, acc[4 * j + 2]);
                acc[4 * j + 3] = fmaf(w[u], v[u][j].w, acc[4 * j + 3]);
            }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int d = 4 * (lane + 32 * j);
        if (F32) {
            float* o = static_cast<float*>(out) + (q * kH + h) * int64_t(kD);
            *reinterpret_cast<float4*>(o + d) =
                make_float4(acc[4 * j] * inv, acc[4 * j + 1] * inv, acc[4 * j + 2] * inv, acc[4 * j + 3] * inv);
        } else {
            uint16_t* o = static_cast<uint16_t*>(out) + (q * kH + h) * int64_t(kD);
            const uint32_t lo = uint32_t(bf16_bits(acc[4 * j] * inv)) | (uint32_t(bf16_bits(acc[4 * j + 1] * inv)) << 16);
            const uint32_t hi = uint32_t(bf16_bits(acc[4 * j + 2] * inv)) | (uint32_t(bf16_bits(acc[4 * j + 3] * inv)) << 16);
            *reinterpret_cast<uint2*>(o + d) = make_uint2(lo, hi);
        }
    }
    if (lse && lane == 0) lse[q * kH + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

template <int E, bool CLUSTER>
static csa2_status launch_split(dim3 grid, cudaStream_t s, const uint16_t* q, const uint8_t* kv_codes,
                                const uint8_t* kv_scales, int64_t n_rows, const int64_t* kv_start,
                                const int32_t* n_visible, const int32_t* topk, int k, uint8_t* swa,
                                const uint16_t* swa_new, int window, float sm_scale, float* part_o,
                                float* part_ml, int splits, void* out, bool out_f32, float* out_lse,
                                Status* st) {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(attn_split_kernel<E, CLUSTER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnSmem<E>))) != cudaSuccess)
            return CSA2_ERR_CUDA;
        done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(AttnSmem<E>);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (CLUSTER) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = grid.x;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    timer_begin(K_ATTN_SPLIT, s);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_split_kernel<E, CLUSTER>, q, kv_codes, kv_scales, n_rows,
                                             kv_start, n_visible, topk, k, swa, swa_new, window, sm_scale,
                                             part_o, part_ml, splits, out, out_f32, out_lse, st);
    timer_end(K_ATTN_SPLIT, s);
    return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_sparse_attn(const void* q_bf16, int64_t n_q, const uint8_t* kv_codes,
                                        const uint8_t* kv_scales, int64_t n_rows,
                                        const int64_t* kv_start, const int32_t* n_visible,
                                        const int32_t* topk, int k, uint8_t* swa,
                                        const void* swa_new_bf16, int window, float sm_scale, void* out,
                                        int out_dtype, float* out_lse, void* ws, size_t ws_bytes,
                                        csa2_stream_t stream) {
    if (n_q < 0 || n_rows < 0 || k < 0 || k > kMaxTopk || window < 0 || window > kMaxWindow)
        return CSA2_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || !(sm_scale < FLT_MAX)) return CSA2_ERR_INVALID_ARG;
    if (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32) return CSA2_ERR_INVALID_ARG;
    if (!q_bf16 || !kv_codes || !kv_scales || !kv_start || !n_visible || !out) return CSA2_ERR_INVALID_ARG;
    if (k > 0 && !topk) return CSA2_ERR_INVALID_ARG;
    if (window > 0 && !swa) return CSA2_ERR_INVALID_ARG;
    if (swa_new_bf16 && (window == 0 || !aligned16(swa_new_bf16))) return CSA2_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(kv_codes) || !aligned16(out) || (swa && !aligned16(swa)))
        return CSA2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv_scales) & 7) return CSA2_ERR_INVALID_ARG;
    if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
    const AttnWs L = attn_ws(n_q, k, window);
    if (!ws || !aligned16(ws) || ws_bytes < L.total) return CSA2_ERR_WORKSPACE;
    if (n_q == 0) return CSA2_OK;
    cudaStream_t s = cudaStream_t(stream);
    char* base = static_cast<char*>(ws);
    Status* st = reinterpret_cast<Status*>(base);
    float* part_o = reinterpret_cast<float*>(base + L.part_o);
    float* part_ml = reinterpret_cast<float*>(base + L.part_ml);
    const uint16_t* q = static_cast<const uint16_t*>(q_bf16);
    const uint16_t* sn = static_cast<const uint16_t*>(swa_new_bf16);
    const bool f32 = out_dtype == CSA2_OUT_F32;
    // merge through cluster shared memory only when every cluster of the
    // launch can be resident at once (a cluster needs `splits` free SMs in
    // one GPC); otherwise clusters run in waves and the workspace merge wins
    const bool cluster = L.splits <= 8 && n_q * L.splits <= 64;
    const dim3 grid(static_cast<unsigned>(L.splits), static_cast<unsigned>(n_q));
    csa2_status e = CSA2_OK;
#define CSA2_SPLIT(E_, C_)                                                                              \
    e = launch_split<E_, C_>(grid, s, q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, \
                             sn, window, sm_scale, part_o, part_ml, L.splits, out, f32, out_lse, st)
#define CSA2_SPLIT_E(C_)                      \
    switch (L.entries) {                      \
        case 80: CSA2_SPLIT(80, C_); break;   \
        case 64: CSA2_SPLIT(64, C_); break;   \
        case 48: CSA2_SPLIT(48, C_); break;   \
        case 32: CSA2_SPLIT(32, C_); break;   \
        default: CSA2_SPLIT(16, C_); break;   \
    }
    if (cluster) {
        CSA2_SPLIT_E(true)
    } else {
        CSA2_SPLIT_E(false)
    }
#undef CSA2_SPLIT_E
#undef CSA2_SPLIT
    if (e != CSA2_OK) return e;
    if (cluster) return launch_status();
    timer_begin(K_ATTN_MERGE, s);
    if (f32)
        attn_merge_kernel<true><<<dim3(unsigned(n_q), kH / 8), 256, 0, s>>>(part_o, part_ml, L.splits, out, out_lse);
    else
        attn_merge_kernel<false><<<dim3(unsigned(n_q), kH / 8), 256, 0, s>>>(part_o, part_ml, L.splits, out, out_lse);
    timer_end(K_ATTN_MERGE, s);
    return launch_status();
}
