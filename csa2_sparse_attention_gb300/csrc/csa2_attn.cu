// Sparse attention over the selected FP4 latents plus the FP8 window, with
// one merged softmax.
//
// [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", §二: main
// attention has 64 heads of dim 512 over one shared latent per entry, each
// layer keeps its own query and window KV; [T3] "DeepSeek-V4.1-Flash：全局 KV
// 仅 890 B/token，百万上下文怎么做成的？", 第三刀: the FP4 main KV is dequantized
// before attention and the window KV stays FP8.
//
// Split-K over entries: CTA (split, query) takes 64 entries, gathers and
// dequantizes them into shared memory (exact in bf16), computes S = Q C^T
// (bf16 MMA, fp32 accumulate), the split's softmax statistics (m, l), and
// O_s = P C with P split into f16 hi + lo parts (C converted in place to f16,
// still exact), so the partial output carries ~2^-22 relative error.  A merge
// kernel combines the splits with their log-sum-exp weights and rounds to
// bf16 once.
#include "csa2_common.cuh"
#include "csa2_timer.cuh"
#include "csa2_layout.cuh"

#include <cfloat>

namespace csa2 {

constexpr int kAttnThreads = 256;
constexpr int kE = kAttnSplit;     // 64 entries per CTA
constexpr int kH = CSA2_ATTN_HEADS;
constexpr int kD = CSA2_LATENT_DIM;
constexpr int kSStride = kE + 4;   // fp32 S row stride
constexpr int kPStride = kE + 8;   // f16 P row stride (144 B rows)

struct AttnSmem {
    uint4 q[kH * kD / 8];          // bf16 [64][512], 16-byte chunks swizzled
    uint4 c[kE * kD / 8];          // bf16 then f16 [64][512], swizzled
    float s[kH * kSStride];
    __half p_hi[kH * kPStride];
    __half p_lo[kH * kPStride];
    uint32_t lut4[256];            // E2M1 pair -> bf16x2 (unscaled)
    uint16_t lut8[256];            // E4M3 byte -> bf16
    int ok[kE];                    // entry valid
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
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(
    const uint16_t* __restrict__ qg, const uint8_t* __restrict__ kv_codes,
    const uint8_t* __restrict__ kv_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, const int32_t* __restrict__ topk, int k,
    const uint8_t* __restrict__ swa, int window, float sm_scale, int32_t max_visible,
    float* __restrict__ part_o, float* __restrict__ part_ml, int splits, Status* st) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    AttnSmem& S = *reinterpret_cast<AttnSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int split = blockIdx.x;
    const int64_t q = blockIdx.y;

    // tables: E2M1 pair -> bf16x2, E4M3 -> bf16 (exact)
    {
        const int b = tid;
        const float e2m1[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        const float lo = (b & 8 ? -1.f : 1.f) * e2m1[b & 7];
        const float hi = (b & 128 ? -1.f : 1.f) * e2m1[(b >> 4) & 7];
        S.lut4[b] = uint32_t(bf16_bits(lo)) | (uint32_t(bf16_bits(hi)) << 16);
        S.lut8[b] = bf16_bits(e4m3_value(uint32_t(b)));
    }
    // Q (bf16 [64][512]) into swizzled shared memory
    const uint16_t* qsrc = qg + q * (kH * kD);
    for (int i = tid; i < kH * kD / 8; i += kAttnThreads) {
        const int r = i >> 6, c = i & 63;
        cp_async16(smem_addr(reinterpret_cast<uint8_t*>(S.q) + swz(r, c)), qsrc + r * kD + c * 8);
    }
    // per-query validity (reported once per query)
    int32_t n = 0;
    {
        const int64_t ks = kv_start[q];
        const int32_t nv = n_visible[q];
        const bool report = split == 0 && tid == 0;
        if (ks < 0) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_KV_START, int32_t(q), int32_t(ks));
        } else if (nv < 0 || nv > max_visible) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_VISIBLE, int32_t(q), nv);
        } else if (ks + nv > n_rows) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_ROWS, int32_t(q), nv);
        } else {
            n = nv;
        }
    }
    const int64_t ks = kv_start[q];
    const int nw = n < window ? n : window;
    __syncthreads();  // tables ready

    // gather + dequantize: thread -> (entry e = tid/4, quarter qq = tid%4)
    {
        const int e = tid >> 2, qq = tid & 3;
        const int ge = split * kE + e;
        uint8_t* crow = reinterpret_cast<uint8_t*>(S.c);
        bool ok = false;
        if (ge < k) {
            const int32_t p = topk[q * k + ge];
            if (p >= 0 && p < n) {
                ok = true;
                const int64_t row = ks + p;
                const uint4* src = reinterpret_cast<const uint4*>(kv_codes + row * 256 + qq * 64);
                const uint2 sc = __ldg(reinterpret_cast<const uint2*>(kv_scales + row * 32 + qq * 8));
                const uint32_t scw[2] = {sc.x, sc.y};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 v = __ldg(src + j);
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    // 16 code bytes = 32 channels = groups 2j, 2j+1 of this quarter
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t sb = (scw[(2 * j + h) >> 2] >> (8 * ((2 * j + h) & 3))) & 0xFF;
                        const uint32_t s16 = S.lut8[sb];  // scale as bf16 (exact)
                        const uint32_t s2 = s16 | (s16 << 16);
                        // 8 code bytes (words 2h, 2h+1) = 16 channels, two per byte
                        uint32_t outw[8];
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const uint32_t w = wv[2 * h + m];
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb)
                                outw[4 * m + bb] = bf16x2_mul(S.lut4[(w >> (8 * bb)) & 0xFF], s2);
                        }
                        // 8 bytes = 16 channels = 2 chunks of 8 channels
                        const int chunk = qq * 16 + 4 * j + 2 * h;
                        *reinterpret_cast<uint4*>(crow + swz(e, chunk)) =
                            make_uint4(outw[0], outw[1], outw[2], outw[3]);
                        *reinterpret_cast<uint4*>(crow + swz(e, chunk + 1)) =
                            make_uint4(outw[4], outw[5], outw[6], outw[7]);
                    }
                }
            } else if (p < -1 || p >= n) {
                if (qq == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_TOPK, int32_t(q), p);
            }
        } else if (ge - k < nw) {
            ok = true;
            const int64_t pos = int64_t(n - nw) + (ge - k);
            const int64_t slot = pos % window;
            const uint4* src = reinterpret_cast<const uint4*>(swa + (q * window + slot) * kD + qq * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = __ldg(src + j);
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
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

    // S = Q C^T: warp -> heads 16*(warp%4).., entries 32*(warp/4)..
    const int hg = warp & 3, eh = warp >> 2;
    {
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const uint32_t qb = smem_addr(S.q), cb = smem_addr(S.c);
        const int arow = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int brow = 32 * eh + (lane & 7) + 8 * (lane >> 4);
#pragma unroll 4
        for (int kk = 0; kk < kD / 16; ++kk) {
            uint32_t a[4], b01[4], b23[4];
            ldsm_x4(qb + swz(arow, 2 * kk + (lane >> 4)), a);
            ldsm_x4(cb + swz(brow, 2 * kk + ((lane >> 3) & 1)), b01);
            ldsm_x4(cb + swz(brow + 16, 2 * kk + ((lane >> 3) & 1)), b23);
            mma_bf16(acc[0], a, b01[0], b01[1]);
            mma_bf16(acc[1], a, b01[2], b01[3]);
            mma_bf16(acc[2], a, b23[0], b23[1]);
            mma_bf16(acc[3], a, b23[2], b23[3]);
        }
        const int r = 16 * hg + (lane >> 2);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 32 * eh + 8 * j + 2 * (lane & 3);
            S.s[r * kSStride + c] = acc[j][0];
            S.s[r * kSStride + c + 1] = acc[j][1];
            S.s[(r + 8) * kSStride + c] = acc[j][2];
            S.s[(r + 8) * kSStride + c + 1] = acc[j][3];
        }
    }
    __syncthreads();

    // softmax statistics of this split: thread -> (head tid/4, 16 entries)
    {
        const int h = tid >> 2, c0 = (tid & 3) * 16;
        float x[16], m = -INFINITY;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            x[j] = S.ok[c0 + j] ? sm_scale * S.s[h * kSStride + c0 + j] : -INFINITY;
            m = fmaxf(m, x[j]);
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float p = x[j] == -INFINITY ? 0.f : expf(x[j] - m);
            l += p;
            const __half hi = __float2half_rn(p);
            S.p_hi[h * kPStride + c0 + j] = hi;
            S.p_lo[h * kPStride + c0 + j] = __float2half_rn(p - __half2float(hi));
        }
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if ((tid & 3) == 0) {
            float* ml = part_ml + ((q * splits + split) * kH + h) * 2;
            ml[0] = m;
            ml[1] = l;
        }
    }
    // C from bf16 to f16 in place (exact for FP4 and E4M3 values)
    {
        uint32_t* cw = reinterpret_cast<uint32_t*>(S.c);
        for (int i = tid; i < kE * kD / 2; i += kAttnThreads) {
            const uint32_t v = cw[i];
            const __half2 h = __floats2half2_rn(bf16_lo(v), bf16_hi(v));
            cw[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    __syncthreads();

    // O_s = P C: warp -> heads 16*hg.., dims 256*(warp/4).. in two passes of 128
    {
        const int dh = warp >> 2;
        const uint32_t ph = smem_addr(S.p_hi), pl = smem_addr(S.p_lo), cb = smem_addr(S.c);
        const int arow = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1);
        float* out = part_o + (q * splits + split) * int64_t(kH * kD);
        for (int pass = 0; pass < 2; ++pass) {
            const int d0 = 256 * dh + 128 * pass;  // first dim of this pass
            float acc[16][4];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kE / 16; ++ks) {
                uint32_t ahi[4], alo[4];
                const uint32_t aoff = uint32_t((arow * kPStride + 16 * ks + 8 * (lane >> 4)) * 2);
                ldsm_x4(ph + aoff, ahi);
                ldsm_x4(pl + aoff, alo);
                const int erow = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
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
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int c = d0 + 8 * j + 2 * (lane & 3);
                *reinterpret_cast<float2*>(out + r * kD + c) = make_float2(acc[j][0], acc[j][1]);
                *reinterpret_cast<float2*>(out + (r + 8) * kD + c) = make_float2(acc[j][2], acc[j][3]);
            }
        }
    }
}

// grid (n_q, 8): 8 heads per CTA, 256 threads, 16 dims per thread.
__global__ void __launch_bounds__(256) attn_merge_kernel(const float* __restrict__ part_o,
                                                         const float* __restrict__ part_ml, int splits,
                                                         uint16_t* __restrict__ out, float* __restrict__ lse) {
    const int64_t q = blockIdx.x;
    const int h = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int lane = lane_id();
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[((q * splits + s) * kH + h) * 2]);
    float L = 0.f;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float* ml = part_ml + ((q * splits + s) * kH + h) * 2;
            if (ml[0] == -INFINITY) continue;
            const float a = expf(ml[0] - M);
            L = fmaf(a, ml[1], L);
            const float4* src = reinterpret_cast<const float4*>(part_o + ((q * splits + s) * kH + h) * int64_t(kD));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 v = src[lane + 32 * j];
                acc[4 * j] = fmaf(a, v.x, acc[4 * j]);
                acc[4 * j + 1] = fmaf(a, v.y, acc[4 * j + 1]);
                acc[4 * j + 2] = fmaf(a, v.z, acc[4 * j + 2]);
                acc[4 * j + 3] = fmaf(a, v.w, acc[4 * j + 3]);
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* o = out + (q * kH + h) * int64_t(kD);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int d = 4 * (lane + 32 * j);
        const uint32_t lo = uint32_t(bf16_bits(acc[4 * j] * inv)) | (uint32_t(bf16_bits(acc[4 * j + 1] * inv)) << 16);
        const uint32_t hi = uint32_t(bf16_bits(acc[4 * j + 2] * inv)) | (uint32_t(bf16_bits(acc[4 * j + 3] * inv)) << 16);
        *reinterpret_cast<uint2*>(o + d) = make_uint2(lo, hi);
    }
    if (lse && lane == 0) lse[q * kH + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

static csa2_status prepare_attn_kernel() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
    if (done[dev]) return CSA2_OK;
    if (cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sizeof(AttnSmem))) != cudaSuccess)
        return CSA2_ERR_CUDA;
    done[dev] = true;
    return CSA2_OK;
}

}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_sparse_attn(const void* q_bf16, int64_t n_q, const uint8_t* kv_codes,
                                        const uint8_t* kv_scales, int64_t n_rows,
                                        const int64_t* kv_start, const int32_t* n_visible,
                                        const int32_t* topk, int k, const uint8_t* swa, int window,
                                        float sm_scale, void* out_bf16, float* out_lse, void* ws,
                                        size_t ws_bytes, csa2_stream_t stream) {
    if (n_q < 0 || n_rows < 0 || k < 0 || k > kMaxTopk || window < 0 || window > kMaxWindow)
        return CSA2_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || !(sm_scale < FLT_MAX)) return CSA2_ERR_INVALID_ARG;
    if (!q_bf16 || !kv_codes || !kv_scales || !kv_start || !n_visible || !out_bf16) return CSA2_ERR_INVALID_ARG;
    if (k > 0 && !topk) return CSA2_ERR_INVALID_ARG;
    if (window > 0 && !swa) return CSA2_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(kv_codes) || !aligned16(out_bf16) || (swa && !aligned16(swa)))
        return CSA2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv_scales) & 7) return CSA2_ERR_INVALID_ARG;
    if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
    const AttnWs L = attn_ws(n_q, k, window);
    if (!ws || !aligned16(ws) || ws_bytes < L.total) return CSA2_ERR_WORKSPACE;
    if (n_q == 0) return CSA2_OK;
    csa2_status e = prepare_attn_kernel();
    if (e != CSA2_OK) return e;
    cudaStream_t s = cudaStream_t(stream);
    char* base = static_cast<char*>(ws);
    Status* st = reinterpret_cast<Status*>(base);
    float* part_o = reinterpret_cast<float*>(base + L.part_o);
    float* part_ml = reinterpret_cast<float*>(base + L.part_ml);
    const int32_t max_visible = int32_t(n_rows < INT32_MAX ? n_rows : INT32_MAX);
    dim3 grid(unsigned(L.splits), unsigned(n_q));
    timer_begin(K_ATTN_SPLIT, s);
    attn_split_kernel<<<grid, kAttnThreads, sizeof(AttnSmem), s>>>(
        static_cast<const uint16_t*>(q_bf16), kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k,
        swa, window, sm_scale, max_visible, part_o, part_ml, L.splits, st);
    timer_end(K_ATTN_SPLIT, s);
    timer_begin(K_ATTN_MERGE, s);
    attn_merge_kernel<<<dim3(unsigned(n_q), kH / 8), 256, 0, s>>>(part_o, part_ml, L.splits,
                                                                 static_cast<uint16_t*>(out_bf16), out_lse);
    timer_end(K_ATTN_MERGE, s);
    return launch_status();
}
