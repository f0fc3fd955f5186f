// KV append: fused RoPE + FP4 quantization, plain FP4 for indexer rows, FP8
// for window latents.
//
// [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", §三 and [T3]
// "DeepSeek-V4.1-Flash：全局 KV 仅 890 B/token，百万上下文怎么做成的？", 第三刀:
// the main KV is stored as E2M1 with an E4M3 scale per 16 channels, quantized
// after RoPE; the window KV stays FP8.
//
// One thread per group of 16 channels (dim/16 threads per row): each thread
// reads 32 contiguous bytes of bf16, rotates its 8 channel pairs, quantizes
// and writes 8 code bytes + 1 scale byte.  The kernel is bound by HBM
// (1024 B read + 288 B written per 512-channel row).
#include "csa2_common.cuh"
#include "csa2_timer.cuh"
#include "csa2_layout.cuh"

#include <cmath>

namespace csa2 {

// Table rows [0, n_hi): cos/sin(hi * 1024 * w_i); rows [n_hi, n_hi + 1024):
// cos/sin(lo * w_i), w_i = theta^(-2i/dim), computed in fp64 on the device.
// The buffer holds the rows twice: as float2 (fast path) and then as double2
// (exact fallback near rounding ties).
__global__ void rope_table_kernel(float theta, int dim, int n_hi, float2* t32, double2* t64) {
    grid_dep_wait();
    grid_dep_launch();
    const int half = dim / 2;
    const int64_t total = int64_t(n_hi + 1024) * half;
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const int row = int(t / half), i = int(t % half);
        const double w = pow(double(theta), -2.0 * double(i) / double(dim));
        const double p = row < n_hi ? double(row) * 1024.0 : double(row - n_hi);
        double s, c;
        sincos(p * w, &s, &c);
        t32[t] = make_float2(float(c), float(s));
        t64[t] = make_double2(c, s);
    }
}

// Nearest-even E4M3 byte of v >= 0 held in fp64, saturating at 448: the
// fp32-rounded guess is off by at most one step; the midpoint test 2v vs
// a + b is exact in fp64.
__device__ __forceinline__ uint32_t e4m3_rne_f64(double v) {
    if (v >= 448.0) return 0x7E;
    const uint32_t g = e4m3x2_rn_sat(float(v), 0.f) & 0x7F;
    uint32_t best = g;
    double bv = double(e4m3_value(g));
#pragma unroll
    for (int d = -1; d <= 1; d += 2) {
        const int c = int(g) + d;
        if (c < 0 || c > 0x7E) continue;
        const double cv = double(e4m3_value(uint32_t(c)));
        // exact: compare 2v with the sum of the two candidates
        const bool closer = (cv < bv) ? (2.0 * v < cv + bv) : (2.0 * v > cv + bv);
        const bool tie = (2.0 * v == cv + bv);
        if (closer || (tie && (c & 1) == 0)) { best = uint32_t(c); bv = cv; }
    }
    return best;
}

// E2M1 code of x / s for s > 0 by exact fp64 comparisons (ties to even).
__device__ __forceinline__ uint32_t e2m1_code_f64(double x, double s) {
    const double a = fabs(x);
    uint32_t c = 0;
    c += (a > 0.25 * s);
    c += (a >= 0.75 * s);
    c += (a > 1.25 * s);
    c += (a >= 1.75 * s);
    c += (a > 2.5 * s);
    c += (a >= 3.5 * s);
    c += (a > 5.0 * s);
    return c | (signbit(x) ? 8u : 0u);
}

// E2M1 pair via the hardware conversion (nearest-even, saturating at 6, sign
// kept): low nibble from `lo`.
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}\n"
        : "=h"(r) : "f"(hi), "f"(lo));
    return r & 0xFF;
}

// FP4 append.  TPR = dim/16 threads per row.  LAYOUT: CSA2_LAYOUT_ROWS,
// CSA2_LAYOUT_BLOCK8 (scales in their own plane) or CSA2_LAYOUT_BLOCK8R
// (576-byte records: a block's codes, then its scales; `scales` unused).
template <int DIM, int LAYOUT>
__global__ void __launch_bounds__(256, 3) quantize_fp4_kernel(
    const uint4* __restrict__ x, int64_t n, const int64_t* __restrict__ pos,
    const float2* __restrict__ table, int n_hi, int64_t max_pos,
    const int64_t* __restrict__ dst_row, int64_t n_rows, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, Status* st) {
    constexpr int TPR = DIM / 16;
    constexpr int RPB = 256 / TPR;  // rows per block per iteration
    grid_dep_wait();
    grid_dep_launch();
    const int g = threadIdx.x % TPR;
    const int64_t stride = int64_t(gridDim.x) * RPB;
    // the next row's input, position and destination are loaded while the
    // current one is converted (two rows in flight per thread)
    int64_t i = blockIdx.x * int64_t(RPB) + threadIdx.x / TPR;
    uint4 na = make_uint4(0, 0, 0, 0), nb = na;
    int64_t np = 0, nrow = 0;
    auto fetch = [&](int64_t r) {
        if (r < n) {
            const uint4* src = x + r * (DIM / 8) + 2 * g;  // 8 bf16 per uint4
            na = __ldg(src);
            nb = __ldg(src + 1);
            np = pos != nullptr ? __ldg(pos + r) : 0;
            nrow = dst_row ? __ldg(dst_row + r) : r;
        }
    };
    fetch(i);
    for (; i < n; i += stride) {
        const uint4 a = na, b = nb;
        const int64_t p = np, row = nrow;
        fetch(i + stride);
        if (row < 0 || row >= n_rows) {
            if (g == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_DST_ROW, int32_t(i), int32_t(row));
            continue;
        }
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float v[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[2 * j] = bf16_lo(w[j]);
            v[2 * j + 1] = bf16_hi(w[j]);
        }
        uint32_t cw[2];
        uint32_t sb;
        if (pos == nullptr) {
            sb = quantize_group16(v, cw);  // bf16 inputs: exact comparisons
        } else {
            if (p < 0 || p >= max_pos) {
                if (g == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_POSITION, int32_t(i), int32_t(p));
                continue;
            }
            // fp32 rotation by angle addition from the table; bnd bounds its
            // error (table rounding, products) with a wide safety factor
            const int64_t rh = (p >> 10) * (DIM / 2) + 8 * g;
            const int64_t rl = (int64_t(n_hi) + (p & 1023)) * (DIM / 2) + 8 * g;
            const float4* th = reinterpret_cast<const float4*>(table + rh);
            const float4* tl = reinterpret_cast<const float4*>(table + rl);
            // bnd[j] bounds the fp32 error of pair j's two outputs.  The table
            // entries are within 2^-25 of cos/sin, so c, s carry at most
            // 1.5 * 2^-23 and y = x0 c - x1 s at most 2.5 * 2^-23 (|x0| + |x1|)
            // after its two roundings; 2^-21 (|x0| + |x1|) covers that.
            float y[16], bnd[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 h = __ldg(th + j), l = __ldg(tl + j);
                const float c0 = fmaf(h.x, l.x, -h.y * l.y), s0 = fmaf(h.y, l.x, h.x * l.y);
                const float c1 = fmaf(h.z, l.z, -h.w * l.w), s1 = fmaf(h.w, l.z, h.z * l.w);
                const float x0 = v[4 * j], x1 = v[4 * j + 1], x2 = v[4 * j + 2], x3 = v[4 * j + 3];
                y[4 * j] = fmaf(x0, c0, -x1 * s0);
                y[4 * j + 1] = fmaf(x0, s0, x1 * c0);
                y[4 * j + 2] = fmaf(x2, c1, -x3 * s1);
                y[4 * j + 3] = fmaf(x2, s1, x3 * c1);
                bnd[2 * j] = 0x1p-21f * (fabsf(x0) + fabsf(x1));
                bnd[2 * j + 1] = 0x1p-21f * (fabsf(x2) + fabsf(x3));
            }
            float amax = 0.f, bmax = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(y[e]));
#pragma unroll
            for (int j = 0; j < 8; ++j) bmax = fmaxf(bmax, bnd[j]);
            // amax / 6 by a multiply: its error (< 2^-22 relative) sits inside mq
            const float q6 = amax * (1.0f / 6.0f);
            const float mq = fmaf(q6, 0x1p-20f, bmax * (1.0f / 6.0f) * 1.001f);
            sb = e4m3x2_rn_sat(q6, 0.f) & 0xFF;
            // a tie of the scale inside the margin: resolve in fp64
            const uint32_t span = e4m3x2_rn_sat(fmaxf(q6 - mq, 0.f), q6 + mq);
            bool risky = (span & 0xFF) != (span >> 8);
            const float sc = e4m3_value(sb);
            cw[0] = cw[1] = 0;
            if (sc > 0.f) {
                const float inv = __frcp_rn(sc);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float r0 = y[2 * j] * inv, r1 = y[2 * j + 1] * inv;
                    cw[j >> 2] |= e2m1x2_rn_sat(r0, r1) << (8 * (j & 3));
                    const float a0 = fabsf(r0), a1 = fabsf(r1);
                    const float m0 = fmaf(a0, 0x1p-22f, bnd[j] * inv * 1.001f);
                    const float m1 = fmaf(a1, 0x1p-22f, bnd[j] * inv * 1.001f);
                    risky |= e2m1x2_rn_sat(fmaxf(a0 - m0, 0.f), fmaxf(a1 - m1, 0.f)) !=
                             e2m1x2_rn_sat(a0 + m0, a1 + m1);
                }
            }
            if (risky) {
                // fp64 rotation from the fp64 table and exact quantization
                const double2* t64 = reinterpret_cast<const double2*>(table + int64_t(n_hi + 1024) * (DIM / 2));
                double z[16], a64 = 0.0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const double2 h = t64[rh + j], l = t64[rl + j];
                    const double c = fma(h.x, l.x, -h.y * l.y), sn = fma(h.y, l.x, h.x * l.y);
                    const double x0 = v[2 * j], x1 = v[2 * j + 1];
                    z[2 * j] = fma(x0, c, -x1 * sn);
                    z[2 * j + 1] = fma(x0, sn, x1 * c);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) a64 = fmax(a64, fabs(z[e]));
                sb = e4m3_rne_f64(a64 / 6.0);
                const double s64 = double(e4m3_value(sb));
                cw[0] = cw[1] = 0;
                if (s64 > 0.0) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) cw[e >> 3] |= e2m1_code_f64(z[e], s64) << (4 * (e & 7));
                }
            }
        }
        int64_t off;
        if (LAYOUT == CSA2_LAYOUT_BLOCK8R)
            off = (row >> 3) * 576 + (g >> 1) * 128 + (row & 7) * 16 + (g & 1) * 8;
        else if (LAYOUT == CSA2_LAYOUT_BLOCK8)
            off = (row >> 3) * 512 + (g >> 1) * 128 + (row & 7) * 16 + (g & 1) * 8;
        else
            off = row * (DIM / 2) + 8 * g;
        *reinterpret_cast<uint2*>(codes + off) = make_uint2(cw[0], cw[1]);
        if (LAYOUT == CSA2_LAYOUT_BLOCK8R)
            codes[(row >> 3) * 576 + 512 + (row & 7) * 8 + g] = uint8_t(sb);
        else
            scales[row * (DIM / 16) + g] = uint8_t(sb);
    }
}

// FP8 append: each thread converts 16 channels to 16 E4M3 bytes.
template <int DIM>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(
    const uint4* __restrict__ x, int64_t n, const int64_t* __restrict__ dst_row, int64_t n_rows,
    uint8_t* __restrict__ dst, Status* st) {
    constexpr int TPR = DIM / 16;
    constexpr int RPB = 256 / TPR;
    grid_dep_wait();
    grid_dep_launch();
    const int g = threadIdx.x % TPR;
    for (int64_t i = blockIdx.x * int64_t(RPB) + threadIdx.x / TPR; i < n;
         i += int64_t(gridDim.x) * RPB) {
        const int64_t row = dst_row ? __ldg(dst_row + i) : i;
        if (row < 0 || row >= n_rows) {
            if (g == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_DST_ROW, int32_t(i), int32_t(row));
            continue;
        }
        const uint4* src = x + i * (DIM / 8) + 2 * g;
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t p0 = e4m3x2_rn_sat(bf16_lo(w[2 * j]), bf16_hi(w[2 * j]));
            const uint32_t p1 = e4m3x2_rn_sat(bf16_lo(w[2 * j + 1]), bf16_hi(w[2 * j + 1]));
            o[j] = p0 | (p1 << 16);
        }
        *reinterpret_cast<uint4*>(dst + row * DIM + 16 * g) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Blocks for `rows` rows: one per rows_per_block rows, at most the blocks
// that are resident at once (per_sm per SM), which then stride the rows.
static int grid_for(int64_t rows, int rows_per_block, int per_sm = 16) {
    int64_t g = ceil_div<int64_t>(rows, rows_per_block);
    const int64_t cap = int64_t(sm_count()) * per_sm;
    return int(g < 1 ? 1 : (g > cap ? cap : g));
}
constexpr int kFp4BlocksPerSm = 3;  // quantize_fp4_kernel's launch bound

}  // namespace csa2

using namespace csa2;

extern "C" size_t csa2_rope_table_bytes(int dim, int64_t max_pos) {
    if (dim <= 0 || dim % 2 || max_pos <= 0) return 0;
    const int64_t n_hi = ceil_div<int64_t>(max_pos, 1024);
    return size_t(n_hi + 1024) * size_t(dim / 2) * (sizeof(float2) + sizeof(double2));
}

extern "C" csa2_status csa2_rope_table_init(float theta, int dim, int64_t max_pos, void* table,
                                            csa2_stream_t stream) {
    if (!table || !aligned16(table) || dim <= 0 || dim % 16 || max_pos <= 0 ||
        max_pos > (int64_t(1) << 31) || !(theta > 1.0f))
        return CSA2_ERR_INVALID_ARG;
    const int n_hi = int(ceil_div<int64_t>(max_pos, 1024));
    float2* t32 = static_cast<float2*>(table);
    double2* t64 = reinterpret_cast<double2*>(t32 + int64_t(n_hi + 1024) * (dim / 2));
    timer_begin(K_ROPE_TABLE, cudaStream_t(stream));
    launch(rope_table_kernel, 256, 256, 0, cudaStream_t(stream), 1, theta, dim, n_hi, t32, t64);
    timer_end(K_ROPE_TABLE, cudaStream_t(stream));
    return launch_status();
}

extern "C" csa2_status csa2_quantize_append(const void* x_bf16, int64_t n, int dim, int fmt,
                                            int layout, const int64_t* pos,
                                            const void* rope_table, int64_t rope_max_pos,
                                            const int64_t* dst_row, int64_t n_rows,
                                            uint8_t* dst_codes, uint8_t* dst_scales, void* ws,
                                            size_t ws_bytes, csa2_stream_t stream) {
    if (n < 0 || n_rows < 0) return CSA2_ERR_INVALID_ARG;
    if (!ws || ws_bytes < CSA2_STATUS_BYTES || !aligned16(ws)) return CSA2_ERR_WORKSPACE;
    if (n == 0) return CSA2_OK;
    if (!x_bf16 || !dst_codes || !aligned16(x_bf16) || !aligned16(dst_codes))
        return CSA2_ERR_INVALID_ARG;
    if (dim != 128 && dim != 512) return CSA2_ERR_UNSUPPORTED;
    if (dst_row == nullptr && n > n_rows) return CSA2_ERR_INVALID_ARG;
    Status* st = static_cast<Status*>(ws);
    cudaStream_t s = cudaStream_t(stream);
    const uint4* x = static_cast<const uint4*>(x_bf16);
    if (fmt == CSA2_FMT_FP8) {
        if (layout != CSA2_LAYOUT_ROWS || pos != nullptr) return CSA2_ERR_UNSUPPORTED;
        timer_begin(K_QUANT_FP8, s);
        if (dim == 512)
            launch(quantize_fp8_kernel<512>, grid_for(n, 8), 256, 0, s, 1, x, n, dst_row, n_rows, dst_codes, st);
        else
            launch(quantize_fp8_kernel<128>, grid_for(n, 32), 256, 0, s, 1, x, n, dst_row, n_rows, dst_codes, st);
        timer_end(K_QUANT_FP8, s);
        return launch_status();
    }
    if (fmt != CSA2_FMT_FP4) return CSA2_ERR_UNSUPPORTED;
    if (layout != CSA2_LAYOUT_ROWS && layout != CSA2_LAYOUT_BLOCK8 && layout != CSA2_LAYOUT_BLOCK8R)
        return CSA2_ERR_UNSUPPORTED;
    if (layout == CSA2_LAYOUT_BLOCK8R ? dst_scales != nullptr : !dst_scales) return CSA2_ERR_INVALID_ARG;
    if (layout != CSA2_LAYOUT_ROWS && (dim != 128 || n_rows % 8)) return CSA2_ERR_UNSUPPORTED;
    int n_hi = 0;
    const float2* table = nullptr;
    if (pos != nullptr) {
        if (!rope_table || !aligned16(rope_table) || rope_max_pos <= 0) return CSA2_ERR_INVALID_ARG;
        n_hi = int(ceil_div<int64_t>(rope_max_pos, 1024));
        table = static_cast<const float2*>(rope_table);
    }
    timer_begin(K_QUANT_FP4, s);
    if (dim == 512)
        launch(quantize_fp4_kernel<512, CSA2_LAYOUT_ROWS>, grid_for(n, 8, kFp4BlocksPerSm), 256, 0, s, 1,
            x, n, pos, table, n_hi, rope_max_pos, dst_row, n_rows, dst_codes, dst_scales, st);
    else if (layout == CSA2_LAYOUT_BLOCK8R)
        launch(quantize_fp4_kernel<128, CSA2_LAYOUT_BLOCK8R>, grid_for(n, 32, kFp4BlocksPerSm), 256, 0, s, 1,
            x, n, pos, table, n_hi, rope_max_pos, dst_row, n_rows, dst_codes, dst_scales, st);
    else if (layout == CSA2_LAYOUT_BLOCK8)
        launch(quantize_fp4_kernel<128, CSA2_LAYOUT_BLOCK8>, grid_for(n, 32, kFp4BlocksPerSm), 256, 0, s, 1,
            x, n, pos, table, n_hi, rope_max_pos, dst_row, n_rows, dst_codes, dst_scales, st);
    else
        launch(quantize_fp4_kernel<128, CSA2_LAYOUT_ROWS>, grid_for(n, 32, kFp4BlocksPerSm), 256, 0, s, 1,
            x, n, pos, table, n_hi, rope_max_pos, dst_row, n_rows, dst_codes, dst_scales, st);
    timer_end(K_QUANT_FP4, s);
    return launch_status();
}
