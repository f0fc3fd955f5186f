// Device helpers shared by the CSA2 kernels: number formats, status word,
// order-preserving keys, warp/block reductions.
//
// Formats: [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", §三:
// the main KV is E2M1 (MXFP4 family) with one E4M3 scale per 16 channels and
// the window KV stays FP8; [T2] blog "DeepSeek V4.1 Flash vs V4 Pro",
// 黑科技之三: like NVFP4 without its second-level global scale.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/csa2.h"

namespace csa2 {

// ---------------------------------------------------------------- status
// The first 256 bytes of every workspace: int32 {status, detail0..2}.
struct Status {
    int32_t code;
    int32_t detail[3];
};

enum BoundsCheck : int32_t {
    CHK_DST_ROW = 1,     // append: destination row outside the plane
    CHK_POSITION = 2,    // append: RoPE position outside the table
    CHK_KV_START = 3,    // index/attn: kv_start not a multiple of 8 or negative
    CHK_VISIBLE = 4,     // index/attn: n_visible > max_visible or < 0
    CHK_ROWS = 5,        // index/attn: kv_start + n_visible > n_rows
    CHK_POOL = 6,        // reindex: pool block outside [0, ceil(n/8))
    CHK_TOPK = 7,        // attn: topk entry outside [-1, n)
};

__device__ __forceinline__ void record(Status* st, int32_t code, int32_t which, int32_t item,
                                       int32_t value) {
    if (st == nullptr) return;
    if (atomicCAS(&st->code, 0, code) == 0) {
        st->detail[0] = which;
        st->detail[1] = item;
        st->detail[2] = value;
    }
}

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ---------------------------------------------------------------- E4M3
// Value of an E4M3FN byte from its fields: bias 7, exponent 0 is subnormal
// (m/8 * 2^-6), 0x7F / 0xFF are NaN.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 0xF, m = b & 7;
    float v = (e == 0) ? float(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    if ((b & 0x7F) == 0x7F) v = __uint_as_float(0x7FC00000u);
    return (b & 0x80) ? -v : v;
}

// Nearest-even E4M3 of two floats, saturating to +-448; byte of `lo` in
// bits 0-7, byte of `hi` in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------- E2M1
// Code of |x| / s for s > 0 by exact comparison with the midpoints
// s*{0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} (each product is exact in fp32):
// above a midpoint rounds up; on a midpoint goes to the even code; the count
// saturates at 7 (value 6).  The IEEE sign of x is kept in bit 3.
__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
    const float a = fabsf(x);
    uint32_t c = 0;
    c += (a > 0.25f * s);                        // 0 | 1, tie -> 0 (even)
    c += (a >= 0.75f * s);                       // 1 | 2, tie -> 2
    c += (a > 1.25f * s);                        // 2 | 3, tie -> 2
    c += (a >= 1.75f * s);                       // 3 | 4, tie -> 4
    c += (a > 2.5f * s);                         // 4 | 5, tie -> 4
    c += (a >= 3.5f * s);                        // 5 | 6, tie -> 6
    c += (a > 5.0f * s);                         // 6 | 7, tie -> 6
    return c | ((__float_as_uint(x) >> 28) & 8u);
}

// Quantize 16 floats (one group): returns the scale byte, writes 8 code
// bytes (even channel in the low nibble) to codes[0..1] as two uint32.
// s = RNE_E4M3(amax / 6) saturating; s == 0 gives all-zero codes.
__device__ __forceinline__ uint32_t quantize_group16(const float (&v)[16], uint32_t (&codes)[2]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t sbyte = e4m3x2_rn_sat(__fdiv_rn(amax, 6.0f), 0.f) & 0xFF;
    const float s = e4m3_value(sbyte);
    codes[0] = codes[1] = 0;
    if (s > 0.f) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            codes[i >> 3] |= e2m1_code(v[i], s) << (4 * (i & 7));
    }
    return sbyte;
}

// Two E2M1 codes in the low byte of `b` (low nibble first) as f16x2, low
// nibble in the low half.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t b) {
    uint32_t r;
    const uint16_t h = static_cast<uint16_t>(b & 0xFF);
    asm("{\n .reg .b8 t, u;\n mov.b16 {t, u}, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n"
        : "=r"(r) : "h"(h));
    return r;
}

// ---------------------------------------------------------------- keys
// Order-preserving map float -> uint32 (larger float, larger key); -0 and
// +0 map to the same key.
__device__ __forceinline__ uint32_t float_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization, so it may become resident while
// the previous kernel of the stream is still running.  grid_dep_wait()
// returns once that kernel has completed and its memory is visible (at once
// when there is none); nothing written by earlier work in the stream may be
// read, and nothing may be written to global memory, before it.
// grid_dep_launch() then lets the next kernel start its own launch.  A kernel
// allocates TMEM only after grid_dep_wait(), so it never waits on columns
// held by its predecessor.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename T>
__host__ __device__ constexpr T ceil_div(T a, T b) { return (a + b - 1) / b; }

}  // namespace csa2

// Host-side helpers shared by the entry points.
namespace csa2 {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
csa2_status launch_status();  // maps cudaGetLastError to a csa2_status
int sm_count();               // the current device's multiprocessors (queried once per device)
uint64_t wait_limit_ns();      // the bounded waits' limit, passed to every launch (2 s by default)

// Launches `kernel` on `s` with programmatic stream serialization (see
// grid_dep_wait) and, when cluster > 1, clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, unsigned cluster,
                   Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
}  // namespace csa2
