// Sparse attention over the selected FP4 latents plus the FP8 window, with
// one merged softmax.
//
// [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", §二: main
// attention has 64 heads of dim 512 over one shared latent per entry, each
// layer keeps its own query and window KV; [T3] "DeepSeek-V4.1-Flash：全局 KV
// 仅 890 B/token，百万上下文怎么做成的？", 第三刀: the FP4 main KV is dequantized
// before attention and the window KV stays FP8.
//
// Split-K over entries on the 5th-generation tensor cores.  CTA (split,
// query) takes 128 entries: it gathers them and decodes them into shared
// memory as f16 with the hardware E2M1/E4M3 conversions (every FP4 value
// times its E4M3 scale and every E4M3 value is exact in f16), converts Q to
// f16 with a per-query power-of-two scale (exact except for elements far
// below max|Q|), computes S^T = C Q^T with one tcgen05 MMA chain (M = 128
// entries, N = 64 heads, K = 512, fp32 accumulate in TMEM), takes the
// split's softmax statistics (m, l) from registers (a transposing warp
// reduction), and computes O^T = C^T P^T (M = 4 x 128 dims, K = 128
// entries) with P split into f16 hi + lo parts side by side as one N = 128
// operand: on this tensor core an M = 128 MMA takes the same time at
// N = 128 as at N = 64, so the lo part costs no extra MMAs (the partial
// output carries ~2^-21 relative error from P).  One shared-memory copy of
// C serves both products: K-major
// for the first, MN-major for the second.  The splits of a query form one
// thread-block cluster when all clusters of the launch can be resident
// together: each CTA parks its fp32 partial in its own shared memory and
// reduces one slice of the dims over its peers through distributed shared
// memory.  Otherwise the partials go to the workspace and a merge kernel
// combines them.  Either way the result is rounded once, to fp32 or bf16.
// Small batches spread the 64 heads over two or four clusters per query
// (each CTA then takes in a part of Q and exchanges a part of the partial),
// and somewhat larger batches (16-19 queries of 640 entries) take two head
// groups over splits of 160 entries, so that the CTAs still fit one per SM.
//
// Optionally the kernel also appends the current token's window latent: the
// bf16 row for position n-1 is rounded to E4M3 (as csa2_quantize_append FP8
// does), written to its ring slot, and used for that entry.
#include "csa2_common.cuh"
#include "csa2_timer.cuh"
#include "csa2_layout.cuh"
#include "csa2_tc.cuh"

#include <cfloat>

#include <cooperative_groups.h>

namespace csa2 {

constexpr int kAttnThreads = 256;
constexpr int kH = CSA2_ATTN_HEADS;
constexpr int kD = CSA2_LATENT_DIM;

constexpr int kTcE = 128;          // entries per CTA = M of S^T
constexpr uint32_t kTcCols = 512;  // TMEM columns: S^T [0, 64); then O^T, 4 blocks of 128 (the first over S^T)

template <int E>
struct AttnTcSmemT {
    uint8_t r0[64 * 1024];         // Q f16 (B of S^T); then P^T hi/lo f16 [0, 32K) and softmax partials
    uint8_t c[E * 1024];           // C [E entries][512] f16; then the fp32 partial (cluster merge)
    int ok[E];                     // entry valid
    uint32_t qmax[kAttnThreads / 32];  // per-warp max |Q| (bf16 magnitude bits)
    float ml[kH][2];               // this split's (m, l) per head
    uint64_t bar;                  // MMA completion (phase 0: S, phase 1: O)
    uint32_t tmem;
};
using AttnTcSmem = AttnTcSmemT<kTcE>;
// 160 entries per CTA (two head groups of 32): 320 threads, two S^T tiles
constexpr int kTcE2 = 160;
constexpr int kAttnThreads2 = 320;
static_assert(sizeof(AttnTcSmemT<kTcE2>) + 1024 <= 227 * 1024, "shared memory of the 160-entry form");

// canonical no-swizzle K-major offsets: rows of 512 16-bit elements, 16-byte
// chunk c of row r -> (r/8)*8192 + c*128 + (r%8)*16
__device__ __forceinline__ uint32_t row512(int r, int c) { return uint32_t((r >> 3) * 8192 + c * 128 + (r & 7) * 16); }
// P^T [128 entries][NB] f16, MN-major B operand of O^T: 8-entry groups of
// 16 NB bytes, 8-column chunks of 128 B; with NB = 2 x the CTA's heads,
// column n < NB/2 is head n's hi part, NB/2 + n its lo part.
template <int NB = 128>
__device__ __forceinline__ uint32_t pmn(int e, int n) {
    return uint32_t((e >> 3) * (16 * NB) + (n >> 3) * 128 + (e & 7) * 16 + (n & 7) * 2);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint16_t bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// The eight E2M1 codes of w (low nibble of each byte first) as four f16x2,
// exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b8 a, b, c, d;\n mov.b32 {a, b, c, d}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n"
        " cvt.rn.f16x2.e2m1x2 %2, c;\n cvt.rn.f16x2.e2m1x2 %3, d;\n}\n"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}
// The four E4M3 bytes of w (byte 0 first) as two f16x2, exact (E4M3
// subnormals are f16 normals).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
        " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}\n"
        : "=r"(o[0]), "=r"(o[1]) : "r"(w));
}

// One quarter (128 channels) of an FP4 latent row: 4 x 16 bytes of E2M1
// codes and 8 E4M3 scales, as f16 into row e of C.  Code times scale has at
// most 5 significant bits and lies in [2^-10, 2688]: exact in f16.
__device__ __forceinline__ void fp4_quarter_to_c(const uint4* v, uint2 sc, uint8_t* c, int e, int qq) {
    uint32_t sw[4];  // scales of groups (0,1), (2,3), (4,5), (6,7) as f16x2
    e4m3x4_to_f16x2(sc.x, sw);
    e4m3x4_to_f16x2(sc.y, sw + 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // scale groups 2j, 2j+1 of this quarter
            const uint32_t s2 = __byte_perm(sw[j], 0, h ? 0x3232 : 0x1010);
            uint32_t outw[8];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                e2m1x8_to_f16x2(wv[2 * h + m], outw + 4 * m);
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) outw[4 * m + bb] = h2_mul(outw[4 * m + bb], s2);
            }
            const int chunk = qq * 16 + 4 * j + 2 * h;
            *reinterpret_cast<uint4*>(c + row512(e, chunk)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
            *reinterpret_cast<uint4*>(c + row512(e, chunk + 1)) = make_uint4(outw[4], outw[5], outw[6], outw[7]);
        }
    }
}

// One quarter (128 channels) of an FP8 window row (8 x 16 bytes) as f16
// into row e of C.
__device__ __forceinline__ void fp8_quarter_to_c(const uint4* v, uint8_t* c, int e, int qq) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t outw[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) e4m3x4_to_f16x2(wv[m], outw + 2 * m);
        const int chunk = qq * 16 + 2 * j;
        *reinterpret_cast<uint4*>(c + row512(e, chunk)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        *reinterpret_cast<uint4*>(c + row512(e, chunk + 1)) = make_uint4(outw[4], outw[5], outw[6], outw[7]);
    }
}

// grid (HG splits, n_q), 256 threads (320 with E = 160), one CTA per SM.  CTA x takes split
// x % splits for the 64 / HG heads of head group x / splits.  The split's
// unnormalized partial O_s = sum_j exp(l_j - m_s) c_j (fp32 [heads][512])
// and (m_s, l_s) per head go to the workspace, or (CLUSTER, one cluster per
// head group of a query) are merged across the cluster.  With HG head
// groups each CTA takes in 1/HG of Q and exchanges 1/HG of the partial
// bytes, for HG times the CTAs: the launch form for small batches.  With
// E = 160 entries per CTA (two head groups, 320 threads) a query's 640
// entries take 4 splits, so 16 queries fill 128 SMs in two head groups: C
// is stored with entries 128 .. 159 first (rows 0 .. 31), then 0 .. 127, so
// that S^T is two M = 128 tiles (storage rows 32 .. 159, and rows 0 .. 127
// of which only the first 32 are kept) and O^T runs over the storage order.
// win_shared: the window rows come from swa [n_rows][512] at row kv_start +
// position (a window over a sequence the queries share) instead of each
// query's ring swa [n_q][window][512] at slot position mod window.
template <bool CLUSTER, int HG, int E = kTcE>
__global__ void __launch_bounds__(E == kTcE ? kAttnThreads : kAttnThreads2, 1) attn_tc_kernel(
    const uint16_t* __restrict__ qg, const uint8_t* __restrict__ kv_codes,
    const uint8_t* __restrict__ kv_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, const int32_t* __restrict__ topk, int k,
    uint8_t* __restrict__ swa, const uint16_t* __restrict__ swa_new, int window, bool win_shared, float sm_scale,
    float* __restrict__ part_o, float* __restrict__ part_ml, int splits, void* __restrict__ out,
    bool out_f32, float* __restrict__ out_lse, Status* st, uint64_t wlim) {
    static_assert(HG == 1 || ((HG == 2 || HG == 4) && CLUSTER), "head groups are merged inside their cluster");
    constexpr int NH = kH / HG;  // heads of this CTA
    constexpr int NB = 2 * NH;   // P^T columns: hi parts, then lo parts
    constexpr int NJ = 16 / HG;  // 16-byte chunks of Q per thread
    constexpr int NC = NH >= 32 ? 4 : NH / 8;  // 8-head chunks of a softmax warp
    static_assert(E == kTcE || (E == kTcE2 && HG == 2), "160 entries per CTA with two head groups only");
    constexpr int T = E == kTcE ? kAttnThreads : kAttnThreads2;  // threads
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    AttnTcSmemT<E>& S = *reinterpret_cast<AttnTcSmemT<E>*>(smem_raw);
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int split = int(blockIdx.x) % splits, hg = int(blockIdx.x) / splits;
    const int64_t q = blockIdx.y;

    if (tid == 0) {
        mbar_init(&S.bar, 1);
        mbar_init_fence();
    }
    grid_dep_wait();
    grid_dep_launch();
    // every load of the thread first: the query's row range, its entry, Q
    const int64_t ks = kv_start[q];
    const int32_t nv = n_visible[q];
    // the sequence (top-k entries, then window entries) in groups of 32:
    // split s takes groups s, s + splits, s + 2 splits, ... (E / 32 of them),
    // so the splits get about the same mix and each warp one kind of entry
    const int ent = tid % E, qa = tid / E;  // entry; channel quarters qa, qa + 2
    // C row of entry e: itself, or (160 entries) 128 .. 159 first
    auto srow = [](int e) { return E == kTcE ? e : (e < kTcE ? e + (E - kTcE) : e - kTcE); };
    const int ge = ((ent >> 5) * splits + split) * 32 + (ent & 31);
    const int32_t pre = ge < k ? topk[q * k + ge] : -1;
    if (warp == 0) tmem_alloc(&S.tmem, kTcCols);
    // Q chunk j of this thread (16 bytes): head 8 (g / 16) + lane % 8 of the
    // CTA's heads, chunk 4 (g % 16) + lane / 8 with g = NJ warp + j.  A
    // quarter-warp covers 8 heads (8 distinct bank groups in the canonical
    // layout); an instruction reads 64 contiguous bytes of each of 8 rows.
    auto q_chunk = [&](int j) {
        const int g = NJ * warp + j;
        return (8 * (g >> 4) + (lane & 7)) * 64 + 4 * (g & 15) + (lane >> 3);
    };
    const bool qw = T == kAttnThreads || warp < kAttnThreads / 32;  // warps that carry Q
    uint4 qv[NJ];
    if (qw) {
        const uint4* qsrc = reinterpret_cast<const uint4*>(qg + q * (kH * kD) + hg * (NH * kD));
#pragma unroll
        for (int j = 0; j < NJ; ++j) qv[j] = __ldg(qsrc + q_chunk(j));
    }
    // the current token's bf16 window latent (two channels per thread), loaded
    // now by the split that holds its entry when the context fills the window
    // (the usual case), so it does not wait for the context length
    const bool pre_new = swa_new != nullptr && window > 0 && ((k + window - 1) >> 5) % splits == split;
    const uint32_t x_new =
        pre_new && tid < kD / 2 ? __ldg(reinterpret_cast<const uint32_t*>(swa_new + q * kD) + tid) : 0u;
    int32_t n = 0;  // per-query validity, reported once per query
    {
        const bool report = split == 0 && hg == 0 && tid == 0;
        if (ks < 0) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_KV_START, int32_t(q), int32_t(ks));
        } else if (nv < 0 || ks + nv > n_rows) {
            if (report) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_ROWS, int32_t(q), nv);
        } else {
            n = nv;
        }
    }
    const int nw = n < window ? n : window;
    // the current token's window entry, when this call appends it: its
    // position in this CTA (uniform over the CTA) or -1
    int cur_e = -1;
    if (swa_new != nullptr && nw > 0) {
        const int cur_ge = k + nw - 1, grp = cur_ge >> 5;
        if (grp % splits == split) cur_e = (grp / splits) * 32 + (cur_ge & 31);
    }
    // this thread's row: 0 none (zeros), 1 FP4 latent, 2 FP8 window, 3 the current token
    int kind = 0;
    uint4 rv[16];
    uint2 rs0 = make_uint2(0, 0), rs1 = make_uint2(0, 0);
    if (ge < k) {
        const int32_t p = pre;
        if (p >= 0 && p < n) {
            kind = 1;
            const int64_t row = ks + p;
            const uint4* src = reinterpret_cast<const uint4*>(kv_codes + row * 256);
            const uint2* ssrc = reinterpret_cast<const uint2*>(kv_scales + row * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                rv[j] = __ldg(src + qa * 4 + j);
                rv[4 + j] = __ldg(src + (qa + 2) * 4 + j);
            }
            rs0 = __ldg(ssrc + qa);
            rs1 = __ldg(ssrc + qa + 2);
        } else if (p < -1 || p >= n) {
            if (qa == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_TOPK, int32_t(q), p);
        }
    } else if (ge - k < nw) {
        if (ent == cur_e) {
            kind = 3;
        } else {
            kind = 2;
            const int64_t pos = int64_t(n - nw) + (ge - k);
            const uint4* ring = reinterpret_cast<const uint4*>(
                swa + (win_shared ? ks + pos : q * window + pos % window) * kD);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                rv[j] = ring[qa * 8 + j];
                rv[8 + j] = ring[(qa + 2) * 8 + j];
            }
        }
    }
    if (cur_e >= 0 && tid < kD / 2) {  // E4M3 of the current token's bf16 latent, two channels per thread: ring and C
        uint8_t* ring = swa + (q * window + int64_t(n - 1) % window) * kD;
        const uint32_t x = pre_new ? x_new : __ldg(reinterpret_cast<const uint32_t*>(swa_new + q * kD) + tid);
        const uint32_t b2 = e4m3x2_rn_sat(bf16_lo(x), bf16_hi(x));
        if (hg == 0) reinterpret_cast<uint16_t*>(ring)[tid] = static_cast<uint16_t>(b2);
        uint32_t h2[2];
        e4m3x4_to_f16x2(b2, h2);
        *reinterpret_cast<uint32_t*>(S.c + row512(srow(cur_e), tid >> 2) + (tid & 3) * 4) = h2[0];
    }
    // Q is stored as f16 times 2^-qs, qs chosen so that max|Q| 2^-qs lies in
    // [2^14, 2^15): exact for every element above max|Q| 2^-28, the rest within
    // 2^-25 absolute (scaled), far below the fp32 accumulation error
    {
        uint32_t am = 0;
#pragma unroll
        for (int j = 0; j < NJ && qw; ++j) {
            am = __vmaxu2(am, __vmaxu2(qv[j].x & 0x7FFF7FFFu, qv[j].y & 0x7FFF7FFFu));
            am = __vmaxu2(am, __vmaxu2(qv[j].z & 0x7FFF7FFFu, qv[j].w & 0x7FFF7FFFu));
        }
        am = __reduce_max_sync(0xffffffffu, max(am & 0xFFFFu, am >> 16));
        if (lane == 0 && qw) S.qmax[warp] = am;
    }
    __syncthreads();  // max |Q| per warp, the current token's row, the barrier
    int qs = 0;
    {
        uint32_t am = 0;
#pragma unroll
        for (int w = 0; w < kAttnThreads / 32; ++w) am = max(am, S.qmax[w]);
        if (am != 0) qs = int(am >> 7) - 127 - 14;  // bf16 exponent of max|Q| minus 14
        qs = qs < -126 ? -126 : (qs > 126 ? 126 : qs);
        const float qf = __uint_as_float(uint32_t(127 - qs) << 23);  // 2^-qs
#pragma unroll
        for (int j = 0; j < NJ && qw; ++j) {
            const int i = q_chunk(j);
            const uint32_t wv[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
            uint32_t o[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const __half2 h = __floats2half2_rn(__uint_as_float(wv[m] << 16) * qf,
                                                    __uint_as_float(wv[m] & 0xFFFF0000u) * qf);
                o[m] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(S.r0 + row512(i >> 6, i & 63)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    // dequantize this thread's row into C
    const int er = srow(ent);
    if (kind == 1) {
        fp4_quarter_to_c(rv, rs0, S.c, er, qa);
        fp4_quarter_to_c(rv + 4, rs1, S.c, er, qa + 2);
    } else if (kind == 2) {
        fp8_quarter_to_c(rv, S.c, er, qa);
        fp8_quarter_to_c(rv + 8, S.c, er, qa + 2);
    } else if (kind == 0) {
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2)
            for (int c = (qa + 2 * h2) * 16; c < (qa + 2 * h2) * 16 + 16; ++c)
                *reinterpret_cast<uint4*>(S.c + row512(er, c)) = make_uint4(0, 0, 0, 0);
    }
    if (qa == 0) S.ok[ent] = kind != 0;
    const float sm_eff = sm_scale * __uint_as_float(uint32_t(127 + qs) << 23);  // logits scale of the f16 S
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    const uint32_t sm_c = smem_addr(S.c), sm_r0 = smem_addr(S.r0);

    // S^T = C Q^T: 32 MMAs of K = 16 dims per 128-entry tile (160 entries:
    // storage rows 32 .. 159 into columns [0, NH), rows 0 .. 127 into
    // [NH, 2 NH), whose first 32 rows are entries 128 .. 159)
    if (tid == 0) {
        constexpr uint32_t id = idesc_f16(128, NH, 0, false, false);
#pragma unroll 1
        for (int t = 0; t < (E == kTcE ? 1 : 2); ++t) {
            const uint32_t a0 = sm_c + (E == kTcE || t == 1 ? 0u : uint32_t(E - kTcE) / 8 * 8192);
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_f16_ss(tmem + NH * t, umma_desc(a0 + kk * 256, 128, 8192), umma_desc(sm_r0 + kk * 256, 128, 8192),
                           id, kk > 0);
        }
        tc_commit(&S.bar);
    }
    // ok_mma: the MMAs issued so far are done.  A wait that gives up leaves
    // them in flight: the CTA then writes nothing more into C or the Q/P
    // area (their operands), takes part in the cluster barriers only, and
    // waits for them once more before TMEM is released.
    bool ok_mma = __syncthreads_and(mbar_wait(&S.bar, 0, wlim));
    uint32_t pending = ok_mma ? 0u : 1u;  // 1 + the parity of the MMA commit still outstanding
    tc_fence_after();

    // softmax statistics from the registers: warp -> entries 32 (warp % 4) +
    // lane, heads 32 (warp / 4) + j of the CTA's (warps 4..7 idle with 32
    // heads or fewer; with 16, columns 16..31 of the load are not S and are
    // masked).  P^T (f16 hi parts in columns [0, NH), lo parts in
    // [NH, NB) of the B operand) goes to the consumed Q area.
    // With 160 entries warps 0..3 take entries 32 warp + lane (tile 0) and
    // warp 4 entries 128 + lane (tile 1, lanes 0..31).
    uint8_t* pt = S.r0;
    float(*red)[kH] = reinterpret_cast<float(*)[kH]>(S.r0 + 32 * 1024);  // per entry row block, per head
    constexpr int NR = E / 32 > 4 ? E / 32 : 4;  // entry row blocks
    const int qd = warp & 3, hf = E == kTcE ? warp >> 2 : 0;
    const int rb = E == kTcE ? qd : warp;  // this warp's row block
    const int e = 32 * rb + lane;
    const bool sw = E == kTcE ? (HG == 1 || hf < (NH + 31) / 32) : warp < NR;
    if (ok_mma) {
        float x[32];
        if (sw) {
            uint32_t r[32];
            tmem_ld32(tmem + (uint32_t(32 * qd) << 16) + 32 * hf + (rb >= 4 ? NH : 0), r);
            tmem_ld_wait();
            const bool oke = S.ok[e];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = (oke && j < NH) ? sm_eff * __uint_as_float(r[j]) : -INFINITY;
        }
        // transpose-reduce: in the round with offset o each lane keeps half
        // of its values and takes the partner's matching half, so lane l
        // ends with head 32 hf + l
        auto reduce = [&](float(&v)[32], bool is_max) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < o; ++i) {
                    const float send = up ? v[i] : v[i + o];
                    const float keep = up ? v[i + o] : v[i];
                    const float got = __shfl_xor_sync(0xffffffffu, send, o);
                    v[i] = is_max ? fmaxf(keep, got) : keep + got;
                }
            }
            return v[0];
        };
        if (sw) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = x[j];
            red[rb][32 * hf + lane] = reduce(v, true);
        }
        __syncthreads();
        const int hl = 32 * hf + lane;
        float mh = 0.f;
        if (sw) {
            mh = red[0][hl];
#pragma unroll
            for (int b = 1; b < NR; ++b) mh = fmaxf(mh, red[b][hl]);  // this split's max
        }
        float lh = 0.f;
        if (sw) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float m = __shfl_sync(0xffffffffu, mh, j);
                x[j] = x[j] == -INFINITY ? 0.f : __expf(x[j] - m);
                v[j] = x[j];
            }
            lh = reduce(v, false);
        }
#pragma unroll
        for (int c = 0; c < NC && sw; ++c) {  // P^T hi and lo, 8 heads per 16-byte store
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float a = x[8 * c + 2 * t], b = x[8 * c + 2 * t + 1];
                const __half2 h2 = __floats2half2_rn(a, b);
                const float2 hb = __half22float2(h2);
                const __half2 l2 = __floats2half2_rn(a - hb.x, b - hb.y);
                hi[t] = *reinterpret_cast<const uint32_t*>(&h2);
                lo[t] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            *reinterpret_cast<uint4*>(pt + pmn<NB>(srow(e), 32 * hf + 8 * c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(pt + pmn<NB>(srow(e), NH + 32 * hf + 8 * c)) =
                make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        __syncthreads();  // every read of the maxima is done
        if (sw) red[rb][hl] = lh;
        __syncthreads();
        if (rb == 0 && sw) {  // (m, l) of head hl
            float l = red[0][hl] + red[1][hl] + red[2][hl] + red[3][hl];
#pragma unroll
            for (int b = 4; b < NR; ++b) l += red[b][hl];
            if (CLUSTER) {
                S.ml[hl][0] = mh;
                S.ml[hl][1] = l;
            } else {
                float* ml = part_ml + ((q * splits + split) * kH + hl) * 2;
                ml[0] = mh;
                ml[1] = l;
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // O^T = C^T P^T: 4 blocks of 128 dims (C is the MN-major A operand), each
    // into NB TMEM columns: heads' hi parts, then their lo parts (an M = 128
    // MMA costs the same at N = 128 as at N = 64).  Block 0 overwrites S^T,
    // which has been read.
    if (tid == 0 && ok_mma) {
        constexpr uint32_t id = idesc_f16(128, NB, 0, true, true);
        const uint32_t pb = smem_addr(pt);
        for (int mb = 0; mb < 4; ++mb) {
            const uint32_t d = tmem + NB * mb;
            for (int kk = 0; kk < E / 16; ++kk)
                mma_f16_ss(d, umma_desc(sm_c + mb * 2048 + kk * 16384, 8192, 128),
                           umma_desc(pb + kk * (32 * NB), 16 * NB, 128), id, kk > 0);
        }
        tc_commit(&S.bar);
    }
    if (ok_mma) {
        ok_mma = __syncthreads_and(mbar_wait(&S.bar, 1, wlim));
        if (!ok_mma) pending = 2u;
    }
    tc_fence_after();
    // warp -> dims 32*(warp%4) + lane of blocks 2*(warp/4), +1: to the
    // workspace, or (CLUSTER) to this CTA's shared memory (C is consumed)
    float* X = CLUSTER ? reinterpret_cast<float*>(S.c) : part_o + (q * splits + split) * int64_t(kH * kD);
    if (ok_mma && warp < 8) {
        for (int b2 = 0; b2 < 2; ++b2) {
            const int mb = 2 * (warp >> 2) + b2;
            const int dim = mb * 128 + 32 * (warp & 3) + lane;
            if (NH >= 32) {
#pragma unroll
                for (int half = 0; half < NH / 32; ++half) {
                    uint32_t rh[32], rl[32];
                    tmem_ld32(tmem + (uint32_t(32 * (warp & 3)) << 16) + NB * mb + 32 * half, rh);
                    tmem_ld32(tmem + (uint32_t(32 * (warp & 3)) << 16) + NB * mb + NH + 32 * half, rl);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        X[(32 * half + j) * kD + dim] = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
                }
            } else {  // 16 heads: hi and lo parts in one 32-column load
                uint32_t r[32];
                tmem_ld32(tmem + (uint32_t(32 * (warp & 3)) << 16) + NB * mb, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < NH; ++j) X[j * kD + dim] = __uint_as_float(r[j]) + __uint_as_float(r[NH + j]);
            }
        }
    } else if (tid == 0) {
        record(st, CSA2_ERR_TIMEOUT, 2, int32_t(q), split);
    }
    if (CLUSTER) {
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every partial and (m, l) of the query is visible
        const int rank = int(cluster.block_rank());
        float(*wts)[8] = reinterpret_cast<float(*)[8]>(S.r0);  // P is consumed: merge weights a_s / L
        if (pending == 0 && tid < NH) {  // merge weights of the CTA's head tid
            float mp[8], lp[8], M = -INFINITY;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                mp[p] = -INFINITY;
                lp[p] = 0.f;
                if (p < splits) {
                    const float2 v = *reinterpret_cast<const float2*>(cluster.map_shared_rank(&S.ml[tid][0], p));
                    mp[p] = v.x;
                    lp[p] = v.y;
                }
                M = fmaxf(M, mp[p]);
            }
            float L = 0.f, a[8];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                a[p] = (M == -INFINITY || mp[p] == -INFINITY) ? 0.f : __expf(mp[p] - M);
                L = fmaf(a[p], lp[p], L);
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int p = 0; p < 8; ++p) wts[tid][p] = a[p] * inv;
            if (rank == 0 && out_lse) out_lse[q * kH + hg * NH + tid] = L > 0.f ? M + logf(L) : -INFINITY;
        }
        __syncthreads();
        // this CTA reduces dims [lo, hi) (whole float4s) over all peers
        const int per = ((kD / 4 + splits - 1) / splits) * 4;
        const int lo = rank * per, hi = min(kD, lo + per);
        const int w4 = (hi - lo) / 4;
        const float4* px[8];
#pragma unroll
        for (int p = 0; p < 8; ++p)
            px[p] = reinterpret_cast<const float4*>(cluster.map_shared_rank(X, p < splits ? p : 0));
        for (int idx = tid; pending == 0 && idx < NH * w4; idx += T) {
            const int h = idx / w4, d4 = lo / 4 + idx % w4;
            float4 v[8];
#pragma unroll
            for (int p = 0; p < 8; ++p)
                v[p] = p < splits ? px[p][h * (kD / 4) + d4] : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float wgt = p < splits ? wts[h][p] : 0.f;
                o.x = fmaf(wgt, v[p].x, o.x);
                o.y = fmaf(wgt, v[p].y, o.y);
                o.z = fmaf(wgt, v[p].z, o.z);
                o.w = fmaf(wgt, v[p].w, o.w);
            }
            const int64_t oi = (q * kH + hg * NH + h) * int64_t(kD) + 4 * d4;
            if (out_f32) {
                *reinterpret_cast<float4*>(static_cast<float*>(out) + oi) = o;
            } else {
                const uint32_t a0 = uint32_t(bf16_bits(o.x)) | (uint32_t(bf16_bits(o.y)) << 16);
                const uint32_t a1 = uint32_t(bf16_bits(o.z)) | (uint32_t(bf16_bits(o.w)) << 16);
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + oi) = make_uint2(a0, a1);
            }
        }
        cluster.sync();  // peers are done reading this CTA's shared memory
    }
    if (tid == 0 && pending != 0) mbar_wait(&S.bar, pending - 1, kDrainNs);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTcCols);
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
    grid_dep_wait();
    grid_dep_launch();
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

// One CTA per query, for batches of many queries (prefill chunks): the
// query's entries in 128-entry chunks, one after another, with an online
// softmax, so no partial outputs and no merge.  Chunk c holds sequence
// entries [128 c, 128 c + 128) (top-k entries, then window entries).  S^T of
// a chunk goes to TMEM columns 256..319; O^T accumulates over the chunks in
// columns 0..255 (4 blocks of 128 dims x 64 heads: P's f16 hi and lo parts
// are two MMAs into the same columns, as the 512 columns cannot also hold
// them side by side), and is rescaled in TMEM whenever a head's running
// maximum rises.  The next chunk's index and rows are loaded while the
// current chunk's MMAs and softmax run.
constexpr uint32_t kQColO = 0, kQColS = 256, kQCols = 512;
// Batches of at least this many queries take attn_query_kernel: one wave of
// (split, query) CTAs no longer holds them, and one CTA per query avoids the
// fp32 partials and their merge.
constexpr int64_t kAttnQueryMin = 128;
struct AttnQSmem {
    uint8_t q[64 * 1024];             // Q f16 (B of S^T), for every chunk
    uint8_t c[kTcE * 1024];           // C of the current chunk
    uint8_t p[32 * 1024];             // P^T hi/lo of the current chunk
    float red[4][kH];                 // per lane quadrant, per head
    float m[kH], l[kH], alpha[kH];    // running max and sum, this chunk's rescale factor
    int ok[kTcE];                     // entry valid
    uint32_t qmax[kAttnThreads / 32];
    uint64_t bar;                     // MMA completion (per chunk: phase 0 S, phase 1 O)
    uint32_t tmem;
};

__global__ void __launch_bounds__(kAttnThreads, 1) attn_query_kernel(
    const uint16_t* __restrict__ qg, const uint8_t* __restrict__ kv_codes,
    const uint8_t* __restrict__ kv_scales, int64_t n_rows, const int64_t* __restrict__ kv_start,
    const int32_t* __restrict__ n_visible, const int32_t* __restrict__ topk, int k,
    uint8_t* __restrict__ swa, const uint16_t* __restrict__ swa_new, int window, bool win_shared, float sm_scale,
    void* __restrict__ out, bool out_f32, float* __restrict__ out_lse, Status* st, uint64_t wlim) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    AttnQSmem& S = *reinterpret_cast<AttnQSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int64_t q = blockIdx.x;

    if (tid == 0) {
        mbar_init(&S.bar, 1);
        mbar_init_fence();
    }
    grid_dep_wait();
    grid_dep_launch();
    const int64_t ks = kv_start[q];
    const int32_t nv = n_visible[q];
    const int ent = tid & (kTcE - 1), qa = tid >> 7;  // entry of a chunk; channel quarters qa, qa + 2
    const int32_t pre0 = ent < k ? topk[q * k + ent] : -1;
    if (warp == 0) tmem_alloc(&S.tmem, kQCols);
    auto q_chunk = [&](int j) {  // as in attn_tc_kernel
        const int g = 16 * warp + j;
        return (8 * (g >> 4) + (lane & 7)) * 64 + 4 * (g & 15) + (lane >> 3);
    };
    uint4 qv[16];
    {
        const uint4* qsrc = reinterpret_cast<const uint4*>(qg + q * (kH * kD));
#pragma unroll
        for (int j = 0; j < 16; ++j) qv[j] = __ldg(qsrc + q_chunk(j));
    }
    int32_t n = 0;
    if (ks < 0) {
        if (tid == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_KV_START, int32_t(q), int32_t(ks));
    } else if (nv < 0 || ks + nv > n_rows) {
        if (tid == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_ROWS, int32_t(q), nv);
    } else {
        n = nv;
    }
    const int nw = n < window ? n : window;
    const int cur_ge = (swa_new != nullptr && nw > 0) ? k + nw - 1 : -1;  // the current token's entry
    const int nchunks = (k + window + kTcE - 1) / kTcE;

    // this thread's row of sequence entry ge: kind 0 none (zeros), 1 FP4
    // latent, 2 FP8 window, 3 the current token
    int kind = 0;
    uint4 rv[16];
    uint2 rs0 = make_uint2(0, 0), rs1 = make_uint2(0, 0);
    auto load_row = [&](int ge, int32_t p) {
        kind = 0;
        if (ge < k) {
            if (p >= 0 && p < n) {
                kind = 1;
                const int64_t row = ks + p;
                const uint4* src = reinterpret_cast<const uint4*>(kv_codes + row * 256);
                const uint2* ssrc = reinterpret_cast<const uint2*>(kv_scales + row * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    rv[j] = __ldg(src + qa * 4 + j);
                    rv[4 + j] = __ldg(src + (qa + 2) * 4 + j);
                }
                rs0 = __ldg(ssrc + qa);
                rs1 = __ldg(ssrc + qa + 2);
            } else if (p < -1 || p >= n) {
                if (qa == 0) record(st, CSA2_ERR_DEVICE_BOUNDS, CHK_TOPK, int32_t(q), p);
            }
        } else if (ge - k < nw) {
            if (ge == cur_ge) {
                kind = 3;
            } else {
                kind = 2;
                const int64_t pos = int64_t(n - nw) + (ge - k);
                const uint4* ring = reinterpret_cast<const uint4*>(
                    swa + (win_shared ? ks + pos : q * window + pos % window) * kD);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    rv[j] = ring[qa * 8 + j];
                    rv[8 + j] = ring[(qa + 2) * 8 + j];
                }
            }
        }
    };
    load_row(ent, pre0);

    // Q as f16 times 2^-qs (as in attn_tc_kernel)
    {
        uint32_t am = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            am = __vmaxu2(am, __vmaxu2(qv[j].x & 0x7FFF7FFFu, qv[j].y & 0x7FFF7FFFu));
            am = __vmaxu2(am, __vmaxu2(qv[j].z & 0x7FFF7FFFu, qv[j].w & 0x7FFF7FFFu));
        }
        am = __reduce_max_sync(0xffffffffu, max(am & 0xFFFFu, am >> 16));
        if (lane == 0) S.qmax[warp] = am;
    }
    if (tid < kH) {
        S.m[tid] = -INFINITY;
        S.l[tid] = 0.f;
    }
    __syncthreads();  // max |Q| per warp, the running statistics, the barrier
    int qs = 0;
    {
        uint32_t am = 0;
#pragma unroll
        for (int w = 0; w < kAttnThreads / 32; ++w) am = max(am, S.qmax[w]);
        if (am != 0) qs = int(am >> 7) - 127 - 14;
        qs = qs < -126 ? -126 : (qs > 126 ? 126 : qs);
        const float qf = __uint_as_float(uint32_t(127 - qs) << 23);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = q_chunk(j);
            const uint32_t wv[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
            uint32_t o[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const __half2 h = __floats2half2_rn(__uint_as_float(wv[m] << 16) * qf,
                                                    __uint_as_float(wv[m] & 0xFFFF0000u) * qf);
                o[m] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(S.q + row512(i >> 6, i & 63)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    const float sm_eff = sm_scale * __uint_as_float(uint32_t(127 + qs) << 23);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    const uint32_t sm_c = smem_addr(S.c), sm_q = smem_addr(S.q), pb = smem_addr(S.p);
    const int qd = warp & 3, hf = warp >> 2, e = 32 * qd + lane, hl = 32 * hf + lane;
    float(*red)[kH] = S.red;
    // ok: every wait so far succeeded.  pend (thread 0): 1 + the parity of a
    // commit issued but not yet seen complete, else 0
    bool ok = true;
    uint32_t pend = 0;

    for (int c = 0; c < nchunks; ++c) {
        const int ge = c * kTcE + ent;
        // the next chunk's index, in flight while this chunk is processed
        const int ge2 = ge + kTcE;
        const int32_t pre_next = ge2 < k ? topk[q * k + ge2] : -1;
        if (c > 0) {  // C and P are free once the previous chunk's O MMA is done
            const bool w = __syncthreads_and(ok && mbar_wait(&S.bar, 1, wlim));
            if (w) pend = 0;
            ok = w;
            tc_fence_after();
        }
        if (cur_ge >= c * kTcE && cur_ge < (c + 1) * kTcE) {
            // two channels per thread: to the ring and into C
            const int ce = cur_ge - c * kTcE;
            uint8_t* ring = swa + (q * window + int64_t(n - 1) % window) * kD;
            const uint32_t x = __ldg(reinterpret_cast<const uint32_t*>(swa_new + q * kD) + tid);
            const uint32_t b2 = e4m3x2_rn_sat(bf16_lo(x), bf16_hi(x));
            reinterpret_cast<uint16_t*>(ring)[tid] = static_cast<uint16_t>(b2);
            uint32_t h2[2];
            e4m3x4_to_f16x2(b2, h2);
            if (ok) *reinterpret_cast<uint32_t*>(S.c + row512(ce, tid >> 2) + (tid & 3) * 4) = h2[0];
        }
        if (ok) {  // dequantize this thread's row into C
            if (kind == 1) {
                fp4_quarter_to_c(rv, rs0, S.c, ent, qa);
                fp4_quarter_to_c(rv + 4, rs1, S.c, ent, qa + 2);
            } else if (kind == 2) {
                fp8_quarter_to_c(rv, S.c, ent, qa);
                fp8_quarter_to_c(rv + 8, S.c, ent, qa + 2);
            } else if (kind == 0) {
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2)
                    for (int cc = (qa + 2 * h2) * 16; cc < (qa + 2 * h2) * 16 + 16; ++cc)
                        *reinterpret_cast<uint4*>(S.c + row512(ent, cc)) = make_uint4(0, 0, 0, 0);
            }
            if (qa == 0) S.ok[ent] = kind != 0;
        }
        // the next chunk's rows, in flight during this chunk's MMAs and softmax
        if (c + 1 < nchunks) load_row(ge2, pre_next);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // S^T = C Q^T (32 MMAs of K = 16 dims)
        if (tid == 0 && ok) {
            constexpr uint32_t id = idesc_f16(128, 64, 0, false, false);
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_f16_ss(tmem + kQColS, umma_desc(sm_c + kk * 256, 128, 8192), umma_desc(sm_q + kk * 256, 128, 8192),
                           id, kk > 0);
            tc_commit(&S.bar);
            pend = 1;
        }
        {
            const bool w = __syncthreads_and(ok && mbar_wait(&S.bar, 0, wlim));
            if (w) pend = 0;
            ok = w;
        }
        tc_fence_after();

        // softmax against the running maximum; P^T hi/lo into S.p
        float alpha_l = 1.f;  // this lane's head hl: rescale factor of the accumulated O
        if (ok) {
            float x[32];
            {
                uint32_t r[32];
                tmem_ld32(tmem + (uint32_t(32 * qd) << 16) + kQColS + 32 * hf, r);
                tmem_ld_wait();
                const bool oke = S.ok[e];
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = oke ? sm_eff * __uint_as_float(r[j]) : -INFINITY;
            }
            auto reduce = [&](float(&v)[32], bool is_max) {  // lane l ends with head 32 hf + l
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < o; ++i) {
                        const float send = up ? v[i] : v[i + o];
                        const float keep = up ? v[i + o] : v[i];
                        const float got = __shfl_xor_sync(0xffffffffu, send, o);
                        v[i] = is_max ? fmaxf(keep, got) : keep + got;
                    }
                }
                return v[0];
            };
            {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = x[j];
                red[qd][hl] = reduce(v, true);
            }
            __syncthreads();
            const float m_old = S.m[hl];
            const float mc = fmaxf(fmaxf(red[0][hl], red[1][hl]), fmaxf(red[2][hl], red[3][hl]));
            const float m_new = fmaxf(m_old, mc);
            alpha_l = m_old == -INFINITY ? 0.f : __expf(m_old - m_new);
            float lh;
            {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float m = __shfl_sync(0xffffffffu, m_new, j);
                    x[j] = x[j] == -INFINITY ? 0.f : __expf(x[j] - m);
                    v[j] = x[j];
                }
                lh = reduce(v, false);
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float a = x[8 * cc + 2 * t], b = x[8 * cc + 2 * t + 1];
                    const __half2 h2 = __floats2half2_rn(a, b);
                    const float2 hb = __half22float2(h2);
                    const __half2 l2 = __floats2half2_rn(a - hb.x, b - hb.y);
                    hi[t] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[t] = *reinterpret_cast<const uint32_t*>(&l2);
                }
                *reinterpret_cast<uint4*>(S.p + pmn(e, 32 * hf + 8 * cc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(S.p + pmn(e, 64 + 32 * hf + 8 * cc)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            __syncthreads();  // every read of the maxima is done
            red[qd][hl] = lh;
            __syncthreads();
            if (qd == 0) {
                const float lc = red[0][hl] + red[1][hl] + red[2][hl] + red[3][hl];
                S.l[hl] = S.l[hl] * alpha_l + lc;
                S.m[hl] = m_new;
                S.alpha[hl] = alpha_l;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // rescale the accumulated O where a head's maximum rose (uniform:
        // every warp reads the same factors)
        if (ok && c > 0) {
            const bool any = __any_sync(0xffffffffu, S.alpha[lane] != 1.f || S.alpha[lane + 32] != 1.f);
            if (any) {
                for (int b2 = 0; b2 < 2; ++b2) {
                    const int mb = 2 * (warp >> 2) + b2;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t ta = tmem + (uint32_t(32 * (warp & 3)) << 16) + kQColO + 64 * mb + 32 * half;
                        uint32_t r[32];
                        tmem_ld32(ta, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            r[j] = __float_as_uint(__uint_as_float(r[j]) * S.alpha[32 * half + j]);
                        tmem_st32(ta, r);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
            }
        }

        // O^T += C^T P^T: per block of 128 dims, the hi part then the lo part
        // into the same 64 columns
        if (tid == 0 && ok) {
            constexpr uint32_t id = idesc_f16(128, 64, 0, true, true);
            for (int mb = 0; mb < 4; ++mb) {
                const uint32_t d = tmem + kQColO + 64 * mb;
                for (int part = 0; part < 2; ++part)
                    for (int kk = 0; kk < kTcE / 16; ++kk)
                        mma_f16_ss(d, umma_desc(sm_c + mb * 2048 + kk * 16384, 8192, 128),
                                   umma_desc(pb + part * 1024 + kk * 4096, 2048, 128), id,
                                   c > 0 || part > 0 || kk > 0);
            }
            tc_commit(&S.bar);
            pend = 2;
        }
    }
    {
        const bool w = __syncthreads_and(ok && mbar_wait(&S.bar, 1, wlim));
        if (w) pend = 0;
        ok = w;
    }
    tc_fence_after();
    if (ok) {  // O / l, rounded once; warp -> dims 32 (warp % 4) + lane of blocks 2 (warp / 4), +1
        for (int b2 = 0; b2 < 2; ++b2) {
            const int mb = 2 * (warp >> 2) + b2;
            const int dim = mb * 128 + 32 * (warp & 3) + lane;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                tmem_ld32(tmem + (uint32_t(32 * (warp & 3)) << 16) + kQColO + 64 * mb + 32 * half, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int h = 32 * half + j;
                    const float L = S.l[h];
                    const float o = L > 0.f ? __uint_as_float(r[j]) / L : 0.f;
                    const int64_t oi = (q * kH + h) * int64_t(kD) + dim;
                    if (out_f32)
                        static_cast<float*>(out)[oi] = o;
                    else
                        static_cast<uint16_t*>(out)[oi] = bf16_bits(o);
                }
            }
        }
        if (out_lse && tid < kH) {
            const float L = S.l[tid];
            out_lse[q * kH + tid] = L > 0.f ? S.m[tid] + logf(L) : -INFINITY;
        }
    } else if (tid == 0) {
        record(st, CSA2_ERR_TIMEOUT, 5, int32_t(q), 0);
    }
    if (tid == 0 && pend != 0) mbar_wait(&S.bar, pend - 1, kDrainNs);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kQCols);
}

// Opt the variants into their shared memory and note how many clusters of
// `splits` CTAs can be resident at once (0 when clusters are unavailable),
// for 128 entries per CTA and (max_clusters2) for 160.
template <class Kernel>
static int max_active_clusters(Kernel kernel, int threads, size_t smem, int c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(c), 1, 1);
    cfg.blockDim = dim3(unsigned(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        n = 0;
        cudaGetLastError();
    }
    return n;
}

static csa2_status prepare_attn_tc(int splits, int splits2, int* max_clusters, int* max_clusters2) {
    static bool done[64] = {};
    static int cached[64][9] = {}, cached2[64][9] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(attn_tc_kernel<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnTcSmem))) != cudaSuccess ||
            cudaFuncSetAttribute(attn_tc_kernel<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnTcSmem))) != cudaSuccess ||
            cudaFuncSetAttribute(attn_tc_kernel<true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnTcSmem))) != cudaSuccess ||
            cudaFuncSetAttribute(attn_tc_kernel<true, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnTcSmem))) != cudaSuccess ||
            cudaFuncSetAttribute(attn_tc_kernel<true, 2, kTcE2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnTcSmemT<kTcE2>))) != cudaSuccess ||
            cudaFuncSetAttribute(attn_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(AttnQSmem))) != cudaSuccess)
            return CSA2_ERR_CUDA;
        for (int c = 1; c <= 8; ++c) {
            cached[dev][c] = max_active_clusters(attn_tc_kernel<true, 1>, kAttnThreads, sizeof(AttnTcSmem), c);
            cached2[dev][c] =
                max_active_clusters(attn_tc_kernel<true, 2, kTcE2>, kAttnThreads2, sizeof(AttnTcSmemT<kTcE2>), c);
        }
        done[dev] = true;
    }
    *max_clusters = (splits >= 1 && splits <= 8) ? cached[dev][splits] : 0;
    *max_clusters2 = (splits2 >= 1 && splits2 <= 8) ? cached2[dev][splits2] : 0;
    return CSA2_OK;
}

}  // namespace csa2

using namespace csa2;

// csa2_sparse_attn and csa2_sparse_attn_prefill: swa is a ring per query
// (win_shared false) or rows of the shared sequence (true).
static csa2_status sparse_attn(const void* q_bf16, int64_t n_q, const uint8_t* kv_codes, const uint8_t* kv_scales,
                               int64_t n_rows, const int64_t* kv_start, const int32_t* n_visible,
                               const int32_t* topk, int k, uint8_t* swa, const void* swa_new_bf16, int window,
                               bool win_shared, float sm_scale, void* out, int out_dtype, float* out_lse, void* ws,
                               size_t ws_bytes, cudaStream_t s) {
    if (n_q < 0 || n_rows < 0 || k < 0 || k > kMaxTopk || window < 0 || window > kMaxWindow)
        return CSA2_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || !(sm_scale < FLT_MAX)) return CSA2_ERR_INVALID_ARG;
    if (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32) return CSA2_ERR_INVALID_ARG;
    if (!q_bf16 || !kv_codes || !kv_scales || !kv_start || !n_visible || !out) return CSA2_ERR_INVALID_ARG;
    if (k > 0 && !topk) return CSA2_ERR_INVALID_ARG;
    if (window > 0 && !swa) return CSA2_ERR_INVALID_ARG;
    if (swa_new_bf16 && (window == 0 || win_shared || !aligned16(swa_new_bf16))) return CSA2_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(kv_codes) || !aligned16(out) || (swa && !aligned16(swa)))
        return CSA2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv_scales) & 7) return CSA2_ERR_INVALID_ARG;
    if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;  // grid.y of the split kernel (the per-query kernel uses grid.x)
    const AttnWs L = attn_ws(n_q, k, window);
    if (!ws || !aligned16(ws) || ws_bytes < L.total) return CSA2_ERR_WORKSPACE;
    if (n_q == 0) return CSA2_OK;
    char* base = static_cast<char*>(ws);
    Status* st = reinterpret_cast<Status*>(base);
    float* part_o = reinterpret_cast<float*>(base + L.part_o);
    float* part_ml = reinterpret_cast<float*>(base + L.part_ml);
    const uint16_t* q = static_cast<const uint16_t*>(q_bf16);
    const uint16_t* sn = static_cast<const uint16_t*>(swa_new_bf16);
    const bool f32 = out_dtype == CSA2_OUT_F32;
    int max_clusters = 0, max_clusters2 = 0;
    const int splits2 = (k + window + kTcE2 - 1) / kTcE2;  // splits of 160 entries
    csa2_status e = prepare_attn_tc(L.splits, splits2, &max_clusters, &max_clusters2);
    if (e != CSA2_OK) return e;
    if (n_q >= kAttnQueryMin && k + window > 0) {
        // many queries: one CTA per query over all its entries, no merge
        timer_begin(K_ATTN_SPLIT, s);
        const cudaError_t lq = launch(attn_query_kernel, dim3(unsigned(n_q)), kAttnThreads, sizeof(AttnQSmem), s, 1,
                                      q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, sn, window,
                                      win_shared, sm_scale, out, f32, out_lse, st, wait_limit_ns());
        timer_end(K_ATTN_SPLIT, s);
        return lq == cudaSuccess ? launch_status() : CSA2_ERR_CUDA;
    }
    // one cluster per query when every cluster of the launch is resident at
    // once; one cluster per half or quarter of the heads when those fit too,
    // with at most one CTA per multiprocessor; else halves of the heads over
    // fewer splits of 160 entries
    const bool cluster = L.splits <= 8 && n_q <= max_clusters;
    auto fits = [&](int hg) { return cluster && hg * n_q <= max_clusters && hg * n_q * L.splits <= sm_count(); };
    const int hg = fits(4) ? 4 : fits(2) ? 2 : 1;
    const bool e160 = hg == 1 && cluster && splits2 < L.splits && splits2 <= 8 && 2 * n_q <= max_clusters2 &&
                      2 * n_q * splits2 <= sm_count();
    const dim3 grid(static_cast<unsigned>(e160 ? 2 * splits2 : L.splits * hg), static_cast<unsigned>(n_q), 1);
    timer_begin(K_ATTN_SPLIT, s);
    const cudaError_t le =
        e160      ? launch(attn_tc_kernel<true, 2, kTcE2>, grid, kAttnThreads2, sizeof(AttnTcSmemT<kTcE2>), s,
                           unsigned(splits2), q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, sn,
                           window, win_shared, sm_scale, part_o, part_ml, splits2, out, f32, out_lse, st,
                           wait_limit_ns())
        : hg == 4 ? launch(attn_tc_kernel<true, 4>, grid, kAttnThreads, sizeof(AttnTcSmem), s, unsigned(L.splits), q,
                           kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, sn, window, win_shared,
                           sm_scale, part_o, part_ml, L.splits, out, f32, out_lse, st, wait_limit_ns())
        : hg == 2 ? launch(attn_tc_kernel<true, 2>, grid, kAttnThreads, sizeof(AttnTcSmem), s, unsigned(L.splits), q,
                           kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, sn, window, win_shared,
                           sm_scale, part_o, part_ml, L.splits, out, f32, out_lse, st, wait_limit_ns())
        : cluster ? launch(attn_tc_kernel<true, 1>, grid, kAttnThreads, sizeof(AttnTcSmem), s, unsigned(L.splits), q,
                           kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, sn, window, win_shared,
                           sm_scale, part_o, part_ml, L.splits, out, f32, out_lse, st, wait_limit_ns())
                  : launch(attn_tc_kernel<false, 1>, grid, kAttnThreads, sizeof(AttnTcSmem), s, 1, q, kv_codes,
                           kv_scales, n_rows, kv_start, n_visible, topk, k, swa, sn, window, win_shared, sm_scale,
                           part_o, part_ml, L.splits, out, f32, out_lse, st, wait_limit_ns());
    timer_end(K_ATTN_SPLIT, s);
    if (le != cudaSuccess) return CSA2_ERR_CUDA;
    if (cluster) return launch_status();
    timer_begin(K_ATTN_MERGE, s);
    if (f32)
        launch(attn_merge_kernel<true>, dim3(unsigned(n_q), kH / 8), 256, 0, s, 1, part_o, part_ml, L.splits, out,
               out_lse);
    else
        launch(attn_merge_kernel<false>, dim3(unsigned(n_q), kH / 8), 256, 0, s, 1, part_o, part_ml, L.splits, out,
               out_lse);
    timer_end(K_ATTN_MERGE, s);
    return launch_status();
}

extern "C" csa2_status csa2_sparse_attn(const void* q_bf16, int64_t n_q, const uint8_t* kv_codes,
                                        const uint8_t* kv_scales, int64_t n_rows,
                                        const int64_t* kv_start, const int32_t* n_visible,
                                        const int32_t* topk, int k, uint8_t* swa,
                                        const void* swa_new_bf16, int window, float sm_scale, void* out,
                                        int out_dtype, float* out_lse, void* ws, size_t ws_bytes,
                                        csa2_stream_t stream) {
    return sparse_attn(q_bf16, n_q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k, swa, swa_new_bf16,
                       window, false, sm_scale, out, out_dtype, out_lse, ws, ws_bytes, cudaStream_t(stream));
}

extern "C" csa2_status csa2_sparse_attn_prefill(const void* q_bf16, int64_t n_q, const uint8_t* kv_codes,
                                                const uint8_t* kv_scales, int64_t n_rows,
                                                const int64_t* kv_start, const int32_t* n_visible,
                                                const int32_t* topk, int k, const uint8_t* swa_rows, int window,
                                                float sm_scale, void* out, int out_dtype, float* out_lse,
                                                void* ws, size_t ws_bytes, csa2_stream_t stream) {
    return sparse_attn(q_bf16, n_q, kv_codes, kv_scales, n_rows, kv_start, n_visible, topk, k,
                       const_cast<uint8_t*>(swa_rows), nullptr, window, true, sm_scale, out, out_dtype, out_lse, ws,
                       ws_bytes, cudaStream_t(stream));
}
