// ABI utilities: version, status strings, workspace sizing, status word.
#include "csa2_common.cuh"
#include "csa2_layout.cuh"
#include "csa2_timer.cuh"

#include <atomic>
#include <vector>

namespace csa2 {
csa2_status launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

int sm_count() {
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// ---- instrumentation: launch counter and per-kernel event pairs
static std::atomic<int64_t> g_launches{0};
struct KernelTimer {
    bool on = false;
    int used = 0;
    std::vector<cudaEvent_t> ev;  // 2 per recorded launch
};
static KernelTimer g_timer[K_COUNT];

void timer_begin(int id, cudaStream_t s) {
    KernelTimer& t = g_timer[id];
    if (t.on && 2 * t.used + 1 < int(t.ev.size())) cudaEventRecord(t.ev[2 * t.used], s);
}
void timer_end(int id, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    KernelTimer& t = g_timer[id];
    if (t.on && 2 * t.used + 1 < int(t.ev.size())) {
        cudaEventRecord(t.ev[2 * t.used + 1], s);
        ++t.used;
    }
}

static const char* kKernelNames[K_COUNT] = {
    "scan_blockmax", "select_blocks", "pool_score", "select_topk", "attn_split",
    "attn_merge", "quantize_fp4", "quantize_fp8", "rope_table"};
}  // namespace csa2

using namespace csa2;

extern "C" int csa2_abi_version(void) { return 1; }

extern "C" const char* csa2_status_string(csa2_status s) {
    switch (s) {
        case CSA2_OK: return "ok";
        case CSA2_ERR_INVALID_ARG: return "invalid argument";
        case CSA2_ERR_UNSUPPORTED: return "unsupported shape or format";
        case CSA2_ERR_CUDA: return "CUDA error";
        case CSA2_ERR_TIMEOUT: return "device wait timed out";
        case CSA2_ERR_DEVICE_BOUNDS: return "device bounds check failed (item skipped)";
        case CSA2_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

extern "C" size_t csa2_workspace_bytes(int op, int64_t n_q, int32_t max_visible, int pool_blocks,
                                       int topk) {
    if (n_q < 0 || max_visible < 0) return 0;
    switch (op) {
        case CSA2_OP_APPEND: return CSA2_STATUS_BYTES;
        case CSA2_OP_INDEX_FULL:
            if (pool_blocks < 1 || topk < 1) return 0;
            return index_full_ws(n_q, max_visible, pool_blocks, topk).total;
        case CSA2_OP_INDEX_REINDEX:
            if (pool_blocks < 1 || topk < 1) return 0;
            return reindex_ws(n_q, pool_blocks).total;
        case CSA2_OP_SPARSE_ATTN: {
            if (topk < 0) return 0;
            size_t m = 0;  // the split count depends on the window: take the largest
            for (int win = 0; win <= kMaxWindow; ++win) {
                const size_t t = attn_ws(n_q, topk, win).total;
                m = t > m ? t : m;
            }
            return m;
        }
        default: return 0;
    }
}

extern "C" csa2_status csa2_status_reset(void* ws, csa2_stream_t stream) {
    if (!ws) return CSA2_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, CSA2_STATUS_BYTES, cudaStream_t(stream)) == cudaSuccess
               ? CSA2_OK : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_status_fetch(const void* ws, int32_t out[4], csa2_stream_t stream) {
    if (!ws || !out) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = cudaStream_t(stream);
    if (cudaMemcpyAsync(out, ws, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return CSA2_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

extern "C" int64_t csa2_launch_count(void) { return g_launches.load(); }

static std::atomic<uint64_t> g_wait_ns{2000000000ull};
uint64_t csa2::wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

extern "C" csa2_status csa2_debug_wait_limit(int64_t ns) {
    if (ns < 0) return CSA2_ERR_INVALID_ARG;
    g_wait_ns.store(ns == 0 ? 2000000000ull : uint64_t(ns), std::memory_order_relaxed);
    return CSA2_OK;
}

extern "C" const char* csa2_kernel_name(int kernel_id) {
    return (kernel_id >= 0 && kernel_id < K_COUNT) ? kKernelNames[kernel_id] : "unknown";
}

extern "C" csa2_status csa2_timer_enable(int kernel_id, int max_launches) {
    if (kernel_id < 0 || kernel_id >= K_COUNT || max_launches < 1 || max_launches > 100000)
        return CSA2_ERR_INVALID_ARG;
    KernelTimer& t = g_timer[kernel_id];
    for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
    t.ev.assign(size_t(2 * max_launches), nullptr);
    for (auto& e : t.ev)
        if (cudaEventCreate(&e) != cudaSuccess) return CSA2_ERR_CUDA;
    t.used = 0;
    t.on = true;
    return CSA2_OK;
}

extern "C" csa2_status csa2_timer_read(int kernel_id, double* total_ms, int32_t* launches) {
    if (kernel_id < 0 || kernel_id >= K_COUNT || !total_ms || !launches) return CSA2_ERR_INVALID_ARG;
    KernelTimer& t = g_timer[kernel_id];
    double sum = 0.0;
    for (int i = 0; i < t.used; ++i) {
        if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess) return CSA2_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess) return CSA2_ERR_CUDA;
        sum += ms;
    }
    *total_ms = sum;
    *launches = t.used;
    for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
    t.ev.clear();
    t.used = 0;
    t.on = false;
    return CSA2_OK;
}
