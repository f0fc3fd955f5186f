// Launch accounting and optional per-kernel event timing (instrumentation,
// off by default; the compute path does not depend on it).
#pragma once

#include <cuda_runtime.h>

namespace csa2 {

enum KernelId {
    K_SCAN = 0,
    K_SELECT_BLOCKS = 1,
    K_POOL_SCORE = 2,
    K_SELECT_TOPK = 3,
    K_ATTN_SPLIT = 4,
    K_ATTN_MERGE = 5,
    K_QUANT_FP4 = 6,
    K_QUANT_FP8 = 7,
    K_ROPE_TABLE = 8,
    K_COUNT = 9
};

void timer_begin(int id, cudaStream_t s);
void timer_end(int id, cudaStream_t s);  // also counts the launch

}  // namespace csa2
