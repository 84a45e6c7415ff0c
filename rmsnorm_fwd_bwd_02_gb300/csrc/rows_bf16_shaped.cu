// Row-wise bf16 kernels shaped for the Qwen3 feature counts the workloads
// use: 128 (head_dim, QK-norm), 896 (0.8B decode hidden), 4096 (8B hidden),
// 5120 (14B hidden).
#include "registry.h"
#include "rows.cuh"

namespace rmsk {
//        name     type  E    L  V  G   S  MINB exact
RMSK_ROWS(b_h128,  bf16, 8,  16, 1, 2, 16, 1, true)
RMSK_ROWS(b_h896,  bf16, 8,  16, 7, 1, 16, 2, true)
RMSK_ROWS(b_h4096, bf16, 8, 256, 2, 2,  1, 2, true)
RMSK_ROWS(b_h5120, bf16, 8, 640, 1, 2,  1, 1, true)
} // namespace rmsk
