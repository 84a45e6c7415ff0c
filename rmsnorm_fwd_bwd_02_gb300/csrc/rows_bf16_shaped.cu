// Row-wise bf16 kernels shaped for the Qwen3 feature counts the workloads
// use: 128 (head_dim, QK-norm), 896 (0.8B decode hidden), 4096 (8B hidden),
// 5120 (14B hidden). Layouts chosen by measurement on GB300.
#include "registry.h"
#include "rows.cuh"

namespace rmsk {
//                      |------- forward -------|  |------- backward ------|
//        name     type  E   L  V  G   S MINB exact  L  V  G   S MINB exact
RMSK_ROWS(b_h128,  bf16, 8,  16, 1, 2, 16, 1, true,  16, 1, 4, 16, 2, true)
RMSK_ROWS(b_h896,  bf16, 8,  16, 7, 1, 16, 1, true,  16, 7, 1,  8, 1, true)
RMSK_ROWS(b_h4096, bf16, 8, 128, 4, 2,  1, 4, true, 128, 4, 2,  1, 2, true)
RMSK_ROWS(b_h5120, bf16, 8, 320, 2, 1,  1, 2, true, 640, 1, 1,  1, 2, true)

// Rows 32-byte aligned: the forward moves 32-byte packs (one instruction per
// 16 bf16), the backward is the one above.
//                       |--------- forward ---------|  |-------- backward --------|
//         name      type  E   L  V  G   S MINB exact  E   L  V  G   S MINB exact
RMSK_ROWS2(b_h128w,  bf16, 16,  8, 1, 4, 16, 2, true,  8,  16, 1, 4, 16, 2, true)
RMSK_ROWS2(b_h4096w, bf16, 16, 64, 4, 2,  1, 4, true,  8, 128, 4, 2,  1, 2, true)
RMSK_ROWS2(b_h5120w, bf16, 16,160, 2, 1,  1, 2, true,  8, 640, 1, 1,  1, 2, true)
} // namespace rmsk
