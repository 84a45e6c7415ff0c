// Row-wise fp16 kernels for the Qwen3 feature counts: the bf16 layouts of
// rows_bf16_shaped.cu with fp16 storage.
#include "registry.h"
#include "rows.cuh"

namespace rmsk {
//                      |------- forward -------|  |------- backward ------|
//        name     type E   L  V  G   S MINB exact  L  V  G   S MINB exact
RMSK_ROWS(h_h128,  f16, 8,  16, 1, 2, 16, 1, true,  16, 1, 4, 16, 2, true)
RMSK_ROWS(h_h896,  f16, 8,  16, 7, 1, 16, 1, true,  16, 7, 1,  8, 1, true)
RMSK_ROWS(h_h4096, f16, 8, 128, 4, 2,  1, 4, true, 128, 4, 2,  1, 2, true)
RMSK_ROWS(h_h5120, f16, 8, 320, 2, 1,  1, 2, true, 640, 1, 1,  1, 2, true)

//                       |--------- forward ---------|  |-------- backward --------|
//         name      type E   L  V  G   S MINB exact  E   L  V  G   S MINB exact
RMSK_ROWS2(h_h128w,  f16, 16,  8, 1, 4, 16, 2, true,  8,  16, 1, 4, 16, 2, true)
RMSK_ROWS2(h_h4096w, f16, 16, 64, 4, 2,  1, 4, true,  8, 128, 4, 2,  1, 2, true)
RMSK_ROWS2(h_h5120w, f16, 16,160, 2, 1,  1, 2, true,  8, 640, 1, 1,  1, 2, true)
} // namespace rmsk
