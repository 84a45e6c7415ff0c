// Row-wise fp16 kernels for any other feature count: the bf16 layouts of
// rows_bf16_generic.cu with fp16 storage.
#include "registry.h"
#include "rows.cuh"

namespace rmsk {
//                      |-------- forward --------|  |-------- backward -------|
//        name     type E    L   V  G  S MINB exact    L   V  G  S MINB exact
RMSK_ROWS(h_g32,   f16, 8,   32,  4, 1, 8, 1, false,   32,  4, 1, 8, 1, false)  // H <= 1024
RMSK_ROWS(h_g128,  f16, 8,  128,  4, 1, 1, 1, false,  128,  4, 1, 1, 1, false)  // H <= 4096
RMSK_ROWS(h_g512,  f16, 8,  512,  4, 1, 1, 1, false,  512,  4, 1, 1, 1, false)  // H <= 16384
RMSK_ROWS(h_s32,   f16, 1,   32, 16, 1, 8, 1, false,   32, 16, 1, 8, 1, false)  // H <= 512
RMSK_ROWS(h_s1024, f16, 1, 1024, 16, 1, 1, 1, false, 1024, 16, 1, 1, 1, false)  // H <= 16384
} // namespace rmsk
