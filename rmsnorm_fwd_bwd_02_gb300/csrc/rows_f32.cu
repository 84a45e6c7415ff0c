// Row-wise fp32 kernels.
#include "registry.h"
#include "rows.cuh"

namespace rmsk {
//                       |-------- forward --------|  |-------- backward -------|
//        name     type   E    L   V  G  S MINB exact    L   V  G  S MINB exact
RMSK_ROWS(f_h896,  float, 4,   32,  7, 1, 8, 1, true,    32,  7, 1, 8, 1, true)   // H == 896
RMSK_ROWS(f_g32,   float, 4,   32,  4, 1, 8, 1, false,   32,  4, 1, 8, 1, false)  // H <= 512
RMSK_ROWS(f_g128,  float, 4,  128,  4, 1, 1, 1, false,  128,  4, 1, 1, 1, false)  // H <= 2048
RMSK_ROWS(f_g512,  float, 4,  512,  8, 1, 1, 1, false,  512,  8, 1, 1, 1, false)  // H <= 16384
RMSK_ROWS(f_s32,   float, 1,   32, 16, 1, 8, 1, false,   32, 16, 1, 8, 1, false)  // H <= 512
RMSK_ROWS(f_s1024, float, 1, 1024, 16, 1, 1, 1, false, 1024, 16, 1, 1, 1, false)  // H <= 16384
} // namespace rmsk
