// Row-wise bf16 kernels for any other feature count: 16-byte packs with
// column masking, and the one-element-per-access kernels for rows that are
// not 16-byte aligned.
#include "registry.h"
#include "rows.cuh"

namespace rmsk {
//                      |-------- forward --------|  |-------- backward -------|
//        name     type  E    L   V  G  S MINB exact    L   V  G  S MINB exact
RMSK_ROWS(b_g32,   bf16, 8,   32,  4, 1, 8, 1, false,   32,  4, 1, 8, 1, false)  // H <= 1024
RMSK_ROWS(b_g128,  bf16, 8,  128,  4, 1, 1, 1, false,  128,  4, 1, 1, 1, false)  // H <= 4096
RMSK_ROWS(b_g512,  bf16, 8,  512,  4, 1, 1, 1, false,  512,  4, 1, 1, 1, false)  // H <= 16384
RMSK_ROWS(b_s32,   bf16, 1,   32, 16, 1, 8, 1, false,   32, 16, 1, 8, 1, false)  // H <= 512
RMSK_ROWS(b_s1024, bf16, 1, 1024, 16, 1, 1, 1, false, 1024, 16, 1, 1, 1, false)  // H <= 16384
} // namespace rmsk
