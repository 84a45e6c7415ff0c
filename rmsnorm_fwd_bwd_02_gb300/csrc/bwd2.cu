// Double-backward kernels (bwd2.cuh): 16-byte packs with column masking for
// any H, one exact layout for the Qwen3-8B width, and one element per
// access for rows that are not 16-byte aligned.
#include "bwd2.cuh"
#include "registry.h"

namespace rmsk {

#define RMSK_BWD2(NAME, T, E, L, V, S, MINB, EXACT) \
    const Bwd2Kernel NAME = {#NAME, {E, L, V, 1, S, EXACT},  \
                             (const void *)&rms_bwd2_rows<T, E, L, V, S, MINB, EXACT>};

//        name         type   E    L   V  S MINB exact
RMSK_BWD2(b2_bf_g32,   bf16,  8,   32, 4, 8, 1, false)   // H <= 1024
RMSK_BWD2(b2_bf_g128,  bf16,  8,  128, 4, 1, 1, false)   // H <= 4096
RMSK_BWD2(b2_bf_h4096, bf16,  8,  128, 4, 1, 2, true)    // H == 4096
RMSK_BWD2(b2_bf_g512,  bf16,  8,  512, 4, 1, 1, false)   // H <= 16384
RMSK_BWD2(b2_bf_s1024, bf16,  1, 1024, 16, 1, 1, false)  // unaligned rows
RMSK_BWD2(b2_h_g32,    f16,   8,   32, 4, 8, 1, false)
RMSK_BWD2(b2_h_g128,   f16,   8,  128, 4, 1, 1, false)
RMSK_BWD2(b2_h_h4096,  f16,   8,  128, 4, 1, 2, true)
RMSK_BWD2(b2_h_g512,   f16,   8,  512, 4, 1, 1, false)
RMSK_BWD2(b2_h_s1024,  f16,   1, 1024, 16, 1, 1, false)
RMSK_BWD2(b2_f_g32,    float, 4,   32, 4, 8, 1, false)   // H <= 512
RMSK_BWD2(b2_f_g128,   float, 4,  128, 4, 1, 1, false)   // H <= 2048
RMSK_BWD2(b2_f_g512,   float, 4,  512, 8, 1, 1, false)   // H <= 16384
RMSK_BWD2(b2_f_s1024,  float, 1, 1024, 16, 1, 1, false)

} // namespace rmsk
