// RMSNorm fused with the projection GEMV: the register-fed kernel
// (gemv.cuh) and the bulk-copy fed one (gemv_tma.cuh), bf16 and fp16, an
// 8-row y tile (M <= 8) or one to four 16-row tiles, with and without the
// residual add.
#include "gemv.cuh"
#include "gemv_tma.cuh"
#include "registry.h"

namespace rmsk {

// [plain, residual with r read from L2, residual with r staged]
#define RMSK_GEMV_MT(T, MT, HALF)                              \
    {(const void *)&rms_gemv<T, MT, HALF, false, false>,       \
     (const void *)&rms_gemv<T, MT, HALF, true, false>,        \
     (const void *)&rms_gemv<T, MT, HALF, true, true>}

// [dtype][tiles: 0 = the 8-row tile, 1..4 = that many 16-row tiles][variant]
const GemvKernels gemv_kernels = {
    {{RMSK_GEMV_MT(bf16, 1, true), RMSK_GEMV_MT(bf16, 1, false), RMSK_GEMV_MT(bf16, 2, false),
      RMSK_GEMV_MT(bf16, 3, false), RMSK_GEMV_MT(bf16, 4, false)},
     {RMSK_GEMV_MT(f16, 1, true), RMSK_GEMV_MT(f16, 1, false), RMSK_GEMV_MT(f16, 2, false),
      RMSK_GEMV_MT(f16, 3, false), RMSK_GEMV_MT(f16, 4, false)}}};

#define RMSK_GEMV_TMA_MT(T, MT, HALF, CS)                          \
    {(const void *)&rms_gemv_tma<T, MT, HALF, false, false, CS>,   \
     (const void *)&rms_gemv_tma<T, MT, HALF, true, false, CS>,    \
     (const void *)&rms_gemv_tma<T, MT, HALF, true, true, CS>}

// the bulk-copy fed variants, same indexing; above 16 rows the norm is
// shared by a cluster of kGemvCluster CTAs
const GemvKernels gemv_tma_kernels = {
    {{RMSK_GEMV_TMA_MT(bf16, 1, true, 1), RMSK_GEMV_TMA_MT(bf16, 1, false, 1),
      RMSK_GEMV_TMA_MT(bf16, 2, false, kGemvCluster),
      RMSK_GEMV_TMA_MT(bf16, 3, false, kGemvCluster),
      RMSK_GEMV_TMA_MT(bf16, 4, false, kGemvCluster)},
     {RMSK_GEMV_TMA_MT(f16, 1, true, 1), RMSK_GEMV_TMA_MT(f16, 1, false, 1),
      RMSK_GEMV_TMA_MT(f16, 2, false, kGemvCluster),
      RMSK_GEMV_TMA_MT(f16, 3, false, kGemvCluster),
      RMSK_GEMV_TMA_MT(f16, 4, false, kGemvCluster)}}};

} // namespace rmsk
