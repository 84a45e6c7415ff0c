// RMSNorm fused with the projection, the product on tcgen05 (gemv_umma.cuh):
// bf16 and fp16, with and without the residual add, without a cluster or
// with the norm shared by one.
#include "gemv_umma.cuh"
#include "registry.h"

namespace rmsk {

#define RMSK_GEMV_UMMA(T, RES)                                                        \
    {(const void *)&rms_gemv_umma<T, RES, 1>, (const void *)&rms_gemv_umma<T, RES, kUmmaCluster>}

const GemvUmmaKernels gemv_umma_kernels = {
    {{RMSK_GEMV_UMMA(bf16, false), RMSK_GEMV_UMMA(bf16, true)},
     {RMSK_GEMV_UMMA(f16, false), RMSK_GEMV_UMMA(f16, true)}}};

} // namespace rmsk
