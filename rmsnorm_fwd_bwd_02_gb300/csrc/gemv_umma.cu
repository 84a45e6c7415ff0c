// RMSNorm fused with the projection, the product on tcgen05 with K split
// over a cluster (gemv_umma.cuh): bf16 and fp16, with and without the
// residual add.
#include "gemv_umma.cuh"
#include "registry.h"

namespace rmsk {

const GemvUmmaKernels gemv_umma_kernels = {
    {{(const void *)&rms_gemv_umma<bf16, false>, (const void *)&rms_gemv_umma<bf16, true>},
     {(const void *)&rms_gemv_umma<f16, false>, (const void *)&rms_gemv_umma<f16, true>}}};

} // namespace rmsk
