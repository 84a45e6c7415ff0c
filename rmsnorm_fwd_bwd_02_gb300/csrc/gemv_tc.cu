// RMSNorm fused with the projection, persistent with y held per CTA, the
// product on tcgen05 (gemv_tc.cuh): bf16 and fp16, with and without the
// residual add.
#include "gemv_tc.cuh"
#include "registry.h"

namespace rmsk {

const GemvTcKernels gemv_tc_kernels = {
    {{{(const void *)&rms_gemv_tc<bf16, false, false>, (const void *)&rms_gemv_tc<bf16, false, true>},
      {(const void *)&rms_gemv_tc<bf16, true, false>, (const void *)&rms_gemv_tc<bf16, true, true>}},
     {{(const void *)&rms_gemv_tc<f16, false, false>, (const void *)&rms_gemv_tc<f16, false, true>},
      {(const void *)&rms_gemv_tc<f16, true, false>, (const void *)&rms_gemv_tc<f16, true, true>}}}};

} // namespace rmsk
