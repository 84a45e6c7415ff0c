// Split-row (cluster) forward kernels, every element type, vectorised and
// scalar.
#include "registry.h"
#include "split.cuh"

namespace rmsk {
RMSK_SPLIT(split_bf16_v, bf16, 8)
RMSK_SPLIT(split_bf16_s, bf16, 1)
RMSK_SPLIT(split_f32_v, float, 4)
RMSK_SPLIT(split_f32_s, float, 1)
RMSK_SPLIT(split_f16_v, f16, 8)
RMSK_SPLIT(split_f16_s, f16, 1)
} // namespace rmsk
