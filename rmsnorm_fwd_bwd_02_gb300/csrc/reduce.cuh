// reduce.cuh -- second stage of dw: sum the per-CTA partial rows written by
// the backward kernel, in a fixed order ([P1] "训推加速 Qwen3 实战：从“调包”到手写
// Triton Kernel（含 backward）" §5.4: per-row partials, then a separate
// reduction over rows, no atomics; [P2] trdm.cn news/483216 §3.3: fp32
// partials merged in fp32 by a dedicated reduce kernel for reproducibility).
#pragma once

#include "common.cuh"

namespace rmsk {

// CW columns per CTA, RY threads per column. Thread (tx, ty) adds partial
// rows ty, ty+RY, ty+2RY, ... of column blockIdx.x*CW+tx; the RY sums are
// then added in ty order. With P == 0 (no rows) dw is all zeros. With
// accumulate != 0 the total is added to the dw already there (gradient
// accumulation over micro-batches), after the fixed-order sum.
template <int CW, int RY>
__global__ void __launch_bounds__(CW * RY)
dw_reduce(const float *__restrict__ part, int P, int H, float *__restrict__ dw, int accumulate)
{
    __shared__ float sm[RY][CW + 1];
    // Launched with programmatic serialization after the backward kernel:
    // wait until its partial rows are complete and visible.
    griddep_wait();
    griddep_launch_dependents();
    const int tx = threadIdx.x % CW;
    const int ty = threadIdx.x / CW;
    const int col = blockIdx.x * CW + tx;
    float s = 0.f;
    if (col < H) {
#pragma unroll 8
        for (int b = ty; b < P; b += RY)
            s += __ldcg(part + (int64_t)b * H + col);
    }
    sm[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && col < H) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < RY; ++q)
            t += sm[q][tx];
        dw[col] = accumulate ? dw[col] + t : t;
    }
}

} // namespace rmsk
