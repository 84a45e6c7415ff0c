// params.h -- kernel argument blocks, passed by value; shared by the
// kernels and the host code that launches them. Every [M,H] tensor has its
// own row stride ld (elements between the starts of consecutive rows, >= H;
// H for contiguous rows); a kernel's pack width divides every stride it gets.
#pragma once

#include <stdint.h>

namespace rmsk {

// Row-wise forward (rows.cuh).
struct FwdParams {
    const void *x;   // [M,H]
    const void *r;   // [M,H] residual input (residual variant), else unused
    const void *w;   // [H]
    void *y;         // [M,H]
    void *h;         // [M,H] residual sum out (residual variant), else unused
    float *rstd;     // [M] or nullptr
    int64_t M;
    int H;
    float eps;
    int64_t ldx, ldr, ldy, ldh;   // row strides of x, r, y, h
    // Streamed kernels only: bytes a stage waits for beyond what its copies
    // deliver (0; a test sets it to make waits run out) and the wait limit
    // in microseconds (0 = the default of about one second).
    uint32_t extra_tx;
    uint32_t wait_limit_us;
};

// Row-wise backward (rows.cuh).
struct BwdParams {
    const void *dy;     // [M,H]
    const void *x;      // [M,H] (h for the residual variant)
    const void *w;      // [H]
    const float *rstd;  // [M] or nullptr (recompute)
    const void *dh;     // [M,H] incoming residual-stream gradient, or unused
    void *dx;           // [M,H]
    float *part;        // [gridDim.x, H] fp32 partial dw rows
    int64_t M;
    int H;
    float eps;
    int64_t lddy, ldx, lddh, lddx;   // row strides of dy, x, dh, dx
    uint32_t extra_tx;       // as in FwdParams
    uint32_t wait_limit_us;
};

// Double backward (bwd2.cuh, stream.cuh).
struct Bwd2Params {
    const void *dy;     // [M,H]
    const void *x;      // [M,H] (h for the residual variant)
    const void *w;      // [H]
    const float *rstd;  // [M] or nullptr (recompute)
    const void *gx;     // [M,H] gradient arriving on dx, or nullptr (zero)
    const float *gw;    // [H] gradient arriving on dw, or nullptr (zero)
    void *ddy;          // [M,H]
    void *dx2;          // [M,H]
    float *part;        // [gridDim.x, H] fp32 partial rows of dw2
    int64_t M;
    int H;
    float eps;
    uint32_t extra_tx;       // streamed kernel only, as in FwdParams
    uint32_t wait_limit_us;
};

// Split-row forward (split.cuh).
struct SplitParams {
    const void *x;   // [M,H]
    const void *r;   // [M,H] residual input (residual variant), else unused
    const void *w;   // [H]
    void *y;         // [M,H]
    void *h;         // [M,H] residual sum out (residual variant), else unused
    float *rstd;     // [M] or nullptr
    int H;           // features per row
    int NV;          // packs per row
    int SV;          // packs per CTA (the last ranks may hold fewer or none)
    float eps;
    int64_t ldx, ldr, ldy, ldh;   // row strides of x, r, y, h
    unsigned int *timeouts;       // counts waits for the peers' sums that ran out
    // test hook of the bounded wait: bytes the peers' sums are expected to
    // bring beyond what they do (0), and the wait limit in microseconds (0:
    // about one second)
    uint32_t extra_tx, wait_limit_us;
};

} // namespace rmsk
